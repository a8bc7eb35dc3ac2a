// Streaming rate of one SM through a ring of shared-memory stages filled by
// bulk copies (cp.async.bulk, 16 KB pieces) from HBM, as a function of the
// stage size and of how many SMs stream at once. One producer thread per CTA
// waits for a free stage and issues its pieces; one consumer thread waits for
// the stage, touches one byte and frees it. Timing only.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I include \
//        -o /tmp/bulk_stream_rate resident_expert_routed_gb300/microbench/bulk_stream_rate.cu && /tmp/bulk_stream_rate
//
// With every SM streaming, HBM sets each SM's share; with fewer (the partial
// last round of a persistent GEMM grid) the stages in flight do.
#include <cstdio>

#include "../csrc/common.cuh"

void moe_count_launches(int) {}
int moe_sm_count() { return 0; }
void moe_prof_begin(int, cudaStream_t) {}
void moe_prof_end(int, cudaStream_t) {}

namespace {

__global__ void __launch_bounds__(64, 1) stream(const uint8_t* buf, long window_stages, long iters, int stage,
                                                int ns, int pieces, unsigned* sink) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)ns * stage);
    uint64_t* empty = full + ns;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + ns);
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {                 // producer: stage c of this CTA's interleaved share
        long c = blockIdx.x;
        int s = 0;
        uint32_t r = 0;
        for (long it = 0; it < iters; ++it) {
            if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag)) break;
            mbar_arrive_expect_tx(&full[s], (uint32_t)stage);
            const int piece = stage / pieces;
            for (int p = 0; p < pieces; ++p)
                bulk_load(smem + (size_t)s * stage + p * piece, buf + c * stage + p * piece, (uint32_t)piece, &full[s]);
            c += gridDim.x;
            if (c >= window_stages) c -= window_stages;
            if (++s == ns) { s = 0; ++r; }
        }
    } else if (threadIdx.x == 32) {         // consumer
        unsigned acc = 0;
        int s = 0;
        uint32_t r = 0;
        for (long it = 0; it < iters; ++it) {
            if (!mbar_wait(&full[s], r & 1, abort_flag)) break;
            acc += smem[(size_t)s * stage + (it & 127)];
            mbar_arrive(&empty[s]);
            if (++s == ns) { s = 0; ++r; }
        }
        if (acc == 0xFFFFFFFFu) *sink = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) *sink = 0xDEADu;
}

}  // namespace

int main() {
    const size_t bytes = 4ull << 30;
    uint8_t* buf = nullptr;
    unsigned* sink = nullptr;
    if (cudaMalloc(&buf, bytes) != cudaSuccess || cudaMalloc(&sink, 4) != cudaSuccess) return 1;
    cudaMemset(buf, 1, bytes);
    cudaMemset(sink, 0, 4);
    cudaFuncSetAttribute(stream, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    struct Run { int stage, ns, pieces, grid; } runs[] = {
        {32768, 5, 2, sms}, {32768, 5, 2, sms / 2}, {32768, 5, 2, 40}, {32768, 5, 2, 8},
        {16384, 10, 1, 40}, {16384, 10, 1, 8}, {65536, 3, 4, sms}, {65536, 3, 4, 40}, {65536, 3, 4, 8}};
    int rc = 0;
    for (const Run& R : runs) {
        const size_t smem = (size_t)R.ns * R.stage + 2 * R.ns * 8 + 16 + 1024;
        const long window = (long)(bytes / R.stage), iters = 1000;
        for (int w = 0; w < 2; ++w)
            stream<<<R.grid, 64, smem>>>(buf, window, iters, R.stage, R.ns, R.pieces, sink);
        const int reps = 3;
        cudaEventRecord(a);
        for (int w = 0; w < reps; ++w)
            stream<<<R.grid, 64, smem>>>(buf, window, iters, R.stage, R.ns, R.pieces, sink);
        cudaEventRecord(b);
        cudaEventSynchronize(b);
        const cudaError_t e = cudaGetLastError();
        unsigned hs = 0;
        cudaMemcpy(&hs, sink, 4, cudaMemcpyDeviceToHost);
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, a, b);
        const double gbs = (double)reps * R.grid * iters * R.stage / (ms * 1e-3) / 1e9;
        printf("%2d stages x %3d KB (%d pieces) in flight, %3d CTAs: %7.1f GB/s, %6.1f GB/s per CTA%s%s\n", R.ns,
               R.stage / 1024, R.pieces, R.grid, gbs, gbs / R.grid, e == cudaSuccess ? "" : cudaGetErrorString(e),
               hs == 0xDEADu ? " (a wait timed out)" : "");
        if (e != cudaSuccess || hs == 0xDEADu) rc = 1;
    }
    return rc;
}
