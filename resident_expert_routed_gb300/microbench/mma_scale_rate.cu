// Tensor-pipe cost of MXFP4 scale factors: one CTA per SM, one thread issuing
// tcgen05.mma.kind::mxf4.block_scale (M 128, N 256, K 64) back to back on
// operands resident in shared memory, alone and interleaved with the two ways
// of putting scale factors into TMEM. Timing only (operands are constants).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I include \
//        -o /tmp/mma_scale_rate resident_expert_routed_gb300/microbench/mma_scale_rate.cu && /tmp/mma_scale_rate
//
// Modes: 0 MMAs only; 1 plus six 32x128b.warpx4 scale copies per four MMAs
// (what a stage of the gate/up GEMM needs); 2 plus four warps writing the same
// 24 scale columns per four MMAs with tcgen05.st; 3 bf16 kind::f16 MMAs
// (M 128, N 256, K 16) for reference; 4 the same e2m1 operands and e8m0
// scales under kind::mxf4nvf4 (scale_vec::2X); 5 kind::mxf4nvf4 with
// scale_vec::4X and ue4m3 scales (one scale per 16 elements).
#include <cstdio>

#include "../csrc/common.cuh"

void moe_count_launches(int) {}
int moe_sm_count() { return 0; }
void moe_prof_begin(int, cudaStream_t) {}
void moe_prof_end(int, cudaStream_t) {}

namespace {

__device__ __forceinline__ void cp_atom(uint32_t taddr, uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(128u >> 4) << 32) |
                 ((uint64_t)1 << 46);
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

template <bool VEC4>
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
    if (VEC4)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
}

constexpr int SMEM = 120 * 1024;     // forces one CTA per SM

template <int MODE>
__global__ void __launch_bounds__(160, 1) rate(int n_mma, unsigned long long* ns_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);
    uint8_t* A = smem;                       // 128 x 128 B
    uint8_t* B = smem + 16384;               // 256 x 128 B
    uint8_t* SF = smem + 49152;              // three 1 KB atom pairs
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 52224);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + 52240);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 52244);
    for (int i = threadIdx.x; i < 49152 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x22222222u, 0x11111111u, 0x22222222u, 0x11111111u);
    for (int i = threadIdx.x; i < 3072; i += blockDim.x) SF[i] = MODE == 5 ? 0x38 : 127;     // scale 1 (ue4m3 / e8m0)
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    if (threadIdx.x < 32) { tmem_alloc(tslot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sfc = tmem + 384;         // 24 scale columns after the 256-column accumulator
    if (MODE == 2 && threadIdx.x < 128) {
        const uint32_t base = sfc + ((uint32_t)(threadIdx.x & ~31) << 16);
        const uint4 v = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        for (int it = 0; it < n_mma / 4; ++it) {
            tc_st_x8(base, v, v);
            tc_st_x8(base + 8, v, v);
            tc_st_x8(base + 16, v, v);
            tc_wait_st();
        }
    }
    if (threadIdx.x == (MODE == 2 ? 128 : 0)) {
        const uint32_t sfs = smem_u32(SF);
        for (int q = 0; q < 2; ++q) {
            cp_atom(sfc + 4 * q, sfs + 512 * q);
            cp_atom(sfc + 8 + 8 * q, sfs + 1024 + 512 * q);
            cp_atom(sfc + 12 + 8 * q, sfs + 2048 + 512 * q);
        }
        const uint32_t as = smem_u32(A), bs = smem_u32(B);
        const uint64_t t0 = global_timer_ns();
        for (int i = 0; i < n_mma; ++i) {
            const int kk = i & 3;
            if (MODE == 1 && kk == 0)
                for (int q = 0; q < 2; ++q) {
                    cp_atom(sfc + 4 * q, sfs + 512 * q);
                    cp_atom(sfc + 8 + 8 * q, sfs + 1024 + 512 * q);
                    cp_atom(sfc + 12 + 8 * q, sfs + 2048 + 512 * q);
                }
            if (MODE == 3)
                mma_bf16(tmem, smem_desc_sw128(as + kk * 32), smem_desc_sw128(bs + kk * 32), i != 0);
            else if (MODE == 4)
                mma_nvf4<false>(tmem, smem_desc_sw128(as + kk * 32), smem_desc_sw128(bs + kk * 32),
                                idesc_mxf4(256, (kk & 1) * 2, (kk & 1) * 2), sfc + (kk >> 1) * 4,
                                sfc + 8 + (kk >> 1) * 8, i != 0);
            else if (MODE == 5)     // ue4m3 scale type: bit 23 clear; one whole scale word per MMA
                mma_nvf4<true>(tmem, smem_desc_sw128(as + kk * 32), smem_desc_sw128(bs + kk * 32),
                               idesc_mxf4(256, 0, 0) & ~(1u << 23), sfc + (kk >> 1) * 4, sfc + 8 + (kk >> 1) * 8,
                               i != 0);
            else
                tc_mma_mxf4(tmem, smem_desc_sw128(as + kk * 32), smem_desc_sw128(bs + kk * 32),
                            idesc_mxf4(256, (kk & 1) * 2, (kk & 1) * 2), sfc + (kk >> 1) * 4, sfc + 8 + (kk >> 1) * 8,
                            i != 0);
        }
        tc_commit(bar);
        const bool ok = mbar_wait(bar, 0, abort_flag, MOE_WAIT_LIMIT_NS);
        ns_out[blockIdx.x] = ok ? global_timer_ns() - t0 : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MODE>
double run(const char* name, double flop, int sms, unsigned long long* d_ns) {
    const int n = 8192;
    cudaFuncSetAttribute(rate<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    for (int w = 0; w < 2; ++w) rate<MODE><<<sms, 160, SMEM>>>(n, d_ns);
    if (cudaDeviceSynchronize() != cudaSuccess) { printf("%s: launch failed\n", name); return 0.0; }
    unsigned long long h[1024];
    cudaMemcpy(h, d_ns, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
    unsigned long long tmax = 0;
    bool timed_out = false;
    for (int b = 0; b < sms; ++b) { tmax = h[b] > tmax ? h[b] : tmax; timed_out |= h[b] == 0; }
    const double tflops = timed_out ? 0.0 : flop * n * sms / (tmax * 1e-9) / 1e12;
    printf("%-44s %7.1f ns per MMA  %8.1f TFLOP/s over %d SMs%s\n", name, (double)tmax / n, tflops, sms,
           timed_out ? "  (a wait timed out)" : "");
    return tflops;
}

}  // namespace

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (sms > 1024) sms = 1024;
    unsigned long long* d_ns;
    cudaMalloc(&d_ns, sizeof(unsigned long long) * 1024);
    const double f4 = 128.0 * 256 * 64 * 2, f16 = 128.0 * 256 * 16 * 2;
    const double a = run<0>("mxf4 128x256x64", f4, sms, d_ns);
    const double b = run<1>("mxf4 + 6 tcgen05.cp 32x128b.warpx4 / 4 MMAs", f4, sms, d_ns);
    const double c = run<2>("mxf4 + 4 warps tcgen05.st (24 columns / 4)", f4, sms, d_ns);
    const double e = run<3>("bf16 128x256x16", f16, sms, d_ns);
    const double g = run<4>("mxf4nvf4 2X (e8m0) 128x256x64", f4, sms, d_ns);
    const double h = run<5>("mxf4nvf4 4X (ue4m3) 128x256x64", f4, sms, d_ns);
    printf("{\"mxf4_tflops\": %.1f, \"mxf4_with_scale_copies_tflops\": %.1f, \"mxf4_with_scale_stores_tflops\": %.1f, "
           "\"bf16_tflops\": %.1f, \"mxf4nvf4_2x_tflops\": %.1f, \"mxf4nvf4_4x_tflops\": %.1f, \"sms\": %d}\n",
           a, b, c, e, g, h, sms);
    return 0;
}
