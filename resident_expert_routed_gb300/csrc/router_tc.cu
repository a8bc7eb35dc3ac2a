// Router logits for large batches on the tensor cores, at fp32-class accuracy.
//
// TideLM README items 1-2: every token is scored against all experts. At
// prefill sizes (8192 tokens x 256 experts x d 4096 = 17 GFLOP) fp32 CUDA-core
// throughput would dominate the layer, so the router GEMM runs on tcgen05
// kind::f16 MMAs instead. bf16 alone would lose the 16 low significand bits of
// W and reorder near-tied experts, so W is split exactly into three bf16 parts
// W = W1 + W2 + W3 (8 + 8 + 8 significand bits: the split-bf16 technique of
// Henry, Tang & Heinecke, "Leveraging the bfloat16 artificial intelligence
// datatype for higher-precision computations", 2019); the hidden states are
// bf16 already, every product x * Wi is exact, and the three products are
// accumulated in fp32 in TMEM:
//   partial[z, t, e] = sum_{i in K slice z} x[t,i] (W1 + W2 + W3)[e,i]
// route_select sums the K slices in order and adds the bias, as for the
// CUDA-core router.
//
// The tensor cores' fp32 accumulation does not round each add to nearest (a
// long chain of MMAs into one accumulator drifts by about an ulp of the
// running sum per instruction), so no accumulator lives longer than RT_EPOCH
// K chunks: two TMEM accumulators alternate, and the epilogue warps add each
// finished one into fp32 registers (round to nearest) while the tensor cores
// fill the other.
//
// One CTA per (128-token tile, 128-expert tile, K slice): warp 4 issues TMA
// for the x tile and the three W tiles per 64-element K chunk; warp 5 issues
// 3 x 4 MMAs (M 128, N 128, K 16) per chunk; warps 0-3 (lane = token) drain
// the accumulators and write the row of partials. Waits are bounded as in the
// expert GEMMs.
#include <cuda_bf16.h>

#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace {

constexpr int RT_NS = 3;
constexpr int RT_TILE = 128 * 128;                 // 128 rows x 64 bf16 (128 bytes)
constexpr int RT_STAGE = 4 * RT_TILE;              // x tile + three W tiles
constexpr int RT_EPOCH = 2;                         // K chunks (24 MMAs) per accumulator epoch
constexpr int RT_SMEM = RT_NS * RT_STAGE + (2 * RT_NS + 5) * 8 + 16 + 1024;   // stages, barriers, TMEM slot + flag

__global__ void __launch_bounds__(256) split_router_weights(const float* __restrict__ W, long n,
                                                            __nv_bfloat16* __restrict__ w1, __nv_bfloat16* __restrict__ w2,
                                                            __nv_bfloat16* __restrict__ w3) {
    pdl_trigger();
    pdl_wait();
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const float w = W[i];
        const __nv_bfloat16 a = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(a);        // exact in fp32
        const __nv_bfloat16 b = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(b);       // exact in fp32
        w1[i] = a;
        w2[i] = b;
        w3[i] = __float2bfloat16_rn(r2);
    }
}

// Instruction descriptor for kind::f16: bf16 x bf16 -> fp32, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

MOE_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct RouterMaps {
    CUtensorMap x;       // (d, T) bf16, box 64 x 128
    CUtensorMap w;       // (d, 3E) bf16 (W1 rows, W2 rows, W3 rows), box 64 x 128
};

__global__ void __launch_bounds__(192, 1) router_logits_tc(const __grid_constant__ RouterMaps maps, int T, int E,
                                                           int kchunks, float* __restrict__ partial,
                                                           uint32_t* err, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RT_NS * RT_STAGE);
    uint64_t* empty = full + RT_NS;
    uint64_t* acc_full = empty + RT_NS;      // [2] accumulator b holds a finished epoch
    uint64_t* acc_empty = acc_full + 2;      // [2] accumulator b has been drained
    uint64_t* drain = acc_empty + 2;         // the MMA thread's own MMAs, after an abort
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * 128, e0 = blockIdx.y * 128, z = blockIdx.z;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < RT_NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 128); }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.w);
    }
    if (warp == 5) { tmem_alloc(tmem_slot, 256); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    const uint32_t tmem = *tmem_slot;
    const int kc0 = z * kchunks;
    const int n_epochs = (kchunks + RT_EPOCH - 1) / RT_EPOCH;
    uint32_t issued = 0;                     // stage fills issued by the producer thread

    if (warp == 4) {
        if (lane == 0) {
            for (int c = 0; c < kchunks; ++c) {
                const int s = c % RT_NS;
                const uint32_t r = c / RT_NS;
                if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, wait_ns)) break;
                ++issued;
                uint8_t* st = smem + s * RT_STAGE;
                const int x0 = (kc0 + c) * 64;
                mbar_arrive_expect_tx(&full[s], RT_STAGE);
                tma_load_2d(st, &maps.x, &full[s], x0, t0);
                for (int p = 0; p < 3; ++p) tma_load_2d(st + (p + 1) * RT_TILE, &maps.w, &full[s], x0, p * E + e0);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            for (int c = 0; c < kchunks; ++c) {
                const int s = c % RT_NS;
                const uint32_t r = c / RT_NS;
                const int ep = c / RT_EPOCH, b = ep & 1;
                const bool first = c % RT_EPOCH == 0;
                if (first && !mbar_wait(&acc_empty[b], ((ep >> 1) & 1) ^ 1, abort_flag, wait_ns)) break;
                if (!mbar_wait(&full[s], r & 1, abort_flag, wait_ns)) break;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * RT_STAGE);
                const uint32_t d = tmem + (uint32_t)(b * 128);
                for (int kk = 0; kk < 4; ++kk)
                    for (int p = 0; p < 3; ++p)
                        tc_mma_bf16(d, smem_desc_sw128(st + kk * 32),
                                    smem_desc_sw128(st + (p + 1) * RT_TILE + kk * 32), idesc_bf16(128),
                                    (first && kk == 0 && p == 0) ? 0u : 1u);
                tc_commit(&empty[s]);
                if (c % RT_EPOCH == RT_EPOCH - 1 || c == kchunks - 1) tc_commit(&acc_full[b]);
            }
        }
    } else {
        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
        for (int ep = 0; ep < n_epochs; ++ep) {
            const int b = ep & 1;
            if (!warp_wait(&acc_full[b], (ep >> 1) & 1, abort_flag, wait_ns)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[16], w[16];
                tc_ld_x16(trow + b * 128 + c0, v);
                tc_ld_x16(trow + b * 128 + c0 + 16, w);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    acc[c0 + i] += __uint_as_float(v[i]);
                    acc[c0 + 16 + i] += __uint_as_float(w[i]);
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
        }
        const int t = t0 + warp * 32 + lane;
        if (ok && t < T) {
            float* out = partial + ((size_t)z * T + t) * E + e0;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 16) {
                if (e0 + c0 < E) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4*>(out + c0 + 4 * q) =
                            make_float4(acc[c0 + 4 * q], acc[c0 + 4 * q + 1], acc[c0 + 4 * q + 2], acc[c0 + 4 * q + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {                       // final after the barrier: nothing new is issued past it
        if (warp == 4 && lane == 0) drain_stage_fills(full, RT_NS, issued);
        if (warp == 5 && lane == 0) tc_drain(drain);
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
    if (threadIdx.x == 0 && *abort_flag) record_error(err, MOE_DEV_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
    auto enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool router_tc_eligible(int T, int E, int d) { return T > 64 && d % 64 == 0 && E % 16 == 0; }

int router_tc_splits(int T, int E, int d) {
    const int tiles = ((T + 127) / 128) * ((E + 127) / 128);
    return (tiles < 152 && (d / 64) % 2 == 0) ? 2 : 1;
}

size_t router_tc_split_bytes(int E, int d) { return ((size_t)3 * E * d * 2 + 255) / 256 * 256; }

cudaError_t launch_router_tc(const uint16_t* x, const float* W, int T, int d, int E, int splits, void* wsplit,
                             float* partial, uint32_t* err, uint64_t wait_ns, cudaStream_t s) {
    __nv_bfloat16* w1 = static_cast<__nv_bfloat16*>(wsplit);
    const long n = (long)E * d;
    long blocks = (n + 255) / 256;
    if (blocks > 4L * moe_sm_count()) blocks = 4L * moe_sm_count();
    moe_prof_begin(MK_ROUTER_LOGITS, s);
    cudaError_t e = moe_launch(split_router_weights, dim3((unsigned)blocks), dim3(256), 0, s, W, n, w1, w1 + n,
                               w1 + 2 * n);
    if (e != cudaSuccess) return e;
    RouterMaps maps;
    e = bf16_map(&maps.x, x, (uint64_t)d, (uint64_t)T);
    if (e == cudaSuccess) e = bf16_map(&maps.w, w1, (uint64_t)d, (uint64_t)3 * E);
    if (e != cudaSuccess) return e;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(router_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, RT_SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid((T + 127) / 128, (E + 127) / 128, splits);
    e = moe_launch(router_logits_tc, grid, dim3(192), RT_SMEM, s, maps, T, E, (d / 64) / splits, partial, err, wait_ns);
    moe_prof_end(MK_ROUTER_LOGITS, s);
    moe_count_launches(2);
    return e;
}
