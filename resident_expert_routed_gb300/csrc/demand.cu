// Demand accumulation and the heavy-miss list.
//
// TideLM README, "How adaptive expert loading works":
//   item 1  each pick the router asks for adds its routing score to the
//           demand of its (layer, expert), whether that expert is resident
//           or not;
//   item 2  a pick that had to be substituted adds to the demand as well;
//   item 3  a miss whose score is a big part of its token's routing weight
//           (at least 0.2; at most 16 a step) may be fetched by a hot read.
//
// demand_accumulate: shared-memory histograms over the E experts of one layer
// (u64 fixed point in units of 2^-40, and the max miss share as float bits),
// flushed with one global atomic per touched expert. Integer sums make the
// result independent of the order of the adds.
// hot_miss_select: one CTA ranks the (layer, expert) miss shares with a
// 64-bit key (share bits, inverted flat index) in `cap` block-wide arg-max
// rounds, then clears the shares for the next step.
#include "common.cuh"

namespace {

__global__ void __launch_bounds__(512) demand_accumulate(const int32_t* __restrict__ want_e,
                                                         const float* __restrict__ want_s,
                                                         const int32_t* __restrict__ slot_of, int P, int E,
                                                         unsigned long long* __restrict__ demand,
                                                         float* __restrict__ miss_max) {
    extern __shared__ unsigned long long hist[];                 // [E] demand, then [E] miss bits
    uint32_t* mbits = reinterpret_cast<uint32_t*>(hist + E);
    pdl_trigger();
    for (int e = threadIdx.x; e < E; e += blockDim.x) { hist[e] = 0ull; mbits[e] = 0u; }
    pdl_wait();
    __syncthreads();
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
        const int e = want_e[p];
        if (e < 0 || e >= E) continue;
        const float s = want_s[p];
        atomicAdd(&hist[e], __float2ull_rn(s * 1099511627776.0f));      // s * 2^40
        if (slot_of[e] < 0) atomicMax(&mbits[e], __float_as_uint(s));   // s >= 0: bits order = value order
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (hist[e]) atomicAdd(&demand[e], hist[e]);
        if (mbits[e]) atomicMax(reinterpret_cast<uint32_t*>(miss_max) + e, mbits[e]);
    }
}

__device__ __forceinline__ unsigned long long miss_key(const float* M, int f, float thr) {
    const float m = M[f];
    if (!(m >= thr)) return 0ull;
    return ((unsigned long long)__float_as_uint(m) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)f);
}

constexpr int MAX_CAND = 2048;

__global__ void __launch_bounds__(1024) hot_miss_select(float* __restrict__ M, int n, float thr, int cap,
                                                        int32_t* __restrict__ out_flat,
                                                        float* __restrict__ out_share, int32_t* __restrict__ n_out) {
    __shared__ unsigned long long wbest[32];
    __shared__ unsigned long long picked;
    __shared__ int count;
    __shared__ int n_cand;
    __shared__ unsigned long long cand[MAX_CAND];
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) { picked = ~0ull; count = 0; n_cand = 0; }
    __syncthreads();
    // usual case: few shares pass the threshold; rank them directly by their keys (all distinct)
    for (int f = threadIdx.x; f < n; f += blockDim.x) {
        const unsigned long long key = miss_key(M, f, thr);
        if (key) {
            const int i = atomicAdd(&n_cand, 1);
            if (i < MAX_CAND) cand[i] = key;
        }
    }
    __syncthreads();
    const int C = n_cand;
    if (C <= MAX_CAND) {
        for (int i = threadIdx.x; i < C; i += blockDim.x) {
            const unsigned long long key = cand[i];
            int rank = 0;
            for (int q = 0; q < C; ++q) rank += cand[q] > key;
            if (rank < cap) {
                out_flat[rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
                out_share[rank] = __uint_as_float((uint32_t)(key >> 32));
            }
        }
        if (threadIdx.x == 0) count = C < cap ? C : cap;
        __syncthreads();
        if (threadIdx.x == 0) *n_out = count;
        for (int f = threadIdx.x; f < n; f += blockDim.x) M[f] = 0.0f;
        return;
    }
    // many candidates: `cap` block-wide arg-max rounds, each below the previous pick
    for (int j = 0; j < cap; ++j) {
        const unsigned long long prev = picked;
        unsigned long long best = 0ull;
        for (int f = threadIdx.x; f < n; f += blockDim.x) {
            const unsigned long long key = miss_key(M, f, thr);
            if (key < prev && key > best) best = key;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
            best = o > best ? o : best;
        }
        if ((threadIdx.x & 31) == 0) wbest[threadIdx.x >> 5] = best;
        __syncthreads();
        if (threadIdx.x < 32) {
            unsigned long long b = threadIdx.x < (blockDim.x >> 5) ? wbest[threadIdx.x] : 0ull;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, b, off);
                b = o > b ? o : b;
            }
            if (threadIdx.x == 0) {
                if (b != 0ull) {
                    out_flat[count] = (int32_t)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
                    out_share[count] = __uint_as_float((uint32_t)(b >> 32));
                    ++count;
                }
                picked = b;
            }
        }
        __syncthreads();
        if (picked == 0ull) break;
    }
    if (threadIdx.x == 0) *n_out = count;
    __syncthreads();
    for (int f = threadIdx.x; f < n; f += blockDim.x) M[f] = 0.0f;
}

// demand[i] = floor(demand[i] * q / 2^32) with q <= 2^32 (the product is < 2^96, its high word < 2^32).
__global__ void __launch_bounds__(256) demand_decay(unsigned long long* __restrict__ D, long n,
                                                    unsigned long long q) {
    pdl_trigger();
    pdl_wait();
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const unsigned long long d = D[i];
        D[i] = (__umul64hi(d, q) << 32) | ((d * q) >> 32);
    }
}

}  // namespace

cudaError_t launch_demand_decay(unsigned long long* demand, long n, unsigned long long q, cudaStream_t s) {
    long blocks = (n + 255) / 256;
    if (blocks > 4L * moe_sm_count()) blocks = 4L * moe_sm_count();
    const cudaError_t e = moe_launch(demand_decay, dim3((unsigned)blocks), dim3(256), 0, s, demand, n, q);
    moe_count_launches(1);
    return e;
}

cudaError_t launch_demand(const int32_t* want_e, const float* want_s, const int32_t* slot_of, int T, int k,
                          int layer, int E, unsigned long long* demand, float* miss_max, cudaStream_t s) {
    const int P = T * k;
    int grid = (P + 511) / 512;
    if (grid > 2 * moe_sm_count()) grid = 2 * moe_sm_count();
    const size_t smem = (size_t)E * (sizeof(unsigned long long) + sizeof(uint32_t));
    moe_prof_begin(MK_DEMAND, s);
    const cudaError_t e = moe_launch(demand_accumulate, dim3(grid), dim3(512), smem, s, want_e, want_s, slot_of, P,
                                     E, demand + (size_t)layer * E, miss_max + (size_t)layer * E);
    moe_prof_end(MK_DEMAND, s);
    moe_count_launches(1);
    return e;
}

cudaError_t launch_hot_miss(float* miss_max, int n, float threshold, int cap, int32_t* out_flat, float* out_share,
                            int32_t* n_out, cudaStream_t s) {
    moe_prof_begin(MK_HOT_MISS, s);
    const cudaError_t e = moe_launch(hot_miss_select, dim3(1), dim3(1024), 0, s, miss_max, n, threshold, cap,
                                     out_flat, out_share, n_out);
    moe_prof_end(MK_HOT_MISS, s);
    moe_count_launches(1);
    return e;
}
