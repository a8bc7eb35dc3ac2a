// Router scoring and resident-only top-k with substitution.
//
// TideLM README, "How adaptive expert loading works", items 1-2: the router
// scores every token against all experts; the wanted picks are the top-k over
// all of them, and the picks actually routed are the top-k over the resident
// experts only: a wanted expert that is absent gives its place to the best
// resident expert not yet picked.
//
// Two kernels:
//   router_logits_partial  fp32 register-tiled GEMM over a K slice:
//                          partial[z, t, e] = sum_{i in slice z} x[t,i] W[e,i]
//   (router_logits_rows    up to 4 tokens: one CTA per expert row, the whole
//                          sum over i, no K slices; a batch in host memory is
//                          first copied to the workspace by stage_rows)
//   route_select           one warp per token (one CTA with many slices): sum
//                          the slices in a fixed order (+ bias), softmax,
//                          wanted and resident top-k by redux.sync arg-max
//                          rounds.
// The K split keeps >= ~256 CTAs streaming W_r at decode sizes; the partials
// are small and stay in L2.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int BT = 64, BE = 64, BK = 32;

__global__ void __launch_bounds__(256) router_logits_partial(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ W, int T, int d, int E,
                                                             int kslice, float* __restrict__ partial) {
    __shared__ float xs[BK][BT + 4];
    __shared__ float ws[BK][BE + 4];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;       // 16 x 16 threads, 4 x 4 outputs each
    const int e0 = blockIdx.x * BE, t0 = blockIdx.y * BT;
    const int kbeg = blockIdx.z * kslice, kend = kbeg + kslice;
    float acc[4][4] = {};
    const int lr = tid >> 2, lc = (tid & 3) * 8;   // loader: row, 8 consecutive k
    const int tl = t0 + lr, el = e0 + lr;
    // registers hold the next K tile while the current one is multiplied
    uint4 xv = make_uint4(0, 0, 0, 0);
    float4 wa = make_float4(0, 0, 0, 0), wb = wa;
    auto fetch = [&](int k0) {
        xv = make_uint4(0, 0, 0, 0);
        wa = make_float4(0, 0, 0, 0);
        wb = wa;
        if (tl < T) xv = *reinterpret_cast<const uint4*>(x + (size_t)tl * d + k0 + lc);
        if (el < E) {
            wa = *reinterpret_cast<const float4*>(W + (size_t)el * d + k0 + lc);
            wb = *reinterpret_cast<const float4*>(W + (size_t)el * d + k0 + lc + 4);
        }
    };
    fetch(kbeg);
    for (int k0 = kbeg; k0 < kend; k0 += BK) {
        {   // x tile: 64 tokens x 32 bf16 -> xs[k][t]; W tile: 64 experts x 32 fp32 -> ws[k][e]
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[lc + i][lr] = bf16_bits_to_float(h[i]);
            ws[lc + 0][lr] = wa.x; ws[lc + 1][lr] = wa.y; ws[lc + 2][lr] = wa.z; ws[lc + 3][lr] = wa.w;
            ws[lc + 4][lr] = wb.x; ws[lc + 5][lr] = wb.y; ws[lc + 6][lr] = wb.z; ws[lc + 7][lr] = wb.w;
        }
        __syncthreads();
        if (k0 + BK < kend) fetch(k0 + BK);
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* out = partial + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int e = e0 + tx * 4 + j;
            if (e < E) out[(size_t)t * E + e] = acc[i][j];
        }
    }
}

// A few tokens (T <= ROWS_MAX_T) whose x is in device memory: one CTA per
// expert e reads its whole W_r row, 8 consecutive elements per thread and
// chunk, with every load in flight at once, and writes logits[t, e] (the
// single K slice of the selection's input). W_r is loaded before the wait: no
// kernel of this library writes it, so those loads overlap the end of the
// previous kernel; x, which that kernel may have written, after. Each sum runs
// in a fixed order: a thread's chunks and their elements in K order, the warp's
// butterfly, then the warps in order.
constexpr int ROWS_THREADS = 256, ROWS_MAX_T = 4, ROWS_MAX_CH = 4;    // d <= 8 * 4 * 256 = 8192

__global__ void __launch_bounds__(ROWS_THREADS) router_logits_rows(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ W, int T, int d,
                                                                   int E, float* __restrict__ logits) {
    __shared__ float red[ROWS_THREADS / 32][ROWS_MAX_T];
    pdl_trigger();
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nch = d / 8;
    const float4* wr = reinterpret_cast<const float4*>(W + (size_t)e * d);
    float4 wlo[ROWS_MAX_CH], whi[ROWS_MAX_CH];
#pragma unroll
    for (int j = 0; j < ROWS_MAX_CH; ++j) {
        const int c = tid + j * ROWS_THREADS;
        wlo[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        whi[j] = wlo[j];
        if (c < nch) { wlo[j] = wr[2 * c]; whi[j] = wr[2 * c + 1]; }
    }
    pdl_wait();
    uint4 xv[ROWS_MAX_T][ROWS_MAX_CH];
#pragma unroll
    for (int t = 0; t < ROWS_MAX_T; ++t)
#pragma unroll
        for (int j = 0; j < ROWS_MAX_CH; ++j) {
            const int c = tid + j * ROWS_THREADS;
            xv[t][j] = make_uint4(0u, 0u, 0u, 0u);
            if (t < T && c < nch) xv[t][j] = *reinterpret_cast<const uint4*>(x + (size_t)t * d + 8 * c);
        }
    float acc[ROWS_MAX_T];
#pragma unroll
    for (int t = 0; t < ROWS_MAX_T; ++t) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < ROWS_MAX_CH; ++j) {
            const uint4 h = xv[t][j];
            s = fmaf(__uint_as_float(h.x << 16), wlo[j].x, s);
            s = fmaf(__uint_as_float(h.x & 0xFFFF0000u), wlo[j].y, s);
            s = fmaf(__uint_as_float(h.y << 16), wlo[j].z, s);
            s = fmaf(__uint_as_float(h.y & 0xFFFF0000u), wlo[j].w, s);
            s = fmaf(__uint_as_float(h.z << 16), whi[j].x, s);
            s = fmaf(__uint_as_float(h.z & 0xFFFF0000u), whi[j].y, s);
            s = fmaf(__uint_as_float(h.w << 16), whi[j].z, s);
            s = fmaf(__uint_as_float(h.w & 0xFFFF0000u), whi[j].w, s);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
        acc[t] = s;
    }
    if (lane == 0)
#pragma unroll
        for (int t = 0; t < ROWS_MAX_T; ++t) red[warp][t] = acc[t];
    __syncthreads();
    if (tid < T) {
        float s = red[0][tid];
#pragma unroll
        for (int w = 1; w < ROWS_THREADS / 32; ++w) s += red[w][tid];
        logits[(size_t)tid * E + e] = s;
    }
}

// Order-preserving map of a float onto uint32 (-0 and +0 both map to +0's
// image, so that they tie); 0 is below every float's image and means "none".
__device__ __forceinline__ uint32_t ordered_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The bias and slot of the experts a lane holds (lane + 32 i), padding past E.
// The bias is read before the kernel's wait (no kernel of this library writes
// it); the slot table after it (ring installs and re-plans rewrite it).
template <int VPL>
__device__ __forceinline__ void load_bias(const float* __restrict__ bias, int E, float (&bv)[VPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        bv[i] = (bias && e < E) ? bias[e] : 0.0f;
    }
}
template <int VPL>
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ slot_of, int E, int (&slot)[VPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        slot[i] = e < E ? slot_of[e] : -1;
    }
}

// The float whose ordered_key is u (u != 0); -0 comes back as +0.
__device__ __forceinline__ float key_value(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Rank of (key, expert): larger key first, ties to the lower expert index, as
// one 64-bit value (the key above the inverted index), so that a comparison
// is a single unsigned compare.
__device__ __forceinline__ unsigned long long rank64(uint32_t key, int e) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}

// Bitonic sorting network over a lane's N (key, expert, slot) triples, all in
// registers (every index is a compile-time constant) and without branches
// (each compare-exchange is three selects): afterwards entry 0 ranks ahead of
// entry 1 and so on.
template <int N>
__device__ __forceinline__ void sort_ahead(uint32_t (&key)[N], int (&ex)[N], int (&sl)[N]) {
    unsigned long long r[N];
#pragma unroll
    for (int i = 0; i < N; ++i) r[i] = rank64(key[i], ex[i]);
#pragma unroll
    for (int size = 2; size <= N; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool sw = (r[j] > r[i]) == ((i & size) == 0);   // j must come first
                    const unsigned long long ri = r[i], rj = r[j];
                    const int si = sl[i], sj = sl[j];
                    r[i] = sw ? rj : ri; r[j] = sw ? ri : rj;
                    sl[i] = sw ? sj : si; sl[j] = sw ? si : sj;
                }
            }
#pragma unroll
    for (int i = 0; i < N; ++i) {
        key[i] = (uint32_t)(r[i] >> 32);
        ex[i] = (int)(0xFFFFFFFFu - (uint32_t)r[i]);
    }
}

// Drops a lane's head entry (the warp's pick of this round) when `mine`.
template <int N>
__device__ __forceinline__ void pop_head(bool mine, uint32_t (&key)[N], int (&ex)[N], int (&sl)[N]) {
#pragma unroll
    for (int q = 0; q + 1 < N; ++q) {
        key[q] = mine ? key[q + 1] : key[q];
        ex[q] = mine ? ex[q + 1] : ex[q];
        sl[q] = mine ? sl[q + 1] : sl[q];
    }
    key[N - 1] = mine ? 0u : key[N - 1];
}

// Softmax over all E, wanted top-k over all experts and resident top-k, for
// one token whose logits (bias added) lg[i] (expert lane + 32 i) one warp
// holds. Order by logit (monotone in the score), ties to the lower expert
// index. Each lane sorts its own experts once; every round then takes the
// warp's best head (two redux.sync reductions: the largest key, then the
// lowest expert index among the lanes holding it, with its resident bit) and
// the winning lane drops its head. Every lane knows each round's key and
// expert, so lane j records the j-th wanted pick and lane q the q-th resident
// one, and all picks' weights and stores follow the rounds at once (the
// resident picks' slots read from slot_of). The first k rounds give the
// wanted list and, in the same order, the resident picks among them; when
// fewer than k of those are resident the lanes mask out non-resident experts,
// sort again and continue until k resident picks (or none left).
template <int VPL>
__device__ __forceinline__ void select_token(float (&lg)[VPL], const int (&slot)[VPL], int t, int E, int k,
                                             const int32_t* __restrict__ slot_of,
                                             int32_t* __restrict__ want_e, float* __restrict__ want_s,
                                             int32_t* __restrict__ sel_e, int32_t* __restrict__ sel_slot,
                                             float* __restrict__ sel_w) {
    const int lane = threadIdx.x & 31;
    uint32_t key[VPL];
    int ex[VPL], sl[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? ordered_key(lg[i]) : 0u;
        ex[i] = e;
        sl[i] = slot[i];
    }
    sort_ahead<VPL>(key, ex, sl);
    // softmax over all E: max (the best key), then sum of exp(l - max) in lane and warp order
    const float mx = key_value(__reduce_max_sync(0xFFFFFFFFu, key[0]));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) z += expf(lg[i] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
    const float inv_z = 1.0f / z;

    uint32_t w_key = 0u, r_key = 0u;                      // this lane's wanted / resident pick
    int w_e = -1, r_e = -1;
    int nw = 0, ns = 0;                                   // wanted and resident picks so far
    for (int j = 0; j < k; ++j) {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, key[0]);
        if (m == 0u) break;                               // fewer experts than k
        // lowest expert index among the heads equal to m, its non-resident bit in bit 0
        const uint32_t w = __reduce_min_sync(
            0xFFFFFFFFu, key[0] == m ? ((uint32_t)ex[0] << 1) | (sl[0] < 0 ? 1u : 0u) : 0xFFFFFFFFu);
        const int e = (int)(w >> 1);
        if (lane == j) { w_key = m; w_e = e; }
        if (!(w & 1u)) {
            if (lane == ns) { r_key = m; r_e = e; }
            ++ns;
        }
        ++nw;
        pop_head<VPL>(key[0] == m && ex[0] == e, key, ex, sl);
    }
    if (ns < k) {
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = sl[i] < 0 ? 0u : key[i];
        sort_ahead<VPL>(key, ex, sl);
        for (; ns < k; ++ns) {
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, key[0]);
            if (m == 0u) break;                           // fewer resident experts than k
            const uint32_t w = __reduce_min_sync(0xFFFFFFFFu, key[0] == m ? (uint32_t)ex[0] : 0xFFFFFFFFu);
            if (lane == ns) { r_key = m; r_e = (int)w; }
            pop_head<VPL>(key[0] == m && (uint32_t)ex[0] == w, key, ex, sl);
        }
    }
    // the picks' weights and outputs, one lane per pick; resident positions past the last pick are padding
    const size_t row = (size_t)t * k;
    if (lane < nw) {
        want_e[row + lane] = w_e;
        want_s[row + lane] = expf(key_value(w_key) - mx) * inv_z;
    }
    if (lane < k) {
        const bool real = lane < ns;
        sel_e[row + lane] = real ? r_e : -1;
        sel_slot[row + lane] = real ? slot_of[r_e] : -1;
        sel_w[row + lane] = real ? expf(key_value(r_key) - mx) * inv_z : 0.0f;
    }
}

// One warp per token (few K slices): the slices are summed in slice order;
// U slices' loads are issued together.
template <int VPL>
__global__ void __launch_bounds__(256, 1) route_select(const float* __restrict__ partial, int splits,
                                                    const float* __restrict__ bias,
                                                    const int32_t* __restrict__ slot_of, int T, int E, int k,
                                                    int32_t* __restrict__ want_e, float* __restrict__ want_s,
                                                    int32_t* __restrict__ sel_e, int32_t* __restrict__ sel_slot,
                                                    float* __restrict__ sel_w) {
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    float bv[VPL];
    load_bias<VPL>(bias, E, bv);
    pdl_wait();
    if (t >= T) return;
    int slot[VPL];
    load_slots<VPL>(slot_of, E, slot);
    float lg[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) lg[i] = 0.0f;
    constexpr int U = VPL >= 16 ? 1 : 64 / (VPL * 2);
    int zs = 0;
    for (; zs + U <= splits; zs += U) {
        float v[U][VPL];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const float* pz = partial + ((size_t)(zs + q) * T + t) * E;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int e = lane + 32 * i;
                v[q][i] = e < E ? pz[e] : 0.0f;
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q)
#pragma unroll
            for (int i = 0; i < VPL; ++i) lg[i] += v[q][i];
    }
    for (; zs < splits; ++zs) {
        const float* pz = partial + ((size_t)zs * T + t) * E;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) lg[i] += pz[e];
        }
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) lg[i] += bv[i];
    select_token<VPL>(lg, slot, t, E, k, slot_of, want_e, want_s, sel_e, sel_slot, sel_w);
}

// One CTA of 8 warps per token (many K slices, small batches): warp w sums
// slices w, w + 8, ... in order; warp 0 adds the eight sums in warp order and
// selects. One round of independent loads instead of a chain per token.
template <int VPL>
__global__ void __launch_bounds__(256) route_select_cta(const float* __restrict__ partial, int splits,
                                                        const float* __restrict__ bias,
                                                        const int32_t* __restrict__ slot_of, int T, int E, int k,
                                                        int32_t* __restrict__ want_e, float* __restrict__ want_s,
                                                        int32_t* __restrict__ sel_e, int32_t* __restrict__ sel_slot,
                                                        float* __restrict__ sel_w) {
    __shared__ float part[8][VPL * 32];
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    float bv[VPL];
    int slot[VPL];
    if (warp == 0) load_bias<VPL>(bias, E, bv);
    pdl_wait();
    if (warp == 0) load_slots<VPL>(slot_of, E, slot);
    float acc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = 0.0f;
    // slices warp, warp + 8, ...: up to four rounds' loads are issued before they are summed (in order)
    for (int z0 = warp; z0 < splits; z0 += 32) {
        float v[4][VPL];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int z = z0 + 8 * q;
            const float* pz = partial + ((size_t)z * T + t) * E;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int e = lane + 32 * i;
                v[q][i] = (z < splits && e < E) ? pz[e] : 0.0f;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (z0 + 8 * q < splits)
#pragma unroll
                for (int i = 0; i < VPL; ++i) acc[i] += v[q][i];
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) part[warp][lane + 32 * i] = acc[i];
    __syncthreads();
    if (warp != 0) return;
    float lg[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        lg[i] = part[0][lane + 32 * i];
#pragma unroll
        for (int w = 1; w < 8; ++w) lg[i] += part[w][lane + 32 * i];
        lg[i] += bv[i];
    }
    select_token<VPL>(lg, slot, t, E, k, slot_of, want_e, want_s, sel_e, sel_slot, sel_w);
}

// A batch in page-locked host memory, copied once into device memory (16-byte
// chunks, grid-stride): the routing kernels then read it from HBM instead of
// pulling it across the chip-to-chip link several times.
__global__ void __launch_bounds__(256) stage_rows(const uint4* __restrict__ src, uint4* __restrict__ dst, long n16) {
    pdl_trigger();
    pdl_wait();
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (long)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_rows(const void* src, void* dst, size_t bytes, cudaStream_t s) {
    const long n16 = (long)(bytes / 16);
    long grid = (n16 + 255) / 256;
    if (grid > moe_sm_count()) grid = moe_sm_count();
    const cudaError_t e = moe_launch(stage_rows, dim3((unsigned)grid), dim3(256), 0, s,
                                     static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
    moe_count_launches(1);
    return e;
}

bool router_rows_eligible(int T, int d) { return T <= ROWS_MAX_T && d % 8 == 0 && d <= 8 * ROWS_MAX_CH * ROWS_THREADS; }

int route_splits(int T, int E, int d) {
    const int gx = (E + BE - 1) / BE, gy = (T + BT - 1) / BT;
    int splits = 1;
    const int kblocks = d / BK;
    while (splits * 2 <= 32 && gx * gy * splits * 2 <= 256 && kblocks % (splits * 2) == 0) splits *= 2;
    return splits;
}

cudaError_t launch_route(const RouteLaunch& a, cudaStream_t s) {
    cudaError_t e;
    if (a.wsplit) {
        e = launch_router_tc(a.x, a.w, a.T, a.d, a.E, a.splits, a.wsplit, a.partial, a.err, a.wait_ns, s);
    } else if (a.rows) {
        moe_prof_begin(MK_ROUTER_LOGITS, s);
        e = moe_launch(router_logits_rows, dim3(a.E), dim3(ROWS_THREADS), 0, s, a.x, a.w, a.T, a.d, a.E, a.partial);
        moe_prof_end(MK_ROUTER_LOGITS, s);
        moe_count_launches(1);
    } else {
        dim3 g1((a.E + BE - 1) / BE, (a.T + BT - 1) / BT, a.splits);
        moe_prof_begin(MK_ROUTER_LOGITS, s);
        e = moe_launch(router_logits_partial, g1, dim3(256), 0, s, a.x, a.w, a.T, a.d, a.E, a.d / a.splits,
                       a.partial);
        moe_prof_end(MK_ROUTER_LOGITS, s);
        moe_count_launches(1);
    }
    if (e != cudaSuccess) return e;
    const int vpl = (a.E + 31) / 32;
    const bool per_cta = a.splits >= 8;             // many K slices: one CTA per token
    dim3 g2(per_cta ? a.T : (a.T + 7) / 8);
#define MOE_SEL(V)                                                                                       \
    moe_launch(per_cta ? route_select_cta<V> : route_select<V>, g2, dim3(256), 0, s, a.partial, a.splits, \
               a.bias, a.slot_of, a.T, a.E, a.k, a.want_e, a.want_s, a.sel_e, a.sel_slot, a.sel_w)
    moe_prof_begin(MK_ROUTE_SELECT, s);
    if (vpl <= 1) e = MOE_SEL(1);
    else if (vpl <= 2) e = MOE_SEL(2);
    else if (vpl <= 4) e = MOE_SEL(4);
    else if (vpl <= 8) e = MOE_SEL(8);
    else if (vpl <= 16) e = MOE_SEL(16);
    else e = MOE_SEL(32);
#undef MOE_SEL
    moe_prof_end(MK_ROUTE_SELECT, s);
    moe_count_launches(1);
    return e;
}

// ------------------------------------------------------------------ optional weight renormalisation
namespace {

// w_j / sum of the token's valid weights, summed in pick order; no valid pick: zeros.
__global__ void __launch_bounds__(256) renormalise_weights(const int32_t* __restrict__ sel_slot,
                                                           float* __restrict__ sel_w, int T, int k) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float z = 0.0f;
    for (int j = 0; j < k; ++j)
        if (sel_slot[(size_t)t * k + j] >= 0) z += sel_w[(size_t)t * k + j];
    const float inv = z > 0.0f ? 1.0f / z : 0.0f;
    for (int j = 0; j < k; ++j) {
        const size_t o = (size_t)t * k + j;
        sel_w[o] = sel_slot[o] >= 0 ? sel_w[o] * inv : 0.0f;
    }
}

}  // namespace

extern "C" moe_status moe_renormalise_weights(const int32_t* sel_slot, float* sel_w, int T, int k, void* stream) {
    MOE_RANGE("moe_renormalise_weights");
    if (!sel_slot || !sel_w || T < 1 || k < 1 || k > 32) return MOE_EINVAL;
    const cudaError_t e = moe_launch(renormalise_weights, dim3((T + 255) / 256), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), sel_slot, sel_w, T, k);
    moe_count_launches(1);
    return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

// ------------------------------------------------------------------ routing without a caller workspace
//
// Some callers cannot allocate device memory at the point where they route:
// code running under an allocator that must not grow (a serving loop that
// fixed its memory budget at start-up, a plug-in whose host framework owns all
// allocations), or code that may not synchronise the device, which a cudaMalloc
// can do. For them the split-K partial logits live in this fixed array instead
// of a caller-provided workspace. It is part of the library's image, so every
// GPU that loads the library holds its 4 MiB until the process exits.
namespace {

constexpr size_t kNoAllocPartials = size_t(1) << 20;          // fp32 partial logits: 4 MiB
static __device__ __align__(256) float g_route_partials[kNoAllocPartials];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[64] = {};

// Device address of the array for the current device, looked up once per device.
cudaError_t noalloc_partials(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_partials);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_resident_noalloc(const void* hidden_bf16, const float* w_router, const float* bias,
                                                 const int32_t* slot_of, int T, int d, int E, int k,
                                                 int32_t* want_e, float* want_s, int32_t* sel_e, int32_t* sel_slot,
                                                 float* sel_w, void* stream) {
    MOE_RANGE("moe_route_resident_noalloc");
    if (!hidden_bf16 || !w_router || !slot_of || !want_e || !want_s || !sel_e || !sel_slot || !sel_w)
        return MOE_EINVAL;
    if (T < 1 || d < 32 || d % 32 || E < 1 || k < 1 || k > 32 || k > E) return MOE_EINVAL;
    if (((uintptr_t)hidden_bf16 | (uintptr_t)w_router) & 15) return MOE_EINVAL;
    if (E > 1024) return MOE_EUNSUPPORTED;
    const int splits = route_splits(T, E, d);
    if ((size_t)splits * T * E > kNoAllocPartials) return MOE_EUNSUPPORTED;   // beyond the fixed array
    const int hk = pointer_kind(hidden_bf16);
    if (hk < 0) return MOE_EINVAL;
    float* partials = nullptr;
    if (noalloc_partials(&partials) != cudaSuccess) return MOE_ECUDA;
    RouteLaunch a{};
    a.x = static_cast<const uint16_t*>(hidden_bf16);
    a.w = w_router;
    a.bias = bias;
    a.slot_of = slot_of;
    a.T = T; a.d = d; a.E = E; a.k = k;
    a.splits = splits;
    if (hk == 0 && router_rows_eligible(T, d)) { a.rows = 1; a.splits = 1; }
    a.want_e = want_e; a.want_s = want_s; a.sel_e = sel_e; a.sel_slot = sel_slot; a.sel_w = sel_w;
    a.partial = partials;      // every element read below is written earlier in the same call
    a.wait_ns = moe_wait_limit_ns();
    return launch_route(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK : MOE_ECUDA;
}
