// Re-plan of the one shared expert arena, and the hot-read ring install.
//
// TideLM README, "How adaptive expert loading works":
//   item 1  the arena's contents follow the learned demand history and are
//           planned again from time to time (after a prefill, every few
//           hundred tokens, between requests); all layers draw on a single
//           arena, so layers with more demand hold more of its slots;
//   item 3  (DeepSeek) the largest misses of a step are fetched into extra
//           ring slots beyond the main budget, usable from the step after
//           next, until later fetches wrap around the ring.
//
// arena_replan runs in one CTA (it is off the per-token path): a bitonic sort
// of (demand, currently-main flag, inverted flat id) keys in the workspace,
// then stable compactions of the free main slots and of the newcomers, which
// take those slots in rank order.
#include "common.cuh"

namespace {

constexpr int RP_THREADS = 1024;

// Exclusive stable compaction over [0, len): each thread owns a contiguous
// chunk; returns (through `base`) the count of set predicates in earlier chunks.
__device__ int block_exclusive_count(int local, unsigned long long* part /* smem [RP_THREADS] */, int* total) {
    const int tid = threadIdx.x;
    part[tid] = (unsigned long long)local;
    __syncthreads();
    for (int off = 1; off < RP_THREADS; off <<= 1) {
        unsigned long long v = tid >= off ? part[tid - off] : 0ull;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    const int excl = tid > 0 ? (int)part[tid - 1] : 0;
    *total = (int)part[RP_THREADS - 1];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(RP_THREADS) arena_replan(const unsigned long long* __restrict__ D, int n, int n2,
                                                           int n_main, int n_slots, int32_t* __restrict__ slot_of,
                                                           int32_t* __restrict__ owner, int32_t* __restrict__ loads,
                                                           int32_t* __restrict__ n_loads,
                                                           unsigned long long* __restrict__ kd,
                                                           uint32_t* __restrict__ ks, int32_t* __restrict__ flag,
                                                           int32_t* __restrict__ free_list, uint32_t* err) {
    __shared__ unsigned long long part[RP_THREADS];
    __shared__ int bad;
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    // table consistency: owner[s] = f  <=>  slot_of[f] = s
    for (int s = tid; s < n_slots; s += RP_THREADS) {
        const int f = owner[s];
        if (f >= n || (f >= 0 && slot_of[f] != s)) bad = 1;
    }
    for (int f = tid; f < n; f += RP_THREADS) {
        const int s = slot_of[f];
        if (s >= n_slots || (s >= 0 && owner[s] != f)) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) { record_error(err, MOE_DEV_BAD_TABLE); *n_loads = 0; }
        return;
    }
    // keys: demand, then "in a main slot now", then lower flat id first
    for (int i = tid; i < n2; i += RP_THREADS) {
        if (i < n) {
            const int s = slot_of[i];
            const uint32_t was = (s >= 0 && s < n_main) ? 1u : 0u;
            kd[i] = D[i];
            ks[i] = (was << 30) | (0x3FFFFFFFu - (uint32_t)i);
            flag[i] = 0;
        } else {
            kd[i] = 0ull;
            ks[i] = 0u;
        }
    }
    __syncthreads();
    // bitonic sort, descending by (kd, ks)
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2 / 2; i += RP_THREADS) {
                const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long dl = kd[lo], dh = kd[hi];
                const uint32_t sl = ks[lo], sh = ks[hi];
                const bool lo_less = dl < dh || (dl == dh && sl < sh);
                const bool lo_more = dl > dh || (dl == dh && sl > sh);
                if (desc ? lo_less : lo_more) {
                    kd[lo] = dh; kd[hi] = dl;
                    ks[lo] = sh; ks[hi] = sl;
                }
            }
            __syncthreads();
        }
    }
    const int m = n_main < n ? n_main : n;
    for (int r = tid; r < m; r += RP_THREADS) flag[0x3FFFFFFF - (int)(ks[r] & 0x3FFFFFFFu)] = 1;
    __syncthreads();
    // evict main-set members that fell out
    for (int f = tid; f < n; f += RP_THREADS) {
        const int s = slot_of[f];
        if (s >= 0 && s < n_main && !flag[f]) { owner[s] = -1; slot_of[f] = -1; }
    }
    __syncthreads();
    // free main slots, ascending
    int chunk = (n_main + RP_THREADS - 1) / RP_THREADS;
    int b0 = tid * chunk, b1 = min(n_main, b0 + chunk);
    int local = 0;
    for (int s = b0; s < b1; ++s) local += owner[s] < 0;
    int n_free = 0;
    int w = block_exclusive_count(local, part, &n_free);
    for (int s = b0; s < b1; ++s) if (owner[s] < 0) free_list[w++] = s;
    __syncthreads();
    // newcomers in rank order take them
    chunk = (m + RP_THREADS - 1) / RP_THREADS;
    b0 = tid * chunk;
    b1 = min(m, b0 + chunk);
    local = 0;
    for (int r = b0; r < b1; ++r) local += !((ks[r] >> 30) & 1u);
    int n_new = 0;
    w = block_exclusive_count(local, part, &n_new);
    for (int r = b0; r < b1; ++r) {
        if ((ks[r] >> 30) & 1u) continue;
        const int f = 0x3FFFFFFF - (int)(ks[r] & 0x3FFFFFFFu);
        if (w >= n_free) { record_error(err, MOE_DEV_BAD_TABLE); ++w; continue; }
        const int s = free_list[w];
        const int old = slot_of[f];
        if (old >= n_main) owner[old] = -1;           // promoted out of the ring
        owner[s] = f;
        slot_of[f] = s;
        loads[w] = s;
        ++w;
    }
    if (tid == 0) *n_loads = n_new < n_free ? n_new : n_free;
}

__global__ void ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat, uint32_t* err) {
    pdl_trigger();
    pdl_wait();
    if (slot_of[flat] >= 0) { record_error(err, MOE_DEV_RESIDENT); return; }
    const int old = owner[ring_slot];
    if (old >= 0) slot_of[old] = -1;
    owner[ring_slot] = flat;
    slot_of[flat] = ring_slot;
}

}  // namespace

size_t replan_workspace(int n) {
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    return (size_t)n2 * (8 + 4) + (size_t)n * 4 + (size_t)n * 4 + 256;
}

cudaError_t launch_replan(const unsigned long long* demand, int n, int n_main, int n_slots, int32_t* slot_of,
                          int32_t* owner, int32_t* loads, int32_t* n_loads, void* ws, cudaStream_t s,
                          uint32_t* err) {
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    uint8_t* p = static_cast<uint8_t*>(ws);
    unsigned long long* kd = reinterpret_cast<unsigned long long*>(p);
    uint32_t* ks = reinterpret_cast<uint32_t*>(p + (size_t)n2 * 8);
    int32_t* flag = reinterpret_cast<int32_t*>(p + (size_t)n2 * 12);
    int32_t* free_list = flag + n;
    moe_prof_begin(MK_REPLAN, s);
    const cudaError_t e = moe_launch(arena_replan, dim3(1), dim3(RP_THREADS), 0, s, demand, n, n2, n_main, n_slots,
                                     slot_of, owner, loads, n_loads, kd, ks, flag, free_list, err);
    moe_prof_end(MK_REPLAN, s);
    moe_count_launches(1);
    return e;
}

cudaError_t launch_ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat, cudaStream_t s,
                                uint32_t* err) {
    moe_prof_begin(MK_RING, s);
    const cudaError_t e = moe_launch(ring_install, dim3(1), dim3(1), 0, s, slot_of, owner, ring_slot, flat, err);
    moe_prof_end(MK_RING, s);
    moe_count_launches(1);
    return e;
}
