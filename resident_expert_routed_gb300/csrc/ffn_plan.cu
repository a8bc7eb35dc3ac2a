// Grouping of the routed picks by arena slot, activation quantisation into
// the tensor cores' operand layout, and the weighted combine of the outputs.
//
// TideLM README items 1-2 route each token to resident slots of one shared
// arena; the expert FFN then runs per slot over the rows routed to it. The
// combine adds a token's expert outputs in its own pick order, so the result
// does not depend on how the work was split (colibri cluster page: replies
// are added in the local loop's per-row expert order).
//
// ffn_plan (one CTA): counts picks per slot (shared-memory atomics), gives
//   each slot a segment of positions padded to a multiple of the tile height
//   BN, gives every pick a position in its slot's segment, and writes the GEMM
//   work list: (slot, first position, rows) per tile of at most BN rows.
//   ffn_plan_small computes the same from a sort of (slot, pick) keys, with
//   work in proportion to the picks (arenas of thousands of slots), in one
//   warp for at most 32 picks (and then also packs x for a few tokens).
//   Large batches split it: plan_count (per-CTA histograms), plan_scan (one
//   CTA: per-CTA offsets within each slot, segments, work list), plan_place.
// ffn_prefetch_first (side stream): L2 prefetch of the first K chunks of the
//   weight tiles the gate/up GEMM's CTAs stream first.
// ffn_pack: quantises every token row of x to MXFP4 once (OCP MX v1.0:
//   exponent floor(log2 amax) - 2, round to nearest even, saturate at 6; two
//   codes per byte, even element low) and writes it into row `position` of
//   the gate/up GEMM's activation operand for each of the token's picks, with
//   its scales in the tile's scale atoms, so the GEMM fetches both with plain
//   TMA / bulk copies.
// ffn_combine: out[t] = sum_j sel_w[t,j] * Y[t*k + j], j in order.
#include "common.cuh"

namespace {

constexpr int PLAN_THREADS = 1024;

// From per-slot pick counts cnt[S] (shared memory): each slot's segment of
// positions padded to a multiple of bn (seg), its first work entry (tile_off),
// the work list (slot, first position, rows) and its length. Whole block.
__device__ void plan_slots(const int32_t* cnt, int S, int bn, int32_t* __restrict__ seg,
                           int32_t* __restrict__ tile_off, int4* __restrict__ work, int32_t* __restrict__ n_work,
                           unsigned long long* scan_scratch) {
    const int tid = threadIdx.x;
    // exclusive scan of (padded rows, tiles) per slot; each thread owns a contiguous chunk
    const int chunk = (S + PLAN_THREADS - 1) / PLAN_THREADS;
    const int b0 = tid * chunk, b1 = min(S, b0 + chunk);
    auto packed = [bn](int c) {
        const unsigned long long tiles = (unsigned long long)((c + bn - 1) / bn);
        return (tiles * bn) | (tiles << 32);
    };
    unsigned long long local = 0;
    for (int i = b0; i < b1; ++i) local += packed(cnt[i]);
    unsigned long long total = 0;
    const unsigned long long incl = block_inclusive_scan_u64(local, scan_scratch, &total);
    unsigned long long run = incl - local;
    for (int i = b0; i < b1; ++i) {
        seg[i] = (int32_t)(run & 0xFFFFFFFFull);
        tile_off[i] = (int32_t)(run >> 32);
        run += packed(cnt[i]);
    }
    if (tid == 0) *n_work = (int32_t)(total >> 32);
    __syncthreads();
    for (int i = tid; i < S; i += PLAN_THREADS) {
        const int c = cnt[i];
        const int nt = (c + bn - 1) / bn;
        for (int q = 0; q < nt; ++q) work[tile_off[i] + q] = make_int4(i, seg[i] + q * bn, min(bn, c - q * bn), 0);
    }
}

// Small batches: one CTA counts, scans and places every pick.
__global__ void __launch_bounds__(PLAN_THREADS) ffn_plan(const int32_t* __restrict__ sel_slot, int P, int S, int bn,
                                                         int32_t* __restrict__ pos_of_pair,
                                                         int32_t* __restrict__ pair_of_pos,
                                                         int32_t* __restrict__ seg, int32_t* __restrict__ tile_off,
                                                         int4* __restrict__ work, int32_t* __restrict__ n_work,
                                                         int late_trigger, uint32_t* err) {
    extern __shared__ int32_t cnt[];
    __shared__ unsigned long long scan_scratch[32];
    const int tid = threadIdx.x;
    if (!late_trigger) pdl_trigger();
    for (int i = tid; i < S; i += PLAN_THREADS) cnt[i] = 0;
    pdl_wait();
    if (late_trigger) pdl_trigger();    // after the wait: the pack, launched now, may read x before its own wait
    __syncthreads();
    for (int p = tid; p < P; p += PLAN_THREADS) {
        int s = sel_slot[p];
        if (s >= S) { record_error(err, MOE_DEV_BAD_SLOT); s = -1; }
        pos_of_pair[p] = s >= 0 ? atomicAdd(&cnt[s], 1) : -1;          // rank within the slot for now
    }
    __syncthreads();
    plan_slots(cnt, S, bn, seg, tile_off, work, n_work, scan_scratch);
    for (int p = tid; p < P; p += PLAN_THREADS) {
        const int s = sel_slot[p];
        if (s < 0 || s >= S) continue;
        const int pos = seg[s] + pos_of_pair[p];
        pos_of_pair[p] = pos;
        pair_of_pos[pos] = p;
    }
}

// MXFP4 of one (token t, 32-element block b) of x: 16 bytes of codes and, on
// lane 4g of each group of four lanes, the 4-byte scale word of its 128-element
// group (the four blocks' bytes side by side in the tile's scale atom). Whole
// warps call it together (the word is assembled with shuffles); inactive lanes
// contribute nothing.
__device__ __forceinline__ void pack_quantise(const uint16_t* __restrict__ x, long t, int b, int d, bool active,
                                              uint4& codes, uint32_t& word) {
    codes = make_uint4(0u, 0u, 0u, 0u);
    uint32_t byte = 0;
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(x + t * d + b * 32);
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = src[q];
        const uint16_t* h = reinterpret_cast<const uint16_t*>(v);
        float f[32];
        float amax = 0.0f;
#pragma unroll
        for (int q = 0; q < 32; ++q) { f[q] = bf16_bits_to_float(h[q]); amax = fmaxf(amax, fabsf(f[q])); }
        const int X = mx_shared_exp(amax);
        const float inv = exp2_int(-X);
        codes = make_uint4(e2m1x8(f, inv), e2m1x8(f + 8, inv), e2m1x8(f + 16, inv), e2m1x8(f + 24, inv));
        byte = (uint32_t)(X + 127);
    }
    word = byte;
    word |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
    word |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
    word |= __shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24;
}

// The block's codes and scale word go to the operand row of each of token t's picks.
__device__ __forceinline__ void pack_scatter(const int32_t* __restrict__ pos_of_pair, long t, int b, int k, int d,
                                             int bn, const uint4& codes, uint32_t word, uint8_t* __restrict__ xp,
                                             uint8_t* __restrict__ xsp) {
    for (int j = 0; j < k; ++j) {
        const int pos = pos_of_pair[t * k + j];
        if (pos < 0) continue;
        *reinterpret_cast<uint4*>(xp + (size_t)pos * (d / 2) + b * 16) = codes;
        if ((b & 3) == 0) *reinterpret_cast<uint32_t*>(xsp + operand_scale_offset(pos, b, bn, d)) = word;
    }
}

// At most 32 picks: the plan of ffn_plan_small in one warp, lane = pick, with
// shuffles and ballots instead of block barriers: bitonic sort of the keys
// across the lanes, run heads, and a lane scan of (padded rows, tiles) over
// the heads. Same outputs as the block version.
__device__ __forceinline__ void plan_warp(const int32_t* __restrict__ sel_slot, int P, int S, int bn,
                                          int32_t* __restrict__ pos_of_pair, int32_t* __restrict__ pair_of_pos,
                                          int4* __restrict__ work, int32_t* __restrict__ n_work, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    uint32_t key = 0xFFFFFFFFu;
    if (lane < P) {
        int sl = sel_slot[lane];
        if (sl >= S) { record_error(err, MOE_DEV_BAD_SLOT); sl = -1; }
        if (sl >= 0) key = ((uint32_t)sl << 10) | (uint32_t)lane;
        else pos_of_pair[lane] = -1;
    }
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, key, j);
            const bool up = (lane & k) == 0, lower = (lane & j) == 0;
            key = (up == lower) ? min(key, other) : max(key, other);
        }
    const bool valid = key != 0xFFFFFFFFu;                          // the valid keys come first
    const uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, key, 1);
    const bool head = valid && (lane == 0 || (prev >> 10) != (key >> 10));
    const uint32_t heads = __ballot_sync(0xFFFFFFFFu, head);
    const int n_valid = __popc(__ballot_sync(0xFFFFFFFFu, valid));
    // a head's run ends at the next head (or at the end of the valid keys)
    const uint32_t later = heads & ~((2u << lane) - 1u);
    const int c = head ? (later ? __ffs(later) - 1 : n_valid) - lane : 0;
    const unsigned long long nt = (unsigned long long)((c + bn - 1) / bn);
    const unsigned long long packed = (nt * bn) | (nt << 32);
    unsigned long long incl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    const unsigned long long excl = incl - packed;
    const int seg = (int)(excl & 0xFFFFFFFFull);
    if (head) {
        const int toff = (int)(excl >> 32), r_slot = (int)(key >> 10);
        for (int q = 0; q < (int)nt; ++q) work[toff + q] = make_int4(r_slot, seg + q * bn, min(bn, c - q * bn), 0);
    }
    if (lane == 31) *n_work = (int32_t)(incl >> 32);
    // each valid key: its run's segment start, from the run's head lane
    const uint32_t mine = heads & ((2u << lane) - 1u);
    const int h = mine ? 31 - __clz(mine) : 0;
    const int seg_h = __shfl_sync(0xFFFFFFFFu, seg, h);
    if (valid) {
        const int pick = (int)(key & 1023u);
        const int pos = seg_h + (lane - h);
        pos_of_pair[pick] = pos;
        pair_of_pos[pos] = pick;
    }
}

// Small batches (at most SMALL_PICKS picks), with work in proportion to the
// picks rather than the slots: the (slot, pick) keys are sorted in shared
// memory (bitonic sort of the next power of two >= P), so every used slot is
// one run of equal slots, runs in slot order and each run's picks in pick
// order; block scans give each run's padded segment and first work entry.
// Nothing here visits the S slots one by one, which matters with arenas of
// thousands of slots and a few picks per layer. With `fuse` (few tokens) the
// same CTA then quantises x and writes the operand rows, which saves the pack
// launch: x is complete here, since this kernel runs after its wait.
constexpr int SMALL_PICKS = 1024;
constexpr int SLOT_SCAN_MAX = 2048;                     // arenas up to this many slots plan by counting
constexpr long FUSED_PACK_TASKS = 512;                  // (token, 32-block) tasks: T <= 4 at d = 4096
static_assert(FUSED_PACK_TASKS <= SMALL_PICKS - 32, "the one-warp plan quantises one task per thread of warps 1..");

__global__ void __launch_bounds__(SMALL_PICKS) ffn_plan_small(const int32_t* __restrict__ sel_slot, int P, int S,
                                                              int bn, int32_t* __restrict__ pos_of_pair,
                                                              int32_t* __restrict__ pair_of_pos,
                                                              int4* __restrict__ work, int32_t* __restrict__ n_work,
                                                              int late_trigger, int fuse, const uint16_t* __restrict__ x,
                                                              int T, int k, int d, uint8_t* __restrict__ xp,
                                                              uint8_t* __restrict__ xsp, uint32_t* err) {
    __shared__ uint32_t key[SMALL_PICKS];               // slot << 10 | pick (slot < 2^14), 0xFFFFFFFF = none
    __shared__ int32_t run_start[SMALL_PICKS + 1];
    __shared__ int32_t run_seg[SMALL_PICKS];
    __shared__ unsigned long long scan_scratch[32];
    const int tid = threadIdx.x;
    if (!late_trigger) pdl_trigger();
    pdl_wait();
    if (late_trigger) pdl_trigger();    // after the wait: the pack, launched now, may read x before its own wait
    if (P <= 32) {
        // warp 0 plans; meanwhile warps 1.. quantise x, one (token, 32-block) task per thread
        const int nb = d / 32;
        const long tasks = fuse ? (long)T * nb : 0;
        if (tid < 32) {
            plan_warp(sel_slot, P, S, bn, pos_of_pair, pair_of_pos, work, n_work, err);
            if (!fuse) return;
        } else if (!fuse) {
            return;
        }
        const long i = tid - 32;                                    // task of this thread (warps 1..)
        const bool warp_busy = tid >= 32 && (i & ~31L) < tasks;     // whole warps quantise together
        const bool active = tid >= 32 && i < tasks;
        const long t = active ? i / nb : 0;
        const int b = active ? (int)(i % nb) : 0;
        uint4 codes = make_uint4(0u, 0u, 0u, 0u);
        uint32_t word = 0;
        if (warp_busy) pack_quantise(x, t, b, d, active, codes, word);
        __syncthreads();                                            // the positions are visible to the whole block
        if (active) pack_scatter(pos_of_pair, t, b, k, d, bn, codes, word, xp, xsp);
        return;
    }
    uint32_t kv = 0xFFFFFFFFu;
    if (tid < P) {
        int s = sel_slot[tid];
        if (s >= S) { record_error(err, MOE_DEV_BAD_SLOT); s = -1; }
        if (s >= 0) kv = ((uint32_t)s << 10) | (uint32_t)tid;
        else pos_of_pair[tid] = -1;
    }
    key[tid] = kv;
    int n2 = 32;
    while (n2 < P) n2 <<= 1;                            // keys past P are all 0xFFFFFFFF
    for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            __syncthreads();
            const int ixj = tid ^ j;
            if (tid < n2 && ixj > tid) {
                const uint32_t x = key[tid], y = key[ixj];
                if ((x > y) == ((tid & k) == 0)) { key[tid] = y; key[ixj] = x; }
            }
        }
    __syncthreads();
    const uint32_t me = key[tid];
    const bool valid = me != 0xFFFFFFFFu;               // the valid keys come first
    const bool head = valid && (tid == 0 || (key[tid - 1] >> 10) != (me >> 10));
    unsigned long long n_runs, n_valid;
    const int run = (int)block_inclusive_scan_u64(head ? 1ull : 0ull, scan_scratch, &n_runs) - 1;
    (void)block_inclusive_scan_u64(valid ? 1ull : 0ull, scan_scratch, &n_valid);
    if (head) run_start[run] = tid;
    if (tid == 0) run_start[n_runs] = (int)n_valid;
    __syncthreads();
    // thread r < n_runs: run r's slot, its padded rows and tiles, scanned in slot order
    int c = 0, r_slot = 0;
    if (tid < (int)n_runs) {
        c = run_start[tid + 1] - run_start[tid];
        r_slot = (int)(key[run_start[tid]] >> 10);
    }
    const unsigned long long nt = (unsigned long long)((c + bn - 1) / bn);
    const unsigned long long packed = (nt * bn) | (nt << 32);
    unsigned long long total;
    const unsigned long long excl = block_inclusive_scan_u64(packed, scan_scratch, &total) - packed;
    if (tid < (int)n_runs) {
        const int seg = (int)(excl & 0xFFFFFFFFull), toff = (int)(excl >> 32);
        run_seg[tid] = seg;
        for (int q = 0; q < (int)nt; ++q)
            work[toff + q] = make_int4(r_slot, seg + q * bn, min(bn, c - q * bn), 0);
    }
    if (tid == 0) *n_work = (int32_t)(total >> 32);
    __syncthreads();
    if (valid) {
        const int pick = (int)(me & 1023u);
        const int pos = run_seg[run] + (tid - run_start[run]);
        pos_of_pair[pick] = pos;
        pair_of_pos[pos] = pick;
    }
    if (!fuse) return;
    __syncthreads();                                    // the positions are visible to the whole block
    const int nb = d / 32;
    const long tasks = (long)T * nb;
    for (long i0 = 0; i0 < tasks; i0 += SMALL_PICKS) {  // whole warps iterate together
        const long i = i0 + tid;
        const bool active = i < tasks;
        const long t = active ? i / nb : 0;
        const int b = active ? (int)(i % nb) : 0;
        uint4 codes;
        uint32_t word;
        pack_quantise(x, t, b, d, active, codes, word);
        if (active) pack_scatter(pos_of_pair, t, b, k, d, bn, codes, word, xp, xsp);
    }
}

// Large batches, in three kernels. 1: each CTA counts the picks of its chunk
// per slot (shared-memory histogram) and notes each pick's rank among them.
__global__ void __launch_bounds__(PLAN_THREADS) plan_count(const int32_t* __restrict__ sel_slot, int P, int S,
                                                           int chunk, int32_t* __restrict__ rank,
                                                           int32_t* __restrict__ cta_counts, uint32_t* err) {
    extern __shared__ int32_t cnt[];
    pdl_trigger();
    for (int i = threadIdx.x; i < S; i += PLAN_THREADS) cnt[i] = 0;
    pdl_wait();
    __syncthreads();
    const int p1 = min(P, (blockIdx.x + 1) * chunk);
    for (int p = blockIdx.x * chunk + threadIdx.x; p < p1; p += PLAN_THREADS) {
        int s = sel_slot[p];
        if (s >= S) { record_error(err, MOE_DEV_BAD_SLOT); s = -1; }
        rank[p] = s >= 0 ? atomicAdd(&cnt[s], 1) : -1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += PLAN_THREADS) cta_counts[(size_t)blockIdx.x * S + i] = cnt[i];
}

// 2 (one CTA): per slot, each CTA's offset within the slot (CTA order) and the
// slot's total; then the segments and the work list.
__global__ void __launch_bounds__(PLAN_THREADS) plan_scan(int G, int S, int bn, int32_t* __restrict__ cta_counts,
                                                          int32_t* __restrict__ seg, int32_t* __restrict__ tile_off,
                                                          int4* __restrict__ work, int32_t* __restrict__ n_work) {
    extern __shared__ int32_t cnt[];
    __shared__ unsigned long long scan_scratch[32];
    pdl_trigger();
    pdl_wait();
    for (int i = threadIdx.x; i < S; i += PLAN_THREADS) {
        int run = 0;
        for (int g = 0; g < G; ++g) {
            const int c = cta_counts[(size_t)g * S + i];
            cta_counts[(size_t)g * S + i] = run;
            run += c;
        }
        cnt[i] = run;
    }
    __syncthreads();
    plan_slots(cnt, S, bn, seg, tile_off, work, n_work, scan_scratch);
}

// 3: each pick's position = its slot's segment + its CTA's offset + its rank.
__global__ void __launch_bounds__(256) plan_place(const int32_t* __restrict__ sel_slot, int P, int S, int chunk,
                                                  const int32_t* __restrict__ cta_offsets,
                                                  const int32_t* __restrict__ seg, int32_t* __restrict__ pos_of_pair,
                                                  int32_t* __restrict__ pair_of_pos) {
    pdl_wait();
    pdl_trigger();          // after the wait: the pack, launched now, reads x before its own wait
    const int g = blockIdx.y;
    const int p1 = min(P, (g + 1) * chunk);
    for (int p = g * chunk + blockIdx.x * blockDim.x + threadIdx.x; p < p1; p += gridDim.x * blockDim.x) {
        const int s = sel_slot[p];
        if (s < 0 || s >= S) continue;
        const int pos = seg[s] + cta_offsets[(size_t)g * S + s] + pos_of_pair[p];
        pos_of_pair[p] = pos;
        pair_of_pos[pos] = p;
    }
}

// One thread per (token, 32-element block): the token's 64 bytes of bf16 are
// quantised once (not once per pick), then the 16 bytes of codes go to the
// operand row of each of the token's picks. The four scale bytes of a
// 128-element group sit side by side in the tile's scale atom; d is a multiple
// of 128, so lanes 4g..4g+3 of a warp hold one group of one token and lane 4g
// stores the four bytes as one word.
// With `early` the quantisation runs before the wait for the plan: the plan
// kernel before this one then signals its dependents only after its own wait,
// so this kernel starts once every kernel before the plan, including whatever
// wrote x, has finished; only the positions need the plan. Small batches (too
// little to quantise to hide the later launch) wait first.
__global__ void __launch_bounds__(256) ffn_pack(const uint16_t* __restrict__ x, const int32_t* __restrict__ pos_of_pair,
                                                int T, int k, int d, int bn, int early, uint8_t* __restrict__ xp,
                                                uint8_t* __restrict__ xsp) {
    pdl_trigger();
    if (!early) pdl_wait();
    const int nb = d / 32;
    const long total = (long)T * nb;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;     // whole warps: the grid covers every task
    const bool active = i < total;
    const long t = active ? i / nb : 0;
    const int b = active ? (int)(i % nb) : 0;
    uint4 codes;
    uint32_t word;
    pack_quantise(x, t, b, d, active, codes, word);
    if (early) pdl_wait();                                          // positions are the plan's output
    if (!active) return;
    pack_scatter(pos_of_pair, t, b, k, d, bn, codes, word, xp, xsp);
}

__global__ void __launch_bounds__(256) ffn_combine(const float* __restrict__ Y, const int32_t* __restrict__ sel_slot,
                                                   const float* __restrict__ sel_w, int k, int d, int S,
                                                   float* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int s = sel_slot[(size_t)t * k + j];
        if (s < 0 || s >= S) continue;
        const float w = sel_w[(size_t)t * k + j];
        // streaming load (read once): Y is the largest stream at prefill and need not stay in L2
        const float4 y = __ldcs(reinterpret_cast<const float4*>(Y + ((size_t)t * k + j) * d + c));
        acc.x = fmaf(w, y.x, acc.x);
        acc.y = fmaf(w, y.y, acc.y);
        acc.z = fmaf(w, y.z, acc.z);
        acc.w = fmaf(w, y.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + (size_t)t * d + c) = acc;
}

// Used slots in index order head the plan's work list (its tiles follow the
// slot order), so the gate/up GEMM's persistent grid streams their weights
// first: its CTA b takes feature tile b % m_tiles of the (b / m_tiles)-th used
// slot (one token tile per slot assumed). CTA b of this kernel prefetches the
// same code blocks and scale atoms into L2, so that the prefetches come from
// every SM's copy engine at once. Only the first PREFETCH_CHUNKS 256-element K
// chunks of each tile (the first stages the GEMM streams, 128 KB of codes at
// four chunks) are prefetched: that covers the GEMM's start, while whole tiles
// (544 KB each at d = 4096) went on arriving after the GEMM had read them
// itself and took HBM time from it.
constexpr int PREFETCH_CHUNKS = 4;

__global__ void __launch_bounds__(128) ffn_prefetch_first(const int32_t* __restrict__ sel_slot, int P, int S,
                                                          const uint8_t* __restrict__ arena, long long slot_bytes,
                                                          long long off_codes, long long off_scales, int m_tiles,
                                                          int nc, int atoms) {
    extern __shared__ uint32_t used[];                  // one bit per slot
    __shared__ int slot;
    pdl_trigger();
    const int nw = (S + 31) / 32;
    for (int i = threadIdx.x; i < nw; i += blockDim.x) used[i] = 0;
    pdl_wait();
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int s = sel_slot[p];
        if (s >= 0 && s < S) atomicOr(&used[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int want = (int)blockIdx.x / m_tiles, found = -1;
        for (int i = 0; i < nw && found < 0; ++i) {
            const int c = __popc(used[i]);
            if (want < c) {
                uint32_t m = used[i];
                for (int q = 0; q < want; ++q) m &= m - 1;      // drop the lowest set bits
                found = i * 32 + __ffs(m) - 1;
            } else {
                want -= c;
            }
        }
        slot = found;
    }
    __syncthreads();
    if (slot < 0) return;
    const int mt = (int)blockIdx.x % m_tiles;
    const uint8_t* rec = arena + (size_t)slot * slot_bytes;
    const int npf = nc < PREFETCH_CHUNKS ? nc : PREFETCH_CHUNKS;
    const int apf = 2 * npf < atoms ? 2 * npf : atoms;                  // two scale atoms per chunk
    for (int r = threadIdx.x; r < 2 * npf + 2; r += blockDim.x) {
        if (r < 2 * npf) {
            const int tile = r < npf ? mt : m_tiles + mt;               // up tiles follow the gate tiles
            bulk_prefetch_l2(rec + off_codes + ((size_t)tile * nc + r % npf) * 16384, 16384);
        } else {
            const int tile = r == 2 * npf ? mt : m_tiles + mt;
            bulk_prefetch_l2(rec + off_scales + (size_t)tile * atoms * 512, (uint32_t)apf * 512);
        }
    }
}

}  // namespace

cudaError_t launch_ffn_prefetch(const int32_t* sel_slot, int P, const moe_arena& ar, cudaStream_t s) {
    const int nw = (ar.n_slots + 31) / 32;
    const cudaError_t e = moe_launch(ffn_prefetch_first, dim3((unsigned)moe_sm_count()), dim3(128),
                                     (size_t)nw * 4, s, sel_slot, P, ar.n_slots,
                                     static_cast<const uint8_t*>(ar.base), (long long)ar.slot_bytes,
                                     (long long)ar.off_gu_codes, (long long)ar.off_gu_scales, ar.ffn / 128,
                                     (ar.d + 255) / 256, ar.d / 128);
    moe_count_launches(1);
    return e;
}

cudaError_t launch_ffn_plan(const FfnLaunch& a, cudaStream_t s) {
    const int P = a.T * a.k;
    // batches of 8 tokens or more quantise x while the plan runs (large batches always: their plan ends
    // with plan_place, which signals after its wait)
    const int early = a.plan_ctas > 0 || a.T >= 8 ? 1 : 0;
    // more than 32 picks over an arena of a few thousand slots at most: counting per slot (shared
    // atomics, one scan over the slots) is cheaper than the small plan's sort, which wins on large arenas
    const bool by_slot = a.plan_ctas == 0 && P > 32 && a.S <= SLOT_SCAN_MAX;
    // few tokens: the small plan also packs x (one launch fewer)
    const bool fused = a.plan_ctas == 0 && P <= SMALL_PICKS && !by_slot && (long)a.T * (a.d / 32) <= FUSED_PACK_TASKS;
    const size_t smem = (size_t)a.S * sizeof(int32_t);
    static bool attr_set[64] = {};
    static bool attr_set_multi[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ffn_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    moe_prof_begin(MK_PLAN, s);
    cudaError_t e;
    if (a.plan_ctas > 0) {
        if (dev < 64 && !attr_set_multi[dev]) {
            e = cudaFuncSetAttribute(plan_count, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(plan_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
            if (e != cudaSuccess) return e;
            attr_set_multi[dev] = true;
        }
        const int G = a.plan_ctas, chunk = (P + G - 1) / G;
        e = moe_launch(plan_count, dim3(G), dim3(PLAN_THREADS), smem, s, a.sel_slot, P, a.S, chunk, a.pos_of_pair,
                       a.cta_counts, a.err);
        if (e == cudaSuccess)
            e = moe_launch(plan_scan, dim3(1), dim3(PLAN_THREADS), smem, s, G, a.S, a.bn, a.cta_counts, a.seg,
                           a.tile_off, a.work, a.n_work);
        if (e == cudaSuccess)
            e = moe_launch(plan_place, dim3((chunk + 255) / 256, G), dim3(256), 0, s, a.sel_slot, P, a.S, chunk,
                           static_cast<const int32_t*>(a.cta_counts), static_cast<const int32_t*>(a.seg),
                           a.pos_of_pair, a.pair_of_pos);
        moe_count_launches(2);
    } else {
        if (P <= SMALL_PICKS && !by_slot)
            e = moe_launch(ffn_plan_small, dim3(1), dim3(SMALL_PICKS), 0, s, a.sel_slot, P, a.S, a.bn, a.pos_of_pair,
                           a.pair_of_pos, a.work, a.n_work, fused ? 0 : early, fused ? 1 : 0, a.x, a.T, a.k, a.d,
                           a.xp, a.xsp, a.err);
        else
            e = moe_launch(ffn_plan, dim3(1), dim3(PLAN_THREADS), smem, s, a.sel_slot, P, a.S, a.bn, a.pos_of_pair,
                           a.pair_of_pos, a.seg, a.tile_off, a.work, a.n_work, early, a.err);
    }
    moe_prof_end(MK_PLAN, s);
    if (e != cudaSuccess) return e;
    if (fused) {
        moe_count_launches(1);
        return e;
    }
    const long tasks = (long)a.T * (a.d / 32);
    const long blocks = (tasks + 255) / 256;                // one task per thread (at most 2^20 * 512 / 256)
    moe_prof_begin(MK_PACK, s);
    e = moe_launch(ffn_pack, dim3((unsigned)blocks), dim3(256), 0, s, a.x, a.pos_of_pair, a.T, a.k, a.d, a.bn,
                   early, a.xp, a.xsp);
    moe_prof_end(MK_PACK, s);
    moe_count_launches(2);
    return e;
}

cudaError_t launch_ffn_combine(const FfnLaunch& a, cudaStream_t s) {
    dim3 g(a.T, (a.d / 4 + 255) / 256);
    moe_prof_begin(MK_COMBINE, s);
    const cudaError_t e = moe_launch(ffn_combine, g, dim3(256), 0, s, a.Y, a.sel_slot, a.sel_w, a.k, a.d, a.S,
                                     a.out);
    moe_prof_end(MK_COMBINE, s);
    moe_count_launches(1);
    return e;
}
