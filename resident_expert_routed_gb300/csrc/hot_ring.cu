// The asynchronous hot-read ring (TideLM README, "How adaptive expert loading
// works", item 3, the DeepSeek variant: once a step ends, its largest misses
// are fetched into a dedicated set of ring slots during the following step;
// they can be routed to from the step after that, and stay until newer
// fetches wrap around the ring. "Settings worth knowing": these slots come in
// addition to the main slot budget).
//
// A host object drives it at step boundaries. One call, made after step s
// has been enqueued (including its heavy-miss list):
//   1. installs the experts whose copies the previous call issued (the
//      compute stream waits for those copies): routable from step s + 1;
//   2. reads step s's heavy-miss list (the host waits for step s to finish,
//      as a decode loop does to read its sampled token);
//   3. for each heavy miss with a record in the host store (the stand-in for
//      the drive) that is not already in the ring, takes the next ring slot in
//      FIFO order, removes the slot's current owner from the routing tables on
//      the compute stream (so nothing from step s + 1 on reads the slot), and
//      copies the record into the slot on the copy stream once that removal
//      is done. Those experts are installed by the next call: routable from
//      step s + 2, while step s + 1 ran beside the copies.
// Table updates are small kernels on the compute stream; an install of an
// expert that became resident meanwhile is refused (MOE_DEV_RESIDENT), as for
// moe_ring_install. The GLM-5.3 variant, a synchronous read of a layer's
// heaviest miss into the coldest expert's slot, is moe_hot_read_sync below.
#include <vector>

#include "common.cuh"

namespace {

constexpr int RING_BATCH = 32;

struct RingBatch {
    int n;
    int slot[RING_BATCH];
    int flat[RING_BATCH];
};

// owner[slot] = -1 and slot_of[old owner] = -1 for every slot of the batch.
__global__ void ring_evict_batch(int32_t* slot_of, int32_t* owner, RingBatch b) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x != 0) return;
    for (int i = 0; i < b.n; ++i) {
        const int old = owner[b.slot[i]];
        if (old >= 0 && slot_of[old] == b.slot[i]) slot_of[old] = -1;
        owner[b.slot[i]] = -1;
    }
}

// Make each flat id resident in its slot (slots were emptied by ring_evict_batch).
__global__ void ring_install_batch(int32_t* slot_of, int32_t* owner, RingBatch b, uint32_t* err) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x != 0) return;
    for (int i = 0; i < b.n; ++i) {
        const int f = b.flat[i], s = b.slot[i];
        if (slot_of[f] >= 0) { record_error(err, MOE_DEV_RESIDENT); continue; }
        const int old = owner[s];
        if (old >= 0 && slot_of[old] == s) slot_of[old] = -1;
        owner[s] = f;
        slot_of[f] = s;
    }
}

// ------------------------------------------------------------------ synchronous hot read (GLM-5.3)
//
// README item 3, the GLM-5.3 variant: before a layer's MoE runs, its largest
// miss (a share of at least 0.2 of a token's routing weight; at most 16 such
// reads per step, spread over the layers) is loaded, used for this layer with
// its exact weights, and then stays resident, evicting the expert with the
// least demand. One CTA picks the expert and the victim and updates the
// tables; a grid-wide copy then streams the record from the store (host
// memory the device can address) into the victim's slot. The caller routes
// the layer again before its FFN.

// Block-wide max of a 64-bit key (256 threads).
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
        v = o > v ? o : v;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long r = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = red[w] > r ? red[w] : r;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(256) hot_read_choose(const unsigned long long* __restrict__ store,
                                                       const unsigned long long* __restrict__ D,
                                                       const float* __restrict__ M, int32_t* slot_of,
                                                       int32_t* owner, int layer, int E, float thr,
                                                       int32_t* budget, int32_t* swap) {
    __shared__ unsigned long long red[8];
    pdl_trigger();
    pdl_wait();
    const size_t base = (size_t)layer * E;
    // heaviest servable miss: key (share bits, ~e), larger wins; shares are >= 0 so bits order like values
    unsigned long long best = 0;
    // coldest resident: the lowest demand, then the lowest index: max of ~(demand) then of ~e
    unsigned long long cold = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const float m = M[base + e];
        if (slot_of[base + e] < 0 && store[base + e] != 0ull && m >= thr)
            best = max(best, ((unsigned long long)__float_as_uint(m) << 32) | (0xFFFFFFFFull - (unsigned)e));
        if (slot_of[base + e] >= 0) cold = max(cold, ~D[base + e]);
    }
    best = block_max_u64(best, red);
    const unsigned long long cold_key = block_max_u64(cold, red);      // ~(lowest demand), 0 if none resident
    unsigned long long cold_e = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (slot_of[base + e] >= 0 && ~D[base + e] == cold_key) cold_e = max(cold_e, 0xFFFFFFFFull - (unsigned)e);
    cold_e = block_max_u64(cold_e, red);
    if (threadIdx.x != 0) return;
    swap[0] = swap[1] = swap[2] = -1;
    if (best == 0ull || cold_e == 0ull || *budget <= 0) return;
    const int e_read = (int)(0xFFFFFFFFull - (best & 0xFFFFFFFFull));
    const int e_cold = (int)(0xFFFFFFFFull - cold_e);
    const int slot = slot_of[base + e_cold];
    *budget -= 1;
    slot_of[base + e_cold] = -1;
    slot_of[base + e_read] = slot;
    owner[slot] = (int)(base + e_read);
    swap[0] = (int)(base + e_read);
    swap[1] = slot;
    swap[2] = (int)(base + e_cold);
}

__global__ void __launch_bounds__(256) hot_read_copy(const unsigned long long* __restrict__ store,
                                                     const int32_t* __restrict__ swap, uint8_t* arena,
                                                     long long slot_bytes) {
    pdl_trigger();
    pdl_wait();
    const int f = swap[0];
    if (f < 0) return;
    const uint4* src = reinterpret_cast<const uint4*>(store[f]);
    uint4* dst = reinterpret_cast<uint4*>(arena + (size_t)swap[1] * (size_t)slot_bytes);
    const long long n = slot_bytes / 16;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

extern "C" moe_status moe_hot_read_sync(const uint64_t* store, const uint64_t* demand, const float* miss_max,
                                        int32_t* slot_of, int32_t* owner, const moe_arena* arena, int layer,
                                        int L, int E, float threshold, int32_t* budget, int32_t* swap,
                                        void* stream) {
    MOE_RANGE("moe_hot_read_sync");
    if (!store || !demand || !miss_max || !slot_of || !owner || !arena || !arena->base || !budget || !swap)
        return MOE_EINVAL;
    if (L < 1 || E < 1 || layer < 0 || layer >= L || arena->slot_bytes <= 0 || arena->slot_bytes % 16 ||
        !(threshold >= 0.0f))
        return MOE_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned long long* st = reinterpret_cast<const unsigned long long*>(store);
    cudaError_t e = moe_launch(hot_read_choose, dim3(1), dim3(256), 0, s, st,
                               reinterpret_cast<const unsigned long long*>(demand), miss_max, slot_of, owner, layer,
                               E, threshold, budget, swap);
    if (e == cudaSuccess)
        e = moe_launch(hot_read_copy, dim3((unsigned)(4 * moe_sm_count())), dim3(256), 0, s, st,
                       static_cast<const int32_t*>(swap), static_cast<uint8_t*>(arena->base),
                       (long long)arena->slot_bytes);
    moe_count_launches(2);
    return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

struct moe_hot_ring {
    moe_arena arena;
    int ring_first = 0, n_ring = 0, n_flat = 0, cap = 0;
    std::vector<const void*> records;     // host record of each flat id (or null)
    std::vector<int> ring_flat;           // last flat id copied into each ring slot (host view), -1 = none
    int next = 0;                         // FIFO position in the ring
    RingBatch pending{};                  // copies issued by the previous call, installed by the next
    int32_t* list = nullptr;              // pinned: [0] = count, [1..cap] = flat ids
    cudaEvent_t list_ready = nullptr, evicted = nullptr, copied = nullptr;
    bool copies_in_flight = false;
};

namespace {

cudaError_t launch_batch(bool install, const RingBatch& b, int32_t* slot_of, int32_t* owner, cudaStream_t s) {
    if (b.n == 0) return cudaSuccess;
    cudaError_t e;
    if (install) {
        uint32_t* err = moe_err_word();
        if (!err) return cudaErrorUnknown;
        e = moe_launch(ring_install_batch, dim3(1), dim3(32), 0, s, slot_of, owner, b, err);
    } else {
        e = moe_launch(ring_evict_batch, dim3(1), dim3(32), 0, s, slot_of, owner, b);
    }
    moe_count_launches(1);
    return e;
}

}  // namespace

extern "C" moe_status moe_hot_ring_create(const moe_arena* arena, int ring_first, int n_ring, int n_flat,
                                          const void* const* host_records, int cap, moe_hot_ring** ring) {
    if (!arena || !host_records || !ring || !arena->base || n_flat < 1 || n_ring < 1 || ring_first < 0 ||
        ring_first + n_ring > arena->n_slots || cap < 1 || cap > RING_BATCH || arena->slot_bytes <= 0)
        return MOE_EINVAL;
    *ring = nullptr;
    auto* r = new moe_hot_ring();
    r->arena = *arena;
    r->ring_first = ring_first;
    r->n_ring = n_ring;
    r->n_flat = n_flat;
    r->cap = cap;
    r->records.assign(host_records, host_records + n_flat);
    r->ring_flat.assign(n_ring, -1);
    if (cudaMallocHost(&r->list, sizeof(int32_t) * (1 + cap)) != cudaSuccess ||
        cudaEventCreateWithFlags(&r->list_ready, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&r->evicted, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&r->copied, cudaEventDisableTiming) != cudaSuccess) {
        moe_hot_ring_destroy(r);
        return MOE_ECUDA;
    }
    *ring = r;
    return MOE_OK;
}

extern "C" moe_status moe_hot_ring_step(moe_hot_ring* r, const int32_t* heavy_flat, const int32_t* n_heavy,
                                        int32_t* slot_of, int32_t* owner, void* stream, void* copy_stream,
                                        int32_t* n_fetched) {
    MOE_RANGE("moe_hot_ring_step");
    if (!r || !heavy_flat || !n_heavy || !slot_of || !owner) return MOE_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    if (n_fetched) *n_fetched = 0;
    // 1. install what the previous call copied
    if (r->pending.n > 0) {
        if (cudaStreamWaitEvent(s, r->copied, 0) != cudaSuccess) return MOE_ECUDA;
        if (launch_batch(true, r->pending, slot_of, owner, s) != cudaSuccess) return MOE_ECUDA;
        r->pending.n = 0;
    }
    // 2. this step's heavy-miss list
    if (cudaMemcpyAsync(r->list, n_heavy, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(r->list + 1, heavy_flat, sizeof(int32_t) * r->cap, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaEventRecord(r->list_ready, s) != cudaSuccess || cudaEventSynchronize(r->list_ready) != cudaSuccess)
        return MOE_ECUDA;
    // 3. choose ring slots in FIFO order for the misses the store can serve
    RingBatch b{};
    const int n = r->list[0] < r->cap ? r->list[0] : r->cap;
    for (int i = 0; i < n && b.n < r->n_ring; ++i) {
        const int f = r->list[1 + i];
        if (f < 0 || f >= r->n_flat || !r->records[f]) continue;
        bool in_ring = false;
        for (int q = 0; q < r->n_ring && !in_ring; ++q) in_ring = r->ring_flat[q] == f;
        if (in_ring) continue;
        b.slot[b.n] = r->ring_first + r->next;
        b.flat[b.n] = f;
        r->ring_flat[r->next] = f;
        r->next = (r->next + 1) % r->n_ring;
        ++b.n;
    }
    if (b.n == 0) return MOE_OK;
    if (launch_batch(false, b, slot_of, owner, s) != cudaSuccess || cudaEventRecord(r->evicted, s) != cudaSuccess ||
        cudaStreamWaitEvent(cs, r->evicted, 0) != cudaSuccess)
        return MOE_ECUDA;
    uint8_t* base = static_cast<uint8_t*>(r->arena.base);
    for (int i = 0; i < b.n; ++i)
        if (cudaMemcpyAsync(base + (size_t)b.slot[i] * r->arena.slot_bytes, r->records[b.flat[i]],
                            (size_t)r->arena.slot_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return MOE_ECUDA;
    if (cudaEventRecord(r->copied, cs) != cudaSuccess) return MOE_ECUDA;
    r->pending = b;
    r->copies_in_flight = true;
    if (n_fetched) *n_fetched = b.n;
    return MOE_OK;
}

extern "C" moe_status moe_hot_ring_destroy(moe_hot_ring* r) {
    if (!r) return MOE_OK;
    moe_status st = MOE_OK;
    if (r->copies_in_flight && r->copied && cudaEventSynchronize(r->copied) != cudaSuccess) st = MOE_ECUDA;
    if (r->list) cudaFreeHost(r->list);
    if (r->list_ready) cudaEventDestroy(r->list_ready);
    if (r->evicted) cudaEventDestroy(r->evicted);
    if (r->copied) cudaEventDestroy(r->copied);
    delete r;
    return st;
}

// ------------------------------------------------------------------ refill after a re-plan
//
// README item 1: the arena is planned again from the demand history (after a
// prompt's prefill, every few hundred tokens, between requests), and the
// experts it admits are then read into the slots they were given. The
// re-plan kernel (moe_arena_replan) writes the new tables and the list of
// slots to refill; this host call reads that list once the re-plan has run and
// copies each new owner's record from the host store (the stand-in for the
// drive) on the copy stream; the compute stream then waits for the copies.

extern "C" moe_status moe_arena_refill(const moe_arena* arena, const void* const* host_records, int n_flat,
                                       const int32_t* loads, const int32_t* n_loads, const int32_t* owner,
                                       void* stream, void* copy_stream, int32_t* n_copied) {
    MOE_RANGE("moe_arena_refill");
    if (!arena || !arena->base || !host_records || !loads || !n_loads || !owner || n_flat < 1 ||
        arena->n_slots < 1 || arena->slot_bytes <= 0)
        return MOE_EINVAL;
    if (n_copied) *n_copied = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    int32_t n = 0;
    if (cudaMemcpyAsync(&n, n_loads, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ECUDA;
    if (n < 0 || n > arena->n_slots) return MOE_EINVAL;
    if (n == 0) return MOE_OK;
    std::vector<int32_t> slots(n), own(arena->n_slots);
    if (cudaMemcpyAsync(slots.data(), loads, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(own.data(), owner, sizeof(int32_t) * arena->n_slots, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ECUDA;
    for (int i = 0; i < n; ++i) {                     // every new owner must have a record: else copy nothing
        const int sl = slots[i];
        if (sl < 0 || sl >= arena->n_slots) return MOE_EINVAL;
        const int f = own[sl];
        if (f < 0 || f >= n_flat || !host_records[f]) return MOE_EINVAL;
    }
    cudaEvent_t ready = nullptr, copied = nullptr;
    if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&copied, cudaEventDisableTiming) != cudaSuccess) {
        if (ready) cudaEventDestroy(ready);
        return MOE_ECUDA;
    }
    moe_status st = MOE_OK;
    uint8_t* base = static_cast<uint8_t*>(arena->base);
    if (cudaEventRecord(ready, s) != cudaSuccess || cudaStreamWaitEvent(cs, ready, 0) != cudaSuccess) st = MOE_ECUDA;
    for (int i = 0; i < n && st == MOE_OK; ++i)
        if (cudaMemcpyAsync(base + (size_t)slots[i] * arena->slot_bytes, host_records[own[slots[i]]],
                            (size_t)arena->slot_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
            st = MOE_ECUDA;
    if (st == MOE_OK && (cudaEventRecord(copied, cs) != cudaSuccess || cudaStreamWaitEvent(s, copied, 0) != cudaSuccess))
        st = MOE_ECUDA;
    cudaEventDestroy(ready);                          // released once the work they mark has run
    cudaEventDestroy(copied);
    if (st == MOE_OK && n_copied) *n_copied = n;
    return st;
}
