/*
 * moe_resident.h -- C ABI of one routed-MoE layer step over a partial,
 * demand-learned set of resident experts (hand-written CUDA for sm_103a).
 *
 * The method is the adaptive expert loading of the TideLM README, section
 * "How adaptive expert loading works":
 *   item 1  per (layer, expert) demand, learned from the scores of the
 *           router's picks; a single arena for all layers, planned again
 *           from that history;
 *   item 2  routing is restricted to resident experts: an absent expert's
 *           place goes to the best resident one not yet picked, and the
 *           absent expert's demand is counted anyway;
 *   item 3  misses with a large share of the routing weight (>= 0.2, at
 *           most 16 a step) are fetched by hot reads into extra ring slots.
 * The experts are stored in MXFP4 (README profile table): OCP MX v1.0 e2m1
 * elements with one e8m0 scale per 32 elements.
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers owned by the caller unless a comment says
 *     "host". The library never allocates, frees or synchronises on these
 *     calls; all work is enqueued on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and runs asynchronously.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns MOE_EINVAL (or MOE_ENOMEM for a short workspace,
 *     MOE_EUNSUPPORTED for a size past a documented limit) and launches
 *     nothing. A CUDA launch error returns MOE_ECUDA.
 *   - Data-dependent faults found on the device (a slot id past the arena, an
 *     e8m0 scale byte 0xFF, a bounded wait that ran out) are recorded in a
 *     per-device error word; device code never traps. moe_device_status()
 *     reads and clears it.
 *   - Layouts are row-major. bf16 hidden states are raw 16-bit patterns.
 *   - Ties: equal router scores order by the lower expert index.
 */
#ifndef MOE_RESIDENT_H
#define MOE_RESIDENT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,        /* bad argument (null pointer, size out of range) */
    MOE_ECUDA = 2,         /* a CUDA runtime call or launch failed */
    MOE_ENOMEM = 3,        /* workspace smaller than the matching *_workspace_bytes() */
    MOE_ETIMEOUT = 4,      /* device error word: a bounded wait in a kernel ran out */
    MOE_EDEVICE = 5,       /* device error word: bad slot id / NaN scale / bad table */
    MOE_EUNSUPPORTED = 6,  /* a size past a documented limit */
    MOE_EIO = 7            /* a file could not be read or written (demand history) */
} moe_status;

/* Bits of the device error word (moe_device_status). */
#define MOE_DEV_BAD_SLOT    0x1u   /* a slot id >= arena n_slots was routed */
#define MOE_DEV_NAN_SCALE   0x2u   /* an expert GEMM produced a non-finite value: e2m1 codes and the
                                      quantised activations are finite, so a weight scale byte 0xFF
                                      (e8m0 NaN) was read, or scales large enough to overflow fp32 */
#define MOE_DEV_TIMEOUT     0x4u   /* a pipeline wait gave up after its limit */
#define MOE_DEV_BAD_TABLE   0x8u   /* slot_of / owner tables inconsistent (re-plan, ring) */
#define MOE_DEV_RESIDENT    0x10u  /* ring install of an expert that is already resident */

/*
 * The shared slot arena (README item 1: a single arena serves every layer).
 * Passed by HOST pointer; `base` is a device pointer to n_slots records of
 * slot_bytes each. Slots [0, n_main) form the main arena and the rest the
 * hot-read ring (README item 3); the FFN treats them alike.
 * One slot record holds one expert in MXFP4 (e2m1 codes, two per byte with
 * the even element in the LOW nibble; one e8m0 scale byte per 32 along K).
 * Logically the expert is W_gu [2*ffn, d] (gate rows 0..ffn-1, then up rows
 * ffn..2ffn-1) and W_dn [d, ffn]. The record stores them in the order the
 * tensor cores consume them, so that every pipeline stage is one contiguous
 * copy:
 *   off_gu_codes   (2*ffn/128) * ceil(d/256) * 16384 bytes, tile-major code blocks
 *   off_gu_scales  2*ffn*d/32 bytes, tile-atom order
 *   off_dn_codes   (d/128) * ceil(ffn/256) * 16384 bytes, tile-major code blocks
 *   off_dn_scales  d*ffn/32 bytes, tile-atom order
 * Tiles: rows are grouped in tiles of 128 consecutive logical rows -- tile g
 * is rows 128g..128g+127 (for W_gu the gate tiles come first, then the up
 * tiles). Tile row r is row 128g + r.
 * Tile-major code blocks: for tile g and chunk c of 256 elements along K
 * (128 bytes; zero past the row end), a 16 KB block of 128 rows x 128 bytes
 * at byte (g * ceil(K/256) + c) * 16384; within it, the 16-byte piece q of
 * tile row r is stored at r * 128 + (q ^ (r % 8)) * 16 (the 128-byte swizzle).
 * Tile-atom scales: scale S[row, 4a + k] (K-block 4a + k) of tile row r is at
 * byte (g * (K/128) + a) * 512 + (r % 32) * 16 + (r / 32) * 4 + k.
 * Requirements: base and every offset 256-byte aligned, slot_bytes a multiple
 * of 256, d and ffn multiples of 128.
 */
typedef struct {
    void*   base;
    int64_t slot_bytes;
    int32_t n_slots;
    int32_t d;
    int32_t ffn;
    int32_t reserved;
    int64_t off_gu_codes;
    int64_t off_gu_scales;
    int64_t off_dn_codes;
    int64_t off_dn_scales;
} moe_arena;

/*
 * Router scoring and resident-only top-k with substitution.
 * README items 1-2: the router scores every token against all E experts; the
 * wanted picks are the top-k over all experts; the routed picks come from the
 * resident experts only, an absent wanted expert giving its place to the best
 * resident expert not yet picked.
 *   logit[t,e] = sum_i x[t,i] * W[e,i] + bias[e]   (fp32 accumulation)
 *   score[t,e] = softmax over e of logit[t,e]
 *   want  = top-k of score over all E                (score desc, index asc)
 *   sel   = top-k of score over {e : slot_of[e] >= 0}
 * hidden_bf16 [T,d] bf16; w_router [E,d] fp32; bias [E] fp32 or NULL;
 * slot_of [E] int32 (slot id, -1 = not resident) for this layer.
 * Outputs [T,k]: want_e int32, want_s fp32 (its score); sel_e int32,
 * sel_slot int32, sel_w fp32 (the pick's own score, not renormalised);
 * when fewer than k experts are resident the tail is (-1, -1, 0).
 * workspace: >= moe_workspace_bytes(T, k, d, ffn, E, S) bytes (any ffn, S).
 * hidden_bf16, w_router and workspace must be 16-byte aligned (MOE_EINVAL).
 * hidden_bf16 may be device memory or page-locked host memory (cudaHostAlloc,
 * cudaHostRegister); pageable host memory is refused (MOE_EINVAL). A batch of
 * at most 4 tokens (d <= 8192) in host memory is first copied (once, by a
 * kernel) into the workspace and scored from there, with the same kernels and
 * results as from device memory; a larger one is read in place (there the
 * K-sliced router's reads of it cost less than a separate copy).
 * Up to 4 tokens in device memory (or staged) with d <= 8192, each expert's
 * W_r row is read and summed whole by one CTA; up to 64 tokens, K is split
 * into slices summed in a fixed order by the selection. Batches of more than
 * 64 tokens with d % 64 == 0 and E % 16 == 0 in device memory are scored on
 * the tensor cores: W_r is split exactly into three bf16 parts in the
 * workspace and the products are accumulated in fp32, so the logits match the
 * CUDA-core path up to fp32 rounding order. A batch of more than 64 tokens in
 * host memory is scored on the CUDA cores.
 * Limits: 1 <= k <= 32, k <= E <= 1024, d % 32 == 0, T >= 1.
 */
moe_status moe_route_resident(const void* hidden_bf16, const float* w_router, const float* bias,
                              const int32_t* slot_of, int T, int d, int E, int k,
                              int32_t* want_e, float* want_s,
                              int32_t* sel_e, int32_t* sel_slot, float* sel_w,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Optional renormalisation of the combine weights (the pages say only
 * "score-weighted"; moe_route_resident keeps each pick's own softmax score so
 * that a substitute is not inflated). For callers that want weights summing
 * to one over a token's picks: sel_w[t,j] /= sum of sel_w[t,*] over the picks
 * with sel_slot >= 0 (fp32, summed in pick order); padding picks and tokens
 * without a valid pick get 0. sel_slot int32 [T,k], sel_w fp32 [T,k] in place.
 * Limits: T >= 1, 1 <= k <= 32.
 */
moe_status moe_renormalise_weights(const int32_t* sel_slot, float* sel_w, int T, int k, void* stream);

/*
 * moe_route_resident without a caller workspace (nothing in the TideLM README
 * corresponds to it:
 * this exists for callers of this library that cannot allocate device memory
 * when they route -- e.g. a serving loop whose memory budget was fixed at
 * start-up, or a plug-in whose host framework owns every allocation -- since
 * cudaMalloc can also synchronise the device). Same arguments and limits as
 * moe_route_resident, minus the workspace; it allocates nothing. It always
 * scores on the CUDA cores, so for batches that moe_route_resident scores on
 * the tensor cores (above 64 tokens) the logits can differ in the last fp32
 * bits, and a pick at a near-tie can differ. A batch in page-locked host
 * memory is read in place by the K-sliced router at every size (there is no
 * workspace to copy it into): each K slice reads its rows across the
 * chip-to-chip link, and for up to 4 tokens, which moe_route_resident copies
 * to the device and sums row by row, the fp32 summation order differs, with
 * the same last-bit and near-tie caveat.
 * The split-K partial logits live in one fixed device array of 4 MiB
 * (2^20 fp32) inside the library, held by every GPU that loads the library
 * until the process exits; a call whose partials would not fit
 * (splits * T * E > 2^20, e.g. T above 128 for E = 256) returns
 * MOE_EUNSUPPORTED. Every call on a device shares that array: calls whose
 * work overlaps on the GPU (different streams without ordering) race and
 * corrupt each other's results. Each call writes every element it reads, so
 * nothing needs clearing between calls. The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.
 */
moe_status moe_route_resident_noalloc(const void* hidden_bf16, const float* w_router, const float* bias,
                                      const int32_t* slot_of, int T, int d, int E, int k,
                                      int32_t* want_e, float* want_s,
                                      int32_t* sel_e, int32_t* sel_slot, float* sel_w, void* stream);

/*
 * Demand accumulation (README item 1: each wanted pick adds its score to the
 * demand of its (layer, expert), resident or not; item 2: substituted picks
 * add too) and the miss share (item 3: how much of its token's routing weight
 * a missing expert would have taken).
 *   demand[layer, e]   += round(s * 2^40)   for each wanted pick (t, j)
 *   miss_max[layer, e]  = max(miss_max, s)  for each wanted pick with slot_of[e] < 0
 * want_e, want_s [T,k] as written by moe_route_resident; slot_of [E] of this
 * layer; demand uint64 [L,E] in units of 2^-40 (order-free, deterministic);
 * miss_max fp32 [L,E] (>= 0). Limits: 0 <= layer < L, E <= 1024.
 */
moe_status moe_demand_accumulate(const int32_t* want_e, const float* want_s, const int32_t* slot_of,
                                 int T, int k, int layer, int L, int E,
                                 uint64_t* demand, float* miss_max, void* stream);

/*
 * Heavy-miss list for one step (README item 3: the misses with the largest
 * share, a threshold of 0.2 of a token's routing weight and a cap of 16 per
 * step; the misses of all lanes of a step go into one list). Candidates are (layer, expert) with miss_max >= threshold, ordered
 * by miss_max descending, then flat index layer*E + e ascending; the first
 * `cap` are written. Afterwards miss_max is reset to zero for the next step.
 * out_flat int32 [cap], out_share fp32 [cap], n_out: device int32 (count).
 * Limits: 0 <= cap <= 1024, L*E <= 2^24.
 */
moe_status moe_hot_miss_select(float* miss_max, int L, int E, float threshold, int cap,
                               int32_t* out_flat, float* out_share, int32_t* n_out, void* stream);

/*
 * Grouped SwiGLU expert FFN over the MXFP4 arena with weighted combine
 * (README items 1-2 and the MXFP4 experts of the profile table).
 * For every pick (t, j) with sel_slot[t,j] >= 0, with W the expert in that slot:
 *   xq   = MXFP4(x[t])      (OCP MX: exponent floor(log2 amax) - 2, RNE, saturate)
 *   g, u = Wg xq, Wu xq     (tcgen05 block-scaled MXFP4 MMA, fp32 accumulation)
 *   h    = silu(g) * u,  hq = MXFP4(h)  (blocks of 32 along ffn)
 *   y    = Wd hq
 *   out[t] = sum_j sel_w[t,j] * y(t, j)   (j = 0..k-1 in order: deterministic)
 * hidden_bf16 [T,d]; sel_slot, sel_w [T,k] (as from moe_route_resident);
 * arena: HOST pointer, see moe_arena; out fp32 [T,d] (fully overwritten;
 * a token with no pick gets zeros). hidden_bf16 and out may be device memory
 * or page-locked host memory, which the kernels read and write directly (the
 * batch is read once, the output written once); pageable host memory is
 * refused (MOE_EINVAL).
 * workspace: >= moe_workspace_bytes(T, k, d, ffn, E, arena->n_slots).
 * Limits: 1 <= k <= 32, T*k <= 2^20, n_slots <= 16384, d and ffn multiples of
 * 128, d <= 16384, ffn <= 16384.
 */
moe_status moe_expert_ffn_mxfp4(const void* hidden_bf16, const int32_t* sel_slot, const float* sel_w,
                                const moe_arena* arena, int T, int k, float* out,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Optional, for latency: prefetches into L2 the gate/up weights that
 * moe_expert_ffn_mxfp4 streams first for these picks. Its plan orders the
 * work by slot and its gate/up GEMM runs one CTA per SM, so the first round
 * reads one 128-feature tile of gate and up weights (codes and scales) per SM
 * from the lowest-numbered slots the picks use; this call prefetches exactly
 * those blocks, one SM each. Issue it on a second stream right after the
 * routing, so that HBM serves it while the FFN's plan and pack run (they read
 * little). It reads sel_slot and the arena and writes nothing: results never
 * depend on it. sel_slot int32 [T,k]; arena and limits as for
 * moe_expert_ffn_mxfp4; batches of more than 8,192 picks return MOE_OK
 * without a launch (there the first round is a small part of the GEMM, and
 * every CTA of this call would scan all the picks beside the plan and pack).
 * Measured on GB300 it pays only for a single token through one layer with a
 * cold L2 (about 1 us of 50); from two tokens on, and through consecutive
 * layers, its reads compete with the GEMM's own and the step is slower, so
 * the Python layer step issues it only when asked.
 */
moe_status moe_expert_ffn_prefetch(const int32_t* sel_slot, const moe_arena* arena, int T, int k, void* stream);

/*
 * Re-plan of the one shared arena from the demand history (README item 1: the
 * arena's contents follow the history and are planned again; layers with more
 * demand end up with more of the shared slots).
 *   1. rank every flat id f = layer*E + e by (demand desc, currently in a main
 *      slot first, f asc); the first n_main form the new main set;
 *   2. survivors keep their slots; main-set members that drop out lose theirs;
 *   3. newcomers, in rank order, take the free main slots in ascending order;
 *      a newcomer that sat in a ring slot (>= n_main) leaves it;
 *   4. loads[] lists the main slots given to newcomers (to be refilled by the
 *      caller with the new owners' weights), *n_loads their count.
 * demand uint64 [L,E] (< 2^62); slot_of int32 [L*E] in/out; owner int32
 * [n_slots] in/out (flat id or -1); loads int32 [n_main]; n_loads device int32.
 * workspace: >= moe_replan_workspace_bytes(L, E).
 * Limits: 1 <= n_main <= n_slots, L*E <= 2^22.
 */
moe_status moe_arena_replan(const uint64_t* demand, int L, int E, int n_main, int n_slots,
                            int32_t* slot_of, int32_t* owner, int32_t* loads, int32_t* n_loads,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * Refill after a re-plan (README item 1: once the arena has been planned
 * again, the experts it admitted are read into the slots they were given).
 * Call after moe_arena_replan on `stream` (a HOST call: it synchronises
 * `stream` to read the re-plan's n_loads, loads[] and owner[]). For each slot
 * s in loads[0 .. n_loads) it copies host_records[owner[s]] (arena->slot_bytes
 * bytes, the arena record layout) into slot s with cudaMemcpyAsync on
 * `copy_stream`, after everything enqueued on `stream` so far; `stream` then
 * waits for the copies, so no work enqueued on it afterwards reads a slot
 * before its bytes are in. host_records: host array [n_flat] of host pointers
 * (page-locked, so that the copies run asynchronously), NULL where the store
 * has no copy. If a new owner has no record nothing is copied and MOE_EINVAL
 * is returned (the tables already name it: supply the record, or re-plan).
 * No FFN may be reading the arena on another stream meanwhile.
 * loads int32 [n_main], n_loads device int32, owner int32 [arena->n_slots]
 * (device, after the re-plan); *n_copied (host, may be NULL) = slots copied.
 */
moe_status moe_arena_refill(const moe_arena* arena, const void* const* host_records, int n_flat,
                            const int32_t* loads, const int32_t* n_loads, const int32_t* owner,
                            void* stream, void* copy_stream, int32_t* n_copied);

/*
 * Ring install (README item 3, DeepSeek: a step's largest misses are fetched
 * into extra ring slots and become routable one step later, until newer
 * fetches wrap around the ring). Makes flat id `flat_id` resident in `ring_slot`; the slot's
 * previous owner becomes non-resident. The slot's bytes are written by the
 * caller. An expert that is already resident is left alone and sets
 * MOE_DEV_RESIDENT in the device error word.
 * slot_of int32 [n_flat], owner int32 [n_slots].
 */
moe_status moe_ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat_id,
                            int n_flat, int n_slots, void* stream);

/*
 * Asynchronous hot-read ring (README item 3, DeepSeek: the fetches of a
 * step's largest misses overlap the following step, and the fetched experts
 * can be routed to from the step after it until the ring wraps; "Settings
 * worth knowing": ring slots come in addition to the main budget). A HOST object; one thread drives it, once per step boundary.
 *
 * create: ring slots are arena slots [ring_first, ring_first + n_ring).
 *   host_records: host array [n_flat] of HOST pointers, one expert record
 *   (arena->slot_bytes bytes, the arena record layout) per flat id, or NULL
 *   when the store has no copy (the stand-in for the drive the pages read
 *   from). The pointer array is copied; the records must stay valid and
 *   unchanged until destroy, and should be pinned (cudaHostAlloc) so that the
 *   copies overlap compute. cap: the heavy-miss list's capacity (1..32). The
 *   arena struct is copied.
 * step: call after step s has been enqueued on `stream`, including the
 *   moe_hot_miss_select that wrote heavy_flat [cap] / n_heavy (device).
 *   1. experts copied by the previous call are installed (the stream waits
 *      for their copies): routable from step s + 1;
 *   2. the host waits for step s to finish and reads its heavy-miss list;
 *   3. each listed flat id with a record and not already in the ring takes
 *      the next ring slot in FIFO order: the slot's owner leaves the routing
 *      tables on `stream`, then the record is copied in on `copy_stream`; it
 *      is installed by the next call (routable from step s + 2).
 *   *n_fetched (host, may be NULL) = experts whose copies were issued.
 *   slot_of int32 [n_flat], owner int32 [n_slots] (device). An install of an
 *   expert that became resident in the meantime is refused and sets
 *   MOE_DEV_RESIDENT.
 * destroy: waits for copies in flight, frees the object.
 */
typedef struct moe_hot_ring moe_hot_ring;
moe_status moe_hot_ring_create(const moe_arena* arena, int ring_first, int n_ring, int n_flat,
                               const void* const* host_records, int cap, moe_hot_ring** ring);
moe_status moe_hot_ring_step(moe_hot_ring* ring, const int32_t* heavy_flat, const int32_t* n_heavy,
                             int32_t* slot_of, int32_t* owner, void* stream, void* copy_stream,
                             int32_t* n_fetched);
moe_status moe_hot_ring_destroy(moe_hot_ring* ring);

/*
 * Synchronous hot read of one layer (README item 3, GLM-5.3: before a layer's
 * MoE runs, its largest miss (share >= 0.2; at most 16 such reads a step,
 * spread over the layers) is loaded, used with its exact weights, and stays
 * resident in the slot of the least-demanded expert). Call after
 * moe_demand_accumulate of `layer` and before its FFN; then route the layer
 * again with the updated slot_of, so that the tokens that wanted the expert
 * get it (the wanted picks and the demand are unchanged).
 *   read   = the non-resident expert of the layer with the largest miss share
 *            this step (miss_max >= threshold, ties to the lower index) that
 *            the store holds;
 *   victim = the resident expert of the layer with the lowest demand (ties to
 *            the lower index);
 *   if *budget > 0 and both exist: *budget -= 1; victim leaves the tables,
 *   read takes its slot, and the record store[read] is copied into the slot.
 * store: device array [L*E] of uint64 addresses of expert records (slot_bytes
 *   each, the arena record layout, 16-byte aligned) that the device can read,
 *   e.g. pinned host memory; 0 = not in the store. The addresses are trusted.
 * demand uint64 [L,E]; miss_max fp32 [L,E] (this step's shares, before
 *   moe_hot_miss_select resets them); slot_of int32 [L*E]; owner int32
 *   [n_slots]; budget: device int32, reads left this step (the caller sets
 *   it, e.g. to 16, when a step starts); swap: device int32 [3] out =
 *   (flat read, slot, flat victim), or (-1, -1, -1) when nothing was read.
 */
moe_status moe_hot_read_sync(const uint64_t* store, const uint64_t* demand, const float* miss_max,
                             int32_t* slot_of, int32_t* owner, const moe_arena* arena, int layer, int L, int E,
                             float threshold, int32_t* budget, int32_t* swap, void* stream);

/* Workspace sizes (bytes) for the calls above. */
size_t moe_workspace_bytes(int T, int k, int d, int ffn, int E, int n_slots);
size_t moe_replan_workspace_bytes(int L, int E);

/*
 * Forgetting in the demand history (README "Settings worth knowing": an
 * adaptation setting controls how quickly the resident set tracks a change in
 * traffic; the pages give no formula). Reading: the caller applies an exponential
 * decay between re-plans; every entry is scaled exactly in fixed point:
 *   q = round(factor * 2^32)  (factor in [0, 1]; ties to even)
 *   demand[i] = floor(demand[i] * q / 2^32)        (128-bit product)
 * so factor 1 leaves the table unchanged and 0.5 halves it (floor).
 * demand: device uint64 [n] in units of 2^-40. Bad factor or n < 0: MOE_EINVAL.
 */
moe_status moe_demand_decay(uint64_t* demand, int64_t n, float factor, void* stream);

/*
 * Persistence of the demand history (README item 1: the history "persists
 * across restarts"; "Settings worth knowing": the engine keeps it in a state
 * database). File format, little-endian:
 *   bytes 0-7   magic "MOEDEMD1"
 *   bytes 8-15  int32 L, int32 E
 *   bytes 16-23 int32 fraction bits (40), int32 0
 *   then L*E uint64 demand values, row-major [L, E], in units of 2^-40.
 * demand: device uint64 [L, E]. Both calls order their copy on `stream` and
 * synchronise it (host I/O). save writes `path` whole (a temporary file
 * renamed over it). load checks the header against L and E (MOE_EINVAL on a
 * mismatch or a bad magic) before touching the device; I/O errors give
 * MOE_EIO.
 */
moe_status moe_demand_save(const uint64_t* demand, int L, int E, const char* path, void* stream);
moe_status moe_demand_load(uint64_t* demand, int L, int E, const char* path, void* stream);

/*
 * Reads and clears the current device's error word (synchronises `stream`).
 * Returns MOE_OK, MOE_ETIMEOUT (timeout bit set) or MOE_EDEVICE (any other
 * bit); *bits (host, may be NULL) receives the raw word.
 */
moe_status moe_device_status(void* stream, uint32_t* bits);

/*
 * Bound on every wait inside the library's pipelined kernels (the expert
 * FFN's GEMMs and the tensor-core router), in nanoseconds of wall-clock time
 * counted from the wait's first failed try; ns = 0 restores the default, 2 s.
 * A healthy wait ends in microseconds; the bound exists so that a broken
 * pipeline cannot hang the GPU (failure detection in the spirit of the
 * colibri cluster page, "timeouts": every wait of that cluster is bounded and
 * ends in an error rather than a stall). When a wait
 * runs out, its CTA stops issuing work, waits (at most 0.2 s more) for the
 * bulk copies and tensor-core operations it has already issued, frees its
 * tensor memory and exits; MOE_DEV_TIMEOUT is set in the device error word
 * (moe_device_status then returns MOE_ETIMEOUT) and that call's outputs are
 * not valid. The call's later kernels still run on its unfinished
 * intermediates, so other bits (MOE_DEV_NAN_SCALE) may be set beside
 * MOE_DEV_TIMEOUT. Later calls are unaffected. Process-wide; read when a call
 * launches its kernels, so a CUDA graph keeps the value it was captured with.
 */
moe_status moe_set_wait_limit(uint64_t ns);
uint64_t   moe_get_wait_limit(void);

/*
 * Failure-detection check of the bounded waits: launches one CTA set up like
 * the pipelined kernels (tensor memory allocated, an MMA thread, warps waiting
 * on an mbarrier) whose wait can never be satisfied -- nothing arrives on its
 * barrier. It gives up after the bound in force (moe_set_wait_limit), drains,
 * frees its tensor memory and sets MOE_DEV_TIMEOUT, as a stalled pipeline
 * would; moe_device_status then returns MOE_ETIMEOUT. Takes that long to end:
 * set a short bound first (e.g. 1 ms) and restore it afterwards.
 */
moe_status moe_wait_selftest(void* stream);

/* Static English text for a status code. */
const char* moe_status_str(moe_status s);

/* Number of kernels this library has launched in this process (host counter). */
uint64_t moe_kernel_launches(void);

/*
 * Per-kernel device timing (tracing). When enabled, every kernel launch is
 * bracketed by two CUDA events on its stream; moe_profile_read() waits for
 * the recorded events and returns, per kernel kind, the launch count and the
 * summed device time since the last reset. Off by default; not for use while
 * a stream is being captured into a CUDA graph. The events are created by the
 * library on first use and reused.
 * kind: 0 .. moe_profile_kernel_count()-1; *name is a static string.
 */
moe_status moe_profile_enable(int on);
int        moe_profile_kernel_count(void);
moe_status moe_profile_read(int kind, const char** name, int64_t* launches, double* total_ms);
void       moe_profile_reset(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_RESIDENT_H */
