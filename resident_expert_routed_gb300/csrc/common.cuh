// Shared device helpers for the resident-expert routed MoE kernels (sm_103a).
//
// Thin inline-PTX wrappers for mbarriers, TMA, cp.async, and the tcgen05
// tensor-core / tensor-memory instructions, plus the launcher prototypes each
// kernel file exports to the C-ABI layer (abi.cu). Nothing here allocates.
#pragma once

#include <cuda.h>
#include <cuda_fp4.h>
#include <cuda_runtime.h>

#include <utility>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe_resident.h"

#define MOE_DEV __device__ __forceinline__

// Tracing: every entry point of the C ABI opens an NVTX range named after it
// for the duration of the host call (the enqueue, or the whole call for those
// that synchronise), so a timeline tool shows which library call issued which
// kernels. Without a tool attached NVTX calls return at once.
struct MoeRange {
    explicit MoeRange(const char* name) { nvtxRangePushA(name); }
    ~MoeRange() { nvtxRangePop(); }
    MoeRange(const MoeRange&) = delete;
    MoeRange& operator=(const MoeRange&) = delete;
};
#define MOE_RANGE(name) MoeRange moe_range_guard_(name)

// Default wall-clock bound on any spin-wait inside a kernel (ns); the host
// passes the bound in force (moe_set_wait_limit) to every pipelined kernel. A
// healthy wait ends in microseconds; the bound only exists so that a broken
// pipeline returns with MOE_DEV_TIMEOUT instead of hanging the GPU.
#define MOE_WAIT_LIMIT_NS 2000000000ull
// After a wait has run out, a kernel still waits for the bulk copies and
// tensor-core operations it has already issued (they complete on their own)
// before it frees its tensor memory and exits; those waits use this bound.
#define MOE_DRAIN_LIMIT_NS 200000000ull

// ------------------------------------------------------------------ basic

MOE_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

MOE_DEV uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

MOE_DEV float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// 2^p as a float for p in [-127, 127] (exact; 2^-127 is subnormal).
MOE_DEV float exp2_int(int p) {
    return (p >= -126) ? __uint_as_float((uint32_t)(p + 127) << 23) : __uint_as_float(0x00400000u);
}

// floor(log2(a)) for finite a > 0, from the bit pattern.
MOE_DEV int floor_log2_pos(float a) {
    uint32_t u = __float_as_uint(a);
    int e = (int)((u >> 23) & 0xFF);
    if (e != 0) return e - 127;
    uint32_t m = u & 0x7FFFFF;                  // subnormal: value m * 2^-149
    return (31 - __clz(m)) - 149;
}

// OCP MX v1.0 MXFP4: shared exponent of a block from its amax, clamped to
// [-127, 127]; an all-zero block takes -127 (scale byte 0).
MOE_DEV int mx_shared_exp(float amax) {
    if (!(amax > 0.0f)) return -127;
    int X = floor_log2_pos(amax) - 2;
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Two values (already divided by their block scale) to one byte of e2m1 codes,
// the first in the low nibble: round to nearest, ties to the even code,
// saturating at +-6 (CUDA's fp4 conversion; it agrees value for value with
// the OCP rule the oracle spells out, only the sign bit of a zero may differ).
MOE_DEV uint32_t e2m1x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest);
}

// Eight values to one 32-bit word of e2m1 codes (element 0 in the lowest nibble).
MOE_DEV uint32_t e2m1x8(const float* v, float inv_scale) {
    return e2m1x2(v[0] * inv_scale, v[1] * inv_scale) | (e2m1x2(v[2] * inv_scale, v[3] * inv_scale) << 8) |
           (e2m1x2(v[4] * inv_scale, v[5] * inv_scale) << 16) | (e2m1x2(v[6] * inv_scale, v[7] * inv_scale) << 24);
}

// SwiGLU product silu(g) * u with the fast exponential and division intrinsics.
MOE_DEV float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Byte of the scale of (operand row `pos`, K-block `kb`) in an activation
// operand laid out for the tensor cores: rows are grouped in tiles of `bn`
// (a slot's rows always start a tile), each tile's scales stored as 512-byte
// atoms of four K-blocks, row r of the tile at (r % 32) * 16 + (r / 32) * 4.
MOE_DEV size_t operand_scale_offset(int pos, int kb, int bn, int K) {
    const int tile = pos / bn, r = pos % bn;
    return ((size_t)tile * (K / 128) + (kb >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
}

// Inclusive prefix sum of one 64-bit value per thread across the whole block
// (blockDim.x a multiple of 32, at most 1024). `scratch` is shared memory of
// 32 values; *total receives the block's sum. Contains __syncthreads().
MOE_DEV unsigned long long block_inclusive_scan_u64(unsigned long long v, unsigned long long* scratch,
                                                    unsigned long long* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
    }
    __syncthreads();                       // scratch may still be read by a previous call
    if (lane == 31) scratch[wid] = v;
    __syncthreads();
    if (wid == 0) {
        unsigned long long s = lane < nw ? scratch[lane] : 0ull;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, s, off);
            if (lane >= off) s += o;
        }
        scratch[lane] = s;
    }
    __syncthreads();
    if (wid > 0) v += scratch[wid - 1];
    *total = scratch[nw - 1];
    return v;
}

MOE_DEV void record_error(uint32_t* err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------------ mbarrier

MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

MOE_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false (after
// raising the CTA's abort flag) when about `limit_ns` of wall-clock time pass
// or another role of the CTA has already aborted. The clock is read only
// every 256 failed tries (every 16 under a bound below 1 ms): a %globaltimer
// read on every wait costs pipeline time, and a healthy wait ends long before
// its first read.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
    const uint32_t every = limit_ns >= 1000000ull ? 255u : 15u;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & every) == every) {
            if (*abort_flag) return false;
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 >= limit_ns) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// The same wait for all 32 lanes of a warp; the outcome is made warp-uniform
// so that a time-out can never split a warp across different sync points.
MOE_DEV bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort_flag, limit_ns);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// Wait for an operation this thread issued itself (a bulk copy's bytes, a
// tcgen05.commit) after an abort: ignores the abort flag, bounded by
// MOE_DRAIN_LIMIT_NS.
MOE_DEV bool mbar_drain(uint64_t* bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 >= MOE_DRAIN_LIMIT_NS) return false;
        }
    }
}

// A producer that has issued `issued` stage fills (fill i into stage i % ns,
// each completing one phase of full[i % ns]) and stops early: wait until the
// bytes of the last fill of every stage have landed. Earlier fills of a stage
// have completed already (the producer waited for their stage to be consumed
// before refilling it).
MOE_DEV void drain_stage_fills(uint64_t* full, int ns, uint32_t issued) {
    for (int s = 0; s < ns; ++s) {
        if (issued <= (uint32_t)s) break;
        const uint32_t last = (uint32_t)s + (uint32_t)ns * ((issued - 1u - (uint32_t)s) / (uint32_t)ns);
        (void)mbar_drain(&full[s], (last / (uint32_t)ns) & 1u);
    }
}

MOE_DEV void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOE_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------ TMA and bulk copies

MOE_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 1-D bulk async copy global -> shared (16-byte aligned addresses, size a multiple of 16).
MOE_DEV void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// L2 policy that evicts the lines it covers first (createpolicy, the whole
// access): for data read once, so that it does not push out what later
// kernels reuse.
MOE_DEV uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_load with an L2 cache policy (l2_evict_first_policy for weights streamed once).
MOE_DEV void bulk_load_hint(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bulk prefetch of global bytes into L2 (16-byte aligned, a multiple of 16 bytes; no completion).
MOE_DEV void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes)
                 : "memory");
}
MOE_DEV void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05

MOE_DEV void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
MOE_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive (once) on an mbarrier when every tcgen05 op issued so far by this thread has completed.
MOE_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// After an abort: wait (bounded) until every tcgen05 operation this thread
// has issued has completed. `bar` is an mbarrier of count 1 used only for this.
MOE_DEV void tc_drain(uint64_t* bar) {
    tc_commit(bar);
    (void)mbar_drain(bar, 0);
}

// D[tmem] (+)= A[smem] * B[smem]^T, e2m1 x e2m1 with e8m0 block-32 scales from TMEM.
MOE_DEV void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                         uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Each lane of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
MOE_DEV void tc_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
MOE_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each lane of the warp writes 8 consecutive 32-bit columns of its own TMEM lane.
MOE_DEV void tc_st_x8(uint32_t taddr, uint4 lo, uint4 hi) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"r"(taddr), "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                 : "memory");
}
MOE_DEV void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand tile with 128-byte rows in
// the 128-byte swizzle layout written by TMA (8-row groups 1024 B apart).
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(16u >> 4) << 16;      // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;    // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;               // descriptor version for the sm_100 family
    d |= (uint64_t)2 << 61;               // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::mxf4 (e2m1 x e2m1, e8m0 scales, fp32
// accumulator), both operands K-major, M = 128, N = n; sfid selects the byte
// pair of the scale column used by this MMA (0 or 2).
__host__ __device__ constexpr uint32_t idesc_mxf4(int n, int sfid_a, int sfid_b) {
    return ((uint32_t)(sfid_b & 3) << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(128 >> 4) << 24) | ((uint32_t)(sfid_a & 3) << 29);
}

// ------------------------------------------------------------------ launchers (host side)

struct RouteLaunch {
    const uint16_t* x; const float* w; const float* bias; const int32_t* slot_of;
    int T, d, E, k, splits;
    int32_t* want_e; float* want_s; int32_t* sel_e; int32_t* sel_slot; float* sel_w;
    float* partial;
    void* wsplit;           // non-null: tensor-core router, W split into three bf16 parts here
    uint32_t* err;          // device error word (tensor-core router's bounded waits)
    uint64_t wait_ns;       // bound on each wait of the tensor-core router
    int rows;               // 1: one CTA per expert row (few tokens in device memory; splits = 1)
};
bool router_rows_eligible(int T, int d);
// A batch in page-locked host memory that the row-per-CTA router can take is copied once into the
// routing workspace, after the partial logits, and scored from there.
cudaError_t launch_stage_rows(const void* src, void* dst, size_t bytes, cudaStream_t s);
bool router_tc_eligible(int T, int E, int d);
int pointer_kind(const void* p);      // 0 device, 1 page-locked host, -1 pageable host
int router_tc_splits(int T, int E, int d);
size_t router_tc_split_bytes(int E, int d);
cudaError_t launch_router_tc(const uint16_t* x, const float* W, int T, int d, int E, int splits, void* wsplit,
                             float* partial, uint32_t* err, uint64_t wait_ns, cudaStream_t s);
cudaError_t launch_route(const RouteLaunch& a, cudaStream_t s);
int route_splits(int T, int E, int d);

cudaError_t launch_demand(const int32_t* want_e, const float* want_s, const int32_t* slot_of, int T, int k,
                          int layer, int E, unsigned long long* demand, float* miss_max, cudaStream_t s);
cudaError_t launch_demand_decay(unsigned long long* demand, long n, unsigned long long q, cudaStream_t s);
cudaError_t launch_hot_miss(float* miss_max, int n, float threshold, int cap, int32_t* out_flat, float* out_share,
                            int32_t* n_out, cudaStream_t s);

struct FfnLaunch {
    const uint16_t* x; const int32_t* sel_slot; const float* sel_w; const moe_arena* arena;
    int T, k, d, F, S, bn;
    float* out;
    // workspace: positions are slot-sorted and padded so that every slot starts a tile of bn rows
    int32_t* pos_of_pair;   // [T*k]
    int32_t* pair_of_pos;   // [pad_max]
    int32_t* seg;           // [S]  first position of each slot
    int32_t* tile_off;      // [S]  first work entry of each slot
    int4* work;             // [work_max] (slot, first position, rows)
    int32_t* n_work;
    uint8_t* xp;            // [pad_max, d/2]   gate/up activation operand (MXFP4 codes)
    uint8_t* xsp;           // [work_max * d/128 * 512] its scales, tile atoms
    uint8_t* hq;            // [pad_max, F/2]   down activation operand
    uint8_t* hsp;           // [work_max * F/128 * 512]
    float* Y;               // [T*k, d] one fp32 row per pick
    int32_t* cta_counts;    // [plan_ctas, S] per-CTA pick counts, then offsets (large batches)
    int plan_ctas;          // 0: one-CTA plan
    int work_max, pad_max;
    uint32_t* err;
    uint64_t wait_ns;       // bound on each wait of the GEMM pipelines
};
cudaError_t launch_ffn_plan(const FfnLaunch& a, cudaStream_t s);
cudaError_t launch_ffn_prefetch(const int32_t* sel_slot, int P, const moe_arena& ar, cudaStream_t s);
cudaError_t launch_ffn_gemms(const FfnLaunch& a, cudaStream_t s, int* n_launches);
cudaError_t launch_ffn_combine(const FfnLaunch& a, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t wait_ns, cudaStream_t s);

cudaError_t launch_replan(const unsigned long long* demand, int n, int n_main, int n_slots, int32_t* slot_of,
                          int32_t* owner, int32_t* loads, int32_t* n_loads, void* ws, cudaStream_t s,
                          uint32_t* err);
cudaError_t launch_ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat, cudaStream_t s,
                                uint32_t* err);

// Programmatic dependent launch. Every kernel of the library is launched with
// moe_launch (programmatic stream serialisation allowed) and starts with
// pdl_trigger() then, after any prologue that touches no input, pdl_wait()
// before reading anything: so the next kernel on the stream is launched and
// runs its own prologue while this one finishes, and every kernel still sees
// all the memory of everything launched before it (each grid completes only
// after its wait, so completion is transitive down the stream).
MOE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t moe_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The device error word of the current device (abi.cu); null if it cannot be found.
uint32_t* moe_err_word();

// The bound on every wait of the pipelined kernels now in force (moe_set_wait_limit; abi.cu).
uint64_t moe_wait_limit_ns();

// Kernel launch counter kept by abi.cu.
void moe_count_launches(int n);
int moe_sm_count();

// Kernel kinds for the optional per-launch event timing (abi.cu).
enum MoeKernelKind {
    MK_ROUTER_LOGITS = 0, MK_ROUTE_SELECT, MK_DEMAND, MK_HOT_MISS, MK_PLAN, MK_PACK, MK_GEMM_GATE_UP,
    MK_GEMM_DOWN, MK_COMBINE, MK_REPLAN, MK_RING, MK_COUNT
};
void moe_prof_begin(int kind, cudaStream_t s);
void moe_prof_end(int kind, cudaStream_t s);
