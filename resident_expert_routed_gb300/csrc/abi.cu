// C ABI of the resident-expert routed MoE layer step (include/moe_resident.h).
//
// Host-side argument checks, workspace carving, the per-device error word and
// the launch sequence of each entry point. Every step of the computation runs
// in the kernels of route.cu, demand.cu, ffn_plan.cu, ffn_gemm.cu and
// replan.cu; nothing here computes on the host.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

size_t replan_workspace(int n);

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{MOE_WAIT_LIMIT_NS};

// One error word per device; its device address is looked up once per device.
__device__ uint32_t g_err_word;

constexpr int MAX_DEV = 64;
uint32_t* g_err_ptr[MAX_DEV] = {};
int g_sm_count[MAX_DEV] = {};
std::mutex g_mu;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev < MAX_DEV ? dev : -1;
}

uint32_t* err_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    if (g_err_ptr[dev]) return g_err_ptr[dev];
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<uint32_t*>(p);
    }
    return g_err_ptr[dev];
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int bn_for(int T) { return T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128; }

// Workspace of the FFN, carved in this order (every piece 256-byte aligned).
// Positions are slot-sorted with every slot's segment padded to a multiple of
// the tile height bn, so at most work_max tiles and pad_max = work_max * bn rows.
struct FfnCarve {
    size_t pos_of_pair, pair_of_pos, seg, tile_off, work, n_work, xp, xsp, hq, hsp, Y, cta_counts, total;
    int work_max, pad_max, bn, plan_ctas;
};

// Batches of at least this many picks plan with several CTAs (2048 picks each, at most 64).
constexpr size_t kPlanMultiPicks = 8192;
constexpr long kPrefetchMaxPicks = 8192;        // moe_expert_ffn_prefetch scans the picks in every CTA

FfnCarve ffn_carve(int T, int k, int d, int F, int S) {
    FfnCarve c{};
    c.bn = bn_for(T);
    const size_t P = (size_t)T * k;
    const size_t U = P < (size_t)S ? P : (size_t)S;
    c.work_max = (int)(U + (P + c.bn - 1) / c.bn);
    c.pad_max = c.work_max * c.bn;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    c.pos_of_pair = take(P * 4);
    c.pair_of_pos = take((size_t)c.pad_max * 4);
    c.seg = take((size_t)S * 4);
    c.tile_off = take((size_t)S * 4);
    c.work = take((size_t)c.work_max * 16);
    c.n_work = take(4);
    c.xp = take((size_t)c.pad_max * d / 2);
    c.xsp = take((size_t)c.work_max * (d / 128) * 512);
    c.hq = take((size_t)c.pad_max * F / 2);
    c.hsp = take((size_t)c.work_max * (F / 128) * 512);
    c.Y = take(P * d * 4);
    c.plan_ctas = P >= kPlanMultiPicks ? (int)std::min<size_t>(64, (P + 2047) / 2048) : 0;
    c.cta_counts = take((size_t)c.plan_ctas * S * 4);
    c.total = o;
    return c;
}

// Routing workspace: the split-K partial logits of the CUDA-core router (then,
// for batches the row-per-CTA router takes, room for such a batch in host
// memory, copied there once and scored from there), or, for batches the
// tensor-core router can take, the larger of that and its three bf16 parts of
// W_r followed by its partials (a larger batch in host memory is scored by the
// K-sliced CUDA-core router in place).
size_t route_bytes(int T, int E, int d) {
    size_t simt = align_up((size_t)route_splits(T, E, d) * T * E * 4, 256);
    if (router_rows_eligible(T, d)) simt += align_up((size_t)T * d * 2, 256);   // a host batch, staged here
    if (!router_tc_eligible(T, E, d)) return simt;
    return std::max(simt, router_tc_split_bytes(E, d) + align_up((size_t)router_tc_splits(T, E, d) * T * E * 4, 256));
}

}  // namespace

// Where a caller's buffer lives: 0 device memory (or a pointer the runtime does
// not know, e.g. without a device), 1 page-locked host memory that the kernels
// read and write directly (over the chip-to-chip link on this platform), -1
// pageable host memory, which they cannot touch.
int pointer_kind(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (at.type == cudaMemoryTypeHost) return 1;
    if (at.type == cudaMemoryTypeUnregistered) return -1;
    return 0;
}

namespace {

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ECUDA; }

// ------------------------------------------------------------------ optional per-launch event timing
const char* const kKernelNames[MK_COUNT] = {"router_logits_partial", "route_select", "demand_accumulate",
                                            "hot_miss_select", "ffn_plan", "ffn_pack", "ffn_gemm_gate_up",
                                            "ffn_gemm_down", "ffn_combine", "arena_replan", "ring_install"};
struct ProfRec {
    int kind;
    cudaEvent_t a, b;
};
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_open;        // recorded, not yet read
std::vector<cudaEvent_t> g_prof_pool;    // free events
cudaEvent_t g_prof_pending = nullptr;    // begin event of the launch in flight (per library; one host thread)
int64_t g_prof_n[MK_COUNT] = {};
double g_prof_ms[MK_COUNT] = {};

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

}  // namespace

// The device error word of the current device, for other translation units.
uint32_t* moe_err_word() { return err_word(); }

void moe_prof_begin(int kind, cudaStream_t s) {
    (void)kind;
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_pending = prof_event();
    cudaEventRecord(g_prof_pending, s);
}

void moe_prof_end(int kind, cudaStream_t s) {
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_pending) return;
    cudaEvent_t b = prof_event();
    cudaEventRecord(b, s);
    g_prof_open.push_back({kind, g_prof_pending, b});
    g_prof_pending = nullptr;
}

static void prof_drain() {   // caller holds g_prof_mu
    for (const ProfRec& r : g_prof_open) {
        float ms = 0.f;
        cudaEventSynchronize(r.b);
        cudaEventElapsedTime(&ms, r.a, r.b);
        g_prof_n[r.kind] += 1;
        g_prof_ms[r.kind] += ms;
        g_prof_pool.push_back(r.a);
        g_prof_pool.push_back(r.b);
    }
    g_prof_open.clear();
}

void moe_count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

uint64_t moe_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int moe_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 148;
    if (!g_sm_count[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 148;
    }
    return g_sm_count[dev];
}

extern "C" {

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_EINVAL: return "invalid argument";
        case MOE_ECUDA: return "CUDA error";
        case MOE_ENOMEM: return "workspace too small";
        case MOE_ETIMEOUT: return "device wait timed out";
        case MOE_EDEVICE: return "device reported bad data (slot id, scale byte or table)";
        case MOE_EUNSUPPORTED: return "size beyond a documented limit";
        case MOE_EIO: return "file could not be read or written";
    }
    return "unknown status";
}

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status moe_set_wait_limit(uint64_t ns) {
    g_wait_limit_ns.store(ns == 0 ? MOE_WAIT_LIMIT_NS : ns, std::memory_order_relaxed);
    return MOE_OK;
}

uint64_t moe_get_wait_limit(void) { return moe_wait_limit_ns(); }

moe_status moe_wait_selftest(void* stream) {
    MOE_RANGE("moe_wait_selftest");
    uint32_t* err = err_word();
    if (!err) return MOE_ECUDA;
    return cuda_status(launch_wait_selftest(err, moe_wait_limit_ns(), static_cast<cudaStream_t>(stream)));
}

moe_status moe_profile_enable(int on) {
    g_prof_on.store(on != 0);
    return MOE_OK;
}

int moe_profile_kernel_count(void) { return MK_COUNT; }

moe_status moe_profile_read(int kind, const char** name, int64_t* launches, double* total_ms) {
    if (kind < 0 || kind >= MK_COUNT) return MOE_EINVAL;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof_drain();
    if (name) *name = kKernelNames[kind];
    if (launches) *launches = g_prof_n[kind];
    if (total_ms) *total_ms = g_prof_ms[kind];
    return MOE_OK;
}

void moe_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof_drain();
    for (int i = 0; i < MK_COUNT; ++i) { g_prof_n[i] = 0; g_prof_ms[i] = 0.0; }
}

size_t moe_workspace_bytes(int T, int k, int d, int ffn, int E, int n_slots) {
    if (T < 1 || k < 1 || d < 1 || E < 1) return 0;
    size_t r = route_bytes(T, E, d);
    if (ffn > 0 && n_slots > 0) {
        const size_t f = ffn_carve(T, k, d, ffn, n_slots).total;
        if (f > r) r = f;
    }
    return r;
}

size_t moe_replan_workspace_bytes(int L, int E) {
    if (L < 1 || E < 1) return 0;
    return replan_workspace(L * E);
}

moe_status moe_route_resident(const void* hidden_bf16, const float* w_router, const float* bias,
                              const int32_t* slot_of, int T, int d, int E, int k, int32_t* want_e, float* want_s,
                              int32_t* sel_e, int32_t* sel_slot, float* sel_w, void* workspace, size_t ws_bytes,
                              void* stream) {
    MOE_RANGE("moe_route_resident");
    if (!hidden_bf16 || !w_router || !slot_of || !want_e || !want_s || !sel_e || !sel_slot || !sel_w || !workspace)
        return MOE_EINVAL;
    if (T < 1 || d < 32 || d % 32 || E < 1 || k < 1 || k > 32 || k > E) return MOE_EINVAL;
    if (((uintptr_t)hidden_bf16 | (uintptr_t)w_router | (uintptr_t)workspace) & 15) return MOE_EINVAL;
    if (E > 1024) return MOE_EUNSUPPORTED;
    if ((size_t)T * E > ((size_t)1 << 31)) return MOE_EUNSUPPORTED;
    if (ws_bytes < route_bytes(T, E, d)) return MOE_ENOMEM;
    int hk = pointer_kind(hidden_bf16);
    if (hk < 0) return MOE_EINVAL;
    RouteLaunch a{};
    a.x = static_cast<const uint16_t*>(hidden_bf16);
    if (hk == 1 && router_rows_eligible(T, d)) {      // a few host tokens: one copy across the link, then HBM
        void* staged = static_cast<uint8_t*>(workspace) + align_up((size_t)route_splits(T, E, d) * T * E * 4, 256);
        const cudaError_t se = launch_stage_rows(hidden_bf16, staged, (size_t)T * d * 2, static_cast<cudaStream_t>(stream));
        if (se != cudaSuccess) return cuda_status(se);
        a.x = static_cast<const uint16_t*>(staged);
        hk = 0;
    }
    a.w = w_router;
    a.bias = bias;
    a.slot_of = slot_of;
    a.T = T; a.d = d; a.E = E; a.k = k;
    a.splits = route_splits(T, E, d);
    a.want_e = want_e; a.want_s = want_s; a.sel_e = sel_e; a.sel_slot = sel_slot; a.sel_w = sel_w;
    a.partial = static_cast<float*>(workspace);
    a.err = err_word();
    if (!a.err) return MOE_ECUDA;
    a.wait_ns = moe_wait_limit_ns();
    if (hk == 0 && router_rows_eligible(T, d)) {      // few tokens: whole rows, no K slices
        a.rows = 1;
        a.splits = 1;
    }
    if (hk == 0 && router_tc_eligible(T, E, d)) {     // the tensor maps need device memory
        a.wsplit = workspace;
        a.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + router_tc_split_bytes(E, d));
        a.splits = router_tc_splits(T, E, d);
    }
    return cuda_status(launch_route(a, static_cast<cudaStream_t>(stream)));
}

moe_status moe_demand_accumulate(const int32_t* want_e, const float* want_s, const int32_t* slot_of, int T, int k,
                                 int layer, int L, int E, uint64_t* demand, float* miss_max, void* stream) {
    MOE_RANGE("moe_demand_accumulate");
    if (!want_e || !want_s || !slot_of || !demand || !miss_max) return MOE_EINVAL;
    if (T < 1 || k < 1 || k > 32 || E < 1 || L < 1 || layer < 0 || layer >= L) return MOE_EINVAL;
    if (E > 1024) return MOE_EUNSUPPORTED;
    return cuda_status(launch_demand(want_e, want_s, slot_of, T, k, layer, E,
                                     reinterpret_cast<unsigned long long*>(demand), miss_max,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_hot_miss_select(float* miss_max, int L, int E, float threshold, int cap, int32_t* out_flat,
                               float* out_share, int32_t* n_out, void* stream) {
    MOE_RANGE("moe_hot_miss_select");
    if (!miss_max || !n_out || L < 1 || E < 1 || cap < 0) return MOE_EINVAL;
    if (cap > 0 && (!out_flat || !out_share)) return MOE_EINVAL;
    if (cap > 1024 || (long)L * E > (1L << 24)) return MOE_EUNSUPPORTED;
    return cuda_status(launch_hot_miss(miss_max, L * E, threshold, cap, out_flat, out_share, n_out,
                                       static_cast<cudaStream_t>(stream)));
}

// The arena record and batch limits that the expert FFN (and its prefetch) rely on.
static moe_status arena_status(const moe_arena* arena, int T, int k) {
    if (!arena->base) return MOE_EINVAL;
    const int d = arena->d, F = arena->ffn, S = arena->n_slots;
    if (T < 1 || k < 1 || k > 32 || d < 128 || F < 128 || d % 128 || F % 128 || S < 1) return MOE_EINVAL;
    if (arena->slot_bytes <= 0 || arena->slot_bytes % 256) return MOE_EINVAL;
    const uintptr_t b = reinterpret_cast<uintptr_t>(arena->base);
    if (b % 256 || arena->off_gu_codes % 256 || arena->off_gu_scales % 256 || arena->off_dn_codes % 256 ||
        arena->off_dn_scales % 256)
        return MOE_EINVAL;
    const int64_t guc = (int64_t)(F / 64) * ((d + 255) / 256) * 16384, gus = (int64_t)2 * F * d / 32;
    const int64_t dnc = (int64_t)(d / 128) * ((F + 255) / 256) * 16384, dns = (int64_t)d * F / 32;
    auto inside = [&](int64_t off, int64_t len) { return off >= 0 && off + len <= arena->slot_bytes; };
    if (!inside(arena->off_gu_codes, guc) || !inside(arena->off_gu_scales, gus) || !inside(arena->off_dn_codes, dnc) ||
        !inside(arena->off_dn_scales, dns))
        return MOE_EINVAL;
    if (S > 16384 || d > 16384 || F > 16384 || (long)T * k > (1L << 20)) return MOE_EUNSUPPORTED;
    return MOE_OK;
}

moe_status moe_expert_ffn_prefetch(const int32_t* sel_slot, const moe_arena* arena, int T, int k, void* stream) {
    MOE_RANGE("moe_expert_ffn_prefetch");
    if (!sel_slot || !arena) return MOE_EINVAL;
    const moe_status as = arena_status(arena, T, k);
    if (as != MOE_OK) return as;
    if ((long)T * k > kPrefetchMaxPicks) return MOE_OK;        // large batches: nothing to hide it behind
    return cuda_status(launch_ffn_prefetch(sel_slot, T * k, *arena, static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn_mxfp4(const void* hidden_bf16, const int32_t* sel_slot, const float* sel_w,
                                const moe_arena* arena, int T, int k, float* out, void* workspace, size_t ws_bytes,
                                void* stream) {
    MOE_RANGE("moe_expert_ffn_mxfp4");
    if (!hidden_bf16 || !sel_slot || !sel_w || !arena || !out || !workspace) return MOE_EINVAL;
    const moe_status as = arena_status(arena, T, k);
    if (as != MOE_OK) return as;
    const int d = arena->d, F = arena->ffn, S = arena->n_slots;
    const FfnCarve c = ffn_carve(T, k, d, F, S);
    if (ws_bytes < c.total) return MOE_ENOMEM;
    if (pointer_kind(hidden_bf16) < 0 || pointer_kind(out) < 0) return MOE_EINVAL;
    uint32_t* err = err_word();
    if (!err) return MOE_ECUDA;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    FfnLaunch a{};
    a.x = static_cast<const uint16_t*>(hidden_bf16);
    a.sel_slot = sel_slot;
    a.sel_w = sel_w;
    a.arena = arena;
    a.T = T; a.k = k; a.d = d; a.F = F; a.S = S;
    a.bn = c.bn;
    a.out = out;
    a.pos_of_pair = reinterpret_cast<int32_t*>(w + c.pos_of_pair);
    a.pair_of_pos = reinterpret_cast<int32_t*>(w + c.pair_of_pos);
    a.seg = reinterpret_cast<int32_t*>(w + c.seg);
    a.tile_off = reinterpret_cast<int32_t*>(w + c.tile_off);
    a.work = reinterpret_cast<int4*>(w + c.work);
    a.n_work = reinterpret_cast<int32_t*>(w + c.n_work);
    a.xp = w + c.xp;
    a.xsp = w + c.xsp;
    a.hq = w + c.hq;
    a.hsp = w + c.hsp;
    a.Y = reinterpret_cast<float*>(w + c.Y);
    a.cta_counts = reinterpret_cast<int32_t*>(w + c.cta_counts);
    a.plan_ctas = c.plan_ctas;
    a.work_max = c.work_max;
    a.pad_max = c.pad_max;
    a.err = err;
    a.wait_ns = moe_wait_limit_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_ffn_plan(a, s);
    if (e == cudaSuccess) e = launch_ffn_gemms(a, s, nullptr);
    if (e == cudaSuccess) e = launch_ffn_combine(a, s);
    return cuda_status(e);
}

moe_status moe_arena_replan(const uint64_t* demand, int L, int E, int n_main, int n_slots, int32_t* slot_of,
                            int32_t* owner, int32_t* loads, int32_t* n_loads, void* workspace, size_t ws_bytes,
                            void* stream) {
    MOE_RANGE("moe_arena_replan");
    if (!demand || !slot_of || !owner || !loads || !n_loads || !workspace) return MOE_EINVAL;
    if (L < 1 || E < 1 || n_main < 1 || n_slots < n_main) return MOE_EINVAL;
    if ((long)L * E > (1L << 22)) return MOE_EUNSUPPORTED;
    if (n_main > L * E) return MOE_EINVAL;
    if (ws_bytes < replan_workspace(L * E)) return MOE_ENOMEM;
    uint32_t* err = err_word();
    if (!err) return MOE_ECUDA;
    return cuda_status(launch_replan(reinterpret_cast<const unsigned long long*>(demand), L * E, n_main, n_slots,
                                     slot_of, owner, loads, n_loads, workspace, static_cast<cudaStream_t>(stream),
                                     err));
}

moe_status moe_ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat_id, int n_flat, int n_slots,
                            void* stream) {
    MOE_RANGE("moe_ring_install");
    if (!slot_of || !owner || n_flat < 1 || n_slots < 1) return MOE_EINVAL;
    if (ring_slot < 0 || ring_slot >= n_slots || flat_id < 0 || flat_id >= n_flat) return MOE_EINVAL;
    uint32_t* err = err_word();
    if (!err) return MOE_ECUDA;
    return cuda_status(launch_ring_install(slot_of, owner, ring_slot, flat_id, static_cast<cudaStream_t>(stream), err));
}

moe_status moe_device_status(void* stream, uint32_t* bits) {
    uint32_t* err = err_word();
    if (!err) return MOE_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ECUDA;
    if (h) {
        const uint32_t zero = 0;
        if (cudaMemcpyAsync(err, &zero, 4, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ECUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ECUDA;
    }
    if (bits) *bits = h;
    if (!h) return MOE_OK;
    return (h & MOE_DEV_TIMEOUT) ? MOE_ETIMEOUT : MOE_EDEVICE;
}

}  // extern "C"

// ------------------------------------------------------------------ demand history: decay and persistence

moe_status moe_demand_decay(uint64_t* demand, int64_t n, float factor, void* stream) {
    MOE_RANGE("moe_demand_decay");
    if (n < 0 || !(factor >= 0.0f && factor <= 1.0f) || (n > 0 && !demand)) return MOE_EINVAL;
    if (n == 0) return MOE_OK;
    const unsigned long long q = (unsigned long long)std::nearbyint((double)factor * 4294967296.0);
    return cuda_status(launch_demand_decay(reinterpret_cast<unsigned long long*>(demand), (long)n, q,
                                           static_cast<cudaStream_t>(stream)));
}

namespace {

constexpr char kDemandMagic[8] = {'M', 'O', 'E', 'D', 'E', 'M', 'D', '1'};

struct DemandHeader {
    char magic[8];
    int32_t L, E, frac_bits, zero;
};
static_assert(sizeof(DemandHeader) == 24, "demand file header");

}  // namespace

moe_status moe_demand_save(const uint64_t* demand, int L, int E, const char* path, void* stream) {
    MOE_RANGE("moe_demand_save");
    if (!demand || !path || L < 1 || E < 1) return MOE_EINVAL;
    const size_t n = (size_t)L * E;
    std::vector<uint64_t> host(n);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host.data(), demand, n * sizeof(uint64_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ECUDA;
    DemandHeader h{};
    std::memcpy(h.magic, kDemandMagic, 8);
    h.L = L;
    h.E = E;
    h.frac_bits = 40;
    const std::string tmp = std::string(path) + ".tmp";
    FILE* f = std::fopen(tmp.c_str(), "wb");
    if (!f) return MOE_EIO;
    const bool ok = std::fwrite(&h, sizeof h, 1, f) == 1 && std::fwrite(host.data(), sizeof(uint64_t), n, f) == n;
    if (std::fclose(f) != 0 || !ok || std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return MOE_EIO;
    }
    return MOE_OK;
}

moe_status moe_demand_load(uint64_t* demand, int L, int E, const char* path, void* stream) {
    MOE_RANGE("moe_demand_load");
    if (!demand || !path || L < 1 || E < 1) return MOE_EINVAL;
    FILE* f = std::fopen(path, "rb");
    if (!f) return MOE_EIO;
    DemandHeader h{};
    if (std::fread(&h, sizeof h, 1, f) != 1) { std::fclose(f); return MOE_EIO; }
    if (std::memcmp(h.magic, kDemandMagic, 8) != 0 || h.L != L || h.E != E || h.frac_bits != 40) {
        std::fclose(f);
        return MOE_EINVAL;
    }
    const size_t n = (size_t)L * E;
    std::vector<uint64_t> host(n);
    const bool ok = std::fread(host.data(), sizeof(uint64_t), n, f) == n;
    std::fclose(f);
    if (!ok) return MOE_EIO;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(demand, host.data(), n * sizeof(uint64_t), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}
