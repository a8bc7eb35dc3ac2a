// Oracle for the resident-expert routed MoE layer step.
//
// TEST INFRASTRUCTURE ONLY. Plain, slow, single-threaded C++ in float64. It
// shares no code, header, table or constant with the CUDA library; only the
// tests, the bench's CPU-baseline leg and the package smoke check call it.
//
// What it computes follows the TideLM README ("How adaptive expert loading
// works", items 1-3): the router scores every token against all experts and
// routes to resident experts only (an absent wanted expert gives its place to
// the best resident expert not yet picked), adds each wanted pick's score to
// the demand of its (layer, expert), lists the misses with a large share of
// the routing weight (>= 0.2, at most 16 a step), and runs the expert FFN over the resident weights
// ("native MXFP4" experts, profile table) with a score-weighted combine.
// The number formats follow the OCP Microscaling (MX) Formats v1.0 spec:
// e2m1 elements, e8m0 shared scales, blocks of 32.
//
// Where the pages leave a step open, the reading taken is stated beside the
// function that takes it. Every function is pinned by tests/test_oracle_pins.py
// against hand-worked cases, closed forms, invariants or brute force.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

extern "C" {

// ---------------------------------------------------------------- number formats

// e2m1 element (OCP MX v1.0, FP4 E2M1): bit 3 sign, bits 2..1 exponent
// (bias 1), bit 0 mantissa. Exponent 0 is subnormal: value 0.5 * m.
double or_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

// e8m0 shared scale (OCP MX v1.0): 2^(byte - 127); 0xFF is NaN.
double or_e8m0_value(int byte) {
    if ((byte & 0xFF) == 0xFF) return std::nan("");
    return std::ldexp(1.0, (byte & 0xFF) - 127);
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// Round |a| (already divided by the block scale) to the e2m1 grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}: nearest, ties to the even code, saturating
// at 6. Returns the 3-bit magnitude code.
static int e2m1_round_mag(double a) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    if (a >= 6.0) return 7;
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = std::fabs(a - grid[c]), db = std::fabs(a - grid[best]);
        if (dc < db || (dc == db && (c % 2 == 0))) best = c;
    }
    return best;
}

// MXFP4 quantisation of one vector of length n (n % 32 == 0), OCP MX v1.0
// section on conversion: per 32-block, X = floor(log2(amax)) - 2 (2 = emax of
// e2m1), clamped to [-127, 127]; scale byte X + 127; element code =
// round-to-nearest-even of v / 2^X on the e2m1 grid, saturating at +-6, sign
// bit set for v < 0. An all-zero block gets scale byte 0 and zero codes.
// codes: n/2 bytes, element 2i in the low nibble of byte i.
void or_quantise_mxfp4(const double* v, int n, uint8_t* codes, uint8_t* scales) {
    for (int b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[b * 32 + i]));
        int X;
        if (amax == 0.0) {
            X = -127;
        } else {
            int ex;
            std::frexp(amax, &ex);      // amax = f * 2^ex, f in [0.5, 1)
            X = (ex - 1) - 2;           // floor(log2(amax)) - 2
            X = std::min(127, std::max(-127, X));
        }
        scales[b] = (uint8_t)(X + 127);
        for (int i = 0; i < 32; ++i) {
            double x = v[b * 32 + i];
            int mag = (amax == 0.0) ? 0 : e2m1_round_mag(std::fabs(x) / std::ldexp(1.0, X));
            int code = mag | (x < 0.0 ? 8 : 0);
            int idx = b * 32 + i;
            if (idx % 2 == 0) codes[idx / 2] = (uint8_t)code;
            else codes[idx / 2] = (uint8_t)(codes[idx / 2] | (code << 4));
        }
    }
}

// Dequantise an MXFP4 vector of length n (codes n/2 bytes, scales n/32 bytes).
void or_dequantise_mxfp4(const uint8_t* codes, const uint8_t* scales, int n, double* out) {
    double value[16];
    for (int c = 0; c < 16; ++c) value[c] = or_e2m1_value(c);
    for (int b = 0; b < n / 32; ++b) {
        double sc = or_e8m0_value(scales[b]);
        for (int i = b * 32; i < b * 32 + 32; ++i) {
            int c = (i % 2 == 0) ? (codes[i / 2] & 0xF) : (codes[i / 2] >> 4);
            out[i] = value[c] * sc;
        }
    }
}

// ---------------------------------------------------------------- router

// Router logits and scores for T tokens (README item 1: "the router's own
// demand"; reading: logits + bias, then softmax over all E experts).
//   logit[t,e] = sum_i x[t,i] * W[e,i] + b[e]      (bf16 x, fp32 W, f64 sum)
//   score[t,e] = exp(logit - max) / sum_e' exp(logit' - max)
void or_router(const uint16_t* x_bf16, const float* W, const float* bias,
               int T, int d, int E, double* logits, double* scores) {
    for (int t = 0; t < T; ++t) {
        double* lt = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += bf16_to_double(x_bf16[(size_t)t * d + i]) * (double)W[(size_t)e * d + i];
            lt[e] = acc + (bias ? (double)bias[e] : 0.0);
        }
        double mx = lt[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, lt[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += std::exp(lt[e] - mx);
        for (int e = 0; e < E; ++e) scores[(size_t)t * E + e] = std::exp(lt[e] - mx) / z;
    }
}

// Wanted top-k over all experts and resident top-k with substitution
// (README item 2: routing is restricted to resident experts, and an absent
// wanted expert gives its place to the best resident expert not yet picked).
// Order: score descending, ties to the lower expert index. The selected list
// is the top-k of the scores restricted to {e : slot_of[e] >= 0}; when fewer
// than k experts are resident it is padded with expert -1, slot -1, weight 0.
// The combine weight of a pick is its own softmax score (no renormalisation).
void or_topk(const double* scores, const int32_t* slot_of, int T, int E, int k,
             int32_t* want_e, double* want_s,
             int32_t* sel_e, int32_t* sel_slot, double* sel_w) {
    std::vector<int> idx(E);
    for (int t = 0; t < T; ++t) {
        const double* s = scores + (size_t)t * E;
        std::iota(idx.begin(), idx.end(), 0);
        std::sort(idx.begin(), idx.end(), [&](int a, int b) {
            if (s[a] != s[b]) return s[a] > s[b];
            return a < b;
        });
        for (int j = 0; j < k; ++j) {
            want_e[(size_t)t * k + j] = idx[j];
            want_s[(size_t)t * k + j] = s[idx[j]];
        }
        int j = 0;
        for (int r = 0; r < E && j < k; ++r) {
            int e = idx[r];
            if (slot_of[e] >= 0) {
                sel_e[(size_t)t * k + j] = e;
                sel_slot[(size_t)t * k + j] = slot_of[e];
                sel_w[(size_t)t * k + j] = s[e];
                ++j;
            }
        }
        for (; j < k; ++j) {
            sel_e[(size_t)t * k + j] = -1;
            sel_slot[(size_t)t * k + j] = -1;
            sel_w[(size_t)t * k + j] = 0.0;
        }
    }
}

// Demand recording (README item 1: each wanted pick adds its routing score to
// the demand of its (layer, expert), resident or not; item 2: substituted
// picks add too). D[layer*E + e] += s for each wanted pick. The miss share
// M[layer*E + e] = max(M, s) over the wanted picks of non-resident experts
// (item 3: how much of its token's routing weight a missing expert would have
// taken; reading: the share is the softmax score).
void or_demand(const int32_t* want_e, const double* want_s, const int32_t* slot_of,
               int T, int k, int layer, int E, double* D, double* M) {
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = want_e[(size_t)t * k + j];
            double s = want_s[(size_t)t * k + j];
            size_t f = (size_t)layer * E + e;
            D[f] += s;
            if (slot_of[e] < 0) M[f] = std::max(M[f], s);
        }
}

// Forgetting in the demand history (README "Settings worth knowing": an
// adaptation setting controls how quickly the resident set tracks a change in
// traffic; no formula is given). Reading: exponential decay applied between re-plans to
// the stored table, which keeps demand as an integer count of 2^-40 units.
// The factor is rounded to a multiple of 2^-32 (ties to even) and each entry
// becomes the floor of its exact product with it.
void or_demand_decay_fixed(uint64_t* D, int64_t n, double factor) {
    const unsigned __int128 q = (unsigned __int128)std::nearbyint(factor * 4294967296.0);
    for (int64_t i = 0; i < n; ++i) D[i] = (uint64_t)(((unsigned __int128)D[i] * q) >> 32);
}

// Optional renormalisation of the combine weights over a token's k picks
// (reading R2 keeps the raw scores; this is the alternative): w_j / sum_j w_j
// over the valid picks (sel_slot >= 0), in pick order; a token without a
// valid pick keeps zeros.
void or_renormalise(const int32_t* sel_slot, double* sel_w, int T, int k) {
    for (int t = 0; t < T; ++t) {
        double z = 0.0;
        for (int j = 0; j < k; ++j)
            if (sel_slot[(size_t)t * k + j] >= 0) z += sel_w[(size_t)t * k + j];
        for (int j = 0; j < k; ++j) {
            double& w = sel_w[(size_t)t * k + j];
            w = (sel_slot[(size_t)t * k + j] >= 0 && z > 0.0) ? w / z : 0.0;
        }
    }
}

// Synchronous hot read of one layer (README item 3, GLM-5.3: before a layer's
// MoE runs, its largest miss is loaded, used with its exact weights, and stays
// resident in the slot of the least-demanded expert). Reading: the read expert
// is the non-resident expert of the layer with the largest miss share this
// step (>= threshold, ties to the lower index) that the store holds; the
// coldest expert is the resident one with the lowest demand (ties to the
// lower index); nothing happens when the step's read budget is spent or
// either is missing. out = (read expert, victim expert), or (-1, -1).
void or_hot_read_choose(const double* M, const double* D, const int32_t* slot_of, const uint8_t* in_store,
                        int E, double threshold, int budget, int32_t* out) {
    out[0] = out[1] = -1;
    if (budget <= 0) return;
    int best = -1, cold = -1;
    for (int e = 0; e < E; ++e) {
        if (slot_of[e] < 0 && in_store[e] && M[e] >= threshold && (best < 0 || M[e] > M[best])) best = e;
        if (slot_of[e] >= 0 && (cold < 0 || D[e] < D[cold])) cold = e;
    }
    if (best < 0 || cold < 0) return;
    out[0] = best;
    out[1] = cold;
}

// Heavy misses (README item 3: the misses with the largest share; the share
// threshold is 0.2 of a token's routing weight and the cap 16 per step). Candidates are the (layer, expert) with
// M >= threshold, ordered by M descending then flat index ascending; the first
// `cap` are returned. M is then reset to zero for the next step.
void or_hot_miss_select(double* M, int L, int E, double threshold, int cap,
                        int32_t* out_flat, double* out_share, int32_t* n_out) {
    std::vector<int> cand;
    for (int f = 0; f < L * E; ++f)
        if (M[f] >= threshold) cand.push_back(f);
    std::sort(cand.begin(), cand.end(), [&](int a, int b) {
        if (M[a] != M[b]) return M[a] > M[b];
        return a < b;
    });
    int n = std::min<int>(cap, (int)cand.size());
    for (int i = 0; i < n; ++i) {
        out_flat[i] = cand[i];
        out_share[i] = M[cand[i]];
    }
    *n_out = n;
    for (int f = 0; f < L * E; ++f) M[f] = 0.0;
}

// ---------------------------------------------------------------- expert FFN

// An expert's weights dequantised once to f64: gate/up [2F, d] and down [d, F].
struct DeqExpert {
    std::vector<double> gu, dn;
};

static void dequantise_expert(const uint8_t* gu_codes, const uint8_t* gu_scales, const uint8_t* dn_codes,
                              const uint8_t* dn_scales, int d, int F, DeqExpert* e) {
    e->gu.resize((size_t)2 * F * d);
    e->dn.resize((size_t)d * F);
    for (int r = 0; r < 2 * F; ++r)
        or_dequantise_mxfp4(gu_codes + (size_t)r * (d / 2), gu_scales + (size_t)r * (d / 32), d,
                            e->gu.data() + (size_t)r * d);
    for (int o = 0; o < d; ++o)
        or_dequantise_mxfp4(dn_codes + (size_t)o * (F / 2), dn_scales + (size_t)o * (F / 32), F,
                            e->dn.data() + (size_t)o * F);
}

// One (token, expert) pair of the SwiGLU expert FFN over MXFP4 weights.
//   xq      = MXFP4(x)                           (activation quantised, OCP rule)
//   g_f     = sum_i Wg[f,i] * xq_i,  u_f = sum_i Wu[f,i] * xq_i   (f64, exact products)
//   h_f     = silu(g_f) * u_f,  silu(z) = z / (1 + e^-z)
//   hq      = MXFP4(h)  (blocks of 32 along the ffn dimension)
//   y_o     = sum_f Wd[o,f] * hq_f
// Weights: gate/up rows 0..F-1 gate, F..2F-1 up; down [d, F].
static void expert_pair_deq(const uint16_t* x_bf16, int d, int F, const DeqExpert& e, double* y,
                            uint8_t* xq_codes, uint8_t* xq_scales, double* h_out,
                            uint8_t* hq_codes, uint8_t* hq_scales) {
    std::vector<double> x(d), xq(d), h(F), hq(F);
    std::vector<uint8_t> xc(d / 2), xs(d / 32), hc(F / 2), hs(F / 32);
    for (int i = 0; i < d; ++i) x[i] = bf16_to_double(x_bf16[i]);
    or_quantise_mxfp4(x.data(), d, xc.data(), xs.data());
    or_dequantise_mxfp4(xc.data(), xs.data(), d, xq.data());
    for (int f = 0; f < F; ++f) {
        const double* wg = e.gu.data() + (size_t)f * d;
        const double* wu = e.gu.data() + (size_t)(F + f) * d;
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) g += wg[i] * xq[i];
        for (int i = 0; i < d; ++i) u += wu[i] * xq[i];
        h[f] = g / (1.0 + std::exp(-g)) * u;
    }
    or_quantise_mxfp4(h.data(), F, hc.data(), hs.data());
    or_dequantise_mxfp4(hc.data(), hs.data(), F, hq.data());
    for (int o = 0; o < d; ++o) {
        const double* wd = e.dn.data() + (size_t)o * F;
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += wd[f] * hq[f];
        y[o] = acc;
    }
    if (xq_codes) std::memcpy(xq_codes, xc.data(), d / 2);
    if (xq_scales) std::memcpy(xq_scales, xs.data(), d / 32);
    if (h_out) std::memcpy(h_out, h.data(), sizeof(double) * F);
    if (hq_codes) std::memcpy(hq_codes, hc.data(), F / 2);
    if (hq_scales) std::memcpy(hq_scales, hs.data(), F / 32);
}

void or_expert_pair(const uint16_t* x_bf16, int d, int F,
                    const uint8_t* gu_codes, const uint8_t* gu_scales,
                    const uint8_t* dn_codes, const uint8_t* dn_scales,
                    double* y,
                    uint8_t* xq_codes, uint8_t* xq_scales, double* h_out,
                    uint8_t* hq_codes, uint8_t* hq_scales) {
    DeqExpert e;
    dequantise_expert(gu_codes, gu_scales, dn_codes, dn_scales, d, F, &e);
    expert_pair_deq(x_bf16, d, F, e, y, xq_codes, xq_scales, h_out, hq_codes, hq_scales);
}

// The routed FFN with score-weighted combine for T tokens (README items 1-2;
// the combine adds a token's picks in its rank order j = 0..k-1).
// sel_u[t,j] indexes the expert arrays (n_u experts, stacked), -1 = no pick.
//   out[t] = sum_j sel_w[t,j] * y(t, sel_u[t,j])
// Each expert is dequantised once; every pick's y is kept, then combined.
void or_ffn(const uint16_t* x_bf16, const int32_t* sel_u, const double* sel_w,
            int T, int k, int d, int F, int n_u,
            const uint8_t* gu_codes, const uint8_t* gu_scales,
            const uint8_t* dn_codes, const uint8_t* dn_scales,
            double* out) {
    size_t guc = (size_t)2 * F * (d / 2), gus = (size_t)2 * F * (d / 32);
    size_t dnc = (size_t)d * (F / 2), dns = (size_t)d * (F / 32);
    std::vector<double> y((size_t)T * k * d, 0.0);
    DeqExpert e;
    for (int u = 0; u < n_u; ++u) {
        bool used = false;
        for (size_t p = 0; p < (size_t)T * k; ++p) used = used || sel_u[p] == u;
        if (!used) continue;
        dequantise_expert(gu_codes + u * guc, gu_scales + u * gus, dn_codes + u * dnc, dn_scales + u * dns,
                          d, F, &e);
        for (size_t p = 0; p < (size_t)T * k; ++p)
            if (sel_u[p] == u)
                expert_pair_deq(x_bf16 + (p / k) * d, d, F, e, y.data() + p * d,
                                nullptr, nullptr, nullptr, nullptr, nullptr);
    }
    for (int t = 0; t < T; ++t) {
        double* o = out + (size_t)t * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int j = 0; j < k; ++j) {
            size_t p = (size_t)t * k + j;
            if (sel_u[p] < 0) continue;
            double w = sel_w[p];
            for (int i = 0; i < d; ++i) o[i] += w * y[p * d + i];
        }
    }
}

// ---------------------------------------------------------------- arena re-plan

// Re-plan of the one shared arena (README item 1: a single arena serves every
// layer, so layers with more demand hold more of its slots; its contents are
// planned again from the demand history). Slots [0, n_main) are the main arena, slots
// [n_main, n_slots) the hot-read ring.
//   1. Rank every (layer, expert) flat id f by (D desc, currently in a main
//      slot first, f asc); the first n_main form the new main set.
//   2. Survivors (old and new main set) keep their slots. Main-set members that
//      fall out lose their slot (slot_of = -1, owner = -1).
//   3. Newcomers, in rank order, take the free main slots in ascending slot
//      order. A newcomer that sat in a ring slot leaves it (owner = -1).
//   4. loads[] lists the main slots given to newcomers, in that order.
// slot_of: [L*E] in/out, owner: [n_slots] in/out.
void or_replan(const double* D, int L, int E, int n_main, int n_slots,
               int32_t* slot_of, int32_t* owner, int32_t* loads, int32_t* n_loads) {
    int n = L * E;
    std::vector<int> rank(n);
    std::iota(rank.begin(), rank.end(), 0);
    auto in_main = [&](int f) { return slot_of[f] >= 0 && slot_of[f] < n_main; };
    std::vector<char> was_main(n);
    for (int f = 0; f < n; ++f) was_main[f] = in_main(f) ? 1 : 0;
    std::sort(rank.begin(), rank.end(), [&](int a, int b) {
        if (D[a] != D[b]) return D[a] > D[b];
        if (was_main[a] != was_main[b]) return was_main[a] > was_main[b];
        return a < b;
    });
    int m = std::min(n_main, n);
    std::vector<char> now_main(n, 0);
    for (int r = 0; r < m; ++r) now_main[rank[r]] = 1;
    for (int f = 0; f < n; ++f)
        if (was_main[f] && !now_main[f]) {
            owner[slot_of[f]] = -1;
            slot_of[f] = -1;
        }
    std::vector<int> free_slots;
    for (int s = 0; s < n_main; ++s)
        if (owner[s] < 0) free_slots.push_back(s);
    int nl = 0;
    for (int r = 0; r < m; ++r) {
        int f = rank[r];
        if (was_main[f]) continue;
        if (slot_of[f] >= n_main) owner[slot_of[f]] = -1;     // leaves its ring slot
        int s = free_slots[nl];
        owner[s] = f;
        slot_of[f] = s;
        loads[nl++] = s;
    }
    *n_loads = nl;
}

// Install expert `flat` in ring slot `ring_slot` (README item 3, DeepSeek: a
// step's largest misses are fetched into extra ring slots and can be routed to
// one step later, until newer fetches wrap around the ring). The slot's previous owner
// becomes non-resident. An expert that is already resident is left alone and
// the call returns 1; otherwise 0.
int or_ring_install(int32_t* slot_of, int32_t* owner, int ring_slot, int flat) {
    if (slot_of[flat] >= 0) return 1;
    int old = owner[ring_slot];
    if (old >= 0) slot_of[old] = -1;
    owner[ring_slot] = flat;
    slot_of[flat] = ring_slot;
    return 0;
}

}  // extern "C"
