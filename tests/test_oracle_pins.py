"""Pins for the oracle: hand-worked cases, closed forms, invariants and brute force.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a swapped index, a transposed operand,
a wrong tie rule) fails at least one of them.
"""
import heapq
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))


# ------------------------------------------------------------------ number formats (OCP MX v1.0)

def test_e2m1_table_exhaustive():
    vals = GOLDEN["e2m1_table"]["values"]
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == vals[code]
        assert math.copysign(1.0, v) == math.copysign(1.0, vals[code])


def test_e8m0_all_bytes():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(128) == 2.0
    assert oracle.e8m0_value(124) == 0.125
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)


def _table_dequant(codes, scales, n):
    """Independent dequantiser: nibble split + the hand-typed table + per-32 scale."""
    table = np.array(GOLDEN["e2m1_table"]["values"], dtype=np.float64)
    codes = np.asarray(codes, np.uint8)
    nib = np.empty(n, np.int64)
    nib[0::2] = codes & 0xF
    nib[1::2] = codes >> 4
    sc = np.ldexp(1.0, np.asarray(scales, np.int64) - 127)
    return table[nib] * np.repeat(sc, 32)


def test_quantise_midpoints_and_signs():
    g = GOLDEN["quantise_block"]
    codes, scales = oracle.quantise_mxfp4(np.array(g["input"]))
    assert scales[0] == g["expected_scale_byte"]
    got = _table_dequant(codes, scales, 32)
    exp = np.array(g["expected_value"])
    assert np.array_equal(got, exp)
    assert np.array_equal(np.signbit(got), np.signbit(exp))     # -0.1 -> -0, -0.25 -> -0


def test_quantise_saturates():
    g = GOLDEN["quantise_saturate"]
    v = np.zeros(32)
    v[:4] = g["input_head"]
    codes, scales = oracle.quantise_mxfp4(v)
    assert scales[0] == g["expected_scale_byte"]
    assert np.array_equal(_table_dequant(codes, scales, 32)[:4], g["expected_head"])


@pytest.mark.parametrize("p", range(-8, 9))
def test_quantise_power_of_two_amax(p):
    # amax = 2^p -> shared exponent p - 2; amax itself maps to code 4 (value 4)
    v = np.zeros(64)
    v[5] = 2.0 ** p
    v[40] = -(2.0 ** p) * 0.75     # second block: amax 0.75*2^p -> exponent p-3, value 6*2^(p-3) = 0.75*2^p
    codes, scales = oracle.quantise_mxfp4(v)
    assert scales[0] == 127 + p - 2
    assert scales[1] == 127 + p - 3
    deq = _table_dequant(codes, scales, 64)
    assert deq[5] == 2.0 ** p
    assert deq[40] == -(2.0 ** p) * 0.75
    assert np.count_nonzero(deq) == 2


def test_quantise_zero_block_and_roundtrip_on_grid():
    codes, scales = oracle.quantise_mxfp4(np.zeros(32))
    assert scales[0] == 0 and not codes.any()
    # values already on the grid with a shared exponent are reproduced exactly
    rng = np.random.default_rng(1)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    v = rng.choice(grid, 256) * rng.choice([-1, 1], 256) * 2.0 ** 3
    v[::32] = 6 * 2.0 ** 3       # amax 48 in every block -> exponent 3
    codes, scales = oracle.quantise_mxfp4(v)
    assert np.array_equal(_table_dequant(codes, scales, 256), v)
    assert np.array_equal(oracle.dequantise_mxfp4(codes, scales, 256), v)


def test_quantise_is_nearest_on_grid_random():
    # brute force: every element is the nearest grid point of v / 2^X (clamped at 6)
    rng = np.random.default_rng(2)
    v = rng.standard_normal(32 * 50) * np.repeat(2.0 ** rng.integers(-20, 20, 50), 32)
    codes, scales = oracle.quantise_mxfp4(v)
    deq = _table_dequant(codes, scales, v.size)
    for b in range(50):
        blk = v[b * 32:(b + 1) * 32]
        X = math.floor(math.log2(np.abs(blk).max())) - 2
        assert scales[b] == 127 + X
        grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6]) * 2.0 ** X
        for i in range(32):
            a = abs(blk[i])
            best = np.abs(grid - min(a, 6 * 2.0 ** X)).min()
            assert abs(abs(deq[b * 32 + i]) - min(a, 6 * 2.0 ** X)) == best


# ------------------------------------------------------------------ router and top-k (README items 1-2)

def test_router_hand_worked():
    g = GOLDEN["router_tiny"]
    d, E, k = g["d"], g["E"], g["k"]
    x = np.zeros((1, d), np.float32)
    x[0, g["x_index"]] = g["x_value"]
    W = np.zeros((E, d), np.float32)
    W[:, g["x_index"]] = g["w_col"]
    W[:, 0] = 100.0                              # x is zero there: a transposed W would show it
    b = np.array(g["bias"], np.float32)
    out = oracle.route(synth.f32_to_bf16_bits(x), W, b, np.array(g["slot_of"], np.int32), k)
    assert np.array_equal(out["logits"][0], g["expected_logits"])
    lg = np.array(g["expected_logits"])
    closed = np.exp(lg) / np.exp(lg).sum()
    assert np.allclose(out["scores"][0], closed, rtol=1e-14, atol=0)
    assert list(out["want_e"][0]) == g["expected_want_e"]
    assert list(out["sel_e"][0]) == g["expected_sel_e"]
    assert list(out["sel_slot"][0]) == g["expected_sel_slot"]
    assert np.allclose(out["sel_w"][0], closed[g["expected_sel_e"]], rtol=1e-14)


def test_router_scores_sum_to_one_and_match_logsumexp():
    cfg = synth.TINY
    x = synth.hidden_bf16(cfg.seed, 8, cfg.d)
    W = synth.router_weights(cfg.seed, cfg.E, cfg.d)
    b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma)
    logits, scores = oracle.router(x, W, b)
    assert np.allclose(scores.sum(1), 1.0, rtol=0, atol=1e-14)
    # logits by a library matmul of the decoded operands
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ W.astype(np.float64).T + b.astype(np.float64)
    assert np.allclose(logits, ref, rtol=1e-13, atol=1e-13)
    lse = np.log(np.exp(ref - ref.max(1, keepdims=True)).sum(1, keepdims=True)) + ref.max(1, keepdims=True)
    assert np.allclose(scores, np.exp(ref - lse), rtol=1e-12, atol=0)


def _substitute_view(s_row, resident, k):
    """The README's wording: take the wanted top-k; replace each missing pick, in rank
    order, by the next-best resident expert not already chosen; list by score."""
    order = sorted(range(len(s_row)), key=lambda e: (-s_row[e], e))
    want = order[:k]
    chosen = [e for e in want if resident[e]]
    for e in want:
        if not resident[e]:
            for c in order:
                if resident[c] and c not in chosen:
                    chosen.append(c)
                    break
    return sorted(chosen, key=lambda e: (-s_row[e], e))


def test_topk_all_resident_equals_plain_topk():
    rng = np.random.default_rng(3)
    s = rng.random((20, 16))
    s /= s.sum(1, keepdims=True)
    out = oracle.topk(s, np.arange(16, dtype=np.int32), 4)
    assert np.array_equal(out["want_e"], out["sel_e"])
    assert np.array_equal(out["want_s"], out["sel_w"])
    for t in range(20):
        assert list(out["want_e"][t]) == [-ne for _, ne in heapq.nlargest(4, [(s[t, e], -e) for e in range(16)])]
        assert list(out["want_e"][t]) == list(np.argsort(-s[t], kind="stable")[:4])


def test_topk_single_missing_is_replaced_by_rank_k_plus_1():
    rng = np.random.default_rng(4)
    s = rng.random((30, 16))
    s /= s.sum(1, keepdims=True)
    k = 4
    for t in range(30):
        order = np.argsort(-s[t], kind="stable")
        for miss in range(k):
            slot_of = np.arange(16, dtype=np.int32) + 100
            slot_of[order[miss]] = -1
            out = oracle.topk(s[t:t + 1], slot_of, k)
            expect = [e for e in order[:k + 1] if e != order[miss]]
            assert list(out["sel_e"][0]) == expect
            assert list(out["sel_slot"][0]) == [e + 100 for e in expect]
            assert list(out["want_e"][0]) == list(order[:k])


def test_topk_brute_force_all_masks_E16_k4():
    rng = np.random.default_rng(5)
    T, E, k = 8, 16, 4
    s = rng.random((T, E))
    s[:, 3] = s[:, 9]          # exact ties: the lower expert index goes first
    s /= s.sum(1, keepdims=True)
    for mask in range(1 << E):
        if mask % 97 and bin(mask).count("1") not in (0, 1, 3, 4, 5):
            continue                                          # every 97th mask plus all small sets
        resident = [(mask >> e) & 1 == 1 for e in range(E)]
        slot_of = np.array([e if resident[e] else -1 for e in range(E)], np.int32)
        out = oracle.topk(s, slot_of, k)
        for t in range(T):
            expect = _substitute_view(s[t], resident, k)
            got = [e for e in out["sel_e"][t] if e >= 0]
            assert got == expect, (mask, t)
            nres = sum(resident)
            assert list(out["sel_e"][t][min(k, nres):]) == [-1] * (k - min(k, nres))
            assert all(w == 0.0 for w in out["sel_w"][t][min(k, nres):])


def test_topk_tie_lower_index_first():
    s = np.full((1, 8), 1.0 / 8)
    out = oracle.topk(s, np.array([-1, 0, 1, -1, 2, 3, 4, 5], np.int32), 3)
    assert list(out["want_e"][0]) == [0, 1, 2]
    assert list(out["sel_e"][0]) == [1, 2, 4]


# ------------------------------------------------------------------ demand and heavy misses (README items 1, 3)

def test_demand_sums_and_miss_max():
    rng = np.random.default_rng(6)
    T, E, k, L = 12, 16, 4, 3
    s = rng.random((T, E))
    s /= s.sum(1, keepdims=True)
    slot_of = np.where(rng.random(E) < 0.6, np.arange(E), -1).astype(np.int32)
    out = oracle.topk(s, slot_of, k)
    D = np.zeros((L, E))
    M = np.zeros((L, E))
    oracle.demand(out["want_e"], out["want_s"], slot_of, 1, D, M)
    assert np.isclose(D.sum(), out["want_s"].sum(), rtol=1e-14)
    assert not D[0].any() and not D[2].any()
    # one-hot bookkeeping: D[1, e] = sum of the scores of token rows that wanted e
    ref = np.zeros(E)
    mref = np.zeros(E)
    for t in range(T):
        for j in range(k):
            e = out["want_e"][t, j]
            ref[e] += s[t, e]
            if slot_of[e] < 0:
                mref[e] = max(mref[e], s[t, e])
    assert np.allclose(D[1], ref, rtol=1e-14, atol=0)
    assert np.array_equal(M[1], mref)
    assert not M[1][slot_of >= 0].any()


def test_heavy_miss_hand_worked():
    g = GOLDEN["heavy_miss"]
    M = np.zeros((g["L"], g["E"]))
    flat = M.reshape(-1)
    for i in range(20):
        flat[3 * i] = 0.2 + 0.01 * i
    flat[100] = 0.19999
    flat[101] = 0.5
    flat[61] = 0.5
    keep = M.copy()
    ids, shares = oracle.hot_miss_select(M, 0.2, 16)
    assert list(ids) == g["expected_flat"]
    assert np.array_equal(shares, keep.reshape(-1)[ids])
    assert not M.any()                                   # reset for the next step
    ids, _ = oracle.hot_miss_select(keep.copy(), 0.2, 64)
    assert ids[-1] == 0 and 100 not in ids and len(ids) == 22


# ------------------------------------------------------------------ expert FFN (README profile table: MXFP4 experts)

def _np_pair(x_bits, w, d, F):
    """Second formulation with library matmuls on table-dequantised weights."""
    xq_c, xq_s = oracle.quantise_mxfp4(synth.bf16_bits_to_f32(x_bits).astype(np.float64))
    xq = _table_dequant(xq_c, xq_s, d)
    Wgu = np.stack([_table_dequant(w["gu_codes"][r], w["gu_scales"][r], d) for r in range(2 * F)])
    g = Wgu[:F] @ xq
    u = Wgu[F:] @ xq
    h = g / (1.0 + np.exp(-g)) * u
    hq_c, hq_s = oracle.quantise_mxfp4(h)
    hq = _table_dequant(hq_c, hq_s, F)
    Wd = np.stack([_table_dequant(w["dn_codes"][r], w["dn_scales"][r], F) for r in range(d)])
    return Wd @ hq, h, hq_c, hq_s


def test_expert_pair_matches_matmul_formulation():
    cfg = synth.TINY
    x = synth.hidden_bf16(cfg.seed, 2, cfg.d)
    w = synth.expert_weights(cfg.seed, 0, 5, cfg.d, cfg.ffn)
    for t in range(2):
        o = oracle.expert_pair(x[t], w, cfg.d, cfg.ffn)
        y, h, hc, hs = _np_pair(x[t], w, cfg.d, cfg.ffn)
        assert np.allclose(o["h"], h, rtol=1e-12, atol=1e-12)
        assert np.array_equal(o["hq_codes"], hc) and np.array_equal(o["hq_scales"], hs)
        assert np.allclose(o["y"], y, rtol=1e-12, atol=1e-9)


def test_expert_pair_single_code_closed_form():
    # One non-zero weight per row: g_f = Wg[f, a] * xq[a], u_f = Wu[f, b] * xq[b],
    # and down row o picks hq at one index; the gate/up split and the nibble order show.
    d, F = 64, 64
    w = dict(gu_codes=np.zeros((2 * F, d // 2), np.uint8), gu_scales=np.full((2 * F, d // 32), 127, np.uint8),
             dn_codes=np.zeros((d, F // 2), np.uint8), dn_scales=np.full((d, F // 32), 127, np.uint8))
    for f in range(F):
        w["gu_codes"][f, 1] = 0x20          # gate row f: element 3 (high nibble of byte 1) = code 2 = 1.0
        w["gu_codes"][F + f, 2] = 0x05      # up row f: element 4 (low nibble of byte 2) = code 5 = 3.0
    for o in range(d):
        w["dn_codes"][o, (o % F) // 2] = 0x4 if (o % F) % 2 == 0 else 0x40   # 2.0 at element o % F
    x = np.zeros(d, np.float32)
    x[3], x[4], x[10] = 0.5, 2.0, 4.0       # block amax 4 -> exponent 0: all three exact
    xb = synth.f32_to_bf16_bits(x)
    o = oracle.expert_pair(xb, w, d, F)
    g, u = 1.0 * 0.5, 3.0 * 2.0
    h = g / (1 + math.exp(-g)) * u
    assert np.allclose(o["h"], h, rtol=1e-15)
    hq = _table_dequant(o["hq_codes"], o["hq_scales"], F)
    assert np.allclose(o["y"], 2.0 * hq[np.arange(d) % F], rtol=0, atol=0)
    # h = 1.869 for every f: amax in [1, 2) -> exponent -2, h/0.25 = 7.48 -> saturates at 6 -> 1.5
    assert np.all(hq == 1.5)


def test_ffn_combine_rank_order_and_weights():
    cfg = synth.TINY
    T, k = 3, 2
    x = synth.hidden_bf16(cfg.seed, T, cfg.d)
    ex = [synth.expert_weights(cfg.seed, 0, e, cfg.d, cfg.ffn) for e in (1, 7)]
    sel_u = np.array([[0, 1], [1, -1], [-1, -1]], np.int32)
    sel_w = np.array([[0.25, 0.5], [2.0, 0.0], [0.0, 0.0]])
    out = oracle.ffn(x, sel_u, sel_w, ex, cfg.d, cfg.ffn)
    y00 = oracle.expert_pair(x[0], ex[0], cfg.d, cfg.ffn)["y"]
    y01 = oracle.expert_pair(x[0], ex[1], cfg.d, cfg.ffn)["y"]
    y11 = oracle.expert_pair(x[1], ex[1], cfg.d, cfg.ffn)["y"]
    assert np.allclose(out[0], 0.25 * y00 + 0.5 * y01, rtol=1e-14, atol=1e-14)
    assert np.allclose(out[1], 2.0 * y11, rtol=1e-15)
    assert not out[2].any()


# ------------------------------------------------------------------ re-plan and ring (README items 1, 3)

def test_replan_hand_worked():
    g = GOLDEN["replan"]
    L, E = g["L"], g["E"]
    owner = np.array(g["owner_in"], np.int32)
    slot_of = np.full(L * E, -1, np.int32)
    for s, f in enumerate(owner):
        if f >= 0:
            slot_of[f] = s
    so, ow, loads = oracle.replan(np.array(g["D"], np.float64).reshape(L, E), g["n_main"], slot_of, owner)
    assert list(ow) == g["expected_owner"]
    assert list(loads) == g["expected_loads"]
    for s, f in enumerate(ow):
        if f >= 0:
            assert so[f] == s
    assert (so >= 0).sum() == (ow >= 0).sum()


def _brute_main_set(D, was_main, n_main):
    """Brute force over all subsets: the subset of size n_main that is lexicographically
    best under (sum of D, count of old members, then the smallest flat ids)."""
    n = len(D)
    best, best_key = None, None
    for sub in itertools.combinations(range(n), n_main):
        key = (sum(D[f] for f in sub), sum(was_main[f] for f in sub), [-f for f in sorted(sub)])
        if best_key is None or key > best_key:
            best, best_key = set(sub), key
    return best


def test_replan_brute_force_small():
    rng = np.random.default_rng(7)
    L, E, n_main, n_ring = 2, 4, 4, 2
    for trial in range(60):
        n = L * E
        D = rng.integers(0, 4, n).astype(np.float64)    # small integers: many ties
        flats = rng.permutation(n)
        owner = np.full(n_main + n_ring, -1, np.int32)
        n_old = rng.integers(0, n_main + 1)
        owner[:n_main][rng.permutation(n_main)[:n_old]] = flats[:n_old]
        ring_n = rng.integers(0, n_ring + 1)
        owner[n_main:n_main + ring_n] = flats[n_old:n_old + ring_n]
        slot_of = np.full(n, -1, np.int32)
        for s, f in enumerate(owner):
            if f >= 0:
                slot_of[f] = s
        was_main = [(0 <= slot_of[f] < n_main) for f in range(n)]
        so, ow, loads = oracle.replan(D.reshape(L, E), n_main, slot_of, owner)
        new_main = {int(f) for f in ow[:n_main] if f >= 0}
        assert new_main == _brute_main_set(D, was_main, n_main)
        for f in range(n):                                         # survivors keep their slots
            if was_main[f] and f in new_main:
                assert so[f] == slot_of[f]
        newcomers = [f for f in new_main if not was_main[f]]
        assert len(loads) == len(newcomers)
        assert list(loads) == sorted(loads)                        # free slots in ascending order
        got_order = [int(ow[s]) for s in loads]                    # newcomers by (D desc, flat asc)
        assert got_order == sorted(newcomers, key=lambda f: (-D[f], f))
        for s in range(n_main, n_main + n_ring):                   # ring: untouched unless promoted
            if owner[s] >= 0 and owner[s] in new_main:
                assert ow[s] == -1
            else:
                assert ow[s] == owner[s]
        for s, f in enumerate(ow):
            if f >= 0:
                assert so[f] == s
        assert (so >= 0).sum() == (ow >= 0).sum()


def test_ring_install():
    slot_of = np.array([0, -1, -1, 4], np.int32)
    owner = np.array([0, -1, -1, -1, 3], np.int32)       # slots 0..2 main, 3..4 ring
    assert oracle.ring_install(slot_of, owner, 3, 1) == 0
    assert list(owner) == [0, -1, -1, 1, 3] and slot_of[1] == 3
    assert oracle.ring_install(slot_of, owner, 4, 2) == 0      # evicts flat 3
    assert list(owner) == [0, -1, -1, 1, 2] and slot_of[3] == -1 and slot_of[2] == 4
    assert oracle.ring_install(slot_of, owner, 3, 0) == 1      # already resident: no change
    assert list(owner) == [0, -1, -1, 1, 2]


# ------------------------------------------------------------------ demand forgetting (fixed point)

def test_demand_decay_identity_zero_and_shifts():
    rng = np.random.default_rng(5)
    D = np.concatenate([rng.integers(0, 2**63, 64, dtype=np.uint64),
                        np.array([0, 1, 2, 3, 2**40, 2**64 - 1], dtype=np.uint64)])
    assert np.array_equal(oracle.demand_decay_fixed(D, 1.0), D)                 # factor 1: unchanged
    assert not oracle.demand_decay_fixed(D, 0.0).any()                          # factor 0: forgotten
    for m in range(1, 12):                                                      # 2^-m: a right shift (floor)
        assert np.array_equal(oracle.demand_decay_fixed(D, 2.0 ** -m), D >> np.uint64(m)), m


def test_demand_decay_tracks_the_real_product():
    rng = np.random.default_rng(6)
    D = rng.integers(0, 2**62, 200, dtype=np.uint64)
    prev = np.zeros_like(D)
    for f in (0.001, 0.1, 0.3, 0.5, 0.7, 0.9, 0.99, 0.999999):
        got = oracle.demand_decay_fixed(D, np.float32(f))
        for d, g in zip(D.tolist(), got.tolist()):
            exact = d * float(np.float32(f))
            # factor rounded to a multiple of 2^-32, then floor: within 1 + d * 2^-33 of d * f
            assert abs(g - exact) <= 1 + d * 2.0 ** -33 + exact * 1e-15
        assert np.all(got >= prev)                                                # monotone in the factor
        prev = got


# ------------------------------------------------------------------ synchronous hot read (one layer)

def test_hot_read_choose_hand_case():
    # experts 0..5: 1, 3, 4 resident; 2 and 5 missed with shares 0.25 and 0.6; 5 has no record
    M = np.array([0, 0, 0.25, 0, 0, 0.6])
    D = np.array([0, 7.0, 0, 2.0, 2.0, 0])
    slot_of = np.array([-1, 4, -1, 0, 9, -1], np.int32)
    store = [1, 1, 1, 1, 1, 0]
    # 5 is the heaviest miss but the store cannot serve it; 2 is read; 3 and 4 tie at the lowest
    # demand and the lower index is the coldest
    assert oracle.hot_read_choose(M, D, slot_of, store, 0.2, 1) == (2, 3)
    assert oracle.hot_read_choose(M, D, slot_of, [1] * 6, 0.2, 1) == (5, 3)
    assert oracle.hot_read_choose(M, D, slot_of, store, 0.3, 1) == (-1, -1)     # under the threshold
    assert oracle.hot_read_choose(M, D, slot_of, store, 0.25, 1) == (2, 3)      # the threshold is included
    assert oracle.hot_read_choose(M, D, slot_of, store, 0.2, 0) == (-1, -1)     # the step's budget is spent
    assert oracle.hot_read_choose(M, D, np.full(6, -1, np.int32), store, 0.2, 1) == (-1, -1)   # nothing resident


def test_hot_read_choose_brute_force():
    rng = np.random.default_rng(9)
    for _ in range(300):
        E = int(rng.integers(1, 12))
        M = np.round(rng.random(E), 1) * (rng.random(E) < 0.6)
        D = np.round(rng.random(E) * 4, 0)
        slot_of = np.where(rng.random(E) < 0.5, rng.integers(0, 20, E), -1).astype(np.int32)
        store = (rng.random(E) < 0.8).astype(np.uint8)
        got = oracle.hot_read_choose(M, D, slot_of, store, 0.2, 1)
        cand = [e for e in range(E) if slot_of[e] < 0 and store[e] and M[e] >= 0.2]
        res = [e for e in range(E) if slot_of[e] >= 0]
        if not cand or not res:
            assert got == (-1, -1)
            continue
        best = sorted(cand, key=lambda e: (-M[e], e))[0]
        cold = sorted(res, key=lambda e: (D[e], e))[0]
        assert got == (best, cold)


# ------------------------------------------------------------------ optional weight renormalisation

def test_renormalise_sums_to_one_and_keeps_ratios():
    so = np.array([[3, 1, -1], [-1, -1, -1], [0, 2, 5]], np.int32)
    w = np.array([[0.3, 0.1, 0.0], [0.0, 0.0, 0.0], [0.5, 0.25, 0.25]])
    r = oracle.renormalise(so, w)
    assert np.allclose(r[0], [0.75, 0.25, 0.0]) and np.all(r[1] == 0) and np.allclose(r[2], [0.5, 0.25, 0.25])
    rng = np.random.default_rng(3)
    so = np.where(rng.random((50, 8)) < 0.8, 1, -1).astype(np.int32)
    w = rng.random((50, 8)) * (so >= 0)
    r = oracle.renormalise(so, w)
    valid = (so >= 0).any(1)
    assert np.allclose(r[valid].sum(1), 1.0) and np.all(r[~valid] == 0)
    ratio = np.divide(r, w, out=np.zeros_like(r), where=w > 0)               # one scale per token
    for t in np.flatnonzero(valid):
        x = ratio[t][w[t] > 0]
        assert np.allclose(x, x[0])
