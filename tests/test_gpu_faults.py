"""Device-side checks of the C ABI, made to fire without faulting the GPU.

Each check plants bad data on the host side or shortens a bound, and reads
the result through ``moe_device_status``:

* an e8m0 weight scale byte 0xFF (NaN) in one arena slot sets
  MOE_DEV_NAN_SCALE; picks of other slots are computed as usual;
* inconsistent slot_of / owner tables make ``moe_arena_replan`` set
  MOE_DEV_BAD_TABLE and leave the tables untouched;
* a wait that can never be satisfied gives up after the bound set with
  ``moe_set_wait_limit`` and reports MOE_ETIMEOUT; with a bound too short
  for the real pipelines, the GEMM and router kernels give up the same way,
  and the next call with the default bound is correct again.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import oracle_pool
from tests.cases import device_arena, ffn_within_tolerance, hidden_dev, make_case, oracle_experts, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")


def _ffn(c, arena, sel_slot, sel_w):
    T, cfg = c.x.shape[0], c.cfg
    out = torch.zeros((T, cfg.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_workspace_bytes(T, cfg.k, cfg.d, cfg.ffn, cfg.E, arena.n_slots), dtype=torch.uint8,
                     device="cuda")
    moe.moe_expert_ffn_mxfp4(hidden_dev(c.x), to_dev(sel_slot.astype(np.int32)), to_dev(sel_w.astype(np.float32)),
                             arena, out, ws)
    st = moe.moe_device_status()
    return out.cpu().numpy().astype(np.float64), st


@pytest.mark.parametrize("cfg,T,matrix", [(synth.TINY, 8, "gu"), (synth.TINY, 80, "gu"), (synth.TINY, 80, "dn"),
                                          (synth.DECODE, 8, "dn")],
                         ids=["tiny-T8-gate_up", "tiny-T80-gate_up", "tiny-T80-down", "decode-T8-down"])
def test_nan_weight_scale_sets_error_bit(cfg, T, matrix):
    c = make_case(cfg, T)
    arena = device_arena(cfg, c.owner, c.n_slots)
    ref = oracle.route(c.x, c.W, c.bias, c.slot_of, cfg.k)
    sel_slot, sel_w = ref["sel_slot"], ref["sel_w"]
    used, counts = np.unique(sel_slot[sel_slot >= 0], return_counts=True)
    bad = int(used[np.argmin(counts)])                    # a slot some tokens use and most do not
    off = arena.off_gu_scales if matrix == "gu" else arena.off_dn_scales
    n_scale = (2 * cfg.ffn * cfg.d if matrix == "gu" else cfg.d * cfg.ffn) // 32
    pos = bad * arena.slot_bytes + off + (n_scale * 5) // 7   # a byte inside the matrix's scales
    arena.buf[pos] = 0xFF
    got, (st, bits) = _ffn(c, arena, sel_slot, sel_w)
    assert st == moe.MOE_EDEVICE and bits & moe.MOE_DEV_NAN_SCALE, (st, bits)
    assert not bits & ~moe.MOE_DEV_NAN_SCALE
    # tokens that do not pick the bad slot are unaffected
    clean = ~(sel_slot == bad).any(axis=1)
    assert clean.sum() >= 1
    rows = np.flatnonzero(clean)
    sel_u, experts = oracle_experts(cfg, c.owner, sel_slot[rows])
    exp = oracle.ffn(c.x[rows], sel_u, sel_w[rows].astype(np.float32).astype(np.float64), experts, cfg.d, cfg.ffn)
    ok, fro, mx = ffn_within_tolerance(got[rows], exp)
    assert ok, (fro, mx)
    # the slot repaired: no bit, every token within tolerance
    arena.buf[pos] = 0x7F
    got, st = _ffn(c, arena, sel_slot, sel_w)
    assert st == (moe.MOE_OK, 0)


def test_replan_inconsistent_tables_set_bad_table():
    L, E, n_main, n_ring = 2, 8, 4, 2
    n = L * E
    owner = np.array([0, 3, 5, 9, -1, -1], np.int32)
    slot_of = np.full(n, -1, np.int32)
    for s, f in enumerate(owner):
        if f >= 0:
            slot_of[f] = s
    demand = torch.from_numpy(np.arange(n, dtype=np.int64)[::-1].copy()).cuda().view(L, E)
    ws = torch.empty(moe.moe_replan_workspace_bytes(L, E), dtype=torch.uint8, device="cuda")
    for kind in ("owner", "slot_of"):
        so, ow = slot_of.copy(), owner.copy()
        if kind == "owner":
            ow[4] = 7                                     # slot 4 claims expert 7, whose table entry says -1
        else:
            so[12] = 1                                    # expert 12 claims slot 1, which holds expert 3
        so_d, ow_d = to_dev(so), to_dev(ow)
        loads = torch.full((n_main,), -9, dtype=torch.int32, device="cuda")
        nl = torch.full((1,), -9, dtype=torch.int32, device="cuda")
        moe.moe_arena_replan(demand, n_main, so_d, ow_d, loads, nl, ws)
        st, bits = moe.moe_device_status()
        assert st == moe.MOE_EDEVICE and bits == moe.MOE_DEV_BAD_TABLE, (kind, st, bits)
        assert np.array_equal(so_d.cpu().numpy(), so) and np.array_equal(ow_d.cpu().numpy(), ow)
        assert int(nl.item()) == 0 and bool((loads == -9).all())
    # consistent tables: re-planned as the oracle does, no bit
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    loads = torch.full((n_main,), -9, dtype=torch.int32, device="cuda")
    nl = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_arena_replan(demand, n_main, so_d, ow_d, loads, nl, ws)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
    so_ref, ow_ref, loads_ref = oracle.replan(demand.cpu().numpy().astype(np.float64), n_main, slot_of, owner)
    assert np.array_equal(ow_d.cpu().numpy(), ow_ref) and np.array_equal(so_d.cpu().numpy(), so_ref)


def test_stalled_wait_ends_in_timeout_status():
    old = moe.moe_get_wait_limit()
    try:
        moe.moe_set_wait_limit(1_000_000)                 # 1 ms
        assert moe.moe_get_wait_limit() == 1_000_000
        for _ in range(2):                                # the context stays usable: twice in a row
            moe.moe_wait_selftest()
            st, bits = moe.moe_device_status()
            assert st == moe.MOE_ETIMEOUT and bits == moe.MOE_DEV_TIMEOUT, (st, bits)
    finally:
        moe.moe_set_wait_limit(0)
    assert moe.moe_get_wait_limit() == old == 2_000_000_000


def test_pipelines_give_up_under_a_short_bound_then_recover():
    """With a 1 ns bound the GEMM pipelines (and the tensor-core router) give up at their first wait that
    does not succeed at once: the call reports MOE_ETIMEOUT, and the next call with the default bound gives
    the oracle's results."""
    cfg, T = synth.DECODE, 64
    c = make_case(cfg, T)
    arena = device_arena(cfg, c.owner, c.n_slots)
    ref = oracle.route(c.x, c.W, c.bias, c.slot_of, cfg.k)
    sel_slot, sel_w = ref["sel_slot"], ref["sel_w"]
    outcomes = []
    try:
        moe.moe_set_wait_limit(1)
        # after a pipeline gave up, the call's later kernels read unfinished intermediates (e.g. the down
        # GEMM the gate/up GEMM's missing activation scales), so a non-finite bit may come with the timeout
        after_timeout = moe.MOE_DEV_TIMEOUT | moe.MOE_DEV_NAN_SCALE
        for _ in range(3):
            _, (st, bits) = _ffn(c, arena, sel_slot, sel_w)
            assert (st, bits) == (moe.MOE_OK, 0) or (st == moe.MOE_ETIMEOUT and bits & moe.MOE_DEV_TIMEOUT and
                                                      bits & ~after_timeout == 0), (st, bits)
            outcomes.append(st)
        # the tensor-core router (more than 64 tokens) under the same bound
        cp = make_case(synth.PREFILL, 256)
        k = cfg.k
        o = [torch.empty((256, k), dtype=dt, device="cuda") for dt in (torch.int32, torch.float32, torch.int32,
                                                                        torch.int32, torch.float32)]
        ws = torch.empty(moe.moe_workspace_bytes(256, k, cfg.d, cfg.ffn, cfg.E, cp.n_slots), dtype=torch.uint8,
                         device="cuda")
        moe.moe_route_resident(hidden_dev(cp.x), to_dev(cp.W), to_dev(cp.bias), to_dev(cp.slot_of), k, *o, ws)
        st, bits = moe.moe_device_status()
        assert st in (moe.MOE_OK, moe.MOE_ETIMEOUT) and bits & ~moe.MOE_DEV_TIMEOUT == 0, (st, bits)
        outcomes.append(st)
    finally:
        moe.moe_set_wait_limit(0)
    assert moe.MOE_ETIMEOUT in outcomes, outcomes
    got, st = _ffn(c, arena, sel_slot, sel_w)
    assert st == (moe.MOE_OK, 0)
    exp = oracle_pool.ffn(cfg, c.x, sel_slot, sel_w.astype(np.float32).astype(np.float64), c.owner)
    ok, fro, mx = ffn_within_tolerance(got, exp)
    assert ok, (fro, mx)
