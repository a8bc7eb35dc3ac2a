"""The synchronous hot read of one layer (moe_hot_read_sync) on the GPU, through the C ABI.

TideLM README, item 3 (GLM-5.3): before a layer's MoE runs, its largest miss
is loaded, used with its exact weights, and stays resident in the slot of the
least-demanded expert. The choice and the table update are checked bit-exact against the
oracle fed the GPU's own miss shares and demand; the copied record, the read
budget, and the layer routed again (routing and FFN against the oracle on the
updated table) are checked too.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.cases import ffn_within_tolerance, hidden_dev, ring_case, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")
from resident_expert_routed_gb300.layer import LayerBuffers  # noqa: E402


def _route(buf, x, Wd, bd, so_d):
    moe.moe_route_resident(x, Wd, bd, so_d, buf.k, buf.want_e, buf.want_s, buf.sel_e, buf.sel_slot, buf.sel_w,
                           buf.workspace)


def test_sync_hot_read_replaces_the_coldest_expert():
    # 64 tokens of hidden stream 3 leave heavy misses (found with the oracle); no ring slots
    cfg, T = synth.TINY, 64
    c, arena, slot_of, owner, absent, store, records = ring_case(cfg, 0, T, stream=3)
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    Wd, bd, x = to_dev(c.W), to_dev(c.bias), hidden_dev(c.x)
    buf = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, arena.n_slots)
    demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    store_dev = torch.tensor([r or 0 for r in records], dtype=torch.int64, device="cuda")
    budget = torch.tensor([16], dtype=torch.int32, device="cuda")
    swap = torch.zeros(3, dtype=torch.int32, device="cuda")

    _route(buf, x, Wd, bd, so_d)
    moe.moe_demand_accumulate(buf.want_e, buf.want_s, so_d, 0, demand, miss)
    torch.cuda.synchronize()
    M = miss.cpu().numpy().astype(np.float64).ravel()
    D = demand.cpu().numpy().view(np.uint64).astype(np.float64).ravel()      # < 2^53: exact
    e_read, e_cold = oracle.hot_read_choose(M, D, slot_of, [r is not None for r in records], 0.2, 16)
    assert e_read >= 0 and e_cold >= 0
    moe.moe_hot_read_sync(store_dev, demand, miss, so_d, ow_d, arena, 0, 0.2, budget, swap)
    torch.cuda.synchronize()
    slot = int(slot_of[e_cold])
    assert swap.cpu().tolist() == [e_read, slot, e_cold]
    assert int(budget.item()) == 15
    slot_of[e_cold], slot_of[e_read], owner[slot] = -1, slot, e_read
    assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
    sb = arena.slot_bytes
    i = int(np.flatnonzero(absent == e_read)[0])
    assert torch.equal(arena.buf[slot * sb:(slot + 1) * sb].cpu(), store[i * sb:(i + 1) * sb])

    # the layer routed again: the tokens that wanted the expert now get it; FFN against the oracle
    _route(buf, x, Wd, bd, so_d)
    moe.moe_expert_ffn_mxfp4(x, buf.sel_slot, buf.sel_w, arena, buf.out, buf.workspace)
    torch.cuda.synchronize()
    ref = oracle.route(c.x, c.W, c.bias, slot_of, cfg.k)
    sel = buf.sel_e.cpu().numpy()
    assert np.array_equal(np.sort(sel, 1), np.sort(ref["sel_e"], 1))
    assert (sel == e_read).any() and not (sel == e_cold).any()
    sel_slot = buf.sel_slot.cpu().numpy()
    used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
    idx = {s: j for j, s in enumerate(used)}
    sel_u = np.vectorize(lambda s: idx.get(int(s), -1))(sel_slot).astype(np.int32)
    ex = [synth.expert_weights(cfg.seed, 0, int(owner[s]), cfg.d, cfg.ffn) for s in used]
    exp = oracle.ffn(c.x, sel_u, buf.sel_w.cpu().numpy().astype(np.float64), ex, cfg.d, cfg.ffn)
    ok, fro, mx = ffn_within_tolerance(buf.out.cpu().numpy().astype(np.float64), exp)
    assert ok, (fro, mx)

    # with the step's budget spent nothing is read and the tables stay as they are
    budget.zero_()
    moe.moe_hot_read_sync(store_dev, demand, miss, so_d, ow_d, arena, 0, 0.2, budget, swap)
    torch.cuda.synchronize()
    assert swap.cpu().tolist() == [-1, -1, -1]
    assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
