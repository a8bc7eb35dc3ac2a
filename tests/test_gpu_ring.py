"""The asynchronous hot-read ring (moe_hot_ring_*) on the GPU, through the C ABI.

TideLM README, item 3 (DeepSeek): a step's largest misses are fetched into
extra ring slots during the following step and can be routed to from the step
after it, until newer fetches wrap around the ring. A pinned host store of
expert records stands in for the drive. Checked: the tables after each call
against the oracle's ring install (FIFO order, evictions, experts not yet
routable while their copies are in flight), the copied bytes, and a real
routed step that uses a ring expert, against the oracle's routing and FFN.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.cases import ffn_within_tolerance, hidden_dev, ring_case, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")
from resident_expert_routed_gb300.layer import LayerBuffers, layer_step, step_end  # noqa: E402

N_RING = 2


def _heavy(ids, cap=16):
    flat = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    if ids:
        flat[:len(ids)] = torch.tensor(ids, dtype=torch.int32)
    return flat, torch.tensor([len(ids)], dtype=torch.int32, device="cuda")


def test_ring_fifo_fetch_install_and_evict():
    cfg = synth.TINY
    c, arena, slot_of, owner, absent, store, records = ring_case(cfg, N_RING)
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    ring = moe.HotRing(arena, cfg.resident, N_RING, records)
    a, b, cc = (int(f) for f in absent[:3])
    r0, r1 = cfg.resident, cfg.resident + 1

    # step 1's list names three misses; the ring takes two (FIFO), none routable yet
    assert ring.step(*_heavy([a, b, cc]), so_d, ow_d) == 2
    torch.cuda.synchronize()
    assert so_d[a] == -1 and so_d[b] == -1 and np.array_equal(ow_d.cpu().numpy(), owner)
    # next call installs them: the oracle's ring install in the same FIFO order gives the same tables
    assert ring.step(*_heavy([]), so_d, ow_d) == 0
    torch.cuda.synchronize()
    for slot, f in ((r0, a), (r1, b)):
        assert oracle.ring_install(slot_of, owner, slot, f) == 0
    assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
    sb = arena.slot_bytes
    for slot, f in ((r0, a), (r1, b)):
        i = int(np.flatnonzero(absent == f)[0])
        assert torch.equal(arena.buf[slot * sb:(slot + 1) * sb].cpu(), store[i * sb:(i + 1) * sb])
    # an expert already in the ring is not read again; the next one wraps onto the oldest slot,
    # whose owner leaves the tables at once and whose new owner is routable one call later
    assert ring.step(*_heavy([a, cc]), so_d, ow_d) == 1
    torch.cuda.synchronize()
    assert so_d[a] == -1 and ow_d[r0] == -1 and so_d[cc] == -1 and so_d[b] == r1
    assert ring.step(*_heavy([]), so_d, ow_d) == 0
    torch.cuda.synchronize()
    assert oracle.ring_install(slot_of, owner, r0, cc) == 0
    assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
    ring.close()


def test_ring_experts_are_routed_two_steps_later():
    # 64 tokens of hidden stream 3 leave three heavy misses (found with the oracle); a ring with room
    # for every absent expert, so nothing wraps
    cfg, T, n_ring = synth.TINY, 64, 8
    c, arena, slot_of, owner, absent, store, records = ring_case(cfg, n_ring, T, stream=3)
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    Wd, bd = to_dev(c.W), to_dev(c.bias)
    buf = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, arena.n_slots)
    demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    ring = moe.HotRing(arena, cfg.resident, n_ring, records)
    x = hidden_dev(c.x)
    fetched = []
    for step in range(3):
        tables = (so_d.cpu().numpy().copy(), ow_d.cpu().numpy().copy())     # what this step routes with
        out = layer_step(x, Wd, bd, so_d, arena, demand, miss, 0, buf)
        flat, _, n = step_end(miss, buf)
        heavy = [int(f) for f in flat.cpu().numpy()[:int(n.item())]]
        got = ring.step(flat, n, so_d, ow_d)
        torch.cuda.synchronize()
        ref = oracle.route(c.x, c.W, c.bias, tables[0], cfg.k)
        sel_slot = buf.sel_slot.cpu().numpy()
        assert np.array_equal(np.sort(buf.sel_e.cpu().numpy(), 1), np.sort(ref["sel_e"], 1)), step
        if step == 0:
            assert heavy and got == len(heavy)                  # the drifted bias leaves heavy misses
            fetched = heavy
        if step == 1:                                           # copies in flight: not routable yet
            assert not (sel_slot >= cfg.resident).any()
        if step == 2:                                           # installed by the call after step 1
            assert (sel_slot >= cfg.resident).any()
            ring_owners = tables[1][cfg.resident:]
            assert set(int(f) for f in ring_owners if f >= 0) == set(fetched)
            used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
            idx = {s: i for i, s in enumerate(used)}
            sel_u = np.vectorize(lambda s: idx.get(int(s), -1))(sel_slot).astype(np.int32)
            ex = [synth.expert_weights(cfg.seed, 0, int(tables[1][s]), cfg.d, cfg.ffn) for s in used]
            exp = oracle.ffn(c.x, sel_u, buf.sel_w.cpu().numpy().astype(np.float64), ex, cfg.d, cfg.ffn)
            ok, fro, mx = ffn_within_tolerance(out.cpu().numpy().astype(np.float64), exp)
            assert ok, (fro, mx)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
    ring.close()
