"""Re-plan cadence and slot refill on the GPU (README item 1: the arena is planned again after a prefill,
every few hundred tokens and between requests, and the experts it admits are read into their new slots).

Three layers of 16 experts share an arena of 20 slots, first holding a seeded sample of the 48 experts. Every
step routes a few tokens through each layer and records demand; the Cadence re-plans every 16 tokens,
refills the reassigned slots from a pinned host store (one record per expert) and halves the history. At
each re-plan the tables, the load list, the decayed history and the refilled bytes are checked against the
oracle's re-plan and decay and the generator's records; afterwards a routed layer's FFN is checked against
the oracle on the new owners.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.cases import ffn_within_tolerance, hidden_dev, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")
from resident_expert_routed_gb300.layer import Adaptation, Cadence, LayerBuffers, layer_step  # noqa: E402

ADAPT = synth.LayerConfig("adapt L3 E16 k4 d256 F128 arena20", E=16, k=4, d=256, ffn=128, resident=0, sigma=1.0,
                          seed=0x7EED00B0, L=3, n_main=20)


def _setup(cfg):
    L, E = cfg.L, cfg.E
    slot_of, owner = synth.full_initial_arena(cfg)
    rec = synth.slot_record(cfg.d, cfg.ffn)
    sb = rec["slot_bytes"]
    buf = torch.zeros(cfg.n_main * sb, dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(buf, cfg.d, cfg.ffn, cfg.seed, E, to_dev(owner))
    arena = moe.Arena(buf, sb, cfg.n_main, cfg.d, cfg.ffn, rec["off_gu_codes"], rec["off_gu_scales"],
                      rec["off_dn_codes"], rec["off_dn_scales"])
    store = torch.empty(L * E * sb, dtype=torch.uint8).pin_memory()
    for f in range(L * E):
        store[f * sb:(f + 1) * sb] = torch.from_numpy(synth.expert_slot_bytes(cfg.seed, f // E, f % E, cfg.d, cfg.ffn))
    records = [store.data_ptr() + f * sb for f in range(L * E)]
    return slot_of, owner, arena, store, records


def test_cadence_replans_and_refills_from_the_store():
    cfg, T = ADAPT, 4
    L, E, k = cfg.L, cfg.E, cfg.k
    slot_of, owner, arena, store, records = _setup(cfg)
    Ws = [to_dev(synth.router_weights(cfg.seed, E, cfg.d, layer)) for layer in range(L)]
    bs = [to_dev(synth.router_bias(cfg.seed, E, cfg.sigma, layer)) for layer in range(L)]
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    demand = torch.zeros((L, E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((L, E), dtype=torch.float32, device="cuda")
    buf = LayerBuffers(T, k, E, cfg.d, cfg.ffn, cfg.n_main)
    adapt = Adaptation(demand, so_d, ow_d, arena, cfg.n_main, records, Cadence(every_tokens=16), decay=0.5)
    sb = arena.slot_bytes
    replans = 0
    for step in range(10):
        for layer in range(L):
            x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=1000 + step * L + layer)
            layer_step(hidden_dev(x), Ws[layer], bs[layer], so_d[layer * E:(layer + 1) * E], arena, demand, miss,
                       layer, buf)
        torch.cuda.synchronize()
        D0 = demand.cpu().numpy().view(np.uint64).copy()
        so0, ow0 = so_d.cpu().numpy(), ow_d.cpu().numpy()
        n = adapt.after_step(T)
        torch.cuda.synchronize()
        if (step + 1) % 4 != 0:                           # 16 tokens per re-plan
            assert n == 0 and adapt.replans == replans
            continue
        replans += 1
        assert adapt.replans == replans
        so_ref, ow_ref, loads_ref = oracle.replan(D0.astype(np.float64).reshape(L, E), cfg.n_main, so0, ow0)
        assert np.array_equal(so_d.cpu().numpy(), so_ref) and np.array_equal(ow_d.cpu().numpy(), ow_ref)
        assert n == len(loads_ref) and np.array_equal(adapt.loads.cpu().numpy()[:n], loads_ref)
        got = arena.buf.cpu().numpy()
        for s in loads_ref:                               # the admitted experts' records are in their slots
            f = int(ow_ref[s])
            assert np.array_equal(got[s * sb:(s + 1) * sb],
                                  synth.expert_slot_bytes(cfg.seed, f // E, f % E, cfg.d, cfg.ffn)), (step, s, f)
        assert np.array_equal(demand.cpu().numpy().view(np.uint64), oracle.demand_decay_fixed(D0, np.float32(0.5)))
        assert moe.moe_device_status() == (moe.MOE_OK, 0)
    assert replans == 2 and adapt.loaded > 0
    # a routed layer on the re-planned arena: the FFN reads the refilled slots
    ow = ow_d.cpu().numpy()
    so = so_d.cpu().numpy()
    layer = int(ow[int(adapt.loads[0].item())]) // E
    x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=5000)
    out = layer_step(hidden_dev(x), Ws[layer], bs[layer], so_d[layer * E:(layer + 1) * E], arena, demand, miss,
                     layer, buf)
    torch.cuda.synchronize()
    so_l = so[layer * E:(layer + 1) * E]
    ref = oracle.route(x, synth.router_weights(cfg.seed, E, cfg.d, layer), synth.router_bias(cfg.seed, E, cfg.sigma,
                       layer), so_l, k)
    sel_slot = buf.sel_slot.cpu().numpy()
    assert np.array_equal(np.sort(sel_slot, 1), np.sort(ref["sel_slot"], 1))
    used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
    idx = {s: i for i, s in enumerate(used)}
    sel_u = np.vectorize(lambda s: idx.get(int(s), -1))(sel_slot).astype(np.int32)
    ex = [synth.expert_weights(cfg.seed, int(ow[s]) // E, int(ow[s]) % E, cfg.d, cfg.ffn) for s in used]
    exp = oracle.ffn(x, sel_u, buf.sel_w.cpu().numpy().astype(np.float64), ex, cfg.d, cfg.ffn)
    ok, fro, mx = ffn_within_tolerance(out.cpu().numpy().astype(np.float64), exp)
    assert ok, (fro, mx)
    del store


def test_refill_refuses_a_missing_record_and_copies_nothing():
    cfg = ADAPT
    L, E = cfg.L, cfg.E
    slot_of, owner, arena, store, records = _setup(cfg)
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    # demand that admits experts outside the initial sample
    D = np.zeros((L, E), np.int64)
    absent = np.flatnonzero(slot_of < 0)
    D.ravel()[absent[:5]] = 1 << 40
    demand = to_dev(D)
    before = arena.buf.cpu().clone()
    gone = list(records)
    gone[int(absent[2])] = None                          # the store lacks one of the admitted experts
    adapt = Adaptation(demand, so_d, ow_d, arena, cfg.n_main, gone, Cadence(every_tokens=0))
    with pytest.raises(moe.MoeError) as ei:
        adapt.replan()
    assert ei.value.status == moe.MOE_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(arena.buf.cpu(), before)          # nothing was copied
    # with the record back, the same re-plan (already applied to the tables) refills all five
    n = moe.moe_arena_refill(arena, records, adapt.loads, adapt.n_loads, ow_d)
    torch.cuda.synchronize()
    assert n == 5
    got = arena.buf.cpu().numpy()
    ow = ow_d.cpu().numpy()
    for s in adapt.loads.cpu().numpy()[:n]:
        f = int(ow[s])
        assert np.array_equal(got[s * arena.slot_bytes:(s + 1) * arena.slot_bytes],
                              synth.expert_slot_bytes(cfg.seed, f // E, f % E, cfg.d, cfg.ffn))
    del store


def test_cadence_between_requests_and_after_prefill():
    cfg = ADAPT
    slot_of, owner, arena, store, records = _setup(cfg)
    demand = torch.zeros((cfg.L, cfg.E), dtype=torch.int64, device="cuda")
    adapt = Adaptation(demand, to_dev(slot_of), to_dev(owner), arena, cfg.n_main, records,
                       Cadence(every_tokens=0, after_prefill=True, between_requests=True))
    adapt.after_step(64, prefill=True)
    assert adapt.replans == 1
    assert adapt.request_done() == 0 and adapt.replans == 1     # nothing generated since
    adapt.after_step(3)
    adapt.request_done()
    assert adapt.replans == 2
    torch.cuda.synchronize()
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
    del store
