"""Multi-step GPU runs against the oracle: the hot-read ring and the shared arena.

GLM-like layer: between steps, 64 seeded non-resident experts are installed
in the ring slots (FIFO) and their bytes written; routing and the FFN are then
checked against the oracle on that step's table (README item 3: ring slots on
top of the budget, routable from the step after).

Full decode step: 60 layers share one arena of 10,000 main + 64 ring slots;
each step routes 2 tokens through all layers, records demand, takes the
step's heavy-miss list and installs it in the ring; after 256 steps the arena
is re-planned from the demand history (README item 1). Every layer's routing,
the heavy-miss lists, the demand table, sampled FFN outputs and the re-plan
are checked; the oracle always sees the table the GPU used (a snapshot), so
near-ties cannot cascade across steps.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import oracle_pool
from tests.cases import clear_ranks, ffn_within_tolerance, hidden_dev, near_tie_tokens, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")
from resident_expert_routed_gb300.layer import LayerBuffers, layer_step, step_end  # noqa: E402


def _arena(cfg, n_slots, owner):
    rec = synth.slot_record(cfg.d, cfg.ffn)
    buf = torch.zeros(n_slots * rec["slot_bytes"], dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(buf, cfg.d, cfg.ffn, cfg.seed, cfg.E, to_dev(owner.astype(np.int32)))
    return moe.Arena(buf, rec["slot_bytes"], n_slots, cfg.d, cfg.ffn, rec["off_gu_codes"], rec["off_gu_scales"],
                     rec["off_dn_codes"], rec["off_dn_scales"])


def _fill(arena, cfg, slots, flats):
    synth.fill_slots_device(arena.buf, cfg.d, cfg.ffn, cfg.seed, cfg.E, to_dev(np.asarray(flats, np.int32)),
                            slots=to_dev(np.asarray(slots, np.int32)))


def _check_routing(ref, buf, slot_of, k, E):
    """Routing of one layer call against the oracle (near-tie tokens excluded)."""
    sel = buf.sel_e.cpu().numpy()
    want = buf.want_e.cpu().numpy()
    slot = buf.sel_slot.cpu().numpy()
    _route_matches(ref, (want, sel, slot), slot_of, k, E)
    return sel, slot


def _oracle_ffn(cfg, x, sel_slot, sel_w, owner):
    used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
    idx = {s: i for i, s in enumerate(used)}
    sel_u = np.vectorize(lambda s: idx.get(int(s), -1))(sel_slot).astype(np.int32)
    ex = [synth.expert_weights(cfg.seed, int(owner[s]) // cfg.E, int(owner[s]) % cfg.E, cfg.d, cfg.ffn) for s in used]
    return oracle.ffn(x, sel_u, sel_w.astype(np.float64), ex, cfg.d, cfg.ffn)


def test_glm_layer_with_ring_refills():
    cfg, T, steps = synth.GLM, 16, 3
    W = synth.router_weights(cfg.seed, cfg.E, cfg.d)
    b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma)
    res = synth.resident_set(cfg, b)
    n_slots = cfg.resident + cfg.n_ring
    slot_of = synth.slot_table(cfg, res, cfg.resident)
    owner = np.full(n_slots, -1, np.int32)
    owner[slot_of[res]] = res
    b = synth.drifted_bias(cfg, b)                        # the tide moved: misses happen
    arena = _arena(cfg, n_slots, owner)
    buf = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, n_slots)
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    Wd, bd = to_dev(W), to_dev(b)
    demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    ring_ptr = 0
    for step in range(steps):
        if step > 0:                                      # refill the ring between steps
            cand = synth.ring_candidates(cfg, step, slot_of, cfg.n_ring)
            slots = []
            for f in cand:
                rs = cfg.resident + ring_ptr % cfg.n_ring
                ring_ptr += 1
                moe.moe_ring_install(so_d, ow_d, rs, int(f))
                assert oracle.ring_install(slot_of, owner, rs, int(f)) == 0
                slots.append(rs)
            _fill(arena, cfg, slots, cand)
            torch.cuda.synchronize()
            assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
            assert moe.moe_device_status() == (moe.MOE_OK, 0)
        x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=200 + step)
        out = layer_step(hidden_dev(x), Wd, bd, so_d, arena, demand, miss, 0, buf)
        step_end(miss, buf)
        torch.cuda.synchronize()
        ref = oracle.route(x, W, b, slot_of, cfg.k)
        sel, sel_slot = _check_routing(ref, buf, slot_of, cfg.k, cfg.E)
        if step > 0:
            assert (sel_slot >= cfg.resident).any()       # ring experts are routed to
        rows = np.arange(0, T, 5)
        exp = _oracle_ffn(cfg, x[rows], sel_slot[rows], buf.sel_w.cpu().numpy()[rows], owner)
        ok, fro, mx = ffn_within_tolerance(out.cpu().numpy()[rows].astype(np.float64), exp)
        assert ok, (step, fro, mx)
    del arena


def _route_matches(ref, got, slot_of, k, E):
    """Routing of one layer call (`got`: want_e, sel_e, sel_slot as numpy) against the oracle's: ranks clear of
    their neighbours by more than 1e-5 relative in order, the whole pick sets away from the k-th / (k+1)-th
    near-ties, and the slots of the GPU's picks from the table."""
    want, sel, slot = got
    tie_s = near_tie_tokens(ref["scores"], slot_of >= 0, k)
    tie_w = near_tie_tokens(ref["scores"], np.ones(E, bool), k)
    for t in range(sel.shape[0]):
        if not tie_w[t]:
            assert set(want[t]) == set(ref["want_e"][t])
        if not tie_s[t]:
            assert set(sel[t]) == set(ref["sel_e"][t])
        for ge, re_, mask in ((want, ref["want_e"], np.ones(E, bool)), (sel, ref["sel_e"], slot_of >= 0)):
            clear = clear_ranks(ref["scores"][t], mask, k)
            assert np.array_equal(ge[t][clear], re_[t][clear])
        assert np.array_equal(slot[t], np.where(sel[t] >= 0, slot_of[np.maximum(sel[t], 0)], -1))
    return tie_w


def test_full_decode_256_step_history_and_replan():
    """The full decode step as configured: 60 layers of 256 experts share one arena of 10,000 main + 64 ring
    slots (a seeded sample of the 15,360 experts at first); each step routes 2 tokens through every layer,
    records demand, takes the step's heavy-miss list and installs it in the ring (README item 3). After 256
    steps the arena is re-planned from the accumulated demand history (README item 1).

    Checked against the oracle: every layer call's routing (on the table the GPU used that step, so near-ties
    cannot cascade), every step's heavy-miss list, the demand table after 256 steps, FFN outputs at a few
    (step, layer) points, the re-plan bit-exact (on the GPU's table) and as a resident set (on the oracle's own
    demand), and one routed layer on the re-planned arena."""
    cfg, T, steps = synth.FULL, 2, 256
    L, E, k = cfg.L, cfg.E, cfg.k
    n_slots = cfg.n_main + cfg.n_ring
    slot_of, owner = synth.full_initial_arena(cfg)
    Ws = [synth.router_weights(cfg.seed, E, cfg.d, layer) for layer in range(L)]
    bs = [synth.router_bias(cfg.seed, E, cfg.sigma, layer) for layer in range(L)]
    arena = _arena(cfg, n_slots, owner)
    W_d = to_dev(np.stack(Ws))
    b_d = to_dev(np.stack(bs))
    so_d, ow_d = to_dev(slot_of), to_dev(owner)
    demand = torch.zeros((L, E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((L, E), dtype=torch.float32, device="cuda")
    buf = LayerBuffers(T, k, E, cfg.d, cfg.ffn, n_slots)
    hist = {name: torch.empty((steps, L, T, k), dtype=torch.int32, device="cuda")
            for name in ("want_e", "sel_e", "sel_slot")}
    snaps = np.empty((steps, L * E), np.int32)            # the table each step routed with
    owners = {}                                           # the arena owners at the FFN sample points
    heavy = []
    ring_ptr = 0
    ffn_samples = {(0, 0): None, (97, 31): None, (255, 59): None}
    for step in range(steps):
        snaps[step] = slot_of
        for layer in range(L):
            x = hidden_dev(synth.hidden_bf16(cfg.seed, T, cfg.d, stream=step * L + layer))
            out = layer_step(x, W_d[layer], b_d[layer], so_d[layer * E:(layer + 1) * E], arena, demand, miss,
                             layer, buf)
            for name in hist:
                hist[name][step, layer].copy_(getattr(buf, name))
            if (step, layer) in ffn_samples:
                ffn_samples[(step, layer)] = (out.clone(), buf.sel_slot.clone(), buf.sel_w.clone())
                owners[(step, layer)] = owner.copy()
        flat, share, n = step_end(miss, buf)
        torch.cuda.synchronize()
        got = [int(f) for f in flat.cpu().numpy()[:int(n.item())]]
        heavy.append(got)
        slots = []
        for f in got:                                     # the step's heavy misses go into the ring
            rs = cfg.n_main + ring_ptr % cfg.n_ring
            ring_ptr += 1
            moe.moe_ring_install(so_d, ow_d, rs, f)
            assert oracle.ring_install(slot_of, owner, rs, f) == 0
            slots.append(rs)
        if slots:
            _fill(arena, cfg, slots, got)
    torch.cuda.synchronize()
    assert np.array_equal(so_d.cpu().numpy(), slot_of) and np.array_equal(ow_d.cpu().numpy(), owner)
    assert ring_ptr > cfg.n_ring                          # the ring wrapped: evictions happened
    assert moe.moe_device_status() == (moe.MOE_OK, 0)

    # the oracle routes every (step, layer) call on the table of that step, on several host cores
    jobs = [(layer, step * L + layer, T, snaps[step, layer * E:(layer + 1) * E], False)
            for step in range(steps) for layer in range(L)]
    refs = oracle_pool.route_layers(cfg, jobs)
    H = {name: v.cpu().numpy() for name, v in hist.items()}
    Dref = np.zeros((L, E))
    adds = np.zeros((L, E))
    n_ties = 0
    for step in range(steps):
        Mref = np.zeros((L, E))
        for layer in range(L):
            ref = refs[step * L + layer]
            so_l = snaps[step, layer * E:(layer + 1) * E]
            want = H["want_e"][step, layer]
            tie = _route_matches(ref, (want, H["sel_e"][step, layer], H["sel_slot"][step, layer]), so_l, k, E)
            n_ties += int(tie.sum())
            use = np.where(tie[:, None], want, ref["want_e"])     # near-tie tokens keep the GPU's picks
            ws = np.take_along_axis(ref["scores"], use.astype(np.int64), axis=1)
            oracle.demand(use, ws, so_l, layer, Dref, Mref)
            np.add.at(adds[layer], use.ravel(), 1)
        ids_ref, _ = oracle.hot_miss_select(Mref, 0.2, 16)
        cand = np.sort(Mref.ravel()[Mref.ravel() >= 0.2])[::-1] if Mref.any() else np.zeros(0)
        if not (len(cand) > 16 and abs(cand[15] - cand[16]) <= 1e-5 * cand[15]) and \
                not np.any(np.abs(Mref[Mref > 0] - 0.2) <= 2e-6):
            assert heavy[step] == list(ids_ref), (step, heavy[step], list(ids_ref))
    assert n_ties <= steps * L * T // 100
    Dg = demand.cpu().numpy().astype(np.float64) / 2.0 ** 40
    assert np.all(np.abs(Dg - Dref) <= 1e-5 * Dref + adds * 2.0 ** -41 + 1e-15)

    # FFN outputs at the sample points, on the arena as it was then
    for (step, layer), (out, sel_slot, sel_w) in ffn_samples.items():
        x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=step * L + layer)
        exp = _oracle_ffn(cfg, x, sel_slot.cpu().numpy(), sel_w.cpu().numpy(), owners[(step, layer)])
        ok, fro, mx = ffn_within_tolerance(out.cpu().numpy().astype(np.float64), exp)
        assert ok, (step, layer, fro, mx)

    # re-plan the shared arena from the GPU's demand table; the oracle re-plans the same table bit for bit
    so_ref, ow_ref, loads_ref = oracle.replan(Dg * 2.0 ** 40, cfg.n_main, slot_of, owner)
    loads = torch.full((cfg.n_main,), -1, dtype=torch.int32, device="cuda")
    nl = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(moe.moe_replan_workspace_bytes(L, E), dtype=torch.uint8, device="cuda")
    moe.moe_arena_replan(demand, cfg.n_main, so_d, ow_d, loads, nl, ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
    assert np.array_equal(ow_d.cpu().numpy(), ow_ref) and np.array_equal(so_d.cpu().numpy(), so_ref)
    n_loads = int(nl.item())
    assert n_loads == len(loads_ref) > 0
    assert np.array_equal(loads.cpu().numpy()[:n_loads], loads_ref)
    # ... and on the oracle's own demand the same resident set, up to experts whose demand lies within 1e-5 of
    # the last one admitted
    _, ow_own, _ = oracle.replan(Dref, cfg.n_main, slot_of, owner)
    main_gpu = set(int(f) for f in ow_ref[:cfg.n_main] if f >= 0)
    main_own = set(int(f) for f in ow_own[:cfg.n_main] if f >= 0)
    edge = np.sort(Dref.ravel())[::-1][cfg.n_main - 1]
    for f in main_gpu ^ main_own:
        assert abs(Dref.ravel()[f] - edge) <= 1e-5 * edge + 1e-12, f
    _fill(arena, cfg, loads_ref, ow_ref[loads_ref])       # refill the slots given to newcomers

    # one more step on the re-planned arena: routing and FFN of a layer that gained experts
    layer = int(ow_ref[loads_ref[0]]) // E
    x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=steps * L + layer)
    so_l = so_ref[layer * E:(layer + 1) * E]
    out = layer_step(hidden_dev(x), W_d[layer], b_d[layer], so_d[layer * E:(layer + 1) * E], arena, demand, miss,
                     layer, buf)
    torch.cuda.synchronize()
    ref = oracle.route(x, Ws[layer], bs[layer], so_l, k)
    sel, sel_slot = _check_routing(ref, buf, so_l, k, E)
    exp = _oracle_ffn(cfg, x, sel_slot, buf.sel_w.cpu().numpy(), ow_ref)
    ok, fro, mx = ffn_within_tolerance(out.cpu().numpy().astype(np.float64), exp)
    assert ok, (fro, mx)
    del arena
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [8, 130])
def test_side_stream_step_matches_one_stream(T):
    # the demand update and heavy-miss list (with and without the L2 prefetch) on a second stream, forked
    # after routing and joined at the end of the step, eagerly and under CUDA graph capture: every output
    # equals the one-stream step's
    from resident_expert_routed_gb300.layer import join
    cfg = synth.TINY
    x = [hidden_dev(synth.hidden_bf16(cfg.seed, T, cfg.d, stream=s)) for s in range(3)]
    W, b = to_dev(synth.router_weights(cfg.seed, cfg.E, cfg.d)), to_dev(synth.router_bias(cfg.seed, cfg.E, cfg.sigma))
    res = synth.resident_set(cfg, synth.router_bias(cfg.seed, cfg.E, cfg.sigma))
    n_slots = cfg.resident
    slot_of = synth.slot_table(cfg, res, n_slots)
    owner = np.full(n_slots, -1, np.int32)
    owner[slot_of[res]] = res
    arena = _arena(cfg, n_slots, owner)
    so = to_dev(slot_of)

    def run(side, graph, prefetch=False):
        buf = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, n_slots)
        demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
        miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
        hidden = torch.empty_like(x[0])
        main = torch.cuda.Stream()
        outs = []

        def step():
            layer_step(hidden, W, b, so, arena, demand, miss, 0, buf, main, side, prefetch=prefetch)
            step_end(miss, buf, 0.2, main if side is None else side)
            if side is not None:
                join(main, side)

        g = None
        if graph:
            hidden.copy_(x[0])
            torch.cuda.synchronize()
            with torch.cuda.stream(main):
                step()                                    # warm-up outside the capture
            main.synchronize()
            demand.zero_()
            miss.zero_()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                step()
        for i in range(3):
            torch.cuda.synchronize()
            hidden.copy_(x[i])
            torch.cuda.synchronize()
            if g is not None:
                g.replay()
            else:
                with torch.cuda.stream(main):
                    step()
            torch.cuda.synchronize()
            n = int(buf.hot_n.item())
            outs.append((buf.out.cpu().clone(), buf.sel_slot.cpu().clone(), demand.cpu().clone(), miss.cpu().clone(),
                         buf.hot_flat.cpu()[:n].clone()))
        return outs

    ref = run(None, False)
    for graph, prefetch in ((False, False), (True, False), (False, True), (True, True)):
        got = run(torch.cuda.Stream(), graph, prefetch)
        for r, g in zip(ref, got):
            for a, c in zip(r, g):
                assert torch.equal(a, c)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)


@pytest.mark.parametrize("zero_copy", [True, False], ids=["zero-copy", "copies"])
def test_captured_step_matches_eager_steps(zero_copy):
    # CapturedStep (the batch read from pinned host memory by the kernels, or copied in and out by the graph,
    # around the two-stream step, one CUDA graph per host buffer): its host output, demand and miss tables and
    # heavy-miss list equal those of eager one-stream steps on device copies of the same batches
    from resident_expert_routed_gb300.layer import CapturedStep
    cfg, T = synth.TINY, 40
    xs = [synth.hidden_bf16(cfg.seed, T, cfg.d, stream=s) for s in range(3)]
    host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs]
    W, b = to_dev(synth.router_weights(cfg.seed, cfg.E, cfg.d)), to_dev(synth.router_bias(cfg.seed, cfg.E, cfg.sigma))
    res = synth.resident_set(cfg, synth.router_bias(cfg.seed, cfg.E, cfg.sigma))
    slot_of = synth.slot_table(cfg, res, cfg.resident)
    owner = np.full(cfg.resident, -1, np.int32)
    owner[slot_of[res]] = res
    arena = _arena(cfg, cfg.resident, owner)
    so = to_dev(slot_of)

    def tables():
        return (torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda"),
                torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda"))

    # eager: the capture's own warm-up step (batch 0), then batches 1, 2, 0
    buf_e = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, cfg.resident)
    dem_e, miss_e = tables()
    ref = []
    for i in (0, 1, 2, 0):
        layer_step(hidden_dev(xs[i]), W, b, so, arena, dem_e, miss_e, 0, buf_e)
        step_end(miss_e, buf_e, 0.2)
        torch.cuda.synchronize()
        n = int(buf_e.hot_n.item())
        ref.append((buf_e.out.cpu().clone(), dem_e.cpu().clone(), miss_e.cpu().clone(), buf_e.hot_flat.cpu()[:n].clone()))

    buf_c = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, cfg.resident)
    dem_c, miss_c = tables()
    cap = CapturedStep(host, W, b, so, arena, dem_c, miss_c, 0, buf_c, zero_copy=zero_copy)
    got = []
    torch.cuda.synchronize()
    n = int(buf_c.hot_n.item())
    got.append((cap.host_out.clone(), dem_c.cpu().clone(), miss_c.cpu().clone(), buf_c.hot_flat.cpu()[:n].clone()))
    for i in (1, 2, 0):
        out = cap.run(i)
        torch.cuda.synchronize()
        n = int(buf_c.hot_n.item())
        got.append((out.clone(), dem_c.cpu().clone(), miss_c.cpu().clone(), buf_c.hot_flat.cpu()[:n].clone()))
    for r, g in zip(ref, got):
        for a, c in zip(r, g):
            assert torch.equal(a, c)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)
