"""Edge cases of the layer step on the GPU, against the oracle, through the C ABI.

The sizes at the documented limits (E = 1024 and k = 32 for routing; d and
ffn of 16384 and T*k = 2^20 picks for the FFN) and the degenerate residencies
the method has: every expert resident (the resident picks are plain top-k)
and none resident (every pick is padding, the output is zero, all demand is
missed demand).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.cases import device_arena, ffn_within_tolerance, make_case, oracle_experts, to_dev
from tests.test_gpu_parity import check_route, gpu_ffn, gpu_route

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")

WIDE = synth.LayerConfig("wide E1024 k32 d256 F128 R600", E=1024, k=32, d=256, ffn=128, resident=600, sigma=1.0,
                         seed=0x7EED00B0)
HALF = synth.LayerConfig("half E512 k16 d256 F128 R300", E=512, k=16, d=256, ffn=128, resident=300, sigma=1.0,
                         seed=0x7EED00B1)
ALL = synth.LayerConfig("all-resident E64 k8 d256 F128 R64", E=64, k=8, d=256, ffn=128, resident=64, sigma=1.0,
                        seed=0x7EED00B2)
DEEP = synth.LayerConfig("deep d16384 E8 k2 F128 R8", E=8, k=2, d=16384, ffn=128, resident=8, sigma=1.0,
                         seed=0x7EED00B3)
BROAD = synth.LayerConfig("broad d128 E8 k2 F16384 R8", E=8, k=2, d=128, ffn=16384, resident=8, sigma=1.0,
                          seed=0x7EED00B4)


@pytest.mark.parametrize("cfg,T", [(WIDE, 16), (WIDE, 130), (HALF, 40), (HALF, 200)],
                         ids=["E1024k32-T16", "E1024k32-T130", "E512k16-T40", "E512k16-T200"])
def test_route_at_the_expert_and_pick_limits(cfg, T):
    c = make_case(cfg, T)
    g = gpu_route(c)
    check_route(c, g, np.arange(T))


def test_every_expert_resident_gives_plain_topk():
    c = make_case(ALL, 50)
    g = gpu_route(c)
    ref = check_route(c, g, np.arange(50))
    for t in range(50):
        assert set(g["sel_e"][t]) == set(g["want_e"][t])
        order = np.argsort(g["sel_e"][t])
        assert np.array_equal(g["sel_w"][t][order], g["want_s"][t][np.argsort(g["want_e"][t])])
    # no pick is a miss: the miss shares stay zero and the heavy-miss list is empty
    miss = torch.zeros((1, ALL.E), dtype=torch.float32, device="cuda")
    demand = torch.zeros((1, ALL.E), dtype=torch.int64, device="cuda")
    moe.moe_demand_accumulate(to_dev(g["want_e"]), to_dev(g["want_s"]), to_dev(c.slot_of), 0, demand, miss)
    torch.cuda.synchronize()
    assert not miss.any()
    assert np.allclose(demand.cpu().numpy().astype(np.float64).sum() / 2.0 ** 40, ref["want_s"].sum(), rtol=1e-5)


def test_no_expert_resident():
    cfg, T = synth.TINY, 8
    c = make_case(cfg, T)
    c.slot_of[:] = -1
    owner = np.full(1, -1, np.int32)                       # one empty slot
    arena = device_arena(cfg, owner, 1)
    g = gpu_route(c)
    ref = oracle.route(c.x, c.W, c.bias, c.slot_of, cfg.k)
    assert np.all(g["sel_e"] == -1) and np.all(g["sel_slot"] == -1) and np.all(g["sel_w"] == 0)
    assert np.array_equal(np.sort(g["want_e"], 1), np.sort(ref["want_e"], 1))
    out = gpu_ffn(c, arena, g["sel_slot"], g["sel_w"])
    assert np.all(out == 0)
    # every wanted pick is missed demand; the heavy-miss list is the oracle's
    demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_demand_accumulate(to_dev(g["want_e"]), to_dev(g["want_s"]), to_dev(c.slot_of), 0, demand, miss)
    flat = torch.zeros(16, dtype=torch.int32, device="cuda")
    share = torch.zeros(16, dtype=torch.float32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_hot_miss_select(miss, 0.2, 16, flat, share, n)
    torch.cuda.synchronize()
    D = np.zeros((1, cfg.E))
    M = np.zeros((1, cfg.E))
    oracle.demand(ref["want_e"], ref["want_s"], c.slot_of, 0, D, M)
    ids, _ = oracle.hot_miss_select(M, 0.2, 16)
    assert list(flat.cpu().numpy()[:int(n.item())]) == list(ids)
    assert np.allclose(demand.cpu().numpy().astype(np.float64) / 2.0 ** 40, D, rtol=1e-5, atol=T * cfg.k * 2.0 ** -40)


@pytest.mark.parametrize("cfg,T", [(DEEP, 4), (DEEP, 80), (BROAD, 4), (BROAD, 80)],
                         ids=["d16384-T4", "d16384-T80", "F16384-T4", "F16384-T80"])
def test_ffn_at_the_largest_d_and_ffn(cfg, T):
    c = make_case(cfg, T)
    arena = device_arena(cfg, c.owner, c.n_slots)
    ref = oracle.route(c.x, c.W, c.bias, c.slot_of, cfg.k)
    got = gpu_ffn(c, arena, ref["sel_slot"], ref["sel_w"].astype(np.float32))
    sel_u, experts = oracle_experts(cfg, c.owner, ref["sel_slot"])
    exp = oracle.ffn(c.x, sel_u, ref["sel_w"].astype(np.float32).astype(np.float64), experts, cfg.d, cfg.ffn)
    ok, fro, mx = ffn_within_tolerance(got, exp)
    assert ok, (fro, mx)


def test_ffn_at_the_pick_limit():
    # T * k = 2^20 picks, the largest FFN call; the oracle checks a seeded sample of tokens
    cfg, T = synth.TINY, 1 << 18
    c = make_case(cfg, T)
    arena = device_arena(cfg, c.owner, c.n_slots)
    g = gpu_route(c)
    got = gpu_ffn(c, arena, g["sel_slot"], g["sel_w"])
    rows = np.sort(synth.seeded_permutation(13, synth.T_SAMPLE, T, T)[:24])
    sel_u, experts = oracle_experts(cfg, c.owner, g["sel_slot"][rows])
    exp = oracle.ffn(c.x[rows], sel_u, g["sel_w"][rows].astype(np.float64), experts, cfg.d, cfg.ffn)
    ok, fro, mx = ffn_within_tolerance(got[rows], exp)
    assert ok, (fro, mx)
