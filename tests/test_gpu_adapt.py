"""Demand history on the GPU: forgetting (fixed point) and persistence, through the C ABI.

The TideLM README keeps the demand history over restarts, and a setting there
controls how quickly the resident set tracks a change in traffic. Decay is
checked bit-exact against the oracle's fixed-point restatement; save and load
round-trip the table through the documented file format.
"""
import struct

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")


def _table(L, E, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 2**62, (L, E), dtype=np.uint64)


@pytest.mark.parametrize("factor", [1.0, 0.0, 0.5, 0.9, 0.123456, 0.999])
def test_demand_decay_matches_oracle(factor):
    D = _table(60, 256, 1)
    dev = torch.from_numpy(D.view(np.int64)).cuda()
    moe.moe_demand_decay(dev, factor)
    torch.cuda.synchronize()
    got = dev.cpu().numpy().view(np.uint64)
    assert np.array_equal(got, oracle.demand_decay_fixed(D, np.float32(factor)))


def test_demand_save_load_round_trip(tmp_path):
    D = _table(60, 256, 2)
    dev = torch.from_numpy(D.view(np.int64)).cuda()
    path = str(tmp_path / "demand.bin")
    moe.moe_demand_save(dev, path)
    raw = open(path, "rb").read()
    assert raw[:8] == b"MOEDEMD1" and struct.unpack("<iiii", raw[8:24]) == (60, 256, 40, 0)
    assert np.array_equal(np.frombuffer(raw[24:], dtype="<u8").reshape(60, 256), D)
    back = torch.zeros_like(dev)
    moe.moe_demand_load(back, path)
    torch.cuda.synchronize()
    assert torch.equal(back, dev)
    wrong = torch.zeros((59, 256), dtype=torch.int64, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_demand_load(wrong, path)
    assert ei.value.status == moe.MOE_EINVAL
    assert not wrong.any()


def test_renormalise_weights_matches_oracle():
    from tests.cases import make_case
    from tests.test_gpu_parity import gpu_route
    import synth
    for cfg, T in ((synth.DECODE, 64), (synth.TINY, 8)):
        c = make_case(cfg, T, drift=True)
        g = gpu_route(c)
        so = torch.from_numpy(g["sel_slot"]).cuda()
        w = torch.from_numpy(g["sel_w"]).cuda()
        moe.moe_renormalise_weights(so, w)
        torch.cuda.synchronize()
        ref = oracle.renormalise(g["sel_slot"], g["sel_w"].astype(np.float64))
        assert np.allclose(w.cpu().numpy(), ref, rtol=2e-6, atol=0)
