"""Routing for callers that cannot allocate device memory.

Some users of this library route from places where they may not allocate:
a serving loop that fixed its device-memory budget when it started, or a
plug-in whose host framework owns every allocation (and a cudaMalloc can
also synchronise the device at a bad moment). moe_route_resident_noalloc
serves them: it takes no workspace and keeps its partial logits in a fixed
array inside the library. These checks call it through the C ABI and hold
its results to those of moe_route_resident on the same inputs, on two calls
in a row (the fixed array is reused and keeps the previous call's data).
"""
import numpy as np
import pytest
import torch

import synth
from tests.cases import hidden_dev, make_case, to_dev

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("resident_expert_routed_gb300")


def _outputs(T, k):
    return [torch.full((T, k), -3, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -3.0, dtype=torch.float32, device="cuda"),
            torch.full((T, k), -3, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -3, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -3.0, dtype=torch.float32, device="cuda")]


@pytest.mark.parametrize("cfg,T", [(synth.DECODE, 64), (synth.DECODE, 1), (synth.TINY, 8)],
                         ids=["decode-T64", "decode-T1", "tiny-T8"])
def test_noalloc_matches_workspace_routing_twice(cfg, T):
    for call in range(2):                      # second call reuses the library's array
        c = make_case(cfg, T, stream=40 + call, drift=(call == 1))
        args = (hidden_dev(c.x), to_dev(c.W), to_dev(c.bias), to_dev(c.slot_of), cfg.k)
        ref = _outputs(T, cfg.k)
        ws = torch.empty(moe.moe_workspace_bytes(T, cfg.k, cfg.d, cfg.ffn, cfg.E, c.n_slots),
                         dtype=torch.uint8, device="cuda")
        moe.moe_route_resident(*args, *ref, ws)
        got = _outputs(T, cfg.k)
        moe.moe_route_resident_noalloc(*args, *got)
        torch.cuda.synchronize()
        for name, a, b in zip(("want_e", "want_s", "sel_e", "sel_slot", "sel_w"), got, ref):
            a, b = a.cpu().numpy(), b.cpu().numpy()
            if a.dtype == np.int32:
                assert np.array_equal(a, b), (call, name)                        # indices: bit-exact
            else:
                assert np.allclose(a, b, rtol=1e-5, atol=0), (call, name)        # scores: 1e-5 relative


def test_noalloc_rejects_partials_beyond_the_fixed_array():
    # prefill-sized routing needs 8192 x 256 partial logits, more than the 2^20 the array holds
    cfg, T = synth.PREFILL, 8192
    x = torch.zeros((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((cfg.E, cfg.d), dtype=torch.float32, device="cuda")
    slot_of = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    outs = _outputs(T, cfg.k)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_resident_noalloc(x, W, None, slot_of, cfg.k, *outs)
    assert ei.value.status == moe.MOE_EUNSUPPORTED
    torch.cuda.synchronize()
    assert bool((outs[2] == -3).all())                                         # nothing was launched
