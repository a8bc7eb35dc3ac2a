"""Routing for callers that cannot allocate device memory.

Some users of this library route from places where they may not allocate:
a serving loop that fixed its device-memory budget when it started, or a
plug-in whose host framework owns every allocation (and a cudaMalloc can
also synchronise the device at a bad moment). moe_route_resident_noalloc
serves them: it takes no workspace and keeps its partial logits in a fixed
array inside the library. These checks call it through the C ABI and hold
its results to those of moe_route_resident on the same inputs and to the
oracle's, on two calls in a row (the fixed array is reused and keeps the
previous call's data), from device memory and from page-locked host memory.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.cases import clear_ranks, hidden_dev, make_case, near_tie_tokens, to_dev

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


def _against_oracle(c, got):
    """The no-allocation call's picks against the oracle's: ordered at every rank clear of its neighbours by
    more than 1e-5 relative, as sets away from the k-th / (k+1)-th near-ties; scores within 1e-5."""
    cfg = c.cfg
    ref = oracle.route(c.x, c.W, c.bias, c.slot_of, cfg.k)
    want_e, want_s, sel_e, sel_slot, sel_w = (a.cpu().numpy() for a in got)
    resident = c.slot_of >= 0
    tie_w = near_tie_tokens(ref["scores"], np.ones(cfg.E, bool), cfg.k)
    tie_s = near_tie_tokens(ref["scores"], resident, cfg.k)
    for t in range(c.x.shape[0]):
        s = ref["scores"][t]
        if not tie_w[t]:
            assert set(want_e[t]) == set(ref["want_e"][t]), t
        if not tie_s[t]:
            assert set(sel_e[t]) == set(ref["sel_e"][t]), t
        for ge, re_, mask in ((want_e, ref["want_e"], np.ones(cfg.E, bool)), (sel_e, ref["sel_e"], resident)):
            clear = clear_ranks(s, mask, cfg.k)
            assert np.array_equal(ge[t][clear], re_[t][clear]), t
        assert np.allclose(want_s[t], s[want_e[t]], rtol=1e-5, atol=0)
        v = sel_e[t] >= 0
        assert np.allclose(sel_w[t][v], s[sel_e[t][v]], rtol=1e-5, atol=0)
        assert np.array_equal(sel_slot[t], np.where(v, c.slot_of[np.maximum(sel_e[t], 0)], -1))


@pytest.mark.parametrize("cfg,T", [(synth.DECODE, 64), (synth.DECODE, 2), (synth.TINY, 8)],
                         ids=["decode-T64", "decode-T2", "tiny-T8"])
def test_noalloc_matches_the_oracle(cfg, T):
    for call in range(2):
        c = make_case(cfg, T, stream=50 + call, drift=True)
        got = _outputs(T, cfg.k)
        moe.moe_route_resident_noalloc(hidden_dev(c.x), to_dev(c.W), to_dev(c.bias), to_dev(c.slot_of), cfg.k, *got)
        torch.cuda.synchronize()
        _against_oracle(c, got)


def test_noalloc_pinned_host_batch():
    # a 2-token batch in page-locked host memory: the call has no workspace to copy it into, so the K-sliced
    # router reads it in place (the workspace call copies such a batch to the device first and sums each row
    # whole); the picks agree with the oracle and with the workspace call away from near-ties
    cfg, T = synth.DECODE, 2
    for call in range(2):
        c = make_case(cfg, T, stream=60 + call, drift=(call == 1))
        host_x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        got = _outputs(T, cfg.k)
        moe.moe_route_resident_noalloc(host_x, to_dev(c.W), to_dev(c.bias), to_dev(c.slot_of), cfg.k, *got)
        torch.cuda.synchronize()
        _against_oracle(c, got)
        ref = _outputs(T, cfg.k)
        ws = torch.empty(moe.moe_workspace_bytes(T, cfg.k, cfg.d, cfg.ffn, cfg.E, c.n_slots),
                         dtype=torch.uint8, device="cuda")
        moe.moe_route_resident(host_x, to_dev(c.W), to_dev(c.bias), to_dev(c.slot_of), cfg.k, *ref, ws)
        torch.cuda.synchronize()
        for a, b in ((got[1], ref[1]), (got[4], ref[4])):        # each token's scores, 1e-5 relative
            assert np.allclose(np.sort(a.cpu().numpy(), axis=1), np.sort(b.cpu().numpy(), axis=1), rtol=1e-5, atol=0)
    assert moe.moe_device_status() == (moe.MOE_OK, 0)


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
