"""Oracle for the resident-expert routed MoE layer (TEST INFRASTRUCTURE ONLY).

A plain, slow, single-threaded C++ float64 implementation (``oracle.cpp``)
behind a ctypes wrapper. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. It shares no code with the
CUDA library in ``resident_expert_routed_gb300``; inputs come from ``synth``.

Each wrapper names the passage of the TideLM README ("How adaptive expert
loading works") or of the OCP MX v1.0 spec that its C function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp with g++ (-O2, strict IEEE: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double


def _declare(L):
    L.or_e2m1_value.restype = _D
    L.or_e2m1_value.argtypes = [_I]
    L.or_e8m0_value.restype = _D
    L.or_e8m0_value.argtypes = [_I]
    L.or_quantise_mxfp4.argtypes = [_P, _I, _P, _P]
    L.or_dequantise_mxfp4.argtypes = [_P, _P, _I, _P]
    L.or_router.argtypes = [_P, _P, _P, _I, _I, _I, _P, _P]
    L.or_topk.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P]
    L.or_demand.argtypes = [_P, _P, _P, _I, _I, _I, _I, _P, _P]
    L.or_hot_miss_select.argtypes = [_P, _I, _I, _D, _I, _P, _P, _P]
    L.or_demand_decay_fixed.argtypes = [_P, ctypes.c_int64, _D]
    L.or_hot_read_choose.argtypes = [_P, _P, _P, _P, _I, _D, _I, _P]
    L.or_renormalise.argtypes = [_P, _P, _I, _I]
    L.or_expert_pair.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    L.or_ffn.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    L.or_replan.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P]
    L.or_ring_install.restype = _I
    L.or_ring_install.argtypes = [_P, _P, _I, _I]


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ formats (OCP MX v1.0)

def e2m1_value(code: int) -> float:
    return lib().or_e2m1_value(int(code))


def e8m0_value(byte: int) -> float:
    return lib().or_e8m0_value(int(byte))


def quantise_mxfp4(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 of a float64 vector (len % 32 == 0) -> (codes uint8 [n/2], scales uint8 [n/32])."""
    v = _c(v, np.float64).ravel()
    n = v.size
    codes = np.zeros(n // 2, np.uint8)
    scales = np.zeros(n // 32, np.uint8)
    lib().or_quantise_mxfp4(_ptr(v), n, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantise_mxfp4(codes: np.ndarray, scales: np.ndarray, n: int) -> np.ndarray:
    codes = _c(codes, np.uint8).ravel()
    scales = _c(scales, np.uint8).ravel()
    out = np.zeros(n, np.float64)
    lib().or_dequantise_mxfp4(_ptr(codes), _ptr(scales), n, _ptr(out))
    return out


# ------------------------------------------------------------------ routing (README item 1-2)

def router(x_bf16: np.ndarray, W: np.ndarray, bias: Optional[np.ndarray]):
    """(logits f64 [T,E], scores f64 [T,E]) for bf16-bit hidden [T,d], fp32 W [E,d], fp32 bias [E]."""
    x = _c(x_bf16, np.uint16)
    W = _c(W, np.float32)
    T, d = x.shape
    E = W.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    logits = np.zeros((T, E), np.float64)
    scores = np.zeros((T, E), np.float64)
    lib().or_router(_ptr(x), _ptr(W), _ptr(b), T, d, E, _ptr(logits), _ptr(scores))
    return logits, scores


def topk(scores: np.ndarray, slot_of: np.ndarray, k: int) -> dict:
    """Wanted top-k over all E and resident top-k with substitution (README item 2)."""
    s = _c(scores, np.float64)
    T, E = s.shape
    so = _c(slot_of, np.int32)
    out = dict(want_e=np.zeros((T, k), np.int32), want_s=np.zeros((T, k), np.float64),
               sel_e=np.zeros((T, k), np.int32), sel_slot=np.zeros((T, k), np.int32),
               sel_w=np.zeros((T, k), np.float64))
    lib().or_topk(_ptr(s), _ptr(so), T, E, k, _ptr(out["want_e"]), _ptr(out["want_s"]),
                  _ptr(out["sel_e"]), _ptr(out["sel_slot"]), _ptr(out["sel_w"]))
    return out


def route(x_bf16, W, bias, slot_of, k) -> dict:
    logits, scores = router(x_bf16, W, bias)
    out = topk(scores, slot_of, k)
    out["logits"] = logits
    out["scores"] = scores
    return out


def demand(want_e, want_s, slot_of, layer: int, D: np.ndarray, M: np.ndarray) -> None:
    """In place: D[layer, e] += s for wanted picks; M = max share of non-resident picks (README item 1, 3)."""
    we = _c(want_e, np.int32)
    ws = _c(want_s, np.float64)
    so = _c(slot_of, np.int32)
    assert D.dtype == np.float64 and D.flags.c_contiguous and M.dtype == np.float64 and M.flags.c_contiguous
    T, k = we.shape
    E = D.shape[-1]
    lib().or_demand(_ptr(we), _ptr(ws), _ptr(so), T, k, layer, E, _ptr(D), _ptr(M))


def demand_decay_fixed(D: np.ndarray, factor: float) -> np.ndarray:
    """The stored demand table (uint64, units of 2^-40) after forgetting with `factor` (a new array)."""
    out = np.ascontiguousarray(D, dtype=np.uint64).copy()
    lib().or_demand_decay_fixed(_ptr(out), out.size, float(factor))
    return out


def renormalise(sel_slot, sel_w) -> np.ndarray:
    """Combine weights renormalised over each token's valid picks (a new float64 [T, k] array)."""
    so = _c(sel_slot, np.int32)
    w = np.ascontiguousarray(sel_w, dtype=np.float64).copy()
    T, k = so.shape
    lib().or_renormalise(_ptr(so), _ptr(w), T, k)
    return w


def hot_read_choose(M, D, slot_of, in_store, threshold: float = 0.2, budget: int = 1) -> tuple[int, int]:
    """(expert read, coldest resident it replaces) for one layer's synchronous hot read, or (-1, -1)."""
    Mc, Dc = _c(M, np.float64), _c(D, np.float64)
    so = _c(slot_of, np.int32)
    st = _c(np.asarray(in_store).astype(np.uint8), np.uint8)
    out = np.zeros(2, np.int32)
    lib().or_hot_read_choose(_ptr(Mc), _ptr(Dc), _ptr(so), _ptr(st), Mc.size, float(threshold), int(budget), _ptr(out))
    return int(out[0]), int(out[1])


def hot_miss_select(M: np.ndarray, threshold: float = 0.2, cap: int = 16):
    """(flat ids, shares) of the heavy misses; resets M to zero (README item 3)."""
    assert M.dtype == np.float64 and M.flags.c_contiguous
    L, E = M.shape
    flat = np.zeros(max(cap, 1), np.int32)
    share = np.zeros(max(cap, 1), np.float64)
    n = np.zeros(1, np.int32)
    lib().or_hot_miss_select(_ptr(M), L, E, float(threshold), cap, _ptr(flat), _ptr(share), _ptr(n))
    return flat[:n[0]].copy(), share[:n[0]].copy()


# ------------------------------------------------------------------ expert FFN

def expert_pair(x_row_bf16: np.ndarray, w: dict, d: int, F: int) -> dict:
    """One (token, expert) pair: y [d] plus the intermediate xq, h, hq (README profile table: MXFP4 experts)."""
    x = _c(x_row_bf16, np.uint16).ravel()
    y = np.zeros(d, np.float64)
    xq_c = np.zeros(d // 2, np.uint8)
    xq_s = np.zeros(d // 32, np.uint8)
    h = np.zeros(F, np.float64)
    hq_c = np.zeros(F // 2, np.uint8)
    hq_s = np.zeros(F // 32, np.uint8)
    g = {kk: _c(v, np.uint8) for kk, v in w.items()}
    lib().or_expert_pair(_ptr(x), d, F, _ptr(g["gu_codes"]), _ptr(g["gu_scales"]),
                         _ptr(g["dn_codes"]), _ptr(g["dn_scales"]), _ptr(y),
                         _ptr(xq_c), _ptr(xq_s), _ptr(h), _ptr(hq_c), _ptr(hq_s))
    return dict(y=y, xq_codes=xq_c, xq_scales=xq_s, h=h, hq_codes=hq_c, hq_scales=hq_s)


def ffn(x_bf16: np.ndarray, sel_u: np.ndarray, sel_w: np.ndarray, experts: list, d: int, F: int) -> np.ndarray:
    """out [T,d] f64 = sum_j sel_w[t,j] * y(t, experts[sel_u[t,j]]), j in rank order."""
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    su = _c(sel_u, np.int32)
    k = su.shape[1]
    sw = _c(sel_w, np.float64)
    if len(experts) == 0:
        experts = [dict(gu_codes=np.zeros((2 * F, d // 2), np.uint8), gu_scales=np.zeros((2 * F, d // 32), np.uint8),
                        dn_codes=np.zeros((d, F // 2), np.uint8), dn_scales=np.zeros((d, F // 32), np.uint8))]
    gc = _c(np.stack([e["gu_codes"] for e in experts]), np.uint8)
    gs = _c(np.stack([e["gu_scales"] for e in experts]), np.uint8)
    dc = _c(np.stack([e["dn_codes"] for e in experts]), np.uint8)
    ds = _c(np.stack([e["dn_scales"] for e in experts]), np.uint8)
    out = np.zeros((T, d), np.float64)
    lib().or_ffn(_ptr(x), _ptr(su), _ptr(sw), T, k, d, F, len(experts), _ptr(gc), _ptr(gs), _ptr(dc), _ptr(ds), _ptr(out))
    return out


# ------------------------------------------------------------------ arena (README item 1, 3)

def replan(D: np.ndarray, n_main: int, slot_of: np.ndarray, owner: np.ndarray):
    """Returns (slot_of', owner', loads) after the shared-arena re-plan."""
    Dc = _c(D, np.float64)
    L, E = Dc.shape
    so = _c(slot_of, np.int32).copy()
    ow = _c(owner, np.int32).copy()
    loads = np.zeros(max(n_main, 1), np.int32)
    nl = np.zeros(1, np.int32)
    lib().or_replan(_ptr(Dc), L, E, n_main, ow.size, _ptr(so), _ptr(ow), _ptr(loads), _ptr(nl))
    return so, ow, loads[:nl[0]].copy()


def ring_install(slot_of: np.ndarray, owner: np.ndarray, ring_slot: int, flat: int) -> int:
    """In place; returns 1 when `flat` was already resident (nothing changed)."""
    assert slot_of.dtype == np.int32 and owner.dtype == np.int32
    return lib().or_ring_install(_ptr(slot_of), _ptr(owner), int(ring_slot), int(flat))
