"""Resident-expert routed MoE layer step on GB300 (sm_103a): Python binding.

Same names as the C ABI in ``include/moe_resident.h``. This module only
marshals arguments (torch tensors -> device pointers and sizes) and raises on a
non-OK status; every step of the computation runs in the CUDA kernels of
``libmoe_resident.so``. There is no CPU path: importing this package without
the built library raises.

The method is the adaptive expert loading of the TideLM README ("How adaptive
expert loading works", items 1-3): routing restricted to resident experts with
next-best substitution, score-weighted demand per (layer, expert), heavy-miss
extraction for the hot-read ring, and the grouped MXFP4 SwiGLU expert FFN over
one shared slot arena.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_resident.so")

MOE_OK, MOE_EINVAL, MOE_ECUDA, MOE_ENOMEM, MOE_ETIMEOUT, MOE_EDEVICE, MOE_EUNSUPPORTED, MOE_EIO = range(8)
MOE_DEV_BAD_SLOT, MOE_DEV_NAN_SCALE, MOE_DEV_TIMEOUT, MOE_DEV_BAD_TABLE, MOE_DEV_RESIDENT = 0x1, 0x2, 0x4, 0x8, 0x10

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("moe_route_resident", "moe_route_resident_noalloc", "moe_demand_accumulate", "moe_hot_miss_select", "moe_expert_ffn_mxfp4",
           "moe_arena_replan", "moe_ring_install", "moe_workspace_bytes", "moe_replan_workspace_bytes",
           "moe_device_status", "moe_status_str", "moe_kernel_launches", "moe_profile_enable",
           "moe_profile_kernel_count", "moe_profile_read", "moe_profile_reset", "moe_demand_decay",
           "moe_demand_save", "moe_demand_load", "moe_hot_ring_create", "moe_hot_ring_step", "moe_hot_ring_destroy",
           "moe_hot_read_sync", "moe_renormalise_weights", "moe_expert_ffn_prefetch", "moe_set_wait_limit",
           "moe_get_wait_limit", "moe_wait_selftest", "moe_arena_refill")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class MoeArena(ctypes.Structure):
    """Mirror of ``moe_arena`` (passed by host pointer)."""
    _fields_ = [("base", ctypes.c_void_p), ("slot_bytes", ctypes.c_int64), ("n_slots", ctypes.c_int32),
                ("d", ctypes.c_int32), ("ffn", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("off_gu_codes", ctypes.c_int64), ("off_gu_scales", ctypes.c_int64),
                ("off_dn_codes", ctypes.c_int64), ("off_dn_scales", ctypes.c_int64)]


_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    L.moe_route_resident.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_route_resident_noalloc.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    L.moe_demand_accumulate.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]
    L.moe_hot_miss_select.argtypes = [_P, _I, _I, _F, _I, _P, _P, _P, _P]
    L.moe_expert_ffn_mxfp4.argtypes = [_P, _P, _P, ctypes.POINTER(MoeArena), _I, _I, _P, _P, _SZ, _P]
    L.moe_arena_replan.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_ring_install.argtypes = [_P, _P, _I, _I, _I, _I, _P]
    L.moe_workspace_bytes.restype = _SZ
    L.moe_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
    L.moe_replan_workspace_bytes.restype = _SZ
    L.moe_replan_workspace_bytes.argtypes = [_I, _I]
    L.moe_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
    L.moe_status_str.restype = ctypes.c_char_p
    L.moe_status_str.argtypes = [_I]
    L.moe_kernel_launches.restype = ctypes.c_uint64
    L.moe_kernel_launches.argtypes = []
    L.moe_profile_enable.argtypes = [_I]
    L.moe_profile_kernel_count.restype = _I
    L.moe_profile_kernel_count.argtypes = []
    L.moe_profile_read.argtypes = [_I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(ctypes.c_double)]
    L.moe_profile_reset.restype = None
    L.moe_profile_reset.argtypes = []
    L.moe_demand_decay.argtypes = [_P, ctypes.c_int64, _F, _P]
    L.moe_hot_ring_create.argtypes = [ctypes.POINTER(MoeArena), _I, _I, _I, ctypes.POINTER(ctypes.c_void_p), _I,
                                      ctypes.POINTER(ctypes.c_void_p)]
    L.moe_hot_ring_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_int32)]
    L.moe_hot_ring_destroy.argtypes = [_P]
    L.moe_renormalise_weights.argtypes = [_P, _P, _I, _I, _P]
    L.moe_expert_ffn_prefetch.argtypes = [_P, ctypes.POINTER(MoeArena), _I, _I, _P]
    L.moe_hot_read_sync.argtypes = [_P, _P, _P, _P, _P, ctypes.POINTER(MoeArena), _I, _I, _I, _F, _P, _P, _P]
    L.moe_demand_save.argtypes = [_P, _I, _I, ctypes.c_char_p, _P]
    L.moe_demand_load.argtypes = [_P, _I, _I, ctypes.c_char_p, _P]
    L.moe_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.moe_get_wait_limit.restype = ctypes.c_uint64
    L.moe_get_wait_limit.argtypes = []
    L.moe_wait_selftest.argtypes = [_P]
    L.moe_arena_refill.argtypes = [ctypes.POINTER(MoeArena), ctypes.POINTER(ctypes.c_void_p), _I, _P, _P, _P, _P,
                                   _P, ctypes.POINTER(ctypes.c_int32)]
    for name in ("moe_route_resident", "moe_route_resident_noalloc", "moe_demand_accumulate", "moe_hot_miss_select",
                 "moe_expert_ffn_mxfp4",
                 "moe_arena_replan", "moe_ring_install", "moe_device_status", "moe_profile_enable",
                 "moe_profile_read", "moe_demand_decay", "moe_demand_save", "moe_demand_load", "moe_hot_ring_create",
                 "moe_hot_ring_step", "moe_hot_ring_destroy", "moe_hot_read_sync", "moe_renormalise_weights",
                 "moe_expert_ffn_prefetch", "moe_set_wait_limit", "moe_wait_selftest", "moe_arena_refill"):
        L[name].restype = _I
    _lib = L
    return L


def _check(fn: str, st: int) -> None:
    if st != MOE_OK:
        raise MoeError(fn, st, load().moe_status_str(st).decode())


def _ptr(t, host_ok: bool = False):
    """Pointer of a contiguous CUDA tensor (or, with host_ok, of a pinned host tensor the kernels read directly)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError("expected a CUDA tensor" + (" or a pinned host tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Arena:
    """A device slot arena: ``buf`` uint8 [n_slots * slot_bytes] plus its record layout."""
    buf: torch.Tensor
    slot_bytes: int
    n_slots: int
    d: int
    ffn: int
    off_gu_codes: int
    off_gu_scales: int
    off_dn_codes: int
    off_dn_scales: int

    def struct(self) -> MoeArena:
        return MoeArena(ctypes.c_void_p(self.buf.data_ptr()), self.slot_bytes, self.n_slots, self.d, self.ffn, 0,
                        self.off_gu_codes, self.off_gu_scales, self.off_dn_codes, self.off_dn_scales)


# ------------------------------------------------------------------ entry points (same names as the C ABI)

def moe_workspace_bytes(T: int, k: int, d: int, ffn: int, E: int, n_slots: int) -> int:
    return int(load().moe_workspace_bytes(T, k, d, ffn, E, n_slots))


def moe_replan_workspace_bytes(L: int, E: int) -> int:
    return int(load().moe_replan_workspace_bytes(L, E))


def moe_route_resident(hidden_bf16, w_router, bias, slot_of, k, want_e, want_s, sel_e, sel_slot, sel_w,
                       workspace, stream=None) -> None:
    T, d = hidden_bf16.shape
    E = w_router.shape[0]
    _check("moe_route_resident", load().moe_route_resident(
        _ptr(hidden_bf16, True), _ptr(w_router), _ptr(bias), _ptr(slot_of), T, d, E, k, _ptr(want_e), _ptr(want_s),
        _ptr(sel_e), _ptr(sel_slot), _ptr(sel_w), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_route_resident_noalloc(hidden_bf16, w_router, bias, slot_of, k, want_e, want_s, sel_e, sel_slot, sel_w,
                               stream=None) -> None:
    """moe_route_resident for callers that cannot allocate device memory: no workspace argument.

    The partial logits go to a fixed 4 MiB array inside the library (shared by
    all calls on a device, so calls must not overlap on the GPU); sizes whose
    partials do not fit raise MoeError with MOE_EUNSUPPORTED.
    """
    T, d = hidden_bf16.shape
    E = w_router.shape[0]
    _check("moe_route_resident_noalloc", load().moe_route_resident_noalloc(
        _ptr(hidden_bf16, True), _ptr(w_router), _ptr(bias), _ptr(slot_of), T, d, E, k, _ptr(want_e), _ptr(want_s),
        _ptr(sel_e), _ptr(sel_slot), _ptr(sel_w), _stream(stream)))


def moe_demand_accumulate(want_e, want_s, slot_of, layer, demand, miss_max, stream=None) -> None:
    T, k = want_e.shape
    L, E = demand.shape
    _check("moe_demand_accumulate", load().moe_demand_accumulate(
        _ptr(want_e), _ptr(want_s), _ptr(slot_of), T, k, layer, L, E, _ptr(demand), _ptr(miss_max),
        _stream(stream)))


def moe_hot_miss_select(miss_max, threshold, cap, out_flat, out_share, n_out, stream=None) -> None:
    L, E = miss_max.shape
    _check("moe_hot_miss_select", load().moe_hot_miss_select(
        _ptr(miss_max), L, E, float(threshold), cap, _ptr(out_flat), _ptr(out_share), _ptr(n_out),
        _stream(stream)))


def moe_expert_ffn_mxfp4(hidden_bf16, sel_slot, sel_w, arena: Arena, out, workspace, stream=None) -> None:
    T = hidden_bf16.shape[0]
    k = sel_slot.shape[1]
    st = arena.struct()
    _check("moe_expert_ffn_mxfp4", load().moe_expert_ffn_mxfp4(
        _ptr(hidden_bf16, True), _ptr(sel_slot), _ptr(sel_w), ctypes.byref(st), T, k, _ptr(out, True), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_arena_replan(demand, n_main, slot_of, owner, loads, n_loads, workspace, stream=None) -> None:
    L, E = demand.shape
    _check("moe_arena_replan", load().moe_arena_replan(
        _ptr(demand), L, E, n_main, owner.numel(), _ptr(slot_of), _ptr(owner), _ptr(loads), _ptr(n_loads),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_arena_refill(arena: Arena, records, loads, n_loads, owner, stream=None, copy_stream=None) -> int:
    """Copy the new owners' records into the slots a re-plan gave them (see the header); returns how many.
    `records`: a sequence of n_flat host addresses (int) of expert records, or None where the store has none."""
    n_flat = len(records)
    ptrs = (ctypes.c_void_p * n_flat)(*[r if r else None for r in records])
    st = arena.struct()
    n = ctypes.c_int32(0)
    cs = copy_stream if copy_stream is not None else torch.cuda.current_stream()
    _check("moe_arena_refill", load().moe_arena_refill(
        ctypes.byref(st), ptrs, n_flat, _ptr(loads), _ptr(n_loads), _ptr(owner), _stream(stream),
        ctypes.c_void_p(cs.cuda_stream), ctypes.byref(n)))
    return int(n.value)


def moe_ring_install(slot_of, owner, ring_slot: int, flat_id: int, stream=None) -> None:
    _check("moe_ring_install", load().moe_ring_install(
        _ptr(slot_of), _ptr(owner), ring_slot, flat_id, slot_of.numel(), owner.numel(), _stream(stream)))


def moe_device_status(stream=None) -> tuple[int, int]:
    """(status, raw error bits); reads and clears the device error word."""
    bits = ctypes.c_uint32(0)
    st = load().moe_device_status(_stream(stream), ctypes.byref(bits))
    return st, bits.value


def moe_set_wait_limit(ns: int) -> None:
    """Bound (wall-clock ns) on every wait of the pipelined kernels launched from now on; 0 = the default 2 s."""
    _check("moe_set_wait_limit", load().moe_set_wait_limit(int(ns)))


def moe_get_wait_limit() -> int:
    return int(load().moe_get_wait_limit())


def moe_wait_selftest(stream=None) -> None:
    """Launch the stalled-wait check (see the header); afterwards moe_device_status reports MOE_ETIMEOUT."""
    _check("moe_wait_selftest", load().moe_wait_selftest(_stream(stream)))


def moe_kernel_launches() -> int:
    return int(load().moe_kernel_launches())


def moe_profile_enable(on: bool) -> None:
    _check("moe_profile_enable", load().moe_profile_enable(1 if on else 0))


def moe_profile_reset() -> None:
    load().moe_profile_reset()


def moe_profile_read() -> dict:
    """{kernel name: (launches, total device ms)} for the launches recorded since the last reset."""
    L = load()
    out = {}
    for kind in range(L.moe_profile_kernel_count()):
        name = ctypes.c_char_p()
        n = ctypes.c_int64()
        ms = ctypes.c_double()
        _check("moe_profile_read", L.moe_profile_read(kind, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms)))
        if n.value:
            out[name.value.decode()] = (n.value, ms.value)
    return out


def moe_demand_decay(demand: torch.Tensor, factor: float, stream=None) -> None:
    """demand int64/uint64 [..] in units of 2^-40, scaled in place by factor in [0, 1] (fixed point, floor)."""
    _check("moe_demand_decay", load().moe_demand_decay(_ptr(demand), demand.numel(), float(factor), _stream(stream)))


def moe_demand_save(demand: torch.Tensor, path: str, stream=None) -> None:
    """Write the [L, E] demand history to `path` (see the header for the format)."""
    L, E = demand.shape
    _check("moe_demand_save", load().moe_demand_save(_ptr(demand), L, E, os.fsencode(path), _stream(stream)))


def moe_demand_load(demand: torch.Tensor, path: str, stream=None) -> None:
    """Read an [L, E] demand history written by moe_demand_save into `demand`."""
    L, E = demand.shape
    _check("moe_demand_load", load().moe_demand_load(_ptr(demand), L, E, os.fsencode(path), _stream(stream)))


class HotRing:
    """The asynchronous hot-read ring (moe_hot_ring_*): ring slots [ring_first, ring_first + n_ring) of
    `arena`, filled from `records`, a sequence of n_flat host addresses (int) of expert records or None."""

    def __init__(self, arena: Arena, ring_first: int, n_ring: int, records, cap: int = 16):
        self._keep = arena
        n_flat = len(records)
        self._ptrs = (ctypes.c_void_p * n_flat)(*[r if r else None for r in records])
        self._st = arena.struct()
        h = ctypes.c_void_p()
        _check("moe_hot_ring_create", load().moe_hot_ring_create(
            ctypes.byref(self._st), ring_first, n_ring, n_flat, self._ptrs, cap, ctypes.byref(h)))
        self._h = h
        self.copy_stream = torch.cuda.Stream()

    def step(self, heavy_flat, n_heavy, slot_of, owner, stream=None) -> int:
        """Install last call's copies, read this step's heavy misses, issue their copies; returns how many."""
        n = ctypes.c_int32(0)
        _check("moe_hot_ring_step", load().moe_hot_ring_step(
            self._h, _ptr(heavy_flat), _ptr(n_heavy), _ptr(slot_of), _ptr(owner), _stream(stream),
            ctypes.c_void_p(self.copy_stream.cuda_stream), ctypes.byref(n)))
        return int(n.value)

    def close(self) -> None:
        if self._h:
            _check("moe_hot_ring_destroy", load().moe_hot_ring_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_hot_read_sync(store, demand, miss_max, slot_of, owner, arena: Arena, layer: int, threshold: float,
                      budget, swap, stream=None) -> None:
    """One layer's synchronous hot read (see the header): store int64 [L*E] device-readable record
    addresses (0 = none); budget int32 [1] and swap int32 [3] on the device."""
    L, E = demand.shape
    st = arena.struct()
    _check("moe_hot_read_sync", load().moe_hot_read_sync(
        _ptr(store), _ptr(demand), _ptr(miss_max), _ptr(slot_of), _ptr(owner), ctypes.byref(st), layer, L, E,
        float(threshold), _ptr(budget), _ptr(swap), _stream(stream)))


def moe_expert_ffn_prefetch(sel_slot, arena: Arena, stream=None) -> None:
    """L2 prefetch of the gate/up weights the expert FFN streams first for these picks (see the header)."""
    T, k = sel_slot.shape
    st = arena.struct()
    _check("moe_expert_ffn_prefetch", load().moe_expert_ffn_prefetch(_ptr(sel_slot), ctypes.byref(st), T, k,
                                                                     _stream(stream)))


def moe_renormalise_weights(sel_slot, sel_w, stream=None) -> None:
    """In place: each token's valid combine weights divided by their sum (see the header)."""
    T, k = sel_w.shape
    _check("moe_renormalise_weights", load().moe_renormalise_weights(_ptr(sel_slot), _ptr(sel_w), T, k,
                                                                     _stream(stream)))
