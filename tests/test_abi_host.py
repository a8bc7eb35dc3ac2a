"""Host-side checks of the C-ABI library (no GPU needed).

The library must load, export every function include/moe_resident.h declares,
and reject bad arguments on the host before launching anything.
"""
import ctypes
import os
import re

import pytest

import resident_expert_routed_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_resident.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_route_resident", "moe_demand_accumulate", "moe_hot_miss_select", "moe_expert_ffn_mxfp4",
              "moe_arena_replan"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) <= set(moe.EXPORTS)


def test_status_strings():
    L = moe.load()
    assert L.moe_status_str(0) == b"ok"
    assert L.moe_status_str(3) == b"workspace too small"
    assert L.moe_status_str(99) == b"unknown status"


def test_arena_struct_layout_matches_header():
    # base(8) slot_bytes(8) n_slots d ffn reserved (4 x 4) and four int64 offsets
    assert ctypes.sizeof(moe.MoeArena) == 8 + 8 + 16 + 32
    assert moe.MoeArena.off_gu_codes.offset == 32


def test_workspace_sizes():
    w1 = moe.moe_workspace_bytes(1, 8, 4096, 2048, 256, 166)
    w64 = moe.moe_workspace_bytes(64, 8, 4096, 2048, 256, 166)
    w8k = moe.moe_workspace_bytes(8192, 8, 4096, 2048, 256, 166)
    # large batches route on the tensor cores: three bf16 parts of W_r plus the partial logits
    assert moe.moe_workspace_bytes(8192, 8, 4096, 0, 256, 0) >= 3 * 256 * 4096 * 2 + 8192 * 256 * 4
    assert 0 < w1 < w64 < w8k
    # up to 64 tokens the FFN keeps one fp32 row per pick (T*k*d*4 bytes) for the ordered combine
    assert w64 >= 64 * 8 * 4096 * 4
    # larger batches add into the output directly; they keep the MXFP4 operands of every pick
    assert w8k >= 8192 * 8 * 4096 // 2
    assert moe.moe_workspace_bytes(0, 8, 4096, 2048, 256, 166) == 0
    assert moe.moe_replan_workspace_bytes(60, 256) >= 16384 * 12


NULL = None
FAKE = ctypes.c_void_p(0x1000)      # never dereferenced: every case below fails a host check first


def test_route_rejects_bad_arguments():
    L = moe.load()
    ok = [FAKE] * 4
    outs = [FAKE] * 5
    # null pointer
    assert L.moe_route_resident(NULL, FAKE, NULL, FAKE, 4, 64, 16, 4, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    # k > 32, k > E, d % 32, T < 1
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 4, 64, 64, 33, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 4, 64, 4, 8, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 4, 48, 16, 4, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 0, 64, 16, 4, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    # E beyond the warp-per-token limit
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 4, 64, 2048, 4, *outs, FAKE, 1 << 30, NULL) == moe.MOE_EUNSUPPORTED
    # workspace too small
    assert L.moe_route_resident(*ok[:2], NULL, FAKE, 64, 4096, 256, 8, *outs, FAKE, 16, NULL) == moe.MOE_ENOMEM
    # hidden states, router weights or workspace not 16-byte aligned
    odd = ctypes.c_void_p(0x1002)
    assert L.moe_route_resident(odd, FAKE, NULL, FAKE, 4, 64, 16, 4, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident(FAKE, odd, NULL, FAKE, 4, 64, 16, 4, *outs, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident(FAKE, FAKE, NULL, FAKE, 4, 64, 16, 4, *outs, odd, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_route_resident_noalloc(odd, FAKE, NULL, FAKE, 4, 64, 16, 4, *outs, NULL) == moe.MOE_EINVAL


def _arena(**kw):
    import synth
    rec = synth.slot_record(256, 128)
    a = dict(base=0x100000, slot_bytes=rec["slot_bytes"], n_slots=16, d=256, ffn=128, reserved=0,
             off_gu_codes=rec["off_gu_codes"], off_gu_scales=rec["off_gu_scales"],
             off_dn_codes=rec["off_dn_codes"], off_dn_scales=rec["off_dn_scales"])
    a.update(kw)
    return moe.MoeArena(ctypes.c_void_p(a["base"]), a["slot_bytes"], a["n_slots"], a["d"], a["ffn"], 0,
                        a["off_gu_codes"], a["off_gu_scales"], a["off_dn_codes"], a["off_dn_scales"])


@pytest.mark.parametrize("kw,status", [
    (dict(d=200), moe.MOE_EINVAL),                  # d % 128
    (dict(ffn=96), moe.MOE_EINVAL),                 # ffn % 128
    (dict(base=0x100010), moe.MOE_EINVAL),          # arena base not 256-aligned
    (dict(off_dn_scales=67584 + 100), moe.MOE_EINVAL),   # offset not 256-aligned
    (dict(off_dn_scales=68608), moe.MOE_EINVAL),         # region past the end of the slot
    (dict(slot_bytes=68600), moe.MOE_EINVAL),            # slot size not a multiple of 256
    (dict(n_slots=20000), moe.MOE_EUNSUPPORTED),    # beyond the per-call slot limit
    (dict(), moe.MOE_ENOMEM),                       # valid arena, workspace too small
])
def test_ffn_rejects_bad_arguments(kw, status):
    L = moe.load()
    ar = _arena(**kw)
    st = L.moe_expert_ffn_mxfp4(FAKE, FAKE, FAKE, ctypes.byref(ar), 8, 4, FAKE, FAKE, 64, NULL)
    assert st == status


def test_ffn_rejects_picks_past_the_limit():
    L = moe.load()
    ar = _arena()
    # T * k = 2^20 is the largest call; one token more is refused before anything is touched
    assert L.moe_expert_ffn_mxfp4(FAKE, FAKE, FAKE, ctypes.byref(ar), (1 << 18) + 1, 4, FAKE, FAKE, 1 << 40,
                                  NULL) == moe.MOE_EUNSUPPORTED
    assert L.moe_expert_ffn_mxfp4(FAKE, FAKE, FAKE, ctypes.byref(ar), 1 << 18, 4, FAKE, FAKE, 64,
                                  NULL) == moe.MOE_ENOMEM


def test_other_entry_points_reject_bad_arguments():
    L = moe.load()
    assert L.moe_demand_accumulate(FAKE, FAKE, FAKE, 4, 4, 3, 2, 16, FAKE, FAKE, NULL) == moe.MOE_EINVAL  # layer >= L
    assert L.moe_demand_accumulate(NULL, FAKE, FAKE, 4, 4, 0, 2, 16, FAKE, FAKE, NULL) == moe.MOE_EINVAL
    assert L.moe_hot_miss_select(FAKE, 2, 16, ctypes.c_float(0.2), 2000, FAKE, FAKE, FAKE, NULL) == moe.MOE_EUNSUPPORTED
    assert L.moe_hot_miss_select(FAKE, 2, 16, ctypes.c_float(0.2), 16, NULL, FAKE, FAKE, NULL) == moe.MOE_EINVAL
    assert L.moe_arena_replan(FAKE, 2, 8, 20, 24, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_arena_replan(FAKE, 2, 8, 8, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == moe.MOE_EINVAL
    assert L.moe_arena_replan(FAKE, 2, 8, 8, 10, FAKE, FAKE, FAKE, FAKE, FAKE, 8, NULL) == moe.MOE_ENOMEM
    assert L.moe_ring_install(FAKE, FAKE, 10, 3, 16, 10, NULL) == moe.MOE_EINVAL     # ring slot past the arena
    assert L.moe_ring_install(FAKE, FAKE, 9, 16, 16, 10, NULL) == moe.MOE_EINVAL     # flat id past the table


def test_package_has_no_cpu_fallback():
    # every entry point marshals to the C library and refuses host tensors
    import torch
    x = torch.zeros((2, 64), dtype=torch.int16)
    with pytest.raises(ValueError):
        moe._ptr(x)


def test_demand_history_calls_reject_bad_arguments(tmp_path):
    L = moe.load()
    assert L.moe_demand_decay(FAKE, 16, ctypes.c_float(1.5), NULL) == moe.MOE_EINVAL     # factor above 1
    assert L.moe_demand_decay(FAKE, 16, ctypes.c_float(-0.1), NULL) == moe.MOE_EINVAL
    assert L.moe_demand_decay(FAKE, -1, ctypes.c_float(0.5), NULL) == moe.MOE_EINVAL
    assert L.moe_demand_decay(NULL, 0, ctypes.c_float(0.5), NULL) == moe.MOE_OK          # nothing to do
    missing = str(tmp_path / "none.bin").encode()
    assert L.moe_demand_load(FAKE, 2, 8, missing, NULL) == moe.MOE_EIO
    # a file whose header names another shape, or a bad magic, is refused before the device is touched
    p = tmp_path / "d.bin"
    import struct
    p.write_bytes(b"MOEDEMD1" + struct.pack("<iiii", 3, 8, 40, 0) + bytes(3 * 8 * 8))
    assert L.moe_demand_load(FAKE, 2, 8, str(p).encode(), NULL) == moe.MOE_EINVAL
    p.write_bytes(b"MOEDEMDX" + struct.pack("<iiii", 2, 8, 40, 0) + bytes(2 * 8 * 8))
    assert L.moe_demand_load(FAKE, 2, 8, str(p).encode(), NULL) == moe.MOE_EINVAL
    p.write_bytes(b"MOEDEMD1" + struct.pack("<iiii", 2, 8, 40, 0) + bytes(10))          # truncated
    assert L.moe_demand_load(FAKE, 2, 8, str(p).encode(), NULL) == moe.MOE_EIO
    assert L.moe_demand_save(NULL, 2, 8, str(p).encode(), NULL) == moe.MOE_EINVAL


@pytest.mark.parametrize("kw,status", [
    (dict(d=200), moe.MOE_EINVAL),
    (dict(base=0x100010), moe.MOE_EINVAL),
    (dict(off_dn_scales=68608), moe.MOE_EINVAL),
    (dict(n_slots=20000), moe.MOE_EUNSUPPORTED),
])
def test_ffn_prefetch_checks_the_arena_like_the_ffn(kw, status):
    L = moe.load()
    ar = _arena(**kw)
    assert L.moe_expert_ffn_prefetch(FAKE, ctypes.byref(ar), 8, 4, NULL) == status


def test_ffn_prefetch_skips_large_batches_and_rejects_nulls():
    # more than 8,192 picks: returns MOE_OK without a launch (no GPU needed)
    L = moe.load()
    ar = _arena()
    assert L.moe_expert_ffn_prefetch(FAKE, ctypes.byref(ar), 1024 + 1, 8, NULL) == moe.MOE_OK
    assert L.moe_expert_ffn_prefetch(NULL, ctypes.byref(ar), 8, 4, NULL) == moe.MOE_EINVAL
    assert L.moe_expert_ffn_prefetch(FAKE, None, 8, 4, NULL) == moe.MOE_EINVAL
