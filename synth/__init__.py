"""Seeded synthetic inputs for the resident-expert routed MoE layer.

This module is shared by the CUDA path's tests/bench and by the oracle's
callers. It holds none of the method's arithmetic: it only draws numbers.

Counter-based generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  A stream is keyed by
(seed, tensor id, a, b); value i of a stream is the SplitMix64 output for
state base + (i + 1) * gamma, so any element can be drawn on its own, on the
host (numpy here) or on the device (``csrc/synth_fill.cu``, the same integer
hash for expert weight bytes).

Normals come from Box-Muller in float64 on the host only and are then rounded
to fp32 / bf16, so both sides see the same bits.

Workload recipe (shapes and distributions of the layer configurations this
repository tests and times):

* hidden  x ~ N(0, 1), rounded to bf16 (round to nearest even);
* router  W ~ N(0, 1/d) fp32, bias b = sigma * z, z ~ N(0, 1) (so e^b is
  lognormal(sigma)); the tiny case uses b ~ N(0, 1);
* experts: e2m1 codes uniform on 0..15 (two per byte, low nibble = even
  element), e8m0 scale bytes 127 + U with U uniform on {-6, -5, -4, -3}.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

U64 = np.uint64
GAMMA = U64(0x9E3779B97F4A7C15)
_M1 = U64(0xBF58476D1CE4E5B9)
_M2 = U64(0x94D049BB133111EB)

# tensor ids (stream tags)
T_HIDDEN = 1
T_ROUTER_W = 2
T_BIAS = 3
T_GU_CODES = 4
T_GU_SCALES = 5
T_DN_CODES = 6
T_DN_SCALES = 7
T_MASK = 8
T_SLOTPERM = 9
T_DRIFT = 10
T_RING = 11
T_SAMPLE = 12


def _mix(z):
    """SplitMix64 output function (works on numpy uint64 scalars and arrays)."""
    z = np.asarray(z, dtype=U64)
    z = (z ^ (z >> U64(30))) * _M1
    z = (z ^ (z >> U64(27))) * _M2
    return z ^ (z >> U64(31))


def stream_base(seed: int, tensor_id: int, a: int = 0, b: int = 0) -> np.uint64:
    """Initial SplitMix64 state of the stream (seed, tensor_id, a, b); a, b < 2**28."""
    with np.errstate(over="ignore"):
        key = (U64(tensor_id & 0xFF) << U64(56)) ^ (U64(a & 0xFFFFFFF) << U64(28)) ^ U64(b & 0xFFFFFFF)
        return U64(_mix(U64(seed & 0xFFFFFFFFFFFFFFFF) ^ _mix(key)))


def hash_at(base, idx) -> np.ndarray:
    """Value idx (array) of the stream starting at state ``base``."""
    idx = np.asarray(idx, dtype=U64)
    with np.errstate(over="ignore"):
        return _mix(U64(base) + (idx + U64(1)) * GAMMA)


def uniform01(base, idx) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (hash_at(base, idx) >> U64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normals(seed: int, tensor_id: int, a: int, b: int, n: int) -> np.ndarray:
    """n standard normals (float64), Box-Muller cosine branch, element i from hashes 2i, 2i+1."""
    base = stream_base(seed, tensor_id, a, b)
    i = np.arange(n, dtype=U64)
    u1 = 1.0 - uniform01(base, U64(2) * i)          # (0, 1]
    u2 = uniform01(base, U64(2) * i + U64(1))       # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + U64(0x7FFF) + ((u >> U64(16)) & U64(1))) >> U64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def seeded_permutation(seed: int, tensor_id: int, a: int, n: int) -> np.ndarray:
    """A permutation of 0..n-1: argsort of n hashes (stable, ties impossible in practice)."""
    base = stream_base(seed, tensor_id, a, 0)
    return np.argsort(hash_at(base, np.arange(n, dtype=U64)), kind="stable").astype(np.int64)


# --------------------------------------------------------------------------- experts

def slot_record(d: int, ffn: int) -> dict:
    """Byte layout of one arena slot: gate/up codes, gate/up scales, down codes, down scales.

    gate/up codes  [2F, d/2]  (rows 0..F-1 gate, F..2F-1 up; K contiguous, low nibble = even k)
    gate/up scales [2F, d/32]
    down codes     [d,  F/2]
    down scales    [d,  F/32]
    Every region starts on a 256-byte boundary, and so does every slot.
    """
    def al(x, a=256):
        return (x + a - 1) // a * a
    gu_c = (2 * ffn // 128) * ((d + 255) // 256) * 16384   # tile-major code blocks (pack_codes)
    gu_s = 2 * ffn * d // 32
    dn_c = (d // 128) * ((ffn + 255) // 256) * 16384
    dn_s = d * ffn // 32
    off_gu_codes = 0
    off_gu_scales = al(off_gu_codes + gu_c)
    off_dn_codes = al(off_gu_scales + gu_s)
    off_dn_scales = al(off_dn_codes + dn_c)
    slot_bytes = al(off_dn_scales + dn_s)
    return dict(slot_bytes=slot_bytes, off_gu_codes=off_gu_codes, off_gu_scales=off_gu_scales,
                off_dn_codes=off_dn_codes, off_dn_scales=off_dn_scales,
                gu_codes_bytes=gu_c, gu_scales_bytes=gu_s, dn_codes_bytes=dn_c, dn_scales_bytes=dn_s)


def _code_bytes(seed: int, tid: int, layer: int, expert: int, nbytes: int) -> np.ndarray:
    """Byte j = byte (j % 8) (little end first) of hash j // 8: uniform nibbles."""
    base = stream_base(seed, tid, layer, expert)
    words = hash_at(base, np.arange((nbytes + 7) // 8, dtype=U64))
    return words.view(np.uint8)[:nbytes].copy()


def _scale_bytes(seed: int, tid: int, layer: int, expert: int, nbytes: int) -> np.ndarray:
    """Byte j = 121 + ((hash(j // 32) >> (2 * (j % 32))) & 3): e8m0 exponent 127 + U, U in -6..-3."""
    base = stream_base(seed, tid, layer, expert)
    j = np.arange(nbytes, dtype=U64)
    words = hash_at(base, j >> U64(5))
    two = (words >> (U64(2) * (j & U64(31)))) & U64(3)
    return (U64(121) + two).astype(np.uint8)


def expert_weights(seed: int, layer: int, expert: int, d: int, ffn: int) -> dict:
    """The MXFP4 weights of expert (layer, expert), in the arena's logical layout."""
    return dict(
        gu_codes=_code_bytes(seed, T_GU_CODES, layer, expert, 2 * ffn * d // 2).reshape(2 * ffn, d // 2),
        gu_scales=_scale_bytes(seed, T_GU_SCALES, layer, expert, 2 * ffn * d // 32).reshape(2 * ffn, d // 32),
        dn_codes=_code_bytes(seed, T_DN_CODES, layer, expert, d * ffn // 2).reshape(d, ffn // 2),
        dn_scales=_scale_bytes(seed, T_DN_SCALES, layer, expert, d * ffn // 32).reshape(d, ffn // 32),
    )


def _tile_rows(R: int) -> np.ndarray:
    """[tiles, 128] logical row of each tile row: tile g holds rows 128g..128g+127."""
    return np.arange(R).reshape(-1, 128)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Code bytes [R, K/2] in the arena's tile-major block order.

    For each tile of 128 consecutive rows and each chunk of 256
    elements along K (128 bytes, zero-padded past the row end), one 16 KB block
    of 128 rows x 128 bytes; 16-byte piece c of tile row r is stored at piece
    c ^ (r % 8) of that row (the 128-byte swizzle). Blocks are stored tile by
    tile, chunk by chunk.
    """
    R, Kh = codes.shape
    nkc = (Kh + 127) // 128
    rows = _tile_rows(R)
    tiles = rows.shape[0]
    t = np.zeros((tiles, 128, nkc * 128), np.uint8)
    t[:, :, :Kh] = codes[rows]
    t = t.reshape(tiles, 128, nkc, 8, 16)                 # [tile, r, kc, piece, byte]
    out = np.empty_like(t)
    for rr in range(8):                                    # rows with r % 8 == rr
        rows_r = np.arange(rr, 128, 8)
        for c in range(8):
            out[:, rows_r, :, c ^ rr, :] = t[:, rows_r, :, c, :]
    return np.ascontiguousarray(out.transpose(0, 2, 1, 3, 4)).reshape(-1)


def pack_scales(scales: np.ndarray) -> np.ndarray:
    """Scale bytes [R, K/32] in the arena's tile-atom order (the layout the arena record uses).

    Rows are taken in tiles of 128 consecutive rows, and each tile's scales in
    512-byte atoms of 4 K-blocks: byte (r % 32) * 16 + (r // 32) * 4 + k for
    tile row r and K-block 4a + k of atom a. Tiles, then atoms, are stored in order.
    """
    R, Kb = scales.shape
    rows = _tile_rows(R)
    t = scales[rows]                                   # [tiles, 128, Kb]
    t = t.reshape(t.shape[0], 4, 32, Kb // 4, 4)       # r = 32 j + r0 ; kb = 4 a + k
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def expert_slot_bytes(seed: int, layer: int, expert: int, d: int, ffn: int) -> np.ndarray:
    """One whole slot record (uint8 [slot_bytes]) holding expert (layer, expert).

    Codes are stored in the tile-major block order of ``pack_codes``, scales in
    the tile-atom order of ``pack_scales``.
    """
    rec = slot_record(d, ffn)
    w = expert_weights(seed, layer, expert, d, ffn)
    out = np.zeros(rec["slot_bytes"], dtype=np.uint8)
    out[rec["off_gu_codes"]:rec["off_gu_codes"] + rec["gu_codes_bytes"]] = pack_codes(w["gu_codes"])
    out[rec["off_gu_scales"]:rec["off_gu_scales"] + rec["gu_scales_bytes"]] = \
        pack_scales(w["gu_scales"])
    out[rec["off_dn_codes"]:rec["off_dn_codes"] + rec["dn_codes_bytes"]] = pack_codes(w["dn_codes"])
    out[rec["off_dn_scales"]:rec["off_dn_scales"] + rec["dn_scales_bytes"]] = pack_scales(w["dn_scales"])
    return out


# --------------------------------------------------------------------------- layer configurations

@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """One MoE-layer workload: shapes, resident count and the router bias spread."""
    name: str
    E: int
    k: int
    d: int
    ffn: int
    resident: int            # main-arena residents per layer (single-layer cases)
    sigma: Optional[float]   # bias = sigma * z; None -> bias ~ N(0, 1) with a seeded mask
    seed: int
    L: int = 1
    n_ring: int = 0
    n_main: int = 0          # shared arena size (multi-layer case); 0 -> resident


TINY = LayerConfig("tiny E16 k4 d256 F128 R10", E=16, k=4, d=256, ffn=128, resident=10, sigma=None,
                   seed=0x7EED0000)
DECODE = LayerConfig("decode E256 k8 d4096 F2048 R166", E=256, k=8, d=4096, ffn=2048, resident=166,
                     sigma=1.5, seed=0x7EED0001)
PREFILL = LayerConfig("prefill E256 k8 d4096 F2048 R166 T8192", E=256, k=8, d=4096, ffn=2048, resident=166,
                      sigma=1.5, seed=0x7EED0002)
GLM = LayerConfig("glm-like E256 k8 d6144 F2048 R173+ring64", E=256, k=8, d=6144, ffn=2048, resident=173,
                  sigma=2.0, seed=0x7EED0003, n_ring=64)
FULL = LayerConfig("full decode step L60 E256 k8 d4096 F2048 arena10000+ring64 T2", E=256, k=8, d=4096,
                   ffn=2048, resident=0, sigma=1.5, seed=0x7EED0004, L=60, n_ring=64, n_main=10000)


def hidden_bf16(seed: int, T: int, d: int, stream: int = 0) -> np.ndarray:
    """Hidden states x ~ N(0,1) as bf16 bits, uint16 [T, d]; ``stream`` selects (step, layer)."""
    z = normals(seed, T_HIDDEN, stream, 0, T * d).astype(np.float32)
    return f32_to_bf16_bits(z).reshape(T, d)


def router_weights(seed: int, E: int, d: int, layer: int = 0) -> np.ndarray:
    """Router W ~ N(0, 1/d), fp32 [E, d]."""
    return (normals(seed, T_ROUTER_W, layer, 0, E * d) / math.sqrt(d)).astype(np.float32).reshape(E, d)


def router_bias(seed: int, E: int, sigma: Optional[float], layer: int = 0) -> np.ndarray:
    z = normals(seed, T_BIAS, layer, 0, E)
    s = 1.0 if sigma is None else sigma
    return (s * z).astype(np.float32)


def resident_set(cfg: LayerConfig, bias: np.ndarray, layer: int = 0) -> np.ndarray:
    """Sorted expert ids resident in one layer.

    Tiny case: a fixed seeded mask (first R of a seeded permutation).  Otherwise
    the R experts of highest expected demand; with i.i.d. logit noise that is
    the R largest biases (ties to the lower index).
    """
    if cfg.sigma is None:
        perm = seeded_permutation(cfg.seed, T_MASK, layer, cfg.E)
        return np.sort(perm[:cfg.resident])
    order = np.lexsort((np.arange(cfg.E), -bias.astype(np.float64)))
    return np.sort(order[:cfg.resident])


def slot_table(cfg: LayerConfig, resident: np.ndarray, n_slots: int, layer: int = 0) -> np.ndarray:
    """slot_of[E] (int32, -1 = absent): residents take slots in a seeded order, so slot != expert."""
    slots = seeded_permutation(cfg.seed, T_SLOTPERM, layer, n_slots)[:len(resident)]
    slot_of = np.full(cfg.E, -1, dtype=np.int32)
    slot_of[resident] = slots.astype(np.int32)
    return slot_of


def drifted_bias(cfg: LayerConfig, bias: np.ndarray, layer: int = 0) -> np.ndarray:
    """The bias permuted by a seeded shuffle after the resident set was fixed ("the tide")."""
    perm = seeded_permutation(cfg.seed, T_DRIFT, layer, cfg.E)
    return bias[perm].copy()


def full_initial_arena(cfg: LayerConfig) -> tuple[np.ndarray, np.ndarray]:
    """Multi-layer case: a seeded uniform sample of n_main (layer, expert) ids fills the main slots.

    Returns (slot_of [L*E] int32, owner [n_main + n_ring] int32, -1 = empty).
    """
    n = cfg.L * cfg.E
    chosen = seeded_permutation(cfg.seed, T_SAMPLE, 0, n)[:cfg.n_main]
    owner = np.full(cfg.n_main + cfg.n_ring, -1, dtype=np.int32)
    owner[:cfg.n_main] = chosen.astype(np.int32)
    slot_of = np.full(n, -1, dtype=np.int32)
    slot_of[chosen] = np.arange(cfg.n_main, dtype=np.int32)
    return slot_of, owner


def ring_candidates(cfg: LayerConfig, step: int, slot_of: np.ndarray, count: int) -> np.ndarray:
    """``count`` seeded non-resident expert ids (single layer) to install in the ring between steps."""
    absent = np.flatnonzero(slot_of < 0)
    if len(absent) == 0:
        return absent.astype(np.int32)
    perm = seeded_permutation(cfg.seed, T_RING, step, len(absent))
    return absent[perm[:min(count, len(absent))]].astype(np.int32)


# --------------------------------------------------------------------------- device fill of big arenas

_FILL_SRC = __import__("os").path.join(__import__("os").path.dirname(__file__), "csrc", "synth_fill.cu")
_FILL_LIB = __import__("os").path.join(__import__("os").path.dirname(__file__), "libsynth_fill.so")
_fill = None


def build_fill(force: bool = False) -> str:
    """Compile the device fill kernel (same hash as above) for sm_103a."""
    import os
    import subprocess
    if force or not os.path.exists(_FILL_LIB) or os.path.getmtime(_FILL_LIB) < os.path.getmtime(_FILL_SRC):
        tmp = _FILL_LIB + f".tmp{os.getpid()}"
        subprocess.check_call([os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc"), "-gencode",
                               "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                               "-shared", "-o", tmp, _FILL_SRC])
        os.replace(tmp, _FILL_LIB)
    return _FILL_LIB


def _fill_lib():
    global _fill
    if _fill is None:
        import ctypes
        _fill = ctypes.CDLL(build_fill())
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        _fill.synth_fill_slots.restype = I
        _fill.synth_fill_slots.argtypes = [P, I64, I64, I64, I64, I64, I, I, P, P, I, I, I, ctypes.c_uint64, P]
    return _fill


def fill_slots_device(arena_buf, d: int, ffn: int, seed: int, E: int, flats, slots=None, slot_begin: int = 0,
                      n: int | None = None, stream=None) -> None:
    """Write seeded experts into a device arena (torch uint8 tensor of n_slots * slot_bytes).

    slots is None: slots [slot_begin, slot_begin + n) take expert flats[slot] (an owner table, -1 skips);
    otherwise slot slots[i] takes expert flats[i]. ``flats``/``slots`` are int32 CUDA tensors.
    """
    import ctypes
    import torch
    rec = slot_record(d, ffn)
    if n is None:
        n = int(slots.numel()) if slots is not None else int(flats.numel()) - slot_begin
    s = torch.cuda.current_stream() if stream is None else stream
    err = _fill_lib().synth_fill_slots(
        ctypes.c_void_p(arena_buf.data_ptr()), rec["slot_bytes"], rec["off_gu_codes"], rec["off_gu_scales"],
        rec["off_dn_codes"], rec["off_dn_scales"], d, ffn,
        None if slots is None else ctypes.c_void_p(slots.data_ptr()), ctypes.c_void_p(flats.data_ptr()),
        slot_begin, n, E, ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), ctypes.c_void_p(s.cuda_stream))
    if err != 0:
        raise RuntimeError(f"synth_fill_slots: cudaError {err}")
