"""Seeded layer cases shared by the GPU parity tests, smoke() and the bench.

Builds the host inputs with ``synth``, the device arena (filled by synth's
device generator), and the oracle's view of the experts (regenerated on the
host from the same seeds). Nothing here computes the method.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import synth

# A ragged case: several tiles in every dimension with partial tails.
RAGGED = synth.LayerConfig("ragged E40 k3 d384 F256 R25", E=40, k=3, d=384, ffn=256, resident=25, sigma=1.0,
                           seed=0x7EED00A0)
# Fewer residents than k: padded picks.
SPARSE = synth.LayerConfig("sparse E16 k4 d256 F128 R2", E=16, k=4, d=256, ffn=128, resident=2, sigma=None,
                           seed=0x7EED00A1)

# Routing only: E below one 128-expert tile and an odd number of 64-element K chunks.
ODD = synth.LayerConfig("odd E48 k6 d320 F128 R30", E=48, k=6, d=320, ffn=128, resident=30, sigma=1.0,
                        seed=0x7EED00A2)

# Routing only: the widest rows the row-per-CTA router takes (d = 8192), and one 32-element block wider.
WIDE = synth.LayerConfig("wide E64 k4 d8192 F128 R40", E=64, k=4, d=8192, ffn=128, resident=40, sigma=1.0,
                         seed=0x7EED00A3)
WIDER = synth.LayerConfig("wider E64 k4 d8224 F128 R40", E=64, k=4, d=8224, ffn=128, resident=40, sigma=1.0,
                          seed=0x7EED00A4)


@dataclasses.dataclass
class Case:
    cfg: synth.LayerConfig
    T: int
    x: np.ndarray          # uint16 [T, d] bf16 bits
    W: np.ndarray          # fp32 [E, d]
    bias: np.ndarray       # fp32 [E]
    slot_of: np.ndarray    # int32 [E]
    owner: np.ndarray      # int32 [n_slots] (expert id per slot, -1 empty)
    n_slots: int


def make_case(cfg: synth.LayerConfig, T: int, stream: int = 0, drift: bool = False) -> Case:
    x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream)
    W = synth.router_weights(cfg.seed, cfg.E, cfg.d)
    b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma)
    res = synth.resident_set(cfg, b)
    n_slots = cfg.resident + cfg.n_ring
    slot_of = synth.slot_table(cfg, res, n_slots)
    owner = np.full(n_slots, -1, np.int32)
    owner[slot_of[res]] = res
    if drift:
        b = synth.drifted_bias(cfg, b)
    return Case(cfg, T, x, W, b, slot_of, owner, n_slots)


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def hidden_dev(x_bits: np.ndarray) -> torch.Tensor:
    return to_dev(x_bits.view(np.int16)).view(torch.bfloat16)


def device_arena(cfg: synth.LayerConfig, owner: np.ndarray, n_slots: int):
    import resident_expert_routed_gb300 as moe
    rec = synth.slot_record(cfg.d, cfg.ffn)
    buf = torch.zeros(n_slots * rec["slot_bytes"], dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(buf, cfg.d, cfg.ffn, cfg.seed, cfg.E, to_dev(owner.astype(np.int32)))
    return moe.Arena(buf, rec["slot_bytes"], n_slots, cfg.d, cfg.ffn, rec["off_gu_codes"], rec["off_gu_scales"],
                     rec["off_dn_codes"], rec["off_dn_scales"])


def oracle_experts(cfg: synth.LayerConfig, owner: np.ndarray, sel_slot: np.ndarray):
    """(sel_u, experts) for the oracle FFN: the distinct slots picked, regenerated on the host."""
    used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
    index = {s: i for i, s in enumerate(used)}
    sel_u = np.vectorize(lambda s: index.get(int(s), -1))(sel_slot).astype(np.int32) if sel_slot.size else sel_slot
    experts = []
    for s in used:
        f = int(owner[s])
        experts.append(synth.expert_weights(cfg.seed, f // cfg.E, f % cfg.E, cfg.d, cfg.ffn))
    return sel_u, experts


def rel_frobenius(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def ffn_within_tolerance(got: np.ndarray, ref: np.ndarray) -> tuple[bool, float, float]:
    """The FFN acceptance bar: relative Frobenius <= 5e-3 and max-abs <= 2e-2 * max|ref|."""
    fro = rel_frobenius(got, ref)
    mx = float(np.abs(got - ref).max()) if ref.size else 0.0
    bound = 2e-2 * float(np.abs(ref).max()) if ref.size else 0.0
    return (fro <= 5e-3 and mx <= bound), fro, mx


def near_tie_tokens(scores: np.ndarray, mask: np.ndarray, k: int, rel: float = 1e-5) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th scores over the masked experts lie within `rel` of each other."""
    T = scores.shape[0]
    out = np.zeros(T, bool)
    for t in range(T):
        s = np.sort(scores[t][mask])[::-1]
        if len(s) > k and abs(s[k - 1] - s[k]) <= rel * s[k - 1]:
            out[t] = True
    return out


def clear_ranks(scores_row: np.ndarray, mask: np.ndarray, k: int, rel: float = 1e-5) -> np.ndarray:
    """For the oracle's ranking of the masked experts by score (descending), which of the first k ranks are
    separated from both neighbours (the previous rank and the next one, the (k+1)-th included) by more than
    `rel` relative: at those ranks the expert is fixed whatever the rounding order of the scores."""
    r = np.sort(scores_row[mask])[::-1][:k + 1]
    n = min(k, len(r))
    clear = np.zeros(k, bool)
    for j in range(n):
        above = j == 0 or r[j - 1] - r[j] > rel * r[j - 1]
        below = j + 1 >= len(r) or r[j] - r[j + 1] > rel * r[j]
        clear[j] = above and below
    return clear


def covering_rows(sel_slot: np.ndarray, extra: int = 8, seed: int = 11) -> np.ndarray:
    """A sample of token rows that routes to every slot the batch uses: for each used slot (rarest first) not
    yet covered, the LAST token that picks it (its pick sits at the end of the slot's rows, i.e. in the last,
    usually partial, tile of that slot), plus `extra` seeded rows. Sorted, without repeats."""
    T = sel_slot.shape[0]
    slots, counts = np.unique(sel_slot[sel_slot >= 0], return_counts=True)
    covered = np.zeros(int(sel_slot.max(initial=-1)) + 1, bool)
    rows = set()
    for s in slots[np.argsort(counts, kind="stable")]:
        if covered[s]:
            continue
        t = int(np.flatnonzero((sel_slot == s).any(axis=1))[-1])
        rows.add(t)
        row = sel_slot[t]
        covered[row[row >= 0]] = True
    rng = np.random.default_rng(seed)
    rows.update(int(v) for v in rng.choice(T, size=min(extra, T), replace=False))
    return np.array(sorted(rows), np.int64)


def ring_case(cfg: synth.LayerConfig, n_ring: int, T: int = 8, stream: int = 0):
    """A drifted case with cfg.resident main slots + n_ring ring slots (device arena), its tables, and a
    pinned host store of every absent expert's record (the stand-in for the drive): returns
    (case, arena, slot_of, owner, absent ids, store tensor, per-expert record addresses or None)."""
    import resident_expert_routed_gb300 as moe
    c = make_case(cfg, T, stream=stream, drift=True)
    res = np.flatnonzero(c.slot_of >= 0)
    n_slots = cfg.resident + n_ring
    slot_of = synth.slot_table(cfg, res, cfg.resident)
    owner = np.full(n_slots, -1, np.int32)
    owner[slot_of[res]] = res
    rec = synth.slot_record(cfg.d, cfg.ffn)
    sb = rec["slot_bytes"]
    buf = torch.zeros(n_slots * sb, dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(buf, cfg.d, cfg.ffn, cfg.seed, cfg.E, to_dev(owner))
    arena = moe.Arena(buf, sb, n_slots, cfg.d, cfg.ffn, rec["off_gu_codes"], rec["off_gu_scales"],
                      rec["off_dn_codes"], rec["off_dn_scales"])
    absent = np.flatnonzero(slot_of < 0).astype(np.int32)
    tmp = torch.zeros(len(absent) * sb, dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(tmp, cfg.d, cfg.ffn, cfg.seed, cfg.E, to_dev(absent))
    store = torch.empty(len(absent) * sb, dtype=torch.uint8, pin_memory=True)
    store.copy_(tmp)
    records = [None] * cfg.E
    for i, f in enumerate(absent):
        records[f] = store.data_ptr() + i * sb
    return c, arena, slot_of, owner, absent, store, records
