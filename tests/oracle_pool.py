"""Runs the oracle on several host cores at once (test infrastructure).

The oracle is single-threaded and slow by design. Full-size parity checks
(every token of a 64-token decode batch, a 60-layer history of 256 steps)
split its work into independent pieces -- disjoint groups of tokens, or
separate (step, layer) routing calls -- and run them in worker processes.
Each piece is one unmodified oracle call, so the results are exactly those
of a single call over the same rows.

Workers are started with the ``spawn`` method and import only numpy,
``synth`` and ``oracle`` (never CUDA), so a pool can be created at any point
of a GPU test. Inputs the workers can regenerate (router weights, hidden
states, expert weights) are rebuilt there from their seeds instead of being
pickled across.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing
import os

import numpy as np

_POOL = None


def pool() -> cf.ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2)))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn"))
    return _POOL


def workers() -> int:
    return pool()._max_workers


# ------------------------------------------------------------------ worker side

_W_CACHE: dict = {}


def _router_inputs(cfg, layer):
    import synth
    key = (cfg.name, cfg.seed, layer)
    if key not in _W_CACHE:
        W = synth.router_weights(cfg.seed, cfg.E, cfg.d, layer)
        b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma, layer)
        if len(_W_CACHE) > 64:
            _W_CACHE.clear()
        _W_CACHE[key] = (W, b)
    return _W_CACHE[key]


def _ffn_job(cfg, x, sel_slot, sel_w, owner_of_slot):
    import oracle
    import synth
    used = sorted({int(s) for s in sel_slot.ravel() if s >= 0})
    index = {s: i for i, s in enumerate(used)}
    sel_u = np.array([[index.get(int(s), -1) for s in row] for row in sel_slot], np.int32).reshape(sel_slot.shape)
    experts = []
    for s in used:
        f = int(owner_of_slot[s])
        experts.append(synth.expert_weights(cfg.seed, f // cfg.E, f % cfg.E, cfg.d, cfg.ffn))
    return oracle.ffn(x, sel_u, sel_w, experts, cfg.d, cfg.ffn)


def _route_job(cfg, layer, stream, T, slot_of, drift):
    """The oracle's routing of one seeded batch of one layer (the GPU tests' full-step inputs)."""
    import oracle
    import synth
    W, b = _router_inputs(cfg, layer)
    if drift:
        b = synth.drifted_bias(cfg, b, layer)
    x = synth.hidden_bf16(cfg.seed, T, cfg.d, stream=stream)
    r = oracle.route(x, W, b, slot_of, cfg.k)
    return {kk: r[kk] for kk in ("want_e", "want_s", "sel_e", "sel_slot", "sel_w", "scores")}


def _route_batches_job(cfg, layer, batches):
    """_route_job for several batches of one layer (its router weights generated once)."""
    return [_route_job(cfg, layer, stream, T, so, drift) for (stream, T, so, drift) in batches]


def _route_rows_job(x, W, b, slot_of, k):
    import oracle
    r = oracle.route(x, W, b, slot_of, k)
    return {kk: r[kk] for kk in ("want_e", "want_s", "sel_e", "sel_slot", "sel_w", "scores")}


# ------------------------------------------------------------------ caller side

def ffn(cfg, x: np.ndarray, sel_slot: np.ndarray, sel_w: np.ndarray, owner: np.ndarray,
        groups: int | None = None) -> np.ndarray:
    """oracle.ffn over the tokens x [T, d] with the experts that own the picked slots, split into token
    groups run in parallel; returns the [T, d] float64 output."""
    T = x.shape[0]
    g = max(1, min(T, groups or workers()))
    bounds = np.linspace(0, T, g + 1).astype(int)
    futs = [pool().submit(_ffn_job, cfg, x[a:b], sel_slot[a:b], np.asarray(sel_w[a:b], np.float64), owner)
            for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    return np.concatenate([f.result() for f in futs], axis=0)


def route_rows(x: np.ndarray, W: np.ndarray, b: np.ndarray, slot_of: np.ndarray, k: int,
               groups: int | None = None) -> dict:
    """oracle.route over the token rows of x, in parallel groups of rows; outputs concatenated along T."""
    T = x.shape[0]
    g = max(1, min(T, groups or workers()))
    bounds = np.linspace(0, T, g + 1).astype(int)
    futs = [pool().submit(_route_rows_job, x[a:bb], W, b, slot_of, k) for a, bb in zip(bounds[:-1], bounds[1:])
            if bb > a]
    parts = [f.result() for f in futs]
    return {kk: np.concatenate([p[kk] for p in parts], axis=0) for kk in parts[0]}


def route_layers(cfg, jobs, per_task: int = 32) -> list:
    """The oracle's routing for many (layer, hidden stream, T, slot_of of the layer, drift) calls, in the order
    given; the calls of one layer are grouped into tasks of up to `per_task` calls."""
    by_layer: dict = {}
    for i, (layer, stream, T, so, drift) in enumerate(jobs):
        by_layer.setdefault(layer, []).append((i, (stream, T, so, drift)))
    futs = []
    for layer, items in by_layer.items():
        for a in range(0, len(items), per_task):
            part = items[a:a + per_task]
            futs.append(([i for i, _ in part], pool().submit(_route_batches_job, cfg, layer, [b for _, b in part])))
    out = [None] * len(jobs)
    for idx, f in futs:
        for i, r in zip(idx, f.result()):
            out[i] = r
    return out
