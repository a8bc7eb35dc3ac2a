#!/usr/bin/env python3
"""Throughput of one routed-MoE layer step over a partial expert set on GB300.

A step is one pass of the whole hot path over one batch of synthetic tokens:
router scores + resident-only top-k with substitution, demand accumulation,
the heavy-miss list, and the grouped MXFP4 SwiGLU expert FFN with weighted
combine (TideLM README, "How adaptive expert loading works", items 1-3).

Headline workload: the DeepSeek-like decode layer (E=256, top-8, d=4096,
ffn=2048, 166 of 256 experts resident, router bias sigma=1.5) at T=64 tokens.
The sweep adds T=1, 8, 32 and the 8192-token prefill layer.

Timing: W warm-up steps, then K steps replayed from a CUDA graph, each timed
with CUDA events on the launching stream; between steps the next batch of
hidden states is copied in and L2 is flushed by writing 256 MiB (outside the
timed events). `--gpus N` under torchrun runs N independent replicas (the
layer does not shard across GPUs here) and reports the summed throughput over
the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/sec (decode T=1..64, prefill 8K); % HBM / FP4 roofline"
GATE_UP_BYTES_PER_EXPERT = None   # filled from the slot record


# ------------------------------------------------------------------ setup

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm_gbs=float(j["hbm_gbs"]), bf16_tflops=float(j["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


class Layer:
    """Device-resident inputs of one layer workload (weights, tables, arena, hidden-state pool)."""

    def __init__(self, cfg: synth.LayerConfig, T: int, pool: int, drift: bool = False, ring: int = 0):
        import torch
        import resident_expert_routed_gb300 as moe
        from resident_expert_routed_gb300.layer import LayerBuffers
        self.cfg, self.T = cfg, T
        W = synth.router_weights(cfg.seed, cfg.E, cfg.d)
        b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma)
        res = synth.resident_set(cfg, b)
        self.n_slots = cfg.resident + cfg.n_ring + ring
        # with a hot-read ring the residents keep the main slots and the ring follows them
        self.slot_of_np = synth.slot_table(cfg, res, cfg.resident if ring else self.n_slots)
        owner = np.full(self.n_slots, -1, np.int32)
        owner[self.slot_of_np[res]] = res
        self.owner_np = owner
        if drift:
            b = synth.drifted_bias(cfg, b)
        self.W_np, self.b_np = W, b
        self.W = torch.from_numpy(W).cuda()
        self.bias = torch.from_numpy(b).cuda()
        self.slot_of = torch.from_numpy(self.slot_of_np).cuda()
        rec = synth.slot_record(cfg.d, cfg.ffn)
        self.rec = rec
        buf = torch.zeros(self.n_slots * rec["slot_bytes"], dtype=torch.uint8, device="cuda")
        synth.fill_slots_device(buf, cfg.d, cfg.ffn, cfg.seed, cfg.E, torch.from_numpy(owner).cuda())
        self.arena = moe.Arena(buf, rec["slot_bytes"], self.n_slots, cfg.d, cfg.ffn, rec["off_gu_codes"],
                               rec["off_gu_scales"], rec["off_dn_codes"], rec["off_dn_scales"])
        self.pool_np = [synth.hidden_bf16(cfg.seed, T, cfg.d, stream=100 + i) for i in range(pool)]
        self.pool = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in self.pool_np]
        self.hidden = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
        self.buf = LayerBuffers(T, cfg.k, cfg.E, cfg.d, cfg.ffn, self.n_slots)
        self.demand = torch.zeros((1, cfg.E), dtype=torch.int64, device="cuda")
        self.miss = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")

    def step(self, stream=None, side=None):
        """One layer step; with `side`, the demand update and heavy-miss list run on that second stream,
        beside the expert FFN, and are joined back before the step ends."""
        from resident_expert_routed_gb300.layer import join, layer_step, step_end
        layer_step(self.hidden, self.W, self.bias, self.slot_of, self.arena, self.demand, self.miss, 0, self.buf,
                   stream, side)
        step_end(self.miss, self.buf, 0.2, stream if side is None else side)
        if side is not None:
            join(stream, side)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running (a default timed region of 50
    steps lasts well under a second, steps with their L2 flushes included); only samples taken after the
    sampler is running, i.e. inside the region, are summarised."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.skip = 0

    def _lines(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for line in f if line.strip())
        except OSError:
            return 0

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # the sampler's start-up can take longer than a short timed region: wait (at most 5 s) until it has
        # written its first line, and summarise only the lines written after that (taken while timing)
        t0 = time.perf_counter()
        while self.proc is not None and self._lines() == 0 and time.perf_counter() - t0 < 5.0:
            if self.proc.poll() is not None:
                break
            time.sleep(0.01)
        self.skip = self._lines()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            lines = [line for line in open(self.path) if line.strip()]
            for line in lines[self.skip:]:
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max((num(r[2]) for r in rows if num(r[2]) is not None), default=None),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) for r in rows if num(r[3]) is not None), default=None)}


def measured_traffic(kernel_json: str):
    """DRAM bytes per launch from the committed ncu capture, or None if the kernel source changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", kernel_json)
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha256_prefix"]:
        return None
    return rec["dram_bytes_read"] + rec["dram_bytes_write"]


def measured_fp4_mma():
    """TFLOP/s of back-to-back mxf4 128x256x64 MMAs on resident operands (the package's microbenchmark)."""
    import subprocess
    exe = os.path.join(ROOT, "resident_expert_routed_gb300", "microbench", "mma_scale_rate")
    if not os.path.exists(exe):
        return None
    try:
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120).stdout
        return json.loads([l for l in out.splitlines() if l.startswith("{")][-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def flush_l2(scratch):
    scratch.add_(1)


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, ws, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_ms: float, ws: int, units_per_rank: int):
    """Whole-job rate: every rank processed units_per_rank per step; the job's step is the slowest rank's."""
    step_ms_max = max_over_ranks(step_ms, ws)
    return step_ms_max, ws * units_per_rank / (step_ms_max / 1000.0)


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ timed runs

def timed_graph_steps(layer: Layer, K: int, W: int, scratch, ws: int):
    """Returns (per-step ms list, launches per step, distinct slots per step)."""
    import torch
    import resident_expert_routed_gb300 as moe
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(W, 1)):
            layer.hidden.copy_(layer.pool[i % len(layer.pool)])
            layer.step(stream, side)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = moe.moe_kernel_launches()
    with torch.cuda.graph(graph, stream=stream):
        layer.step(stream, side)
    launches = moe.moe_kernel_launches() - n0
    torch.cuda.synchronize()
    for i in range(3):                     # graph warm-up
        layer.hidden.copy_(layer.pool[i % len(layer.pool)])
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    slots_used = []
    barrier(ws)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    for i in range(K):
        layer.hidden.copy_(layer.pool[i % len(layer.pool)])
        flush_l2(scratch)
        ev[i][0].record(cur)
        graph.replay()
        ev[i][1].record(cur)
    torch.cuda.synchronize()
    barrier(ws)
    ms = [a.elapsed_time(b) for a, b in ev]
    for i in range(min(K, len(layer.pool))):   # distinct slots touched per batch (for the byte count)
        layer.hidden.copy_(layer.pool[i])
        graph.replay()
        torch.cuda.synchronize()
        s = layer.buf.sel_slot.cpu().numpy()
        slots_used.append(int(len(np.unique(s[s >= 0]))))
    return ms, launches, slots_used, graph


def profiled_steps(layer: Layer, K: int, scratch):
    """Per-kernel device time (events around each launch), eager steps with the same L2 flush."""
    import torch
    import resident_expert_routed_gb300 as moe
    moe.moe_profile_reset()
    moe.moe_profile_enable(True)
    stream = torch.cuda.current_stream()
    used = []
    for i in range(K):
        layer.hidden.copy_(layer.pool[i % len(layer.pool)])
        flush_l2(scratch)
        layer.step(stream)
    torch.cuda.synchronize()
    prof = moe.moe_profile_read()
    moe.moe_profile_enable(False)
    return prof


def e2e_steps(layer: Layer, K: int, scratch):
    """Same metric through the public API with host buffers: each step replays a CapturedStep (the kernels read
    the pinned host batch and write the fp32 output into pinned host memory, one CUDA graph) and waits for it."""
    import torch
    from resident_expert_routed_gb300.layer import CapturedStep
    host_in = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in layer.pool_np]
    cap = CapturedStep(host_in, layer.W, layer.bias, layer.slot_of, layer.arena, layer.demand, layer.miss, 0,
                       layer.buf)
    stream = torch.cuda.current_stream()
    for i in range(3):                     # replay warm-up
        cap.run(i % len(host_in))
    torch.cuda.synchronize()
    total = 0.0
    for i in range(K):
        flush_l2(scratch)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cap.run(i % len(host_in))
        b.record(stream)
        b.synchronize()
        total += a.elapsed_time(b)
    h2d = layer.T * layer.cfg.d * 2
    d2h = layer.T * layer.cfg.d * 4
    return total / K, h2d, d2h


# ------------------------------------------------------------------ full decode step: 60 layers, one arena

def full_decode_step(scratch, hbm_gbs: float, K: int = 10, W: int = 3):
    """The 60-layer decode step (2 tokens, E256 k8 d4096 F2048, one arena of 10,000 main + 64 ring slots shared
    by all layers, the main slots a seeded sample of the 15,360 (layer, expert) ids), replayed from one CUDA graph:
    per layer the step (with the demand work on a side stream, joined before the next layer reuses
    the routing buffers), then the step's heavy-miss list."""
    import torch
    import resident_expert_routed_gb300 as moe
    from resident_expert_routed_gb300.layer import LayerBuffers, join, layer_step, step_end
    cfg, T = synth.FULL, 2
    L, E = cfg.L, cfg.E
    n_slots = cfg.n_main + cfg.n_ring
    slot_of, owner = synth.full_initial_arena(cfg)
    rec = synth.slot_record(cfg.d, cfg.ffn)
    abuf = torch.zeros(n_slots * rec["slot_bytes"], dtype=torch.uint8, device="cuda")
    synth.fill_slots_device(abuf, cfg.d, cfg.ffn, cfg.seed, E, torch.from_numpy(owner).cuda())
    arena = moe.Arena(abuf, rec["slot_bytes"], n_slots, cfg.d, cfg.ffn, rec["off_gu_codes"], rec["off_gu_scales"],
                      rec["off_dn_codes"], rec["off_dn_scales"])
    Wd = torch.from_numpy(np.stack([synth.router_weights(cfg.seed, E, cfg.d, l) for l in range(L)])).cuda()
    bd = torch.from_numpy(np.stack([synth.router_bias(cfg.seed, E, cfg.sigma, l) for l in range(L)])).cuda()
    so = torch.from_numpy(slot_of).cuda()
    xs = [torch.from_numpy(synth.hidden_bf16(cfg.seed, T, cfg.d, stream=l).view(np.int16)).cuda()
          .view(torch.bfloat16) for l in range(L)]
    demand = torch.zeros((L, E), dtype=torch.int64, device="cuda")
    miss = torch.zeros((L, E), dtype=torch.float32, device="cuda")
    buf = LayerBuffers(T, cfg.k, E, cfg.d, cfg.ffn, n_slots)
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    used = []                               # distinct slots each layer reads (for the bytes), from an eager pass
    with torch.cuda.stream(stream):
        for l in range(L):
            layer_step(xs[l], Wd[l], bd[l], so[l * E:(l + 1) * E], arena, demand, miss, l, buf, stream)
            stream.synchronize()
            sl = buf.sel_slot.cpu().numpy()
            used.append(len(np.unique(sl[sl >= 0])))

    def step():
        for l in range(L):
            layer_step(xs[l], Wd[l], bd[l], so[l * E:(l + 1) * E], arena, demand, miss, l, buf, stream, side)
            join(stream, side)
        step_end(miss, buf, 0.2, side)
        join(stream, side)

    with torch.cuda.stream(stream):
        for _ in range(max(W, 1)):
            step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    cur = torch.cuda.current_stream()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ms = []
    for _ in range(K):
        flush_l2(scratch)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        graph.replay()
        b.record(cur)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    step_ms = sum(ms) / len(ms)
    expert_bytes = 3 * cfg.d * cfg.ffn // 2 + 3 * cfg.d * cfg.ffn // 32
    step_bytes = sum(used) * expert_bytes + L * E * cfg.d * 4
    out = {"workload": cfg.name, "tokens_per_s": T / (step_ms / 1000.0), "ms_per_step": step_ms, "layers": L,
           "distinct_experts_per_layer": float(np.mean(used)), "step_bytes": step_bytes,
           "step_hbm_frac": step_bytes / (step_ms / 1000.0) / 1e9 / hbm_gbs,
           "step_frac_of_8_tbps": step_bytes / (step_ms / 1000.0) / 1e9 / 8000.0}
    out["history_256"] = replan_after_history(graph, demand, so, torch.from_numpy(owner).cuda(), arena, cfg, 256)
    del graph, abuf, arena
    torch.cuda.empty_cache()
    return out


def replan_after_history(graph, demand, slot_of, owner, arena, cfg, steps: int):
    """The configured demand history: `steps` replays of the full decode step from a cleared table, then the
    re-plan of the shared arena (CUDA events around moe_arena_replan), then the refill of the slots it
    reassigned from pinned host records (CUDA events around moe_arena_refill's copies). The refill's records are
    64 pinned stand-ins reused for every expert: its timing is that of the copy volume; the arena's contents are
    not used afterwards."""
    import torch
    import resident_expert_routed_gb300 as moe
    L, E = cfg.L, cfg.E
    demand.zero_()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        graph.replay()
    torch.cuda.synchronize()
    hist_s = time.perf_counter() - t0
    loads = torch.empty(cfg.n_main, dtype=torch.int32, device="cuda")
    n_loads = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(moe.moe_replan_workspace_bytes(L, E), dtype=torch.uint8, device="cuda")
    so0, ow0 = slot_of.clone(), owner.clone()
    cur = torch.cuda.current_stream()
    times = []
    for _ in range(3):                          # the same re-plan three times, from the same tables
        slot_of.copy_(so0)
        owner.copy_(ow0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        moe.moe_arena_replan(demand, cfg.n_main, slot_of, owner, loads, n_loads, ws)
        b.record(cur)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    n = int(n_loads.item())
    sb = arena.slot_bytes
    stand_in = torch.empty(64 * sb, dtype=torch.uint8).pin_memory()
    records = [stand_in.data_ptr() + (f % 64) * sb for f in range(L * E)]
    copy_stream = torch.cuda.Stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    copied = moe.moe_arena_refill(arena, records, loads, n_loads, owner, cur, copy_stream)
    b.record(cur)
    torch.cuda.synchronize()
    refill_ms = a.elapsed_time(b)
    D = demand.cpu().numpy().astype(np.float64) / 2.0 ** 40
    res = {"steps": steps, "history_wall_s": hist_s, "demand_total": float(D.sum()),
           "experts_with_demand": int((D > 0).sum()), "replan_ms": float(np.median(times)), "n_loads": n,
           "refill_ms": refill_ms, "refill_slots": copied,
           "refill_gb_per_s": copied * sb / (refill_ms / 1000.0) / 1e9 if refill_ms > 0 and copied else None,
           "note": "re-plan of the 10,000-slot main arena over 60 x 256 experts from the 256-step history; the "
                   "refill copies the reassigned slots from pinned host memory (stand-in records)"}
    del stand_in
    return res


# ------------------------------------------------------------------ hot-read ring, on and off

def prefill_chunk_report(layer: Layer, prof: dict) -> dict:
    """The chunk's demand update and heavy-miss list (share >= 0.2, at most 16): the list the last step left,
    the demand it recorded, and the two kernels' average times from the profiled steps."""
    import torch
    layer.demand.zero_()
    layer.hidden.copy_(layer.pool[0])
    layer.step()
    torch.cuda.synchronize()
    n = int(layer.buf.hot_n.item())
    D = layer.demand.cpu().numpy().astype(np.float64) / 2.0 ** 40
    us = {k: 1000.0 * t / c for k, (c, t) in prof.items()}
    return {"heavy_misses": [int(f) for f in layer.buf.hot_flat.cpu().numpy()[:n]],
            "heavy_shares": [float(v) for v in layer.buf.hot_share.cpu().numpy()[:n]],
            "demand_total": float(D.sum()), "experts_with_demand": int((D > 0).sum()),
            "demand_accumulate_us": us.get("demand_accumulate"), "hot_miss_select_us": us.get("hot_miss_select")}


def ring_on_off(T: int, steps: int, n_ring: int = 64):
    """Decode steps (drifted bias, so misses happen) with the asynchronous hot-read ring on and off.

    A pinned host store of every absent expert stands in for the drive. Both modes synchronise the host
    once per step (a decode loop reads its sampled token); the ring's copies run on their own stream.
    """
    import torch
    import resident_expert_routed_gb300 as moe
    cfg = synth.DECODE
    lay = Layer(cfg, T, pool=8, drift=True, ring=n_ring)
    sb = lay.rec["slot_bytes"]
    absent = np.flatnonzero(lay.slot_of_np < 0).astype(np.int32)
    store = torch.empty(len(absent) * sb, dtype=torch.uint8, pin_memory=True)
    tmp = torch.empty(16 * sb, dtype=torch.uint8, device="cuda")
    for i0 in range(0, len(absent), 16):
        part = absent[i0:i0 + 16]
        synth.fill_slots_device(tmp, cfg.d, cfg.ffn, cfg.seed, cfg.E, torch.from_numpy(part).cuda())
        store[i0 * sb:(i0 + len(part)) * sb].copy_(tmp[:len(part) * sb])
    records = [None] * cfg.E
    for i, f in enumerate(absent):
        records[int(f)] = store.data_ptr() + i * sb
    res = {}
    for mode in ("off", "on"):
        lay.slot_of.copy_(torch.from_numpy(lay.slot_of_np))
        owner = torch.from_numpy(lay.owner_np).cuda()
        lay.demand.zero_()
        lay.miss.zero_()
        ring = moe.HotRing(lay.arena, cfg.resident, n_ring, records) if mode == "on" else None
        fetched, t0 = 0, 0.0
        for i in range(3 + steps):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fetched = 0
            lay.hidden.copy_(lay.pool[i % len(lay.pool)])
            lay.step()
            if ring is not None:
                fetched += ring.step(lay.buf.hot_flat, lay.buf.hot_n, lay.slot_of, owner)
            else:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / steps
        if ring is not None:
            ring.close()
        res[f"ring_{mode}"] = {"tokens_per_s": T / dt, "ms_per_step": 1000.0 * dt}
        if mode == "on":
            res["ring_on"]["experts_fetched_per_step"] = fetched / steps
            res["ring_on"]["h2d_gb_per_step"] = fetched / steps * sb / 1e9
    res["workload"] = (f"{cfg.name} with the bias drifted after the resident set was fixed, T={T}, "
                       f"{n_ring} ring slots on top, {len(absent)} absent experts in a pinned host store")
    return res


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)

def oracle_sample_run(cfg: synth.LayerConfig, x_bits, W, bias, slot_of, owner, n_tok: int) -> float:
    """Seconds for the oracle to run the whole step (route, demand, heavy misses, FFN) on n_tok tokens."""
    import oracle
    x = x_bits[:n_tok]
    t0 = time.perf_counter()
    r = oracle.route(x, W, bias, slot_of, cfg.k)
    D = np.zeros((1, cfg.E))
    M = np.zeros((1, cfg.E))
    oracle.demand(r["want_e"], r["want_s"], slot_of, 0, D, M)
    oracle.hot_miss_select(M, 0.2, 16)
    used = sorted({int(s) for s in r["sel_slot"].ravel() if s >= 0})
    index = {s: i for i, s in enumerate(used)}
    sel_u = np.vectorize(lambda s: index.get(int(s), -1))(r["sel_slot"]).astype(np.int32)
    experts = [synth.expert_weights(cfg.seed, int(owner[s]) // cfg.E, int(owner[s]) % cfg.E, cfg.d, cfg.ffn)
               for s in used]
    oracle.ffn(x, sel_u, r["sel_w"], experts, cfg.d, cfg.ffn)
    return time.perf_counter() - t0


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_reference(args, rank, ws):
    """The oracle, as it stands, on the host cores: each step a bounded sample of the headline workload."""
    if rank != 0:
        return
    cfg, T = synth.DECODE, args.T
    W = synth.router_weights(cfg.seed, cfg.E, cfg.d)
    b = synth.router_bias(cfg.seed, cfg.E, cfg.sigma)
    res = synth.resident_set(cfg, b)
    slot_of = synth.slot_table(cfg, res, cfg.resident)
    owner = np.full(cfg.resident, -1, np.int32)
    owner[slot_of[res]] = res
    n_tok = 2
    for i in range(args.warmup):
        oracle_sample_run(cfg, synth.hidden_bf16(cfg.seed, T, cfg.d, stream=100 + i), W, b, slot_of, owner, n_tok)
    secs = 0.0
    for i in range(args.steps):
        secs += oracle_sample_run(cfg, synth.hidden_bf16(cfg.seed, T, cfg.d, stream=100 + i), W, b, slot_of, owner,
                                  n_tok)
    value = n_tok * args.steps / secs
    sample = f"{n_tok} of the {T} tokens of each batch: route, demand, heavy misses and FFN (float64)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name}, T={T}", "reference": "the C++ oracle (no runnable reference code "
                       "exists: the method's pages hold no code)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main

def run_ours(args, rank, ws, local):
    import torch
    import resident_expert_routed_gb300 as moe
    moe.load()
    pk = peaks()
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    cfg, T = synth.DECODE, args.T
    layer = Layer(cfg, T, pool=8)
    rec = layer.rec
    gate_up_bytes = rec["gu_codes_bytes"] + rec["gu_scales_bytes"]
    expert_bytes = gate_up_bytes + rec["dn_codes_bytes"] + rec["dn_scales_bytes"]

    t_wall = time.perf_counter()
    with ClockSampler(local) as clk:
        ms, launches, slots_used, _ = timed_graph_steps(layer, args.steps, args.warmup, scratch, ws)
    wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    step_ms = sum(ms) / len(ms)
    step_ms_max, value = job_throughput(step_ms, ws, T)

    prof = profiled_steps(layer, min(args.steps, 16), scratch)
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    gu = prof.get("ffn_gemm_gate_up", (1, float("nan")))
    u_mean = float(np.mean(slots_used))
    achieved = u_mean * gate_up_bytes / (gu[1] / gu[0] / 1000.0) / 1e9
    roofline = {"bound": "hbm", "kernel": "ffn_gemm_gate_up", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "traffic": measured_traffic("ffn_gemm_gate_up_decode_T64.json"),
                "peak_source": f"{pk['source']} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if pk["source"] == "measured" else "fallback 6800 GB/s",
                "algorithmic_bytes_per_launch": u_mean * gate_up_bytes,
                "units": f"{u_mean:.1f} distinct experts x {gate_up_bytes} B gate/up codes+scales",
                "frac_of_8_tbps": achieved / 8000.0,
                "kernel_ms": gu[1] / gu[0], "dominant_kernel": dom[0]}
    step_bytes = u_mean * expert_bytes + cfg.E * cfg.d * 4
    kernels = {k: {"launches": n, "avg_us": 1000.0 * t / n} for k, (n, t) in prof.items()}

    e2e_ms, h2d, d2h = e2e_steps(layer, min(args.steps, 20), scratch)

    sweep = {}
    if not args.no_sweep:
        for Ts in (1, 8, 32):
            ls = Layer(cfg, Ts, pool=4)
            m, _, su, _ = timed_graph_steps(ls, 20, 3, scratch, 1)
            sm = sum(m) / len(m)
            rate = (np.mean(su) * expert_bytes + cfg.E * cfg.d * 4) / (sm / 1000.0) / 1e9
            sweep[f"decode_T{Ts}"] = {"tokens_per_s": Ts / (sm / 1000.0), "ms_per_step": sm,
                                      "distinct_experts": float(np.mean(su)),
                                      "step_hbm_frac": rate / pk["hbm_gbs"], "step_frac_of_8_tbps": rate / 8000.0}
            del ls
        sweep[f"decode_T{T}"] = {"tokens_per_s": T / (step_ms / 1000.0), "ms_per_step": step_ms,
                                 "distinct_experts": u_mean,
                                 "step_hbm_frac": step_bytes / (step_ms / 1000.0) / 1e9 / pk["hbm_gbs"],
                                 "step_frac_of_8_tbps": step_bytes / (step_ms / 1000.0) / 1e9 / 8000.0}
        sweep["hot_ring"] = ring_on_off(T, 30)
        gcfg = synth.GLM
        g_bytes = 3 * gcfg.d * gcfg.ffn // 2 + 3 * gcfg.d * gcfg.ffn // 32
        for Tg in (1, 16, 64):
            lg = Layer(gcfg, Tg, pool=4)
            m, _, su, _ = timed_graph_steps(lg, 20, 3, scratch, 1)
            sm = sum(m) / len(m)
            rate = (np.mean(su) * g_bytes + gcfg.E * gcfg.d * 4) / (sm / 1000.0) / 1e9
            sweep[f"glm_T{Tg}"] = {"workload": gcfg.name, "tokens_per_s": Tg / (sm / 1000.0), "ms_per_step": sm,
                                   "distinct_experts": float(np.mean(su)),
                                   "step_hbm_frac": rate / pk["hbm_gbs"], "step_frac_of_8_tbps": rate / 8000.0}
            del lg
        if not args.no_full:
            sweep["full_decode_L60_T2"] = full_decode_step(scratch, pk["hbm_gbs"])
        if not args.no_prefill:
            lp = Layer(synth.PREFILL, 8192, pool=2)
            m, _, su, _ = timed_graph_steps(lp, 5, 2, scratch, 1)
            sm = sum(m) / len(m)
            P = 8192 * cfg.k
            flops = P * 6 * cfg.d * cfg.ffn
            # FP4 peak by the nominal dense ratio to bf16 (13.5 / 2.25 PFLOP/s) times the measured bf16 burst;
            # also reported: the datasheet figure and the measured mxf4 MMA rate on resident operands
            fp4_peak = pk["bf16_tflops"] * 6.0
            mma = measured_fp4_mma()
            pprof = profiled_steps(lp, 4, scratch)
            gemm = {}
            for name, fl in (("ffn_gemm_gate_up", 2.0 * P * cfg.d * 2 * cfg.ffn), ("ffn_gemm_down", 2.0 * P * cfg.ffn * cfg.d)):
                n, t = pprof.get(name, (1, float("nan")))
                tf = fl / (t / n / 1000.0) / 1e12
                gemm[name] = {"us": 1000.0 * t / n, "tflops": tf, "frac_fp4_peak": tf / fp4_peak,
                              "frac_fp4_datasheet": tf / 13500.0,
                              "frac_fp4_mma_measured": tf / mma["mxf4_tflops"] if mma else None}
            chunk = prefill_chunk_report(lp, pprof)
            sweep["prefill_T8192"] = {"tokens_per_s": 8192 / (sm / 1000.0), "ms_per_step": sm, "chunk": chunk,
                                      "ffn_tflops": flops / (sm / 1000.0) / 1e12,
                                      "fp4_peak_tflops": fp4_peak,
                                      "fp4_peak_source": f"{pk['source']} bf16 burst x 6 (nominal fp4/bf16 dense ratio)",
                                      "step_frac_fp4_peak": flops / (sm / 1000.0) / 1e12 / fp4_peak,
                                      "fp4_datasheet_tflops": 13500.0,
                                      "fp4_mma_microbench": mma,
                                      "gemms": gemm,
                                      "kernels_us": {k: 1000.0 * t / n for k, (n, t) in pprof.items()},
                                      "distinct_experts": float(np.mean(su))}
            del lp
            torch.cuda.empty_cache()
            ld = Layer(synth.PREFILL, 8192, pool=1, drift=True)
            ld.hidden.copy_(ld.pool[0])
            ld.step()
            torch.cuda.synchronize()
            n = int(ld.buf.hot_n.item())
            sweep["prefill_T8192"]["chunk_drifted"] = {
                "workload": f"{synth.PREFILL.name} with the bias drifted after the resident set was fixed",
                "heavy_misses": [int(f) for f in ld.buf.hot_flat.cpu().numpy()[:n]],
                "heavy_shares": [float(v) for v in ld.buf.hot_share.cpu().numpy()[:n]],
                "demand_total": float(ld.demand.cpu().numpy().astype(np.float64).sum() / 2.0 ** 40)}
            del ld
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # bounded sample: whole T-token batches of the pool until at least 10 s of oracle work (at most 3)
        secs, n_batches = 0.0, 0
        while n_batches < min(3, len(layer.pool_np)) and (secs < 10.0 or n_batches == 0):
            secs += oracle_sample_run(cfg, layer.pool_np[n_batches], layer.W_np, layer.b_np, layer.slot_of_np,
                                      layer.owner_np, T)
            n_batches += 1
        cpu = {"value": n_batches * T / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{n_batches} whole T={T} batch{'es' if n_batches > 1 else ''}: route, demand, heavy "
                         f"misses and FFN in float64, one thread ({secs:.1f} s)", "cpu": cpu_model()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "mxfp4", "data": "synthetic",
                "config": {"workload": f"{cfg.name}, T={T} tokens per layer step (one step = route + demand + "
                                       f"heavy-miss list + expert FFN)",
                           "l2": "flushed between steps (256 MiB write, outside the timed events)",
                           "timing": "CUDA graph replay per step, CUDA events on the launching stream",
                           "parallelism": f"replicas x{ws}"},
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": T / (e2e_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                        "path": "pinned host batch, read by the kernels -> CapturedStep replay (layer_step/step_end through the C ABI in one CUDA graph) -> fp32 output written into pinned host memory"},
                "gpu_launches": launches * args.steps, "clocks": clocks, "kernels": kernels, "sweep": sweep,
                "wall_s": wall}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-full", action="store_true", help="skip the 60-layer decode step of the sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, ws)
    else:
        run_ours(args, rank, ws, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
