"""One routed-MoE layer step as a sequence of C-ABI calls on one stream (or two).

TideLM README, "How adaptive expert loading works", items 1-3, per layer:
route to resident experts (with substitution), record demand and miss shares,
run the expert FFN with the weighted combine; per step, extract the heavy
misses. This module only holds the device buffers and orders the calls; all
arithmetic is in the CUDA library.
"""
from __future__ import annotations

import torch

from . import (Arena, moe_arena_refill, moe_arena_replan, moe_demand_accumulate, moe_demand_decay,
               moe_expert_ffn_mxfp4, moe_expert_ffn_prefetch, moe_hot_miss_select, moe_replan_workspace_bytes,
               moe_route_resident, moe_workspace_bytes)


class LayerBuffers:
    """Preallocated device outputs and workspace for batches of up to T tokens."""

    def __init__(self, T: int, k: int, E: int, d: int, ffn: int, n_slots: int, device="cuda", cap: int = 16):
        dev = torch.device(device)
        self.T, self.k = T, k
        self.want_e = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.want_s = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.sel_e = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.sel_slot = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.sel_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.out = torch.empty((T, d), dtype=torch.float32, device=dev)
        self.workspace = torch.empty(moe_workspace_bytes(T, k, d, ffn, E, n_slots), dtype=torch.uint8, device=dev)
        self.hot_flat = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        self.hot_share = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
        self.hot_n = torch.zeros(1, dtype=torch.int32, device=dev)
        self.cap = cap


def layer_step(hidden: torch.Tensor, w_router: torch.Tensor, bias, slot_of: torch.Tensor, arena: Arena,
               demand: torch.Tensor, miss_max: torch.Tensor, layer: int, buf: LayerBuffers, stream=None,
               side=None, out: torch.Tensor | None = None, prefetch: bool = False) -> torch.Tensor:
    """route -> demand -> expert FFN; returns the output (fp32 [T, d]): buf.out, or `out` when given.

    `hidden` and `out` may be pinned host tensors: the kernels then read the
    batch and write the output in host memory directly.

    With a second stream `side`, the demand update runs there, beside the
    expert FFN (it reads only the routing outputs), and so does the L2
    prefetch of the weights the FFN reads first when `prefetch` is set. The
    caller then runs ``step_end`` on `side` too and calls ``join(stream,
    side)`` before the routing outputs in `buf` are written again (the next
    layer's step when layers share `buf`, else the next step's) and before it
    reads the tables. The prefetch is off by default: it pays only for a
    single token through one layer with a cold L2 (about 1 us of 50); from
    two tokens on, and through consecutive layers, it competes with the
    gate/up GEMM for HBM and the step is slower.
    """
    main = torch.cuda.current_stream() if stream is None else stream
    moe_route_resident(hidden, w_router, bias, slot_of, buf.k, buf.want_e, buf.want_s, buf.sel_e, buf.sel_slot,
                       buf.sel_w, buf.workspace, main)
    if side is None:
        moe_demand_accumulate(buf.want_e, buf.want_s, slot_of, layer, demand, miss_max, main)
    else:
        side.wait_stream(main)
        if prefetch:
            moe_expert_ffn_prefetch(buf.sel_slot, arena, side)
        moe_demand_accumulate(buf.want_e, buf.want_s, slot_of, layer, demand, miss_max, side)
    dst = buf.out if out is None else out
    moe_expert_ffn_mxfp4(hidden, buf.sel_slot, buf.sel_w, arena, dst, buf.workspace, main)
    return dst


def join(stream, side) -> None:
    """The main stream waits for the side stream's work (demand update, heavy-miss list, prefetch)."""
    (torch.cuda.current_stream() if stream is None else stream).wait_stream(side)


def step_end(miss_max: torch.Tensor, buf: LayerBuffers, threshold: float = 0.2, stream=None):
    """Heavy-miss list of the step (README item 3); resets miss_max."""
    moe_hot_miss_select(miss_max, threshold, buf.cap, buf.hot_flat, buf.hot_share, buf.hot_n, stream)
    return buf.hot_flat, buf.hot_share, buf.hot_n


class CapturedStep:
    """A layer step captured once in a CUDA graph and replayed.

    Each replay takes a batch from a pinned host buffer, runs the step (the
    demand update and heavy-miss list on a side stream), and leaves the fp32
    output in the pinned ``host_out``: one graph launch per step instead of one
    host call per kernel. With ``zero_copy`` (the default) the kernels read the
    batch and write the output in host memory directly; otherwise the graph
    copies the batch in and the output out with the copy engines around a
    device-resident step. Everything the step touches is fixed at
    capture (weights, tables, arena, demand and miss tables, ``buf``, the host
    buffers); ``run(i)`` replays the graph of ``host_inputs[i]``, whose contents
    the caller may rewrite between replays. Construction runs one eager step
    (it updates the demand and miss tables like any step) before capturing.
    """

    def __init__(self, host_inputs, w_router: torch.Tensor, bias, slot_of: torch.Tensor, arena: Arena,
                 demand: torch.Tensor, miss_max: torch.Tensor, layer: int, buf: LayerBuffers,
                 host_out: torch.Tensor | None = None, threshold: float = 0.2, zero_copy: bool = True):
        T, d = host_inputs[0].shape
        for h in host_inputs:
            if not h.is_pinned() or h.shape != (T, d) or h.dtype != torch.bfloat16:
                raise ValueError("host inputs must be pinned bf16 [T, d] tensors of one shape")
        self.main, self.side = torch.cuda.Stream(), torch.cuda.Stream()
        self.hidden = None if zero_copy else torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        self.host_out = host_out if host_out is not None else torch.empty((T, d), dtype=torch.float32).pin_memory()
        self.buf = buf

        def body(h_in):
            if zero_copy:
                layer_step(h_in, w_router, bias, slot_of, arena, demand, miss_max, layer, buf, self.main, self.side,
                           out=self.host_out)
            else:
                self.hidden.copy_(h_in, non_blocking=True)
                layer_step(self.hidden, w_router, bias, slot_of, arena, demand, miss_max, layer, buf, self.main,
                           self.side)
            step_end(miss_max, buf, threshold, self.side)
            join(self.main, self.side)
            if not zero_copy:
                self.host_out.copy_(buf.out, non_blocking=True)

        self.main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.main):
            body(host_inputs[0])
        self.main.synchronize()
        self.graphs = []
        for h in host_inputs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.main):
                body(h)
            self.graphs.append(g)

    def run(self, i: int = 0) -> torch.Tensor:
        """Replay the step for host_inputs[i] on the current stream; host_out is valid after a sync."""
        self.graphs[i].replay()
        return self.host_out


class Cadence:
    """When to plan the shared arena again (README item 1: after a prompt's prefill, after every few hundred
    generated tokens, and between requests; "Settings worth knowing" makes the interval a setting).

    Pure host bookkeeping: ``step(tokens, prefill)`` counts the tokens of a finished step and says whether a
    re-plan is due now; ``request_done()`` says so at a request boundary (when anything was generated since
    the last re-plan). ``every_tokens`` = 0 turns the token interval off."""

    def __init__(self, every_tokens: int = 256, after_prefill: bool = True, between_requests: bool = True):
        if every_tokens < 0:
            raise ValueError("every_tokens must be >= 0")
        self.every_tokens = every_tokens
        self.after_prefill = after_prefill
        self.between_requests = between_requests
        self.tokens_since = 0

    def step(self, tokens: int, prefill: bool = False) -> bool:
        self.tokens_since += tokens
        due = (prefill and self.after_prefill) or (self.every_tokens > 0 and self.tokens_since >= self.every_tokens)
        if due:
            self.tokens_since = 0
        return due

    def request_done(self) -> bool:
        due = self.between_requests and self.tokens_since > 0
        if due:
            self.tokens_since = 0
        return due


class Adaptation:
    """Re-plans the shared arena from the demand history on a Cadence and refills the slots it reassigns.

    Each re-plan (README item 1) ranks every (layer, expert) by accumulated demand (moe_arena_replan), copies
    the admitted experts' records from the host store into their new slots on a copy stream
    (moe_arena_refill; the compute stream waits for them), and then scales the history by ``decay`` so that
    demand seen before this re-plan weighs less than demand seen after it ("Settings worth knowing": how
    quickly the resident set follows a change in traffic; decay = 1 keeps the plain sum). ``records``: one
    host address per flat id (layer * E + e) of that expert's record, or None where the store has none."""

    def __init__(self, demand: torch.Tensor, slot_of: torch.Tensor, owner: torch.Tensor, arena: Arena, n_main: int,
                 records, cadence: Cadence | None = None, decay: float = 1.0):
        if not 0.0 <= decay <= 1.0:
            raise ValueError("decay must be in [0, 1]")
        L, E = demand.shape
        self.demand, self.slot_of, self.owner, self.arena = demand, slot_of, owner, arena
        self.n_main, self.records, self.decay = n_main, list(records), decay
        self.cadence = cadence if cadence is not None else Cadence()
        dev = demand.device
        self.loads = torch.empty(n_main, dtype=torch.int32, device=dev)
        self.n_loads = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(moe_replan_workspace_bytes(L, E), dtype=torch.uint8, device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.replans = 0
        self.loaded = 0

    def replan(self, stream=None) -> int:
        """Re-plan now; returns the number of slots refilled."""
        moe_arena_replan(self.demand, self.n_main, self.slot_of, self.owner, self.loads, self.n_loads,
                         self.workspace, stream)
        n = moe_arena_refill(self.arena, self.records, self.loads, self.n_loads, self.owner, stream,
                             self.copy_stream)
        if self.decay < 1.0:
            moe_demand_decay(self.demand, self.decay, stream)
        self.replans += 1
        self.loaded += n
        return n

    def after_step(self, tokens: int, prefill: bool = False, stream=None) -> int:
        """Call after a step's work is enqueued; re-plans when the cadence says so. Returns slots refilled."""
        return self.replan(stream) if self.cadence.step(tokens, prefill) else 0

    def request_done(self, stream=None) -> int:
        return self.replan(stream) if self.cadence.request_done() else 0
