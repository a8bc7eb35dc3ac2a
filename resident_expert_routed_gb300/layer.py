"""One routed-MoE layer step as a sequence of C-ABI calls on one stream (or two).

TideLM README, "How adaptive expert loading works", items 1-3, per layer:
route to resident experts (with substitution), record demand and miss shares,
run the expert FFN with the weighted combine; per step, extract the heavy
misses. This module only holds the device buffers and orders the calls; all
arithmetic is in the CUDA library.
"""
from __future__ import annotations

import torch

from . import (Arena, moe_demand_accumulate, moe_expert_ffn_mxfp4, moe_hot_miss_select, moe_route_resident,
               moe_workspace_bytes)


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
               side=None) -> torch.Tensor:
    """route -> demand -> expert FFN; returns buf.out (fp32 [T, d]).

    With a second stream `side`, the demand update runs there, beside the
    expert FFN (it reads only the routing outputs). The caller then runs
    ``step_end`` on `side` too and calls ``join(stream, side)`` before the next
    step's routing rewrites want_e / want_s, or before it reads the tables.
    """
    main = torch.cuda.current_stream() if stream is None else stream
    moe_route_resident(hidden, w_router, bias, slot_of, buf.k, buf.want_e, buf.want_s, buf.sel_e, buf.sel_slot,
                       buf.sel_w, buf.workspace, main)
    if side is None:
        moe_demand_accumulate(buf.want_e, buf.want_s, slot_of, layer, demand, miss_max, main)
    else:
        side.wait_stream(main)
        moe_demand_accumulate(buf.want_e, buf.want_s, slot_of, layer, demand, miss_max, side)
    moe_expert_ffn_mxfp4(hidden, buf.sel_slot, buf.sel_w, arena, buf.out, buf.workspace, main)
    return buf.out


def join(stream, side) -> None:
    """The main stream waits for the side stream's demand and heavy-miss work."""
    (torch.cuda.current_stream() if stream is None else stream).wait_stream(side)


def step_end(miss_max: torch.Tensor, buf: LayerBuffers, threshold: float = 0.2, stream=None):
    """Heavy-miss list of the step (README item 3); resets miss_max."""
    moe_hot_miss_select(miss_max, threshold, buf.cap, buf.hot_flat, buf.hot_share, buf.hot_n, stream)
    return buf.hot_flat, buf.hot_share, buf.hot_n
