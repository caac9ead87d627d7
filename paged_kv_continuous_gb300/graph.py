"""A whole decode step over L layers captured as one CUDA graph.

koas-w, "errors and solutions", section "CUDA Graph": the engine allocates
fixed-shape static buffers once (input ids, slot_mapping, position ids,
block_table, context_lens), updates their values in place every step, and
replays one captured graph per step, so the step's hundreds of launches are
submitted at once.

``DecodeStepGraph`` captures, for every layer, the two library calls of a
decode step -- ``pa_rope_store_kv`` (or ``pa_store_kv`` when no rotary
tables are given) and then ``pa_decode`` -- both launched with
``PA_LAUNCH_PDL``, so each kernel's start-up overlaps the tail of the one
before.  With ``fused=True`` a layer is one call, ``pa_store_decode`` (or
``pa_rope_store_decode`` with rotary tables, which leaves q as it is), which
also requests its first K/V pages early (``PA_LAUNCH_EARLY_KV``) whenever
the call before it is another layer's, on other pools.  This module only records calls into the graph; every step of
the computation runs in the library's kernels.

Static state (fixed at capture): the batch size, the block-table width, the
per-layer tensors (their addresses are baked into the graph), the split
count and the decode workspace.  Values the caller changes between replays,
in place: the index buffers, through :meth:`DecodeStepGraph.update`, and
each layer's new q / k / v rows (written into the layer tensors given at
construction; with rotary tables and two calls per layer q is rotated in
place, so it must be refilled before every replay; the fused call leaves q
as it is).  The decode kernel partitions its work from
``context_lens`` on the device, so a replay follows new lengths without a
new capture.
"""
from __future__ import annotations

import torch

from . import ops


class DecodeStepGraph:
    """One decode step of ``len(layers)`` layers as a single CUDA graph.

    layers: list of dicts with bf16 CUDA tensors ``q`` [B, Hq, D] (contiguous),
    ``k``, ``v`` [B, Hkv, D] (the step's new token rows), ``k_cache``,
    ``v_cache`` (the layer's pools) and ``out`` [B, Hq, D].
    block_tables int32 [B, max_blocks], context_lens int32 [B], slot_mapping
    int32 [B]: the initial values of the static index buffers (copied).
    positions int32 [B] with cos_table / sin_table float32 [max_position,
    D/2]: rotary embedding of q and k fused into the store.
    fused: one pa_store_decode (pa_rope_store_decode with rotary tables)
    per layer instead of a store and a decode; slot_mapping[b] must then be
    the slot of position context_lens[b] - 1 under the block table.
    """

    def __init__(self, layers, block_tables, context_lens, slot_mapping, scale,
                 positions=None, cos_table=None, sin_table=None, num_splits=0, device=None,
                 fused=False):
        if not layers:
            raise ops.PagedAttentionError("DecodeStepGraph needs at least one layer")
        if (cos_table is None) != (positions is None) or (cos_table is None) != (sin_table is None):
            raise ops.PagedAttentionError("positions, cos_table and sin_table go together")
        self.fused = bool(fused)
        dev = layers[0]["q"].device if device is None else torch.device(device)
        self.layers = layers
        self.scale = float(scale)
        self.rope = cos_table is not None
        # static index buffers: one copy, shared by every layer
        self.block_tables = block_tables.to(dev, torch.int32).clone()
        self.context_lens = context_lens.to(dev, torch.int32).clone()
        self.slot_mapping = slot_mapping.to(dev, torch.int32).clone()
        self.positions = positions.to(dev, torch.int32).clone() if self.rope else None
        self.cos_table = cos_table.to(dev, torch.float32).contiguous() if self.rope else None
        self.sin_table = sin_table.to(dev, torch.float32).contiguous() if self.rope else None
        B, Hq, D = layers[0]["q"].shape
        Hkv = layers[0]["k"].shape[1]
        idx = dev.index if dev.index is not None else torch.cuda.current_device()
        self.num_splits = num_splits or ops.default_splits(Hq, Hkv, idx)
        self.workspace = ops.decode_workspace(Hq, Hkv, self.num_splits, D, dev)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.graph = torch.cuda.CUDAGraph()
        self._capture()

    def _layer_calls(self, x, prev):
        if self.fused:
            # early K/V requests only behind another layer's call on other pools
            early = prev is not None and prev["k_cache"].data_ptr() != x["k_cache"].data_ptr() \
                and prev["v_cache"].data_ptr() != x["v_cache"].data_ptr()
            if self.rope:
                ops.rope_store_decode(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                      self.slot_mapping, self.block_tables, self.context_lens,
                                      self.scale, self.positions, self.cos_table, self.sin_table,
                                      out=x["out"], num_splits=self.num_splits,
                                      workspace=self.workspace, pdl=True, early_kv=early)
            else:
                ops.store_decode(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                 self.slot_mapping, self.block_tables, self.context_lens,
                                 self.scale, out=x["out"], num_splits=self.num_splits,
                                 workspace=self.workspace, pdl=True, early_kv=early)
            return
        if self.rope:
            ops.rope_store_kv(x["q"], x["k"], x["v"], self.positions, self.cos_table,
                              self.sin_table, x["k_cache"], x["v_cache"], self.slot_mapping,
                              q_out=x["q"], error_flags=self.error_word, pdl=True)
        else:
            ops.store_kv(x["k"], x["v"], x["k_cache"], x["v_cache"], self.slot_mapping,
                         error_flags=self.error_word, pdl=True)
        ops.decode(x["q"], x["k_cache"], x["v_cache"], self.block_tables, self.context_lens,
                   self.scale, out=x["out"], num_splits=self.num_splits,
                   workspace=self.workspace, pdl=True)

    def _capture(self):
        # One eager decode call first: kernel attributes (the large dynamic
        # shared memory) are set on a kernel's first launch, which must not
        # happen during capture.  It writes only layer 0's `out`, which every
        # replay rewrites.  The capture itself records the calls without
        # running them, so the pools and q / k / v are left as they are.
        x = self.layers[0]
        ops.decode(x["q"], x["k_cache"], x["v_cache"], self.block_tables, self.context_lens,
                   self.scale, out=x["out"], num_splits=self.num_splits,
                   workspace=self.workspace)
        torch.cuda.synchronize()
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(self.graph, stream=self.stream):
            prev = None
            for x in self.layers:
                self._layer_calls(x, prev)
                prev = x
        torch.cuda.current_stream().wait_stream(self.stream)

    def launches_per_replay(self) -> int:
        return (1 if self.fused else 2) * len(self.layers)

    def update(self, block_tables=None, context_lens=None, slot_mapping=None, positions=None):
        """Write new values into the static index buffers (same shapes), in
        stream order before the next replay."""
        for src, dst, name in ((block_tables, self.block_tables, "block_tables"),
                               (context_lens, self.context_lens, "context_lens"),
                               (slot_mapping, self.slot_mapping, "slot_mapping"),
                               (positions, self.positions, "positions")):
            if src is None:
                continue
            if dst is None:
                raise ops.PagedAttentionError(f"{name}: this graph has no such buffer")
            if tuple(src.shape) != tuple(dst.shape):
                raise ops.PagedAttentionError(
                    f"{name} has shape {tuple(src.shape)}; the graph was captured with "
                    f"{tuple(dst.shape)}")
            dst.copy_(src.to(torch.int32), non_blocking=True)

    def replay(self):
        """Run the captured step on the current stream (after any update)."""
        self.graph.replay()

    def read_error_word(self) -> int:
        """Device error bits of the store calls (and the decode workspace's)."""
        return int(self.error_word.item()) | ops.read_error_word(self.workspace)
