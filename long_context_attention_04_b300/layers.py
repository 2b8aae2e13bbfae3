"""Per-layer orchestration of the attention path: the order of the C-ABI calls of one CSA or
HCA layer step, over device buffers the caller (or the layer object) owns.

The order follows the pages' description of a layer (DeepSeek-V4 hybrid attention,
gxgjx.lffhtl.com/lxrt/355279.html section 混肃穆力机制): compress the block the new token
completes (CSA step one / HCA), refresh the window ring with the new token's row, score and
select entries (CSA step two), run the core attention with window and sink (CSA step three /
HCA), and, in a full block, the grouped output projection (CSA step four).  No arithmetic
happens here; every step is a library call.
"""
from __future__ import annotations

import dataclasses

import torch

from . import api
from .api import AttnParams


def _side_stream(layer) -> torch.cuda.Stream:
    """The layer's second stream (created on first use, on the layer's device)."""
    if getattr(layer, "_side", None) is None:
        layer._side = torch.cuda.Stream(device=layer.kv_cache.device)
    return layer._side


@dataclasses.dataclass
class LayerWeights:
    gamma_kv: torch.Tensor        # [c] fp32
    gamma_q: torch.Tensor         # [c] fp32
    bias_kv: torch.Tensor         # [2m] (CSA) or [m'] (HCA) fp32
    sink: torch.Tensor            # [H] fp32
    bias_idx: torch.Tensor | None = None   # [2m] fp32 (CSA only)


class CsaLayer:
    """One CSA layer for B sequences: KV cache [B, rows, c], indexer keys [B, rows, d_I],
    window ring [B, win_cap, c], plus the index buffer and workspaces of a step of n_q queries.

    Indexer keys in e4m3: pass a uint8 idx_cache with its per-row scales idx_scale [B, rows]
    (fp32); the keys are then compressed into e4m3 and the step's indexer queries are quantised
    (one scale per head) before the e4m3 indexer.  KV rows in e4m3: a uint8 kv_cache with
    kv_scale [B, rows]; the entries are compressed into it and attended over by csa_attend_e4m3."""

    def __init__(self, p: AttnParams, weights: LayerWeights, kv_cache, idx_cache, win_kv, n_q: int = 1,
                 idx_scale=None, kv_scale=None):
        self.p = p
        self.w = weights
        self.kv_cache, self.idx_cache, self.win_kv = kv_cache, idx_cache, win_kv
        self.kv8 = kv_cache.dtype == torch.uint8
        if self.kv8 and kv_scale is None:
            raise ValueError("an e4m3 KV cache needs kv_scale [B, rows]")
        self.kv_scale = kv_scale
        B, rows = kv_cache.shape[:2]
        dev = kv_cache.device
        self.idx = torch.empty((B, n_q, p.topk), dtype=torch.int32, device=dev)
        self.ws_idx = torch.empty(api.csa_indexer_workspace(p, B, n_q, rows), dtype=torch.uint8, device=dev)
        self.ws_att = torch.empty(api.csa_attend_workspace(p, B, n_q), dtype=torch.uint8, device=dev)
        self.e4m3 = idx_cache.dtype == torch.uint8
        if self.e4m3:
            if idx_scale is None:
                raise ValueError("an e4m3 indexer cache needs idx_scale [B, rows]")
            self.idx_scale = idx_scale
            self.q8 = torch.empty((B, n_q, p.idx_heads, p.idx_dim), dtype=torch.uint8, device=dev)
            self.q8_scale = torch.empty((B, n_q, p.idx_heads), dtype=torch.float32, device=dev)

    def compress_keys(self, tok_vi, tok_zi, tok_pos0, first_entry, n_new, stream=None):
        """The indexer-key entries (no RMSNorm, no RoPE), in bf16 or e4m3."""
        if self.e4m3:
            api.compress_kv_ex(True, self.p, tok_vi, tok_zi, tok_pos0, self.w.bias_idx, None, 0, first_entry, n_new,
                               self.idx_cache, cache_scale=self.idx_scale, stream=stream)
        else:
            api.csa_compress_kv(self.p, tok_vi, tok_zi, tok_pos0, self.w.bias_idx, None, 0, first_entry, n_new,
                                self.idx_cache, stream)

    def compress_kv(self, tok_v, tok_z, tok_pos0, first_entry, n_new, stream=None):
        """The KV entries (RMSNorm + RoPE), in bf16 or e4m3."""
        if self.kv8:
            api.compress_kv_ex(True, self.p, tok_v, tok_z, tok_pos0, self.w.bias_kv, self.w.gamma_kv, 1, first_entry,
                               n_new, self.kv_cache, cache_scale=self.kv_scale, stream=stream)
        else:
            api.csa_compress_kv(self.p, tok_v, tok_z, tok_pos0, self.w.bias_kv, self.w.gamma_kv, 1, first_entry,
                                n_new, self.kv_cache, stream)

    def compress(self, tok_v, tok_z, tok_vi, tok_zi, tok_pos0, first_entry, n_new, stream=None):
        """Compress n_new entries per sequence into both caches (KV: RMSNorm + RoPE; keys: neither)."""
        self.compress_kv(tok_v, tok_z, tok_pos0, first_entry, n_new, stream)
        self.compress_keys(tok_vi, tok_zi, tok_pos0, first_entry, n_new, stream)

    def window(self, new_tok_v, new_pos0, stream=None):
        api.lca_window_update(self.p, new_tok_v, new_pos0, self.w.gamma_kv, self.win_kv, stream)

    def select(self, q_idx, w_idx, q_pos, stream=None):
        if self.e4m3:
            api.lca_quantize_rows_e4m3(q_idx, self.q8, self.q8_scale, stream)
            api.csa_indexer_topk_e4m3(self.p, self.q8, self.q8_scale, w_idx, self.idx_cache, self.idx_scale, q_pos,
                                      self.idx, self.ws_idx, stream)
        else:
            api.csa_indexer_topk(self.p, q_idx, w_idx, self.idx_cache, q_pos, self.idx, self.ws_idx, stream)
        return self.idx

    def attend(self, q, q_pos, out, lse=None, stream=None, part="csa_attend"):
        """The attention; `part` may name csa_attend_prepare or csa_attend_prepared to run one half
        (bf16 KV rows only: over e4m3 rows the call is whole)."""
        if self.kv8:
            if part != "csa_attend":
                raise ValueError("the e4m3 attention has no separate halves")
            api.csa_attend_e4m3(self.p, q, self.w.gamma_q, q_pos, self.kv_cache, self.kv_scale, self.idx,
                                self.win_kv, self.w.sink, out, self.ws_att, lse, stream)
        else:
            api.csa_attend(self.p, q, self.w.gamma_q, q_pos, self.kv_cache, self.idx, self.win_kv, self.w.sink, out,
                           self.ws_att, lse, stream, part)

    def step(self, tok_v, tok_z, tok_vi, tok_zi, tok_pos0, first_entry, n_new, new_tok_v, new_pos0,
             q, q_idx, w_idx, q_pos, out, stream=None):
        if n_new:
            self.compress(tok_v, tok_z, tok_vi, tok_zi, tok_pos0, first_entry, n_new, stream)
        self.window(new_tok_v, new_pos0, stream)
        self.select(q_idx, w_idx, q_pos, stream)
        self.attend(q, q_pos, out, stream=stream)

    def step_overlapped(self, tok_v, tok_z, tok_vi, tok_zi, tok_pos0, first_entry, n_new, new_tok_v, new_pos0,
                        q, q_idx, w_idx, q_pos, out, side_prologue=None):
        """The same step on the current stream, with the parts that do not feed the selection (the
        KV entries, the window rows and the query preparation) on a side stream, overlapping the
        key entries, indexer and top-k; the attention waits for both.  `side_prologue(stream)`,
        if given, is issued first on the side stream (e.g. the upload of the side's inputs)."""
        main = torch.cuda.current_stream()
        side = _side_stream(self)
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        if side_prologue is not None:
            side_prologue(side)
        if n_new:
            self.compress_kv(tok_v, tok_z, tok_pos0, first_entry, n_new, side)
        api.lca_window_update(self.p, new_tok_v, new_pos0, self.w.gamma_kv, self.win_kv, side)
        if not self.kv8:
            self.attend(q, q_pos, out, stream=side, part="csa_attend_prepare")
        join.record(side)
        if n_new:
            self.compress_keys(tok_vi, tok_zi, tok_pos0, first_entry, n_new, main)
        self.select(q_idx, w_idx, q_pos, main)
        main.wait_event(join)
        self.attend(q, q_pos, out, stream=main, part="csa_attend" if self.kv8 else "csa_attend_prepared")


class HcaLayer:
    """One HCA layer for B sequences: KV cache [B, rows, c] and window ring [B, win_cap, c].
    KV rows in e4m3: a uint8 kv_cache with kv_scale [B, rows] (fp32)."""

    def __init__(self, p: AttnParams, weights: LayerWeights, kv_cache, win_kv, n_q: int = 1, kv_scale=None):
        self.p = p
        self.w = weights
        self.kv_cache, self.win_kv = kv_cache, win_kv
        self.kv8 = kv_cache.dtype == torch.uint8
        if self.kv8 and kv_scale is None:
            raise ValueError("an e4m3 KV cache needs kv_scale [B, rows]")
        self.kv_scale = kv_scale
        B, rows = kv_cache.shape[:2]
        self.ws_att = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8,
                                  device=kv_cache.device)

    def compress(self, tok_v, tok_z, tok_pos0, first_entry, n_new, stream=None):
        if self.kv8:
            api.compress_kv_ex(False, self.p, tok_v, tok_z, tok_pos0, self.w.bias_kv, self.w.gamma_kv, 1, first_entry,
                               n_new, self.kv_cache, cache_scale=self.kv_scale, stream=stream)
        else:
            api.hca_compress_kv(self.p, tok_v, tok_z, tok_pos0, self.w.bias_kv, self.w.gamma_kv, 1, first_entry,
                                n_new, self.kv_cache, stream)

    def window(self, new_tok_v, new_pos0, stream=None):
        api.lca_window_update(self.p, new_tok_v, new_pos0, self.w.gamma_kv, self.win_kv, stream)

    def attend(self, q, q_pos, out, lse=None, stream=None, part="hca_attend"):
        """The attention; `part` may name hca_attend_prepare or hca_attend_prepared to run one half
        (bf16 KV rows only: over e4m3 rows the call is whole)."""
        if self.kv8:
            if part != "hca_attend":
                raise ValueError("the e4m3 attention has no separate halves")
            api.hca_attend_e4m3(self.p, q, self.w.gamma_q, q_pos, self.kv_cache, self.kv_scale, self.win_kv,
                                self.w.sink, out, self.ws_att, lse, stream)
        else:
            api.hca_attend(self.p, q, self.w.gamma_q, q_pos, self.kv_cache, self.win_kv, self.w.sink, out,
                           self.ws_att, lse, stream, part)

    def step(self, tok_v, tok_z, tok_pos0, first_entry, n_new, new_tok_v, new_pos0, q, q_pos, out, stream=None):
        if n_new:
            self.compress(tok_v, tok_z, tok_pos0, first_entry, n_new, stream)
        self.window(new_tok_v, new_pos0, stream)
        self.attend(q, q_pos, out, stream=stream)

    def step_overlapped(self, tok_v, tok_z, tok_pos0, first_entry, n_new, new_tok_v, new_pos0, q, q_pos, out,
                        side_prologue=None):
        """The same step on the current stream, with the window rows and the query preparation on
        a side stream next to the compression; the attention waits for both.  `side_prologue(stream)`,
        if given, is issued first on the side stream."""
        main = torch.cuda.current_stream()
        side = _side_stream(self)
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        if side_prologue is not None:
            side_prologue(side)
        api.lca_window_update(self.p, new_tok_v, new_pos0, self.w.gamma_kv, self.win_kv, side)
        if not self.kv8:
            self.attend(q, q_pos, out, stream=side, part="hca_attend_prepare")
        join.record(side)
        if n_new:
            self.compress(tok_v, tok_z, tok_pos0, first_entry, n_new, main)
        main.wait_event(join)
        self.attend(q, q_pos, out, stream=main, part="hca_attend" if self.kv8 else "hca_attend_prepared")


class StepGraph:
    """A decode step captured once as a CUDA graph and replayed for every token.

    `fn` issues, on the current stream, everything a step does: the host-to-device copies of the
    step's inputs (from pinned buffers the caller refills), the layer calls, and the copy of the
    result back to pinned host memory.  Replaying the graph runs all of it with one launch from
    the host; the library's calls are plain stream work, so they capture like any other."""

    def __init__(self, fn, warmup: int = 1):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def __call__(self):
        self.graph.replay()


class StagingBuffer:
    """Per-step inputs packed into one device buffer with a pinned host mirror, so that a step
    uploads them with a few large copies (each host-to-device transfer pays a fixed latency of
    tens of microseconds, more than a few MB of payload at link speed).

    `tensors` maps names to device tensors; they are replaced, in place in the dict, by views of
    the packed buffer (16-byte aligned, values copied), and `host[name]` is the matching view of
    the pinned mirror.  `groups` (optional) maps group names to lists of tensor names; each group
    is packed contiguously and can be uploaded on its own, so that the work needing only the
    first group starts while the rest is in flight.  Fill `host[...]`, then `upload(stream,
    group)` (all groups when `group` is None)."""

    def __init__(self, tensors: dict, groups: dict = None):
        if groups is None:
            groups = {None: list(tensors)}
        order = [k for g in groups.values() for k in g]
        if sorted(map(repr, order)) != sorted(map(repr, tensors)):
            raise ValueError("groups must partition the staged tensors")
        offs, total, self.ranges = {}, 0, {}
        for g, keys in groups.items():
            start = total
            for k in keys:
                t = tensors[k]
                offs[k] = total
                total += (t.numel() * t.element_size() + 15) // 16 * 16
            self.ranges[g] = (start, total)
        dev = next(iter(tensors.values())).device
        self.dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        self.host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.host = {}
        for k, t in tensors.items():
            n = t.numel() * t.element_size()
            view = self.dev_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
            view.copy_(t)
            tensors[k] = view
            self.host[k] = self.host_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
            self.host[k].copy_(t)
        self.nbytes = total

    def upload(self, stream=None, group=None):
        a, b = (0, self.nbytes) if group is None else self.ranges[group]
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            self.dev_buf[a:b].copy_(self.host_buf[a:b], non_blocking=True)

