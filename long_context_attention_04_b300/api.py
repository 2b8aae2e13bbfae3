"""Python binding of liblca with the C ABI's names: argument marshalling only.

Every function takes torch CUDA tensors (torch provides the memory and the stream), checks
dtypes and layouts, and passes raw pointers, strides and sizes to the library; all
arithmetic runs in the library's CUDA kernels.  A failure status raises LcaError with the
library's message.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math

import torch

from . import _lib


class LcaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("lca status %d: %s" % (status, message))
        self.status = status


@dataclasses.dataclass
class AttnParams:
    """Mirror of lca_attn_params (names follow the pages' notation)."""
    heads: int = 64
    head_dim: int = 512
    rope_dims: int = 64
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    softmax_scale: float = 0.0      # 0 -> 1/sqrt(head_dim)
    window: int = 128
    ratio: int = 4
    topk: int = 512
    idx_heads: int = 64
    idx_dim: int = 128

    def c(self) -> _lib.lca_attn_params:
        return _lib.lca_attn_params(self.heads, self.head_dim, self.rope_dims, self.rope_base, self.rms_eps,
                                    self.softmax_scale, self.window, self.ratio, self.topk, self.idx_heads,
                                    self.idx_dim)

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.head_dim)


def params_from(shape, **over) -> AttnParams:
    """AttnParams from any object with the same field names (e.g. a workload's layer shape)."""
    kw = {f.name: getattr(shape, f.name) for f in dataclasses.fields(AttnParams) if hasattr(shape, f.name)}
    kw.update(over)
    return AttnParams(**kw)


def _check(status: int):
    if status != 0:
        lib = _lib.load()
        raise LcaError(status, lib.lca_last_error().decode())


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _rows(t: torch.Tensor, name: str) -> int:
    """Batch stride (elements) of a [B, rows, width] tensor whose rows are dense."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("%s must be [B, rows, width] with dense rows" % name)
    return t.stride(0)


def _holds(t, n: int, name: str, exact: bool = False):
    """A dense tensor with at least (or exactly) n elements: the library indexes it as a flat
    array of that length, and cannot see torch's strides or sizes."""
    if t is None:
        return
    if not t.is_contiguous() or (t.numel() != n if exact else t.numel() < n):
        raise ValueError("%s must be a contiguous tensor of %s%d elements, got shape %s"
                         % (name, "" if exact else "at least ", n, tuple(t.shape)))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous int32 tensor" % name)
    return _ptr(t, torch.int32, name)


def _compress(fn, span, p, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new, cache, stream):
    B, n_tok, width = tok_v.shape
    if tok_z.dim() != 2 or tok_z.stride(1) != 1 or tok_z.shape[0] != B:
        raise ValueError("tok_z must be [B, n_tok] with unit inner stride")
    if cache.shape[0] != B or cache.shape[2] != width:
        raise ValueError("cache must be [B, rows, width]")
    _holds(tok_pos0, B, "tok_pos0")
    _holds(first_entry, B, "first_entry")
    _holds(pos_bias, span, "pos_bias")
    _holds(gamma, width, "gamma")
    st = fn(ctypes.byref(p.c()), B, width,
            _ptr(tok_v, torch.bfloat16, "tok_v"), _rows(tok_v, "tok_v"), n_tok,
            _ptr(tok_z, torch.float32, "tok_z"), tok_z.stride(0), _i32(tok_pos0, "tok_pos0"),
            _ptr(pos_bias, torch.float32, "pos_bias"), _ptr(gamma, torch.float32, "gamma"), int(apply_rope),
            _i32(first_entry, "first_entry"), int(n_new),
            _ptr(cache, torch.bfloat16, "cache"), _rows(cache, "cache"), cache.shape[1], _stream(stream))
    _check(st)


def csa_compress_kv(p: AttnParams, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new,
                    cache, stream=None):
    """CSA compression (windows of 2m, stride m) of entries first_entry[b] .. +n_new into cache."""
    _compress(_lib.load().csa_compress_kv, 2 * p.ratio, p, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope,
              first_entry, n_new, cache, stream)


def hca_compress_kv(p: AttnParams, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new,
                    cache, stream=None):
    """HCA compression (non-overlapping windows of m') of entries first_entry[b] .. +n_new into cache."""
    _compress(_lib.load().hca_compress_kv, p.ratio, p, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope,
              first_entry, n_new, cache, stream)


def lca_window_update(p: AttnParams, tok_v, tok_pos0, gamma, win_kv, stream=None):
    """Write RoPE(RMSNorm(v)*gamma, pos) of each token to ring row pos mod win_cap."""
    B, n_tok, _ = tok_v.shape
    _holds(tok_pos0, B, "tok_pos0")
    _holds(gamma, p.head_dim, "gamma")
    st = _lib.load().lca_window_update(
        ctypes.byref(p.c()), B, _ptr(tok_v, torch.bfloat16, "tok_v"), _rows(tok_v, "tok_v"), n_tok,
        _i32(tok_pos0, "tok_pos0"), _ptr(gamma, torch.float32, "gamma"),
        _ptr(win_kv, torch.bfloat16, "win_kv"), _rows(win_kv, "win_kv"), win_kv.shape[1], _stream(stream))
    _check(st)


def _idx_q(q_idx, w_idx, p):
    if q_idx.dim() != 4 or not q_idx.is_contiguous():
        raise ValueError("q_idx must be a contiguous [B, n_q, H_I, d_I] tensor")
    B, n_q, hi, di = q_idx.shape
    if (hi, di) != (p.idx_heads, p.idx_dim):
        raise ValueError("q_idx heads/dim do not match params")
    if tuple(w_idx.shape) != (B, n_q, hi) or not w_idx.is_contiguous():
        raise ValueError("w_idx must be a contiguous [B, n_q, H_I] tensor")
    return B, n_q


def lca_quantize_rows_e4m3(x, q, scale, stream=None):
    """Per-row e4m3 codes q (uint8, x's shape) and scales (float32, one per row of the last dim)
    of the bf16 rows of x."""
    if not x.is_contiguous() or x.dtype != torch.bfloat16:
        raise ValueError("x must be a contiguous bf16 tensor")
    width = x.shape[-1]
    rows = x.numel() // width
    if q.dtype != torch.uint8 or q.numel() != x.numel() or not q.is_contiguous():
        raise ValueError("q must be a contiguous uint8 tensor with x's size")
    _holds(scale, rows, "scale", exact=True)
    st = _lib.load().lca_quantize_rows_e4m3(_ptr(x, torch.bfloat16, "x"), rows, width, _ptr(q, torch.uint8, "q"),
                                            _ptr(scale, torch.float32, "scale"), _stream(stream))
    _check(st)


def compress_kv_ex(csa: bool, p: AttnParams, tok_v, tok_z, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new,
                   cache, cache_scale=None, per_channel=False, stream=None):
    """csa_compress_kv_ex / hca_compress_kv_ex.  per_channel: tok_z [B, n_tok, width] and pos_bias
    [span, width]; a uint8 cache [B, rows, width] is e4m3 with cache_scale [B, rows] (float32)."""
    B, n_tok, width = tok_v.shape
    span = 2 * p.ratio if csa else p.ratio
    if per_channel:
        if tok_z.dim() != 3 or tuple(tok_z.shape) != (B, n_tok, width) or tok_z.stride(2) != 1 or \
                tok_z.stride(1) != width:
            raise ValueError("per-channel tok_z must be [B, n_tok, width] with dense rows")
        _holds(pos_bias, span * width, "pos_bias", exact=True)
    else:
        if tok_z.dim() != 2 or tok_z.stride(1) != 1 or tok_z.shape[0] != B:
            raise ValueError("tok_z must be [B, n_tok] with unit inner stride")
        _holds(pos_bias, span, "pos_bias")
    if cache.shape[0] != B or cache.shape[2] != width:
        raise ValueError("cache must be [B, rows, width]")
    e4m3 = cache.dtype == torch.uint8
    if e4m3:
        if cache_scale is None or cache_scale.dim() != 2 or tuple(cache_scale.shape) != (B, cache.shape[1]) or \
                cache_scale.stride(1) != 1:
            raise ValueError("an e4m3 cache needs cache_scale [B, rows] (float32, unit inner stride)")
    _holds(tok_pos0, B, "tok_pos0")
    _holds(first_entry, B, "first_entry")
    _holds(gamma, width, "gamma")
    var = _lib.lca_compress_variant(int(per_channel), int(e4m3),
                                    _ptr(cache_scale, torch.float32, "cache_scale") if e4m3 else None,
                                    cache_scale.stride(0) if e4m3 else 0)
    lib = _lib.load()
    fn = lib.csa_compress_kv_ex if csa else lib.hca_compress_kv_ex
    st = fn(ctypes.byref(p.c()), ctypes.byref(var), B, width,
            _ptr(tok_v, torch.bfloat16, "tok_v"), _rows(tok_v, "tok_v"), n_tok,
            _ptr(tok_z, torch.float32, "tok_z"), tok_z.stride(0), _i32(tok_pos0, "tok_pos0"),
            _ptr(pos_bias, torch.float32, "pos_bias"), _ptr(gamma, torch.float32, "gamma"), int(apply_rope),
            _i32(first_entry, "first_entry"), int(n_new),
            _ptr(cache, torch.uint8 if e4m3 else torch.bfloat16, "cache"), _rows(cache, "cache"), cache.shape[1],
            _stream(stream))
    _check(st)


def _idx_q8(q8, qs, w, k8, ks, p):
    if q8.dim() != 4 or not q8.is_contiguous() or tuple(q8.shape[2:]) != (p.idx_heads, p.idx_dim):
        raise ValueError("q_idx8 must be a contiguous [B, n_q, H_I, d_I] uint8 tensor")
    B, n_q = q8.shape[0], q8.shape[1]
    _holds(qs, B * n_q * p.idx_heads, "q_scale", exact=True)
    _holds(w, B * n_q * p.idx_heads, "w_idx", exact=True)
    if ks.dim() != 2 or ks.shape[0] != k8.shape[0] or ks.shape[1] < k8.shape[1] or ks.stride(1) != 1:
        raise ValueError("k_scale must be [B, >= rows] with unit inner stride")
    return B, n_q


def csa_indexer_scores_e4m3(p: AttnParams, q_idx8, q_scale, w_idx, k_cache8, k_scale, q_pos, scores, stream=None):
    """csa_indexer_scores over e4m3 queries and keys (codes uint8, per-row float32 scales)."""
    B, n_q = _idx_q8(q_idx8, q_scale, w_idx, k_cache8, k_scale, p)
    if scores.dim() != 3 or scores.stride(2) != 1 or scores.stride(1) != scores.shape[2] or \
            scores.stride(0) != n_q * scores.shape[2]:
        raise ValueError("scores must be a dense [B, n_q, stride] tensor")
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    st = _lib.load().csa_indexer_scores_e4m3(
        ctypes.byref(p.c()), B, n_q, _ptr(q_idx8, torch.uint8, "q_idx8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w_idx, torch.float32, "w_idx"), _ptr(k_cache8, torch.uint8, "k_cache8"), _rows(k_cache8, "k_cache8"),
        _ptr(k_scale, torch.float32, "k_scale"), k_scale.stride(0), k_cache8.shape[1], _i32(q_pos, "q_pos"),
        _ptr(scores, torch.float32, "scores"), scores.shape[2], _stream(stream))
    _check(st)


def csa_indexer_topk_e4m3(p: AttnParams, q_idx8, q_scale, w_idx, k_cache8, k_scale, q_pos, out_idx, workspace,
                          stream=None):
    """csa_indexer_topk over e4m3 queries and keys; workspace from csa_indexer_workspace."""
    B, n_q = _idx_q8(q_idx8, q_scale, w_idx, k_cache8, k_scale, p)
    if tuple(out_idx.shape) != (B, n_q, p.topk):
        raise ValueError("out_idx must be [B, n_q, topk]")
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    st = _lib.load().csa_indexer_topk_e4m3(
        ctypes.byref(p.c()), B, n_q, _ptr(q_idx8, torch.uint8, "q_idx8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w_idx, torch.float32, "w_idx"), _ptr(k_cache8, torch.uint8, "k_cache8"), _rows(k_cache8, "k_cache8"),
        _ptr(k_scale, torch.float32, "k_scale"), k_scale.stride(0), k_cache8.shape[1], _i32(q_pos, "q_pos"),
        _i32(out_idx, "out_idx"), _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st)


def csa_indexer_scores(p: AttnParams, q_idx, w_idx, k_cache, q_pos, scores, stream=None):
    """scores[b, i, j] = sum_h w[b,i,h] ReLU(q[b,i,h] . k[b,j]) for j < n_vis(i), -inf beyond."""
    B, n_q = _idx_q(q_idx, w_idx, p)
    if scores.dim() != 3 or scores.stride(2) != 1 or scores.stride(1) != scores.shape[2] or \
            scores.stride(0) != n_q * scores.shape[2]:
        raise ValueError("scores must be a dense [B, n_q, stride] tensor")
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    st = _lib.load().csa_indexer_scores(
        ctypes.byref(p.c()), B, n_q, _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(w_idx, torch.float32, "w_idx"),
        _ptr(k_cache, torch.bfloat16, "k_cache"), _rows(k_cache, "k_cache"), k_cache.shape[1],
        _i32(q_pos, "q_pos"), _ptr(scores, torch.float32, "scores"), scores.shape[2], _stream(stream))
    _check(st)


def lca_topk(p: AttnParams, scores, q_pos, max_entries, out_idx, stream=None):
    """Top-k (score desc, index asc), ascending indices, -1 padded, per query row of scores."""
    B, n_q, stride = scores.shape
    if tuple(out_idx.shape) != (B, n_q, p.topk):
        raise ValueError("out_idx must be [B, n_q, topk]")
    _holds(scores, B * n_q * stride, "scores", exact=True)
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    st = _lib.load().lca_topk(ctypes.byref(p.c()), B, n_q, _ptr(scores, torch.float32, "scores"), stride,
                              _i32(q_pos, "q_pos"), int(max_entries), _i32(out_idx, "out_idx"), _stream(stream))
    _check(st)


def csa_indexer_workspace(p: AttnParams, batch: int, n_q: int, cache_rows: int) -> int:
    return int(_lib.load().csa_indexer_workspace(ctypes.byref(p.c()), batch, n_q, cache_rows))


def csa_indexer_topk(p: AttnParams, q_idx, w_idx, k_cache, q_pos, out_idx, workspace, stream=None):
    """Indexer scores into the workspace, then top-k into out_idx [B, n_q, k]."""
    B, n_q = _idx_q(q_idx, w_idx, p)
    if tuple(out_idx.shape) != (B, n_q, p.topk):
        raise ValueError("out_idx must be [B, n_q, topk]")
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    st = _lib.load().csa_indexer_topk(
        ctypes.byref(p.c()), B, n_q, _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(w_idx, torch.float32, "w_idx"),
        _ptr(k_cache, torch.bfloat16, "k_cache"), _rows(k_cache, "k_cache"), k_cache.shape[1],
        _i32(q_pos, "q_pos"), _i32(out_idx, "out_idx"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def csa_attend_workspace(p: AttnParams, batch: int, n_q: int) -> int:
    return int(_lib.load().csa_attend_workspace(ctypes.byref(p.c()), batch, n_q))


def hca_attend_workspace(p: AttnParams, batch: int, n_q: int, cache_rows: int) -> int:
    return int(_lib.load().hca_attend_workspace(ctypes.byref(p.c()), batch, n_q, cache_rows))


def _attend_common(q, p, gamma_q, q_pos, sink, out, lse):
    if q.dim() != 4 or not q.is_contiguous() or tuple(q.shape[2:]) != (p.heads, p.head_dim):
        raise ValueError("q must be a contiguous [B, n_q, H, c] tensor matching params")
    B, n_q = q.shape[0], q.shape[1]
    _holds(out, q.numel(), "out", exact=True)
    _holds(lse, B * n_q * p.heads, "lse", exact=True)
    _holds(q_pos, B * n_q, "q_pos", exact=True)
    _holds(gamma_q, p.head_dim, "gamma_q")
    _holds(sink, p.heads, "sink")
    return B, n_q


def csa_attend(p: AttnParams, q, gamma_q, q_pos, kv_cache, idx, win_kv, sink, out, workspace, lse=None,
               stream=None, entry="csa_attend"):
    """Core attention over kv_cache[idx] plus the window rows (see include/lca.h).  `entry`
    selects the whole call or one of its halves (csa_attend_prepare / csa_attend_prepared)."""
    if entry not in ("csa_attend", "csa_attend_prepare", "csa_attend_prepared"):
        raise ValueError("unknown attention entry %r" % (entry,))
    B, n_q = _attend_common(q, p, gamma_q, q_pos, sink, out, lse)
    if tuple(idx.shape) != (B, n_q, p.topk):
        raise ValueError("idx must be [B, n_q, topk]")
    st = getattr(_lib.load(), entry)(
        ctypes.byref(p.c()), B, n_q, _ptr(q, torch.bfloat16, "q"), _ptr(gamma_q, torch.float32, "gamma_q"),
        _i32(q_pos, "q_pos"), _ptr(kv_cache, torch.bfloat16, "kv_cache"), _rows(kv_cache, "kv_cache"),
        kv_cache.shape[1], _i32(idx, "idx"), _ptr(win_kv, torch.bfloat16, "win_kv"), _rows(win_kv, "win_kv"),
        win_kv.shape[1], _ptr(sink, torch.float32, "sink"), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def hca_attend(p: AttnParams, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, workspace, lse=None, stream=None,
               entry="hca_attend"):
    """Dense core attention over the visible entries of kv_cache plus the window rows.  `entry`
    selects the whole call or one of its halves (hca_attend_prepare / hca_attend_prepared)."""
    if entry not in ("hca_attend", "hca_attend_prepare", "hca_attend_prepared"):
        raise ValueError("unknown attention entry %r" % (entry,))
    B, n_q = _attend_common(q, p, gamma_q, q_pos, sink, out, lse)
    st = getattr(_lib.load(), entry)(
        ctypes.byref(p.c()), B, n_q, _ptr(q, torch.bfloat16, "q"), _ptr(gamma_q, torch.float32, "gamma_q"),
        _i32(q_pos, "q_pos"), _ptr(kv_cache, torch.bfloat16, "kv_cache"), _rows(kv_cache, "kv_cache"),
        kv_cache.shape[1], _ptr(win_kv, torch.bfloat16, "win_kv"), _rows(win_kv, "win_kv"), win_kv.shape[1],
        _ptr(sink, torch.float32, "sink"), _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def _kv8(kv8, kv_scale):
    if kv8.dtype != torch.uint8:
        raise TypeError("kv_cache8 must be uint8 (e4m3 codes)")
    if kv_scale.dim() != 2 or kv_scale.shape[0] != kv8.shape[0] or kv_scale.shape[1] < kv8.shape[1] or \
            kv_scale.stride(1) != 1:
        raise ValueError("kv_scale must be [B, >= rows] with unit inner stride")
    return (_ptr(kv8, torch.uint8, "kv_cache8"), _rows(kv8, "kv_cache8"), _ptr(kv_scale, torch.float32, "kv_scale"),
            kv_scale.stride(0), kv8.shape[1])


def csa_attend_e4m3(p: AttnParams, q, gamma_q, q_pos, kv_cache8, kv_scale, idx, win_kv, sink, out, workspace, lse=None,
                    stream=None):
    """csa_attend over an e4m3 compressed cache (codes uint8 [B, rows, c], scales [B, rows])."""
    B, n_q = _attend_common(q, p, gamma_q, q_pos, sink, out, lse)
    if tuple(idx.shape) != (B, n_q, p.topk):
        raise ValueError("idx must be [B, n_q, topk]")
    kv, kv_bs, ks, ks_bs, rows = _kv8(kv_cache8, kv_scale)
    st = _lib.load().csa_attend_e4m3(
        ctypes.byref(p.c()), B, n_q, _ptr(q, torch.bfloat16, "q"), _ptr(gamma_q, torch.float32, "gamma_q"),
        _i32(q_pos, "q_pos"), kv, kv_bs, ks, ks_bs, rows, _i32(idx, "idx"), _ptr(win_kv, torch.bfloat16, "win_kv"),
        _rows(win_kv, "win_kv"), win_kv.shape[1], _ptr(sink, torch.float32, "sink"), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def hca_attend_e4m3(p: AttnParams, q, gamma_q, q_pos, kv_cache8, kv_scale, win_kv, sink, out, workspace, lse=None,
                    stream=None):
    """hca_attend over an e4m3 compressed cache (codes uint8 [B, rows, c], scales [B, rows])."""
    B, n_q = _attend_common(q, p, gamma_q, q_pos, sink, out, lse)
    kv, kv_bs, ks, ks_bs, rows = _kv8(kv_cache8, kv_scale)
    st = _lib.load().hca_attend_e4m3(
        ctypes.byref(p.c()), B, n_q, _ptr(q, torch.bfloat16, "q"), _ptr(gamma_q, torch.float32, "gamma_q"),
        _i32(q_pos, "q_pos"), kv, kv_bs, ks, ks_bs, rows, _ptr(win_kv, torch.bfloat16, "win_kv"),
        _rows(win_kv, "win_kv"), win_kv.shape[1], _ptr(sink, torch.float32, "sink"), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def csa_attend_prepare(p: AttnParams, q, gamma_q, q_pos, kv_cache, idx, win_kv, sink, out, workspace, lse=None,
                       stream=None):
    """The query preparation of csa_attend alone, into the workspace (see include/lca.h)."""
    csa_attend(p, q, gamma_q, q_pos, kv_cache, idx, win_kv, sink, out, workspace, lse, stream, "csa_attend_prepare")


def csa_attend_prepared(p: AttnParams, q, gamma_q, q_pos, kv_cache, idx, win_kv, sink, out, workspace, lse=None,
                        stream=None):
    """The attention of csa_attend alone, on query images a csa_attend_prepare left in the workspace."""
    csa_attend(p, q, gamma_q, q_pos, kv_cache, idx, win_kv, sink, out, workspace, lse, stream, "csa_attend_prepared")


def hca_attend_prepare(p: AttnParams, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, workspace, lse=None,
                       stream=None):
    """The query preparation of hca_attend alone, into the workspace (see include/lca.h)."""
    hca_attend(p, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, workspace, lse, stream, "hca_attend_prepare")


def hca_attend_prepared(p: AttnParams, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, workspace, lse=None,
                        stream=None):
    """The attention of hca_attend alone, on query images an hca_attend_prepare left in the workspace."""
    hca_attend(p, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, workspace, lse, stream, "hca_attend_prepared")


def hca_attend_noalloc(p: AttnParams, q, gamma_q, q_pos, kv_cache, win_kv, sink, out, lse=None, stream=None):
    """hca_attend with its scratch in the library's static device array (no workspace)."""
    B, n_q = _attend_common(q, p, gamma_q, q_pos, sink, out, lse)
    st = _lib.load().hca_attend_noalloc(
        ctypes.byref(p.c()), B, n_q, _ptr(q, torch.bfloat16, "q"), _ptr(gamma_q, torch.float32, "gamma_q"),
        _i32(q_pos, "q_pos"), _ptr(kv_cache, torch.bfloat16, "kv_cache"), _rows(kv_cache, "kv_cache"),
        kv_cache.shape[1], _ptr(win_kv, torch.bfloat16, "win_kv"), _rows(win_kv, "win_kv"), win_kv.shape[1],
        _ptr(sink, torch.float32, "sink"), _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _stream(stream))
    _check(st)


def lca_grouped_oproj(o, Wg, Wm, groups: int, mid, y, stream=None):
    """y = Wm . concat_g(Wg[g] . o_g) for o [B, H, c]; mid [B, groups*d_g] is scratch."""
    B, H, c = o.shape
    if groups < 1 or H % groups or Wg.shape[0] % groups:
        raise ValueError("groups must divide the heads and the rows of Wg")
    d_g = Wg.shape[0] // groups
    d_model = Wm.shape[0]
    for t, n in ((o, "o"), (Wg, "Wg"), (Wm, "Wm"), (mid, "mid"), (y, "y")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    _holds(Wg, groups * d_g * (H // groups) * c, "Wg", exact=True)
    _holds(Wm, d_model * groups * d_g, "Wm", exact=True)
    _holds(mid, B * groups * d_g, "mid")
    _holds(y, B * d_model, "y")
    st = _lib.load().lca_grouped_oproj(B, H, c, groups, d_g, d_model, _ptr(o, torch.bfloat16, "o"),
                                       _ptr(Wg, torch.bfloat16, "Wg"), _ptr(Wm, torch.bfloat16, "Wm"),
                                       _ptr(mid, torch.bfloat16, "mid"), _ptr(y, torch.bfloat16, "y"),
                                       _stream(stream))
    _check(st)


def lca_gemm_bf16(A, B, C, stream=None):
    """C[M, N] = A[M, K] . B[N, K]^T (bf16 in, fp32 accumulation; C bf16, or fp32 through
    lca_gemm_bf16_f32)."""
    M, K = A.shape
    N = B.shape[0]
    if B.dim() != 2 or B.shape[1] != K:
        raise ValueError("B must be [N, K] with A's K")
    if C.dim() != 2 or C.shape[0] < M or C.shape[1] < N:
        raise ValueError("C must be at least [M, N]")
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.stride(1) != 1:
            raise ValueError("%s must have unit stride along its rows" % n)
    lib = _lib.load()
    if C.dtype == torch.float32:
        st = lib.lca_gemm_bf16_f32(M, N, K, _ptr(A, torch.bfloat16, "A"), A.stride(0),
                                   _ptr(B, torch.bfloat16, "B"), B.stride(0), _ptr(C, torch.float32, "C"),
                                   C.stride(0), _stream(stream))
    else:
        st = lib.lca_gemm_bf16(M, N, K, _ptr(A, torch.bfloat16, "A"), A.stride(0),
                               _ptr(B, torch.bfloat16, "B"), B.stride(0), _ptr(C, torch.bfloat16, "C"),
                               C.stride(0), _stream(stream))
    _check(st)


def lca_mhc_workspace(T: int, n: int) -> int:
    return int(_lib.load().lca_mhc_workspace(T, n))


def lca_mhc_pre(x, phi, bias, h, a, c, b_mix, workspace, iters: int = 20, stream=None):
    """Hyper-connection coefficients of every token (a, c sigmoids; b_mix by Sinkhorn-Knopp) and
    the layer input h = sum_i a_i x[i]; x [T, n, d] bf16, phi [2n + n^2, n d] bf16."""
    if x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [T, n, d] tensor")
    T, n, d = x.shape
    K = 2 * n + n * n
    _holds(phi, K * n * d, "phi", exact=True)
    _holds(bias, K, "bias", exact=True)
    _holds(h, T * d, "h", exact=True)
    _holds(a, T * n, "a", exact=True)
    _holds(c, T * n, "c", exact=True)
    _holds(b_mix, T * n * n, "b_mix", exact=True)
    st = _lib.load().lca_mhc_pre(T, n, d, int(iters), _ptr(x, torch.bfloat16, "x"), _ptr(phi, torch.bfloat16, "phi"),
                                 _ptr(bias, torch.float32, "bias"), _ptr(h, torch.bfloat16, "h"),
                                 _ptr(a, torch.float32, "a"), _ptr(c, torch.float32, "c"),
                                 _ptr(b_mix, torch.float32, "b_mix"), _ptr(workspace, None, "workspace"),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)


def lca_mhc_post(x, b_mix, c, y, x_out, stream=None):
    """The streams after the layer: x_out[:, i] = sum_j b_mix[:, i, j] x[:, j] + c[:, i] y."""
    if x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [T, n, d] tensor")
    T, n, d = x.shape
    _holds(b_mix, T * n * n, "b_mix", exact=True)
    _holds(c, T * n, "c", exact=True)
    _holds(y, T * d, "y", exact=True)
    _holds(x_out, T * n * d, "x_out", exact=True)
    st = _lib.load().lca_mhc_post(T, n, d, _ptr(x, torch.bfloat16, "x"), _ptr(b_mix, torch.float32, "b_mix"),
                                  _ptr(c, torch.float32, "c"), _ptr(y, torch.bfloat16, "y"),
                                  _ptr(x_out, torch.bfloat16, "x_out"), _stream(stream))
    _check(st)


def lca_device_error(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word; returns the word."""
    w = ctypes.c_uint32(0)
    _lib.load().lca_device_error(_stream(stream), ctypes.byref(w))
    return int(w.value)


def lca_test_hooks(wait_limit_cycles: int = 0, attend_skip_tile: int = -1):
    """For failure-path tests only: the bound of every kernel wait (cycles; 0 = default) and a
    tile the attention kernel leaves unloaded (-1 = none) on the current device."""
    _check(_lib.load().lca_test_hooks(int(wait_limit_cycles), int(attend_skip_tile)))


def lca_version() -> str:
    return _lib.load().lca_version().decode()
