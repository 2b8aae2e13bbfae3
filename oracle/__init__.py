"""CPU oracle for the CSA/HCA attention path -- TEST INFRASTRUCTURE ONLY.

A plain double-precision C implementation (``oracle.c``) of what the hybrid
compressed attention of DeepSeek-V4 computes, wrapped for numpy.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline leg and its
reference arm) may import this package.  It shares no code with the CUDA library
and the CUDA library never calls it.

bf16 data is passed as numpy ``uint16`` arrays holding the raw bf16 bit patterns;
results come back as float64.

Every function below only marshals arguments; the arithmetic and the citations to
the pages live in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (no fast-math: plain IEEE double)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        D = ctypes.c_double
        lib.orc_compress.argtypes = [I, I, I, P, P, L, L, P, P, D, I, D, L, L, P]
        lib.orc_compress.restype = I
        lib.orc_window_row.argtypes = [I, P, P, D, I, D, L, P]
        lib.orc_window_row.restype = None
        lib.orc_indexer_scores.argtypes = [I, I, P, P, P, L, P]
        lib.orc_indexer_scores.restype = None
        lib.orc_visible_entries.argtypes = [L, I]
        lib.orc_visible_entries.restype = L
        lib.orc_topk.argtypes = [P, L, I, P]
        lib.orc_topk.restype = I
        lib.orc_attend.argtypes = [I, I, I, D, D, D, P, P, L, P, L, P, L, L, P, L, L, P, P, P]
        lib.orc_attend.restype = I
        lib.orc_gemm_bf16.argtypes = [L, L, L, P, P, P]
        lib.orc_gemm_bf16.restype = None
        lib.orc_mhc_coeffs.argtypes = [I, L, I, P, P, P, P, P, P]
        lib.orc_mhc_coeffs.restype = None
        lib.orc_mhc_pre.argtypes = [I, L, P, P, P]
        lib.orc_mhc_pre.restype = None
        lib.orc_mhc_post.argtypes = [I, L, P, P, P, P, P]
        lib.orc_mhc_post.restype = None
        lib.orc_grouped_oproj.argtypes = [I, I, I, I, I, P, P, P, P]
        lib.orc_grouped_oproj.restype = I
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = D
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_quantize_rows_e4m3.argtypes = [L, I, P, P, P]
        lib.orc_quantize_rows_e4m3.restype = None
        lib.orc_dequantize_rows_e4m3.argtypes = [L, I, P, P, P]
        lib.orc_dequantize_rows_e4m3.restype = None
        lib.orc_compress_pc.argtypes = [I, I, I, P, P, L, L, P, P, D, I, D, L, L, P]
        lib.orc_compress_pc.restype = I
        lib.orc_indexer_scores_e4m3.argtypes = [I, I, P, P, P, P, P, L, P]
        lib.orc_indexer_scores_e4m3.restype = None
        lib.orc_attend_e4m3.argtypes = [I, I, I, D, D, D, P, P, L, P, P, L, P, L, L, P, L, L, P, P, P]
        lib.orc_attend_e4m3.restype = I
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def compress(tok_v, tok_z, tok_pos0, bias, gamma, eps, rope_dims, rope_base,
             span, stride, first_entry, n_new):
    """Entries first_entry .. first_entry+n_new-1 of a compressed cache (float64 [n_new, width]).

    tok_v: uint16 [n_tok, width], tok_z: float32 [n_tok] for tokens tok_pos0 .. tok_pos0+n_tok-1.
    CSA: span=2m, stride=m.  HCA: span=stride=m'.  gamma=None skips the RMSNorm.
    """
    lib = _load()
    tok_v = _u16(tok_v)
    tok_z = _f32(tok_z)
    bias = _f32(bias)
    g = None if gamma is None else _f32(gamma)
    n_tok, width = tok_v.shape
    assert tok_z.shape == (n_tok,) and bias.shape == (span,)
    out = np.empty((n_new, width), dtype=np.float64)
    rc = lib.orc_compress(span, stride, width, _ptr(tok_v), _ptr(tok_z), tok_pos0, n_tok,
                          _ptr(bias), _ptr(g), eps, rope_dims, rope_base, first_entry, n_new, _ptr(out))
    if rc != 0:
        raise ValueError("orc_compress: tokens needed by the requested entries are missing (rc=%d)" % rc)
    return out


def window_row(v, gamma, eps, rope_dims, rope_base, pos):
    """Sliding-window row of one token: RMSNorm(v)*gamma, then RoPE at pos (float64 [c])."""
    lib = _load()
    v = _u16(v)
    g = _f32(gamma)
    out = np.empty(v.shape[0], dtype=np.float64)
    lib.orc_window_row(v.shape[0], _ptr(v), _ptr(g), eps, rope_dims, rope_base, pos, _ptr(out))
    return out


def visible_entries(pos: int, ratio: int) -> int:
    return int(_load().orc_visible_entries(pos, ratio))


def indexer_scores(q, w, keys, n_vis):
    """s_j = sum_h w_h ReLU(q_h . k_j) for j < n_vis (float64 [n_vis]).  q: uint16 [H_I, d_I]."""
    lib = _load()
    q = _u16(q)
    w = _f32(w)
    keys = _u16(keys)
    n_heads, dim = q.shape
    assert keys.shape[1] == dim and keys.shape[0] >= n_vis and w.shape == (n_heads,)
    out = np.empty(n_vis, dtype=np.float64)
    lib.orc_indexer_scores(n_heads, dim, _ptr(q), _ptr(w), _ptr(keys), n_vis, _ptr(out))
    return out


def topk(scores, k):
    """Top-k under (score desc, index asc), ascending indices, -1 padded (int32 [k])."""
    lib = _load()
    s = np.ascontiguousarray(scores, dtype=np.float64)
    out = np.empty(k, dtype=np.int32)
    rc = lib.orc_topk(_ptr(s), s.shape[0], k, _ptr(out))
    if rc != 0:
        raise MemoryError("orc_topk")
    return out


def attend(q, gamma_q, pos, comp, sink, win, win_cap, W, rope_dims, rope_base, eps, scale,
           idx=None, n_dense=0):
    """One query's core attention (CSA when idx is given, HCA over comp[:n_dense] otherwise).

    q: uint16 [H, c]; comp: uint16 [rows, c]; win: uint16 [win_cap, c] ring; sink: float32 [H].
    Returns (out float64 [H, c], lse float64 [H]).
    """
    lib = _load()
    q = _u16(q)
    comp = _u16(comp)
    win = _u16(win)
    g = _f32(gamma_q)
    sk = _f32(sink)
    H, c = q.shape
    ix = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((H, c), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    rc = lib.orc_attend(H, c, rope_dims, rope_base, eps, scale, _ptr(q), _ptr(g), pos,
                        _ptr(comp), comp.shape[0], _ptr(ix), 0 if ix is None else ix.shape[0], n_dense,
                        _ptr(win), win_cap, W, _ptr(sk), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("orc_attend: index outside the compressed cache (rc=%d)" % rc)
    return out, lse


def gemm_bf16(A, B):
    """out = A @ B.T in float64 (A: uint16 [M, K], B: uint16 [N, K])."""
    lib = _load()
    A = _u16(A)
    B = _u16(B)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    out = np.empty((M, N), dtype=np.float64)
    lib.orc_gemm_bf16(M, N, K, _ptr(A), _ptr(B), _ptr(out))
    return out


def grouped_oproj(o, Wg, Wm, groups):
    """Grouped output projection of one token: o uint16 [H, c] -> float64 [d_model]."""
    lib = _load()
    o = _u16(o)
    Wg = _u16(Wg)
    Wm = _u16(Wm)
    H, c = o.shape
    G = groups
    d_g = Wg.shape[0] // G
    d_model = Wm.shape[0]
    assert Wg.shape == (G * d_g, (H // G) * c) and Wm.shape == (d_model, G * d_g)
    y = np.empty(d_model, dtype=np.float64)
    rc = lib.orc_grouped_oproj(H, c, G, d_g, d_model, _ptr(o), _ptr(Wg), _ptr(Wm), _ptr(y))
    if rc != 0:
        raise ValueError("orc_grouped_oproj: heads not divisible by groups")
    return y


def mhc_coeffs(x, phi, bias, iters=20):
    """Generated hyper-connection coefficients of one token (manifold-constrained hyper-
    connections): x uint16 [n, d], phi uint16 [2n + n*n, n*d], bias float32 [2n + n*n] ->
    (a [n], c [n], B [n, n]) in float64: sigmoid pre and post weights and the Sinkhorn-Knopp
    projection of exp(z) onto the doubly stochastic matrices (iters row-then-column passes)."""
    lib = _load()
    x = _u16(x)
    phi = _u16(phi)
    b = _f32(bias)
    n, d = x.shape
    assert phi.shape == (2 * n + n * n, n * d) and b.shape == (2 * n + n * n,)
    a = np.empty(n, np.float64)
    c = np.empty(n, np.float64)
    B = np.empty((n, n), np.float64)
    lib.orc_mhc_coeffs(n, d, iters, _ptr(x), _ptr(phi), _ptr(b), _ptr(a), _ptr(c), _ptr(B))
    return a, c, B


def mhc_pre(x, a):
    """The layer input h = sum_i a_i x[i] of one token (x uint16 [n, d], a float64 [n])."""
    lib = _load()
    x = _u16(x)
    n, d = x.shape
    a = np.ascontiguousarray(a, np.float64)
    h = np.empty(d, np.float64)
    lib.orc_mhc_pre(n, d, _ptr(x), _ptr(a), _ptr(h))
    return h


def mhc_post(x, B, c, y):
    """The streams after the layer, x'[i] = sum_j B[i, j] x[j] + c_i y (x uint16 [n, d],
    B float64 [n, n], c float64 [n], y uint16 [d]) -> float64 [n, d]."""
    lib = _load()
    x = _u16(x)
    y = _u16(y)
    n, d = x.shape
    B = np.ascontiguousarray(B, np.float64)
    c = np.ascontiguousarray(c, np.float64)
    xo = np.empty((n, d), np.float64)
    lib.orc_mhc_post(n, d, _ptr(x), _ptr(B), _ptr(c), _ptr(y), _ptr(xo))
    return xo


def e4m3_decode(code: int) -> float:
    """Value of one e4m3 code (NaN for S.1111.111)."""
    return float(_load().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """e4m3 code of a float32 value: nearest, ties to even mantissa, saturating at +-448."""
    return int(_load().orc_e4m3_encode(float(np.float32(x))))


def quantize_rows_e4m3(x):
    """Per-row e4m3 quantisation of bf16 rows x (uint16 [rows, width]): (codes uint8 [rows, width],
    scales float32 [rows]) with scale = amax/448 and code = e4m3(x/scale)."""
    lib = _load()
    x = _u16(x)
    rows, width = x.shape
    q = np.empty((rows, width), dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    lib.orc_quantize_rows_e4m3(rows, width, _ptr(x), _ptr(q), _ptr(sc))
    return q, sc


def dequantize_rows_e4m3(q, scale):
    """scale[r] * e4m3(q[r][i]) as float64 [rows, width]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scale = _f32(scale)
    rows, width = q.shape
    out = np.empty((rows, width), dtype=np.float64)
    lib.orc_dequantize_rows_e4m3(rows, width, _ptr(q), _ptr(scale), _ptr(out))
    return out


def compress_pc(tok_v, tok_z, tok_pos0, bias, gamma, eps, rope_dims, rope_base,
                span, stride, first_entry, n_new):
    """The compressor with per-channel logits tok_z (float32 [n_tok, width]) and per-channel
    offset biases bias (float32 [span, width]); otherwise as compress()."""
    lib = _load()
    tok_v = _u16(tok_v)
    tok_z = _f32(tok_z)
    bias = _f32(bias)
    g = None if gamma is None else _f32(gamma)
    n_tok, width = tok_v.shape
    assert tok_z.shape == (n_tok, width) and bias.shape == (span, width)
    out = np.empty((n_new, width), dtype=np.float64)
    rc = lib.orc_compress_pc(span, stride, width, _ptr(tok_v), _ptr(tok_z), tok_pos0, n_tok,
                             _ptr(bias), _ptr(g), eps, rope_dims, rope_base, first_entry, n_new, _ptr(out))
    if rc != 0:
        raise ValueError("orc_compress_pc: tokens needed by the requested entries are missing (rc=%d)" % rc)
    return out


def indexer_scores_e4m3(q8, qscale, w, k8, kscale, n_vis):
    """Indexer scores over e4m3 rows: q8 uint8 [H_I, d_I] with qscale [H_I], k8 uint8 [rows, d_I]
    with kscale [rows]; float64 [n_vis]."""
    lib = _load()
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    qscale, kscale, w = _f32(qscale), _f32(kscale), _f32(w)
    n_heads, dim = q8.shape
    assert k8.shape[1] == dim and k8.shape[0] >= n_vis and kscale.shape[0] >= n_vis
    out = np.empty(n_vis, dtype=np.float64)
    lib.orc_indexer_scores_e4m3(n_heads, dim, _ptr(q8), _ptr(qscale), _ptr(w), _ptr(k8), _ptr(kscale), n_vis,
                                _ptr(out))
    return out


def attend_e4m3(q, gamma_q, pos, comp8, comp_scale, sink, win, win_cap, W, rope_dims, rope_base, eps, scale,
                idx=None, n_dense=0):
    """attend() over an e4m3 compressed cache: comp8 uint8 [rows, c] with comp_scale float32 [rows]
    (row j read back as comp_scale[j] * e4m3(comp8[j])); the window ring stays bf16."""
    lib = _load()
    q = _u16(q)
    comp8 = np.ascontiguousarray(comp8, dtype=np.uint8)
    cs = _f32(comp_scale)
    win = _u16(win)
    g = _f32(gamma_q)
    sk = _f32(sink)
    H, c = q.shape
    ix = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((H, c), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    rc = lib.orc_attend_e4m3(H, c, rope_dims, rope_base, eps, scale, _ptr(q), _ptr(g), pos,
                             _ptr(comp8), _ptr(cs), comp8.shape[0], _ptr(ix), 0 if ix is None else ix.shape[0],
                             n_dense, _ptr(win), win_cap, W, _ptr(sk), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("orc_attend_e4m3: index outside the compressed cache (rc=%d)" % rc)
    return out, lse
