"""A numpy model of the attention kernel's number formats, checked against the oracle on the
inputs of the attention parity tests (CPU only).

The kernel re-encodes each bf16 KV row to fp16 in shared memory (exact: bf16 carries 8
significant bits, fp16 11), multiplies it with the normalised query split into two fp16
parts (hi = fp16(q), lo = fp16(q - hi)), rounds the probabilities to fp16 for the PV product,
accumulates in fp32 and stores bf16.  The model applies those roundings to a plain
(untiled) softmax attention; tiling and the kernel's accumulation order change the result
by far less than the roundings.  It shows that the formats leave the output at the error
floor set by its own bf16 rounding, and that a single fp16 query part would not: on one of
the test inputs that variant ends above the 2e-2 x RMS bar.

The query normalisation and the exact output come from the oracle; the output rotation is
restated here (and checked against the oracle) because the model rounds after it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import OUT_TOL
from workloads import Rng, bf16_bits

LOG2E = 1.4426950408889634


def _rotate(o, pos, R, base):
    """RoPE at `pos` on the trailing R dims, half-split pairs (d, d + R/2)."""
    o = o.copy()
    c, h = o.shape[-1], R // 2
    ang = pos * base ** (-2.0 * np.arange(h) / R)
    x, y = o[..., c - R:c - R + h].copy(), o[..., c - R + h:].copy()
    o[..., c - R:c - R + h] = x * np.cos(ang) - y * np.sin(ang)
    o[..., c - R + h:] = x * np.sin(ang) + y * np.cos(ang)
    return o


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _case(H, c, R, W, pos, n_vis):
    """One query of the HCA parity test's inputs (same seed and draws), its rows, and the oracle."""
    rng = Rng(15)
    B, n_q, rows, cap = 3, 2, 700, W + 8
    q = rng.normal_bf16((B, n_q, H, c))
    kv = rng.normal_bf16((B, rows, c))
    win = rng.normal_bf16((B, cap, c))
    gamma = (0.5 + torch.rand(c, generator=rng.g)).float().numpy()
    sink = rng.normal_f32((H,)).numpy()
    eps, base, scale = 1e-6, 10000.0, 1.0 / math.sqrt(c)
    qb = bf16_bits(q[0, 0])
    q_hat = np.stack([oracle.window_row(qb[h], gamma, eps, R, base, pos) for h in range(H)])
    t = np.arange(max(0, pos - W + 1), pos + 1)
    K = np.concatenate([kv[0, :n_vis].float().numpy(), win[0, t % cap].float().numpy()]).astype(np.float64)
    ref, _ = oracle.attend(qb, gamma, pos, bf16_bits(kv[0]), sink, bf16_bits(win[0]), cap, W, R, base, eps, scale,
                           n_dense=n_vis)
    return q_hat, K, sink, scale, base, ref


def _model(q_hat, K, sink, scale, parts):
    """Softmax attention with the kernel's formats: fp16 KV, q as `parts` fp16 terms, fp16 P."""
    Kf = K.astype(np.float16).astype(np.float32)
    q32 = q_hat.astype(np.float32)
    hi = q32.astype(np.float16).astype(np.float32)
    S = hi @ Kf.T
    if parts == 2:
        lo = (q32 - hi).astype(np.float16).astype(np.float32)
        S = S + lo @ Kf.T
    x = S * np.float32(scale * LOG2E)
    s2 = sink.astype(np.float32) * np.float32(LOG2E)
    M = np.maximum(x.max(1), s2)
    P = np.exp2(x - M[:, None]).astype(np.float16).astype(np.float32)
    L = P.sum(1) + np.exp2(s2 - M)
    return ((P @ Kf) / L[:, None]).astype(np.float64)


def _err(out, ref):
    return float(np.abs(out - ref).max() / np.sqrt(np.mean(ref * ref)))


@pytest.mark.parametrize("H,c,R,W", [(16, 256, 32, 40), (64, 512, 64, 128), (8, 128, 64, 16)])
def test_kernel_formats_reach_the_bf16_output_floor(H, c, R, W):
    pos, n_vis = 4 * 650 - 1, 650
    q_hat, K, sink, scale, base, ref = _case(H, c, R, W, pos, n_vis)
    # the model's exact arm reproduces the oracle (so the rotation restated here is the oracle's)
    s = q_hat @ K.T * scale
    mx = np.maximum(s.max(1), sink)
    p = np.exp(s - mx[:, None])
    exact = (p @ K) / (p.sum(1) + np.exp(sink - mx))[:, None]
    np.testing.assert_allclose(_rotate(exact, -pos, R, base), ref, rtol=0, atol=1e-9)
    floor = _err(_bf16(ref), ref)                         # the output's own bf16 rounding
    err = _err(_bf16(_rotate(_model(q_hat, K, sink, scale, 2), -pos, R, base)), ref)
    assert err <= floor + 1e-3, (err, floor)
    assert err <= OUT_TOL


def test_a_single_fp16_query_part_crosses_the_bar():
    pos, n_vis = 4 * 650 - 1, 650
    q_hat, K, sink, scale, base, ref = _case(16, 256, 32, 40, pos, n_vis)
    two = _err(_bf16(_rotate(_model(q_hat, K, sink, scale, 2), -pos, 32, base)), ref)
    one = _err(_bf16(_rotate(_model(q_hat, K, sink, scale, 1), -pos, 32, base)), ref)
    assert two <= OUT_TOL < one, (two, one)
