"""Test-side helpers: oracle references over batches and the parity comparisons.

The oracle is the reference; nothing here computes the method itself.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import bf16_bits

# Output tolerance of the attention path: max |gpu - oracle| <= 2e-2 * RMS(oracle output)
OUT_TOL = 2e-2
# Near-tie tolerance of top-k: entries whose oracle score is within 1e-5 * |s_(k)| of the k-th
NEAR_TIE = 1e-5


def u16(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t.cpu())


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float64)


def assert_close_rms(got: np.ndarray, ref: np.ndarray, tol: float = OUT_TOL, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "%s: non-finite values" % what
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert err <= tol * rms, "%s: max abs err %.3e > %.1e * rms %.3e" % (what, err, tol, rms)
    return err / rms if rms > 0 else 0.0


def assert_close_bf16_out(got: np.ndarray, ref: np.ndarray, tol: float = 1e-3, what: str = ""):
    """Element-wise bound for a product with fp32 accumulation and a bf16 result: half an ulp of
    bf16 (2^-8 of the value: 8 significant bits) plus tol x RMS for the accumulation order."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "%s: non-finite values" % what
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = np.abs(ref) * 2.0 ** -8 + tol * rms
    bad = np.abs(got - ref) > bound
    assert not bad.any(), "%s: %d values outside half a bf16 ulp + %.0e x rms (first at %s)" % (
        what, int(bad.sum()), tol, np.argwhere(bad)[0])


def assert_rows_close(got_bf16, ref, what=""):
    """A stored bf16 row equals the oracle's fp64 row up to bf16 rounding (+ fp32 arithmetic)."""
    got = bf16_to_f64(got_bf16)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = 2.0 ** -8 * np.abs(ref) + 2e-3 * rms
    err = np.abs(got - ref)
    assert (err <= bound).all(), "%s: worst %.3e at %s" % (what, float((err - bound).max()), np.argmax(err - bound))


def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """The oracle's fp64 values rounded to bf16 (nearest even) as uint16 bit patterns: how a
    row the oracle computed is stored in a bf16 cache."""
    return bf16_bits(torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16))


def check_topk(gpu_idx: np.ndarray, ref_scores: np.ndarray, k: int, what: str = ""):
    """GPU top-k list vs the oracle's fp64 scores: ascending, -1 padded, and equal to the oracle's
    set except for entries within NEAR_TIE of the k-th score."""
    n = ref_scores.shape[0]
    ref = oracle.topk(ref_scores, k)
    got = np.asarray(gpu_idx)
    take = min(k, n)
    assert (got[take:] == -1).all(), "%s: padding" % what
    sel = got[:take]
    assert (sel >= 0).all() and (sel < n).all(), "%s: index range" % what
    assert (np.diff(sel) > 0).all(), "%s: not strictly ascending" % what
    a, b = set(sel.tolist()), set(ref[:take].tolist())
    diff = a ^ b
    if diff:
        kth = np.sort(ref_scores)[::-1][take - 1]
        tol = NEAR_TIE * max(abs(kth), 1e-30)
        bad = [i for i in diff if abs(ref_scores[i] - kth) > tol]
        assert not bad, "%s: %d entries differ beyond near-ties, e.g. %s" % (what, len(bad), bad[:5])
    return len(diff)


def oracle_attend_batch(p, q, gamma_q, q_pos, kv_cache, win_kv, sink, idx=None, units=None):
    """Oracle attention for (b, i) units (all by default). Returns {(b, i): (out, lse)}."""
    B, n_q = q.shape[:2]
    qb = u16(q)
    kvb = u16(kv_cache)
    wb = u16(win_kv)
    g = f32(gamma_q)
    sk = f32(sink)
    pos = q_pos.cpu().numpy()
    ix = None if idx is None else idx.cpu().numpy()
    res = {}
    for (b, i) in (units or [(b, i) for b in range(B) for i in range(n_q)]):
        kw = dict(idx=ix[b, i]) if ix is not None else dict(n_dense=oracle.visible_entries(int(pos[b, i]), p.ratio))
        res[(b, i)] = oracle.attend(qb[b, i], g, int(pos[b, i]), kvb[b], sk, wb[b], win_kv.shape[1], p.window,
                                    p.rope_dims, p.rope_base, p.rms_eps, p.scale, **kw)
    return res
