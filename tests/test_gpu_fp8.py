"""GPU parity of the FP8 (e4m3) cache variants and the per-channel compressor, through the C ABI.

The e4m3 codes are integers: the GPU quantiser must give the oracle's codes and scales bit for
bit.  The attention over e4m3 rows is held to the bf16 attention's bound against the oracle over
the same decoded rows.  The indexer over e4m3 rows is compared with the oracle evaluating the same bytes (codes
and scales the oracle produced from seeded bf16 inputs), at the bf16 indexer's tolerance, and
its top-k sets must match except at near-ties.  The compressor variants are compared with the
oracle at the bf16 compressor's tolerance (plus e4m3 rounding for the e4m3 cache).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close_rms, assert_rows_close, bf16_to_f64, check_topk, f32, u16
from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.api import AttnParams
from workloads import Rng, bits_to_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield


def dev(t):
    return t.to(DEV)


def quantize_gpu(x):
    width = x.shape[-1]
    q = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    sc = torch.empty(x.numel() // width, dtype=torch.float32, device=DEV)
    api.lca_quantize_rows_e4m3(dev(x).contiguous(), q, sc)
    return q.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("rows,width", [(1, 8), (37, 128), (300, 512), (5, 1024)])
def test_quantize_rows_bit_exact(rows, width):
    """Codes and scales equal the oracle's bit for bit, over rows of very different magnitudes:
    N(0, 1), tiny (subnormal codes), large, an all-zero row, signed zeros, repeated maxima."""
    rng = Rng(60 + width)
    x = rng.normal_bf16((rows, width))
    mags = torch.exp(torch.linspace(-30, 25, rows)).to(torch.bfloat16)
    x = (x.float() * mags.float()[:, None]).to(torch.bfloat16)
    if rows > 2:
        x[1] = 0.0
        x[2, ::2] = -0.0
        x[2, 1::3] = 3.0
        x[2, 2::3] = -3.0
    q, sc = quantize_gpu(x)
    q_ref, sc_ref = oracle.quantize_rows_e4m3(u16(x))
    np.testing.assert_array_equal(sc.view(np.uint32), sc_ref.view(np.uint32))
    np.testing.assert_array_equal(q, q_ref)


def _compress_case(csa, ratio, width, per_channel, seed):
    rng = Rng(seed)
    B = 3
    span = 2 * ratio if csa else ratio
    n_tok = 6 * ratio + (ratio if csa else 0)
    p = AttnParams(heads=8, head_dim=width, rope_dims=64, ratio=ratio)
    tok_v = rng.normal_bf16((B, n_tok, width))
    tok_z = rng.normal_f32((B, n_tok, width) if per_channel else (B, n_tok))
    bias = rng.normal_f32((span, width) if per_channel else (span,), 0.5)
    gamma = (0.5 + torch.rand(width, generator=rng.g)).float()
    pos0 = [0, 40 * ratio, 3000 * ratio]
    first = [0 if p0 == 0 else p0 // ratio + (1 if csa else 0) for p0 in pos0]
    n_new = 6
    rows = max(first) + n_new + 3
    return p, span, tok_v, tok_z, bias, gamma, pos0, first, n_new, rows


@pytest.mark.parametrize("csa,ratio,width", [(True, 4, 512), (True, 4, 128), (False, 128, 512), (False, 8, 256)])
def test_compress_per_channel_matches_oracle(csa, ratio, width):
    p, span, tok_v, tok_z, bias, gamma, pos0, first, n_new, rows = _compress_case(csa, ratio, width, True, 70)
    cache = torch.zeros((3, rows, width), dtype=torch.bfloat16, device=DEV)
    api.compress_kv_ex(csa, p, dev(tok_v), dev(tok_z), dev(torch.tensor(pos0, dtype=torch.int32)), dev(bias),
                       dev(gamma), True, dev(torch.tensor(first, dtype=torch.int32)), n_new, cache, per_channel=True)
    assert api.lca_device_error() == 0
    got = cache.cpu()
    for b in range(3):
        ref = oracle.compress_pc(u16(tok_v[b]), f32(tok_z[b]), pos0[b], f32(bias), f32(gamma), p.rms_eps, 64,
                                 p.rope_base, span, ratio, first[b], n_new)
        assert_rows_close(got[b, first[b]:first[b] + n_new], ref, "compress_pc b=%d" % b)
        assert (got[b, :first[b]] == 0).all() and (got[b, first[b] + n_new:] == 0).all()


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("csa,ratio,width", [(True, 4, 512), (False, 128, 512)])
def test_compress_e4m3_cache(csa, ratio, width, per_channel):
    """The e4m3 cache holds exactly the quantised bf16 row (the same call with a bf16 cache,
    then lca_quantize_rows_e4m3), and reads back close to the oracle's entry."""
    p, span, tok_v, tok_z, bias, gamma, pos0, first, n_new, rows = _compress_case(csa, ratio, width, per_channel,
                                                                                 71)
    args = (dev(tok_v), dev(tok_z), dev(torch.tensor(pos0, dtype=torch.int32)), dev(bias), dev(gamma), True,
            dev(torch.tensor(first, dtype=torch.int32)), n_new)
    c16 = torch.zeros((3, rows, width), dtype=torch.bfloat16, device=DEV)
    api.compress_kv_ex(csa, p, *args, c16, per_channel=per_channel)
    c8 = torch.zeros((3, rows, width), dtype=torch.uint8, device=DEV)
    s8 = torch.full((3, rows), -1.0, device=DEV)
    api.compress_kv_ex(csa, p, *args, c8, cache_scale=s8, per_channel=per_channel)
    assert api.lca_device_error() == 0
    q, sc = quantize_gpu(c16)
    c8h, s8h = c8.cpu().numpy(), s8.cpu().numpy()
    for b in range(3):
        w = slice(first[b], first[b] + n_new)
        np.testing.assert_array_equal(c8h[b, w], q.reshape(3, rows, width)[b, w])
        np.testing.assert_array_equal(s8h[b, w].view(np.uint32), sc.reshape(3, rows)[b, w].view(np.uint32))
        assert (c8h[b, :first[b]] == 0).all() and (s8h[b, :first[b]] == -1.0).all()
        fn = oracle.compress_pc if per_channel else oracle.compress
        ref = fn(u16(tok_v[b]), f32(tok_z[b]), pos0[b], f32(bias), f32(gamma), p.rms_eps, 64, p.rope_base, span,
                 ratio, first[b], n_new)
        back = oracle.dequantize_rows_e4m3(c8h[b, w], s8h[b, w])
        # e4m3 keeps 3 mantissa bits: 2^-4 relative, plus half the smallest step of the row's scale
        bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -9 * s8h[b, w][:, None] + 2e-3 * np.sqrt(np.mean(ref * ref))
        assert (np.abs(back - ref) <= bound).all()


def _e4m3_indexer_inputs(B, n_q, rows, seed, HI=64, DI=128):
    rng = Rng(seed)
    q = rng.normal_bf16((B, n_q, HI, DI))
    w = rng.normal_f32((B, n_q, HI), 1.0 / math.sqrt(HI))
    keys = rng.normal_bf16((B, rows, DI))
    q8, qs = oracle.quantize_rows_e4m3(u16(q).reshape(-1, DI))
    k8, ks = oracle.quantize_rows_e4m3(u16(keys).reshape(-1, DI))
    return (q8.reshape(B, n_q, HI, DI), qs.reshape(B, n_q, HI), w, k8.reshape(B, rows, DI), ks.reshape(B, rows))


def _t(a, dtype=None):
    return dev(torch.from_numpy(np.ascontiguousarray(a)))


@pytest.mark.parametrize("n_q,rows,k", [(1, 700, 64), (2, 1000, 128), (3, 2500, 512), (9, 3000, 1024)])
def test_indexer_e4m3_matches_oracle(n_q, rows, k):
    """Scores over e4m3 rows against the oracle reading the same codes and scales; the top-k
    lists against the oracle's; the fused path (n_q >= 3) equal to scores then lca_topk."""
    B, m = 2, 4
    p = AttnParams(idx_heads=64, idx_dim=128, ratio=m, topk=k)
    q8, qs, w, k8, ks = _e4m3_indexer_inputs(B, n_q, rows, 80 + n_q)
    g = np.random.default_rng(81)
    pos = g.integers(m * rows // 3, m * rows, size=(B, n_q)).astype(np.int32)
    pos[0, 0] = m * rows - 1
    if n_q > 1:
        pos[-1, -1] = m * (k // 2) + 1          # fewer than k visible
    pos_t = _t(pos)
    stride = (rows + 3) // 4 * 4
    scores = torch.full((B, n_q, stride), 7.0, device=DEV)
    api.csa_indexer_scores_e4m3(p, _t(q8), _t(qs), _t(w), _t(k8), _t(ks), pos_t, scores)
    assert api.lca_device_error() == 0
    ws = torch.empty(api.csa_indexer_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    sel = torch.full((B, n_q, k), -7, dtype=torch.int32, device=DEV)
    api.csa_indexer_topk_e4m3(p, _t(q8), _t(qs), _t(w), _t(k8), _t(ks), pos_t, sel, ws)
    plain = torch.empty_like(sel)
    api.lca_topk(p, scores, pos_t, rows, plain)
    assert api.lca_device_error() == 0
    assert torch.equal(sel, plain)
    s_gpu, i_gpu = scores.cpu().numpy(), sel.cpu().numpy()
    for b in range(B):
        for i in range(n_q):
            n_vis = min(oracle.visible_entries(int(pos[b, i]), m), rows)
            ref = oracle.indexer_scores_e4m3(q8[b, i], qs[b, i], w[b, i], k8[b], ks[b], n_vis)
            scale = max(np.abs(ref).max(), 1e-30) if n_vis else 1.0
            np.testing.assert_allclose(s_gpu[b, i, :n_vis].astype(np.float64), ref, rtol=1e-5, atol=1e-5 * scale)
            assert np.isneginf(s_gpu[b, i, n_vis:rows]).all()
            check_topk(i_gpu[b, i], ref, k, "b=%d i=%d" % (b, i))


def test_indexer_e4m3_close_to_bf16_indexer():
    """The e4m3 scores approximate the bf16 indexer's on the rows they were quantised from (three
    mantissa bits per factor; the errors of 128-term dot products mostly cancel)."""
    B, n_q, rows, m = 1, 4, 1500, 4
    p = AttnParams(idx_heads=64, idx_dim=128, ratio=m, topk=256)
    rng = Rng(90)
    q = rng.normal_bf16((B, n_q, 64, 128))
    w = rng.normal_f32((B, n_q, 64), 1.0 / 8)
    keys = rng.normal_bf16((B, rows, 128))
    q8, qs = oracle.quantize_rows_e4m3(u16(q).reshape(-1, 128))
    k8, ks = oracle.quantize_rows_e4m3(u16(keys).reshape(-1, 128))
    pos = _t(np.full((B, n_q), m * rows - 1, dtype=np.int32))
    s8 = torch.empty((B, n_q, rows), device=DEV)
    api.csa_indexer_scores_e4m3(p, _t(q8.reshape(B, n_q, 64, 128)), _t(qs.reshape(B, n_q, 64)), dev(w),
                                _t(k8.reshape(B, rows, 128)), _t(ks.reshape(B, rows)), pos, s8)
    s16 = torch.empty((B, n_q, rows), device=DEV)
    api.csa_indexer_scores(p, dev(q), dev(w), dev(keys), pos, s16)
    a, b = s8.cpu().numpy().ravel(), s16.cpu().numpy().ravel()
    rel = np.sqrt(np.mean((a - b) ** 2)) / np.sqrt(np.mean(b * b))
    assert rel < 0.05, rel


# ------------------------------------------------------------ e4m3 attention ----

def _attend8_inputs(seed, B, n_q, H, c, rows, W, cap):
    rng = Rng(seed)
    kv = rng.normal_bf16((B, rows, c))
    k8, ks = oracle.quantize_rows_e4m3(u16(kv).reshape(-1, c))
    return dict(q=rng.normal_bf16((B, n_q, H, c)), k8=k8.reshape(B, rows, c), ks=ks.reshape(B, rows),
                win=rng.normal_bf16((B, cap, c)), gamma=(0.5 + torch.rand(c, generator=rng.g)).float(),
                sink=rng.normal_f32((H,)))


def _check_attend8(p, d, pos, out, lse, idx=None):
    o, l = out.cpu().float().numpy(), lse.cpu().numpy()
    B, n_q = pos.shape
    for b in range(B):
        for i in range(n_q):
            kw = dict(idx=idx[b, i]) if idx is not None else dict(n_dense=oracle.visible_entries(int(pos[b, i]),
                                                                                                   p.ratio))
            ro, rl = oracle.attend_e4m3(u16(d["q"][b, i]), f32(d["gamma"]), int(pos[b, i]), d["k8"][b], d["ks"][b],
                                        f32(d["sink"]), u16(d["win"][b]), d["win"].shape[1], p.window, p.rope_dims,
                                        p.rope_base, p.rms_eps, p.scale, **kw)
            assert_close_rms(o[b, i], ro, what="e4m3 b=%d i=%d" % (b, i))
            np.testing.assert_allclose(l[b, i], rl, rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))


def test_hca_attend_e4m3_matches_oracle():
    """Dense attention over e4m3 rows against the oracle reading the same codes and scales: ragged,
    full, one-entry and zero-entry row lists; the rows a query cannot see hold NaN codes and NaN
    scales, which must not reach the output."""
    B, n_q, m, rows, H, c, W = 3, 2, 4, 700, 64, 512, 128
    cap = W + 8
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m)
    d = _attend8_inputs(95, B, n_q, H, c, rows, W, cap)
    d["k8"][1, 1:] = 0x7F              # sequence 1 sees at most entry 0
    d["ks"][1, 1:] = np.nan
    pos = np.array([[m * 650 - 1, m * 700 - 1], [4, 0], [m * 333 + 1, m * 129 - 2]], dtype=np.int32)
    out = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    api.hca_attend_e4m3(p, dev(d["q"]), dev(d["gamma"]), _t(pos), _t(d["k8"]), _t(d["ks"]), dev(d["win"]),
                        dev(d["sink"]), out, ws, lse)
    assert api.lca_device_error() == 0
    _check_attend8(p, d, pos, out, lse)


@pytest.mark.parametrize("k,W", [(512, 128), (300, 1)])
def test_csa_attend_e4m3_matches_oracle(k, W):
    """Attention over gathered e4m3 rows (selections with -1 padding, an empty selection) plus bf16
    window rows, against the oracle on the same bytes; unselected rows hold NaN codes."""
    B, n_q, rows, H, c = 2, 2, 3000, 64, 512
    cap = W + 5
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=4, topk=k)
    d = _attend8_inputs(96, B, n_q, H, c, rows, W, cap)
    g = np.random.default_rng(97)
    idx = np.full((B, n_q, k), -1, np.int32)
    counts = [[k, k - 37], [k // 3, 0]]
    used = np.zeros((B, rows), bool)
    for b in range(B):
        for i in range(n_q):
            sel = np.sort(g.choice(rows, counts[b][i], replace=False))
            idx[b, i, :len(sel)] = sel
            used[b, sel] = True
    d["k8"][~used] = 0x7F
    d["ks"][~used] = np.nan
    pos = np.array([[4 * rows - 1, 9000], [3, 700]], dtype=np.int32)
    out = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.csa_attend_workspace(p, B, n_q), dtype=torch.uint8, device=DEV)
    api.csa_attend_e4m3(p, dev(d["q"]), dev(d["gamma"]), _t(pos), _t(d["k8"]), _t(d["ks"]), _t(idx), dev(d["win"]),
                        dev(d["sink"]), out, ws, lse)
    assert api.lca_device_error() == 0
    _check_attend8(p, d, pos, out, lse, idx=idx)
