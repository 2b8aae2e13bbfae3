"""GPU parity of every step of the path against the CPU oracle, through the C ABI.

Sizes are small enough for the oracle to finish in seconds but span several 128-row tiles
and end in a ragged tail.  Tolerances: attention outputs max |err| <= 2e-2 * RMS(oracle);
stored rows within bf16 rounding; top-k sets equal except at near-ties (1e-5 relative).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import (assert_close_bf16_out, assert_close_rms, assert_rows_close, bf16_to_f64, check_topk, f32,
                     oracle_attend_batch, u16)
from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.api import AttnParams
from workloads import Rng, bits_to_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()   # clear any stale device error bits
    yield


def dev(t):
    return t.to(DEV)


# ------------------------------------------------------------------ compress -------

@pytest.mark.parametrize("overlap,ratio,width,rope,norm", [
    (True, 4, 512, True, True),      # CSA KV entries
    (True, 4, 128, False, False),    # CSA indexer keys
    (False, 128, 512, True, True),   # HCA KV entries
    (False, 8, 256, True, True),
])
def test_compress_matches_oracle(overlap, ratio, width, rope, norm):
    rng = Rng(10)
    B = 3
    span = 2 * ratio if overlap else ratio
    n_tok = 6 * ratio + (ratio if overlap else 0)
    p = AttnParams(heads=8, head_dim=width, rope_dims=64, ratio=ratio)
    tok_v = rng.normal_bf16((B, n_tok, width))
    tok_z = rng.normal_f32((B, n_tok))
    bias = rng.normal_f32((span,), 0.5)
    gamma = (0.5 + torch.rand(width, generator=rng.g)).float()
    # sequence 0 starts at position 0 (entry 0's window is clipped); the others deep in a sequence
    pos0 = [0, 40 * ratio, 3000 * ratio]
    first = [0 if p0 == 0 else p0 // ratio + (1 if overlap else 0) for p0 in pos0]
    n_new = 6
    rows = max(first) + n_new + 3
    cache = torch.zeros((B, rows, width), dtype=torch.bfloat16)
    cache_d = dev(cache)
    fn = api.csa_compress_kv if overlap else api.hca_compress_kv
    fn(p, dev(tok_v), dev(tok_z), dev(torch.tensor(pos0, dtype=torch.int32)), dev(bias),
       dev(gamma) if norm else None, rope, dev(torch.tensor(first, dtype=torch.int32)), n_new, cache_d)
    assert api.lca_device_error() == 0
    got = cache_d.cpu()
    for b in range(B):
        ref = oracle.compress(u16(tok_v[b]), f32(tok_z[b]), pos0[b], f32(bias), f32(gamma) if norm else None,
                              p.rms_eps, 64 if rope else 0, p.rope_base, span, ratio, first[b], n_new)
        assert_rows_close(got[b, first[b]:first[b] + n_new], ref, "compress b=%d" % b)
        # rows outside the written range stay untouched
        assert (got[b, :first[b]] == 0).all() and (got[b, first[b] + n_new:] == 0).all()


def test_compress_missing_tokens_sets_device_error_and_skips():
    rng = Rng(11)
    p = AttnParams(head_dim=128, ratio=4)
    tok_v = dev(rng.normal_bf16((1, 8, 128)))
    cache = torch.zeros((1, 10, 128), dtype=torch.bfloat16, device=DEV)
    # entry 3 needs tokens 8..15 but the staging holds 0..7
    api.csa_compress_kv(p, tok_v, dev(rng.normal_f32((1, 8))), dev(torch.tensor([0], dtype=torch.int32)),
                        dev(torch.zeros(8)), None, 0, dev(torch.tensor([3], dtype=torch.int32)), 1, cache)
    assert api.lca_device_error() & 0x1
    assert (cache == 0).all()
    assert api.lca_device_error() == 0     # read clears it


def test_window_update_matches_oracle():
    rng = Rng(12)
    B, n_tok, c, cap = 2, 5, 512, 8
    p = AttnParams(head_dim=c, rope_dims=64)
    tok_v = rng.normal_bf16((B, n_tok, c))
    gamma = (0.5 + torch.rand(c, generator=rng.g)).float()
    pos0 = [6, 1048570]          # wraps around the ring of 8
    win = torch.zeros((B, cap, c), dtype=torch.bfloat16, device=DEV)
    api.lca_window_update(p, dev(tok_v), dev(torch.tensor(pos0, dtype=torch.int32)), dev(gamma), win)
    got = win.cpu()
    for b in range(B):
        for t in range(n_tok):
            pos = pos0[b] + t
            ref = oracle.window_row(u16(tok_v[b, t]), f32(gamma), p.rms_eps, 64, p.rope_base, pos)
            assert_rows_close(got[b, pos % cap], ref, "window b=%d pos=%d" % (b, pos))


# ------------------------------------------------------------ indexer + top-k -------

@pytest.mark.parametrize("HI,DI,rows,k", [(64, 128, 1000, 100), (4, 32, 300, 64), (32, 64, 777, 512)])
def test_indexer_scores_and_topk_match_oracle(HI, DI, rows, k):
    rng = Rng(13)
    B, n_q, m = 2, 3, 4
    p = AttnParams(idx_heads=HI, idx_dim=DI, ratio=m, topk=k)
    q = rng.normal_bf16((B, n_q, HI, DI))
    w = rng.normal_f32((B, n_q, HI), 1.0 / math.sqrt(HI))
    keys = rng.normal_bf16((B, rows, DI))
    # visible entries: all rows, a ragged middle, fewer than k, and zero
    pos = torch.tensor([[m * rows - 1, m * 517 + 2, m * (k // 2) - 1],
                        [m * rows + 50, m * 128 - 1, 0]], dtype=torch.int32)
    stride = (rows + 3) // 4 * 4
    scores = torch.full((B, n_q, stride), 7.0, device=DEV)
    api.csa_indexer_scores(p, dev(q), dev(w), dev(keys), dev(pos), scores)
    err = api.lca_device_error()
    assert err == 0x4   # position (rows + 50) sees more entries than the cache holds: clamped, reported
    out_idx = torch.empty((B, n_q, k), dtype=torch.int32, device=DEV)
    api.lca_topk(p, scores, dev(pos), rows, out_idx)
    assert api.lca_device_error() == 0x4
    s_gpu = scores.cpu().numpy()
    i_gpu = out_idx.cpu().numpy()
    for b in range(B):
        for i in range(n_q):
            n_vis = min(oracle.visible_entries(int(pos[b, i]), m), rows)
            ref = oracle.indexer_scores(u16(q[b, i]), f32(w[b, i]), u16(keys[b]), n_vis)
            got = s_gpu[b, i, :n_vis].astype(np.float64)
            scale = max(np.abs(ref).max(), 1e-30) if n_vis else 1.0
            np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5 * scale)
            assert np.isneginf(s_gpu[b, i, n_vis:rows]).all()
            check_topk(i_gpu[b, i], ref, k, "b=%d i=%d" % (b, i))
    # the combined call gives the same lists
    ws = torch.empty(api.csa_indexer_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    out2 = torch.empty_like(out_idx)
    api.csa_indexer_topk(p, dev(q), dev(w), dev(keys), dev(pos), out2, ws)
    api.lca_device_error()
    assert torch.equal(out2, out_idx)


@pytest.mark.parametrize("B,rows", [(600, 100), (300, 200), (150, 300)])
def test_indexer_many_short_sequences(B, rows):
    """Decode-shaped calls (one query per sequence) with sequences of 1-3 tiles: every CTA walks
    several sequences, so each query-tile buffer is refilled (after the MMAs release it)."""
    rng = Rng(21)
    m, k = 4, 64
    p = AttnParams(idx_heads=64, idx_dim=128, ratio=m, topk=k)
    q = rng.normal_bf16((B, 1, 64, 128))
    w = rng.normal_f32((B, 1, 64), 0.125)
    keys = rng.normal_bf16((B, rows, 128))
    pos = torch.tensor([[m * (rows - (b % 7)) - 1] for b in range(B)], dtype=torch.int32)
    stride = (rows + 3) // 4 * 4
    scores = torch.full((B, 1, stride), 7.0, device=DEV)
    api.csa_indexer_scores(p, dev(q), dev(w), dev(keys), dev(pos), scores)
    assert api.lca_device_error() == 0
    s_gpu = scores.cpu().numpy()
    qb, wf, kb = u16(q), f32(w), u16(keys)
    for b in range(B):
        n_vis = oracle.visible_entries(int(pos[b, 0]), m)
        ref = oracle.indexer_scores(qb[b, 0], wf[b, 0], kb[b], n_vis)
        got = s_gpu[b, 0, :n_vis].astype(np.float64)
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5 * max(np.abs(ref).max(), 1e-30),
                                   err_msg="sequence %d" % b)
        assert np.isneginf(s_gpu[b, 0, n_vis:rows]).all()


@pytest.mark.parametrize("n,k", [(5000, 300), (262144, 1024), (1023, 1024), (32768, 512), (100003, 64)])
def test_topk_exact_on_given_scores_with_ties(n, k):
    """Scores given (not computed): the GPU selection must equal the oracle's exactly, ties included."""
    g = np.random.default_rng(14)
    rows = []
    rows.append(g.integers(-20, 20, n).astype(np.float32))           # heavy ties
    rows.append(np.zeros(n, np.float32))                              # all equal
    r = g.standard_normal(n).astype(np.float32)
    r[g.integers(0, n, n // 10)] = np.sort(r)[-k] if n > k else 0.0   # ties at the boundary
    rows.append(r)
    rows.append(-np.abs(g.standard_normal(n)).astype(np.float32))    # all negative, with -0.0
    rows[-1][::7] = -0.0
    rows[-1][3::7] = 0.0
    rows.append((8.0 * g.standard_normal(n)).astype(np.float32))      # no ties (indexer-like spread)
    r = (-1.0 - g.random(n)).astype(np.float32)                       # 60% share the selected first digit:
    hot = g.random(n) < 0.6                                           # more candidates than one CTA holds
    r[hot] = (1.0 + 0.25 * g.random(int(hot.sum()))).astype(np.float32)
    rows.append(r)
    R = len(rows)
    S = np.stack(rows)[None]                   # [1, R, n]
    stride = (n + 3) // 4 * 4
    Sp = np.full((1, R, stride), -np.inf, np.float32)
    Sp[..., :n] = S
    p = AttnParams(topk=k, ratio=1)
    pos = torch.full((1, R), n - 1, dtype=torch.int32)
    out = torch.empty((1, R, k), dtype=torch.int32, device=DEV)
    api.lca_topk(p, dev(torch.from_numpy(Sp)), dev(pos), n, out)
    got = out.cpu().numpy()
    for r in range(R):
        np.testing.assert_array_equal(got[0, r], oracle.topk(S[0, r].astype(np.float64), k))


# ------------------------------------------------------------------- attention -------

def _attend_inputs(rng, B, n_q, H, c, rows, W, cap):
    return dict(
        q=rng.normal_bf16((B, n_q, H, c)),
        kv=rng.normal_bf16((B, rows, c)),
        win=rng.normal_bf16((B, cap, c)),
        gamma=(0.5 + torch.rand(c, generator=rng.g)).float(),
        sink=rng.normal_f32((H,)),
    )


@pytest.mark.parametrize("H,c,R,W", [(64, 512, 64, 128), (8, 128, 64, 16), (16, 256, 32, 40), (1, 512, 64, 128)])
def test_hca_attend_matches_oracle(H, c, R, W):
    rng = Rng(15)
    B, n_q, m, rows = 3, 2, 4, 700
    cap = W + 8
    p = AttnParams(heads=H, head_dim=c, rope_dims=R, window=W, ratio=m)
    d = _attend_inputs(rng, B, n_q, H, c, rows, W, cap)
    # visible entries: 650 (ragged), 700 (all), 1 (tiny), 0 with a short window, deep positions
    pos = torch.tensor([[m * 650 - 1, m * 700 - 1], [4, 0], [m * 333 + 1, m * 129 - 2]], dtype=torch.int32)
    out = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    api.hca_attend(p, dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"]), dev(d["win"]), dev(d["sink"]), out,
                   ws, lse)
    assert api.lca_device_error() == 0
    ref = oracle_attend_batch(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"])
    o = out.cpu().float().numpy()
    l = lse.cpu().numpy()
    for (b, i), (ro, rl) in ref.items():
        assert_close_rms(o[b, i], ro, what="hca b=%d i=%d" % (b, i))
        np.testing.assert_allclose(l[b, i], rl, rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))


@pytest.mark.parametrize("H,c,k,W", [(64, 512, 512, 128), (8, 128, 64, 16), (64, 512, 300, 1)])
def test_csa_attend_with_injected_indices_matches_oracle(H, c, k, W):
    rng = Rng(16)
    B, n_q, rows = 2, 2, 3000
    cap = W + 5
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=4, topk=k)
    d = _attend_inputs(rng, B, n_q, H, c, rows, W, cap)
    g = np.random.default_rng(17)
    idx = np.full((B, n_q, k), -1, np.int32)
    counts = [[k, k - 37], [k // 3, 0]]
    for b in range(B):
        for i in range(n_q):
            sel = np.sort(g.choice(rows, counts[b][i], replace=False))
            idx[b, i, :len(sel)] = sel
    idx_t = torch.from_numpy(idx)
    pos = torch.tensor([[4 * rows - 1, 9000], [3, 700]], dtype=torch.int32)
    out = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.csa_attend_workspace(p, B, n_q), dtype=torch.uint8, device=DEV)
    api.csa_attend(p, dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"]), dev(idx_t), dev(d["win"]),
                   dev(d["sink"]), out, ws, lse)
    assert api.lca_device_error() == 0
    ref = oracle_attend_batch(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"], idx=idx_t)
    o = out.cpu().float().numpy()
    l = lse.cpu().numpy()
    for (b, i), (ro, rl) in ref.items():
        assert_close_rms(o[b, i], ro, what="csa b=%d i=%d" % (b, i))
        np.testing.assert_allclose(l[b, i], rl, rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_attend_prepare_then_prepared_equals_attend(kind):
    """The query preparation on one stream and the attention on another (joined by an event) give
    the same bits as the single call."""
    rng = Rng(19)
    B, n_q, rows, H, c, W, k = 2, 3, 900, 64, 512, 128, 512
    cap = W + 3
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=4, topk=k)
    d = _attend_inputs(rng, B, n_q, H, c, rows, W, cap)
    pos = torch.tensor([[4 * rows - 1, 2000, 5], [3 * rows, 131, 4 * rows - 9]], dtype=torch.int32)
    g = np.random.default_rng(20)
    idx = torch.from_numpy(np.stack([np.stack([np.sort(g.choice(rows, k, replace=False)) for _ in range(n_q)])
                                     for _ in range(B)]).astype(np.int32))
    args = [dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"])]
    if kind == "csa":
        args.append(dev(idx))
        ws_bytes = api.csa_attend_workspace(p, B, n_q)
    else:
        ws_bytes = api.hca_attend_workspace(p, B, n_q, rows)
    args += [dev(d["win"]), dev(d["sink"])]
    whole, split = (torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV) for _ in range(2))
    lse_w, lse_s = (torch.empty((B, n_q, H), dtype=torch.float32, device=DEV) for _ in range(2))
    ws_w, ws_s = (torch.empty(ws_bytes, dtype=torch.uint8, device=DEV) for _ in range(2))
    getattr(api, kind + "_attend")(p, *args, whole, ws_w, lse_w)
    side, ev = torch.cuda.Stream(), torch.cuda.Event()
    side.wait_stream(torch.cuda.current_stream())
    getattr(api, kind + "_attend_prepare")(p, *args, split, ws_s, lse_s, stream=side)
    ev.record(side)
    torch.cuda.current_stream().wait_event(ev)
    getattr(api, kind + "_attend_prepared")(p, *args, split, ws_s, lse_s)
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    assert torch.equal(whole.view(torch.int16), split.view(torch.int16))
    assert torch.equal(lse_w, lse_s)


def test_attend_reports_out_of_range_indices():
    rng = Rng(18)
    p = AttnParams(heads=8, head_dim=128, window=4, ratio=4, topk=8)
    d = _attend_inputs(rng, 1, 1, 8, 128, 50, 4, 4)
    idx = torch.tensor([[[0, 1, 2, 60, -1, -1, -1, -1]]], dtype=torch.int32)
    out = torch.empty((1, 1, 8, 128), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(api.csa_attend_workspace(p, 1, 1), dtype=torch.uint8, device=DEV)
    api.csa_attend(p, dev(d["q"]), dev(d["gamma"]), dev(torch.tensor([[10]], dtype=torch.int32)), dev(d["kv"]),
                   dev(idx), dev(d["win"]), dev(d["sink"]), out, ws)
    assert api.lca_device_error() & 0x2
    # the bad index is skipped: same as the list without it
    ref = oracle_attend_batch(p, d["q"], d["gamma"], torch.tensor([[10]]), d["kv"], d["win"], d["sink"],
                              idx=torch.tensor([[[0, 1, 2, -1, -1, -1, -1, -1]]], dtype=torch.int32))
    assert_close_rms(out.cpu().float().numpy()[0, 0], ref[(0, 0)][0], what="skip bad index")


# ------------------------------------------------------------- output projection ----

@pytest.mark.parametrize("B,H,c,G,d_g,d", [(4, 64, 512, 8, 1024, 4096), (3, 64, 512, 16, 512, 1000),
                                            (1, 16, 512, 4, 256, 512), (9, 8, 128, 2, 64, 96)])
def test_grouped_oproj_matches_oracle(B, H, c, G, d_g, d):
    rng = Rng(19)
    o = rng.normal_bf16((B, H, c))
    Wg = rng.normal_bf16((G * d_g, (H // G) * c), 0.02)
    Wm = rng.normal_bf16((d, G * d_g), 0.02)
    mid = torch.empty((B, G * d_g), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((B, d), dtype=torch.bfloat16, device=DEV)
    api.lca_grouped_oproj(dev(o), dev(Wg), dev(Wm), G, mid, y)
    got = y.cpu().float().numpy()
    for b in range(B):
        ref = oracle.grouped_oproj(u16(o[b]), u16(Wg), u16(Wm), G)
        assert_close_rms(got[b], ref, what="oproj b=%d" % b)


def test_gemm_matches_oracle():
    rng = Rng(20)
    # the first four take the general kernel; the rest the streaming one (contiguous weights,
    # K a multiple of 2048, N a multiple of 4), with fewer 4-row groups than SMs in the last
    for M, N, K in ((1, 37, 64), (4, 1000, 256), (16, 515, 4096), (3, 8, 8), (5, 124, 8192),
                    (1, 4096, 2048), (2, 1000, 6144), (7, 512, 4096), (4, 640, 8192), (3, 12, 2048)):
        A = rng.normal_bf16((M, K))
        Bm = rng.normal_bf16((N, K))
        C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        api.lca_gemm_bf16(dev(A), dev(Bm), C)
        ref = oracle.gemm_bf16(u16(A), u16(Bm))
        assert_close_bf16_out(C.cpu().float().numpy(), ref, what="gemm %dx%dx%d" % (M, N, K))


# ------------------------------------------------- every indexer dispatch branch ----

@pytest.mark.parametrize("HI,DI,n_q", [(64, 128, 1), (64, 128, 2), (64, 128, 5), (32, 64, 1), (32, 64, 2),
                                       (4, 32, 1)])
def test_indexer_every_dispatch_shape(HI, DI, n_q):
    """One case per kernel instantiation the library dispatches to (queries per tile 1, 2, 4 for
    d_I = 128; 1, 8 for d_I = 64; 4 for d_I = 32), each with a ragged last tile, a query that
    sees fewer entries than k and one that sees none."""
    rng = Rng(22 + n_q)
    B, m, rows, k = 3, 4, 651, 96
    p = AttnParams(idx_heads=HI, idx_dim=DI, ratio=m, topk=k)
    q = rng.normal_bf16((B, n_q, HI, DI))
    w = rng.normal_f32((B, n_q, HI), 1.0 / math.sqrt(HI))
    keys = rng.normal_bf16((B, rows, DI))
    choices = [m * rows - 1, m * 389 + 3, m * (k // 3) + 1, 2, m * 129 - 1]
    pos = torch.tensor([[choices[(b * n_q + i) % len(choices)] for i in range(n_q)] for b in range(B)],
                       dtype=torch.int32)
    stride = (rows + 3) // 4 * 4
    scores = torch.full((B, n_q, stride), 7.0, device=DEV)
    api.csa_indexer_scores(p, dev(q), dev(w), dev(keys), dev(pos), scores)
    assert api.lca_device_error() == 0
    out_idx = torch.empty((B, n_q, k), dtype=torch.int32, device=DEV)
    api.lca_topk(p, scores, dev(pos), rows, out_idx)
    assert api.lca_device_error() == 0
    s_gpu, i_gpu = scores.cpu().numpy(), out_idx.cpu().numpy()
    qb, wf, kb = u16(q), f32(w), u16(keys)
    for b in range(B):
        for i in range(n_q):
            n_vis = oracle.visible_entries(int(pos[b, i]), m)
            ref = oracle.indexer_scores(qb[b, i], wf[b, i], kb[b], n_vis)
            got = s_gpu[b, i, :n_vis].astype(np.float64)
            scale = max(np.abs(ref).max(), 1e-30) if n_vis else 1.0
            np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5 * scale, err_msg="b=%d i=%d" % (b, i))
            assert np.isneginf(s_gpu[b, i, n_vis:rows]).all()
            check_topk(i_gpu[b, i], ref, k, "b=%d i=%d" % (b, i))


# ------------------------------------------- split count, batch position, decode ----

def _attend_call(kind, p, d, pos, idx=None):
    B, n_q = pos.shape
    out = torch.empty((B, n_q, p.heads, p.head_dim), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, p.heads), dtype=torch.float32, device=DEV)
    if kind == "csa":
        ws = torch.empty(api.csa_attend_workspace(p, B, n_q), dtype=torch.uint8, device=DEV)
        api.csa_attend(p, dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"]), dev(idx), dev(d["win"]),
                       dev(d["sink"]), out, ws, lse)
    else:
        ws = torch.empty(api.hca_attend_workspace(p, B, n_q, d["kv"].shape[1]), dtype=torch.uint8, device=DEV)
        api.hca_attend(p, dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"]), dev(d["win"]), dev(d["sink"]),
                       out, ws, lse)
    assert api.lca_device_error() == 0
    return out.cpu().float().numpy(), lse.cpu().numpy()


def _tile(t, reps):
    return t.repeat(reps, *([1] * (t.dim() - 1)))


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_attend_independent_of_split_count(kind):
    """The same two queries alone (each gets many split-K CTAs) and inside a batch of 75 copies
    (one split each): both within the bar of the oracle, and their log-sum-exps agree."""
    rng = Rng(23)
    H, c, W, m, rows, k = 64, 512, 128, 4, 1400, 512
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m, topk=k)
    d1 = _attend_inputs(rng, 1, 2, H, c, rows, W, W + 4)
    pos1 = torch.tensor([[m * rows - 1, m * 777 + 2]], dtype=torch.int32)
    g = np.random.default_rng(24)
    idx1 = torch.from_numpy(np.stack([np.sort(g.choice(rows, k, replace=False)) for _ in range(2)])
                            .astype(np.int32)).view(1, 2, k)
    reps = 75
    dn = dict(d1, q=_tile(d1["q"], reps), kv=_tile(d1["kv"], reps), win=_tile(d1["win"], reps))
    posn, idxn = _tile(pos1, reps), _tile(idx1, reps)
    o1, l1 = _attend_call(kind, p, d1, pos1, idx1)
    on, ln = _attend_call(kind, p, dn, posn, idxn)
    ref = oracle_attend_batch(p, d1["q"], d1["gamma"], pos1, d1["kv"], d1["win"], d1["sink"],
                              idx=idx1 if kind == "csa" else None)
    for i in range(2):
        ro, rl = ref[(0, i)]
        assert_close_rms(o1[0, i], ro, what="alone i=%d" % i)
        for b in (0, 37, reps - 1):
            assert_close_rms(on[b, i], ro, what="batched b=%d i=%d" % (b, i))
            np.testing.assert_allclose(ln[b, i], l1[0, i], rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))
        np.testing.assert_allclose(l1[0, i], rl, rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_attend_independent_of_batch_position(kind):
    """A sequence's result does not depend on where it sits in the batch: the same query at
    batch positions 0 and 5 (same call, same split plan) gives the same bits."""
    rng = Rng(25)
    H, c, W, m, rows, k, B = 64, 512, 128, 4, 900, 256, 6
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m, topk=k)
    d = _attend_inputs(rng, B, 1, H, c, rows, W, W + 2)
    for key in ("q", "kv", "win"):
        d[key][B - 1] = d[key][0]
    pos = torch.tensor([[m * rows - 1 - 7 * b] for b in range(B)], dtype=torch.int32)
    pos[B - 1, 0] = pos[0, 0]
    g = np.random.default_rng(26)
    idx = torch.from_numpy(np.stack([np.sort(g.choice(rows, k, replace=False)) for _ in range(B)])
                           .astype(np.int32)).view(B, 1, k)
    idx[B - 1] = idx[0]
    o, l = _attend_call(kind, p, d, pos, idx)
    assert np.array_equal(o[0], o[B - 1]) and np.array_equal(l[0], l[B - 1])
    assert not np.array_equal(o[0], o[1])


def test_csa_decode_equals_last_prefill_row():
    """A prefill chunk's last query and a decode call for that same token (same selection, same
    caches): the outputs agree within the bar, and each matches the oracle."""
    rng = Rng(27)
    H, c, W, m, k, T = 64, 512, 128, 4, 512, 40
    rows, q0 = 2000, 4 * 2000 - 40
    cap = T + W
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m, topk=k)
    d = _attend_inputs(rng, 1, T, H, c, rows, W, cap)
    pos = torch.arange(q0, q0 + T, dtype=torch.int32).view(1, T)
    g = np.random.default_rng(28)
    idx = torch.from_numpy(np.stack([np.sort(g.choice(rows, k, replace=False)) for _ in range(T)])
                           .astype(np.int32)).view(1, T, k)
    o_pre, l_pre = _attend_call("csa", p, d, pos, idx)
    d1 = dict(d, q=d["q"][:, T - 1:].contiguous())
    o_dec, l_dec = _attend_call("csa", p, d1, pos[:, T - 1:].contiguous(), idx[:, T - 1:].contiguous())
    ref = oracle_attend_batch(p, d1["q"], d["gamma"], pos[:, T - 1:], d["kv"], d["win"], d["sink"],
                              idx=idx[:, T - 1:])[(0, 0)]
    assert_close_rms(o_pre[0, T - 1], ref[0], what="prefill last row")
    assert_close_rms(o_dec[0, 0], ref[0], what="decode")
    assert_close_rms(o_dec[0, 0], o_pre[0, T - 1], what="decode vs prefill")
    np.testing.assert_allclose(l_dec[0, 0], l_pre[0, T - 1], rtol=0, atol=2e-3 * max(1.0, np.abs(ref[1]).max()))


# ------------------------------------------------------------ fp16 input domain ----

@pytest.mark.parametrize("where", ["gamma_q", "kv_row", "window_row", "none"])
def test_attend_reports_values_outside_fp16(where):
    """The products run in fp16: a query or row element beyond 65504 would saturate.  Such a call
    sets LCA_DEVERR_FP16_RANGE; an in-range call right at the edge of the inputs does not."""
    rng = Rng(29)
    H, c, W, m, rows = 8, 256, 16, 4, 300
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m)
    d = _attend_inputs(rng, 1, 1, H, c, rows, W, W)
    pos = torch.tensor([[m * rows - 1]], dtype=torch.int32)
    if where == "gamma_q":
        d["gamma"] = torch.full((c,), 30000.0)     # normalised q ~ N(0, 1) x 30000: tails beyond 65504
    elif where == "kv_row":
        d["kv"][0, 123, 77] = 70000.0
    elif where == "window_row":
        d["win"][0, 5, 200] = -1e30
    else:
        d["gamma"] = torch.full((c,), 2000.0)      # |q| < 6 x 2000 < 65504
        d["kv"][0, 123, 77] = 60000.0
    out = torch.empty((1, 1, H, c), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(api.hca_attend_workspace(p, 1, 1, rows), dtype=torch.uint8, device=DEV)
    api.hca_attend(p, dev(d["q"]), dev(d["gamma"]), dev(pos), dev(d["kv"]), dev(d["win"]), dev(d["sink"]), out, ws)
    err = api.lca_device_error()
    assert err == (0 if where == "none" else 0x10), hex(err)


@pytest.mark.parametrize("M,N,K", [(300, 100, 200), (128, 64, 64), (1000, 300, 1024), (257, 513, 4096),
                                   (17, 24, 16384), (640, 256, 136)])
def test_tensor_core_gemm_matches_oracle(M, N, K):
    """The tensor-core product (M > 16 for bf16 out, any M for fp32 out): ragged M, N and K tails,
    every tile width (N up to 64, 128, 256)."""
    rng = Rng(30)
    A = rng.normal_bf16((M, K))
    Bm = rng.normal_bf16((N, K), 0.05)
    ref = oracle.gemm_bf16(u16(A), u16(Bm))
    C32 = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    api.lca_gemm_bf16(dev(A), dev(Bm), C32)
    assert api.lca_device_error() == 0
    got = C32.cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=2e-6 * rms * math.sqrt(K))
    if M > 16:
        C16 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        api.lca_gemm_bf16(dev(A), dev(Bm), C16)
        assert_close_bf16_out(C16.cpu().float().numpy(), ref, what="gemm %dx%dx%d" % (M, N, K))



@pytest.mark.parametrize("B,n_q,rows,k,mode", [(1, 8, 3000, 1024, "plain"), (2, 5, 2000, 512, "dups"),
                                               (1, 7, 20000, 1024, "dups"), (3, 3, 700, 1024, "plain"),
                                               (1, 64, 5000, 300, "dups"), (1, 6, 30000, 1024, "few"),
                                               (2, 4, 12000, 700, "zero")])
def test_fused_indexer_topk_equals_scores_then_topk(B, n_q, rows, k, mode):
    """The prefill path (four queries per tile) selects the top k inside the indexer.  It must give
    the same lists as the scores written out and selected by lca_topk, and the oracle's sets:
    ragged query groups, queries that see fewer than k entries or none, rows long enough for
    several compactions of the candidate buffers, and equal scores, which the lower index must
    win: repeated key rows (dups), five distinct key rows for the whole row, so that thousands of
    candidates share each score and the compactions must cut by index (few), and zero head
    weights for one query, whose scores are then all zero (zero)."""
    rng = Rng(40 + n_q)
    m, HI, DI = 4, 64, 128
    p = AttnParams(idx_heads=HI, idx_dim=DI, ratio=m, topk=k)
    q = rng.normal_bf16((B, n_q, HI, DI))
    w = rng.normal_f32((B, n_q, HI), 1.0 / math.sqrt(HI))
    keys = rng.normal_bf16((B, rows, DI))
    if mode == "dups":
        keys[:, 1::3] = keys[:, 0::3][:, :keys[:, 1::3].shape[1]]     # row 3i + 1 repeats row 3i
    elif mode == "few":
        keys = keys[:, torch.arange(rows) % 5]
    elif mode == "zero":
        w[0, 2] = 0.0
    g = np.random.default_rng(41)
    pos = torch.from_numpy(g.integers(m * rows // 2, m * rows, size=(B, n_q)).astype(np.int32))
    pos[0, 0] = m * rows - 1
    pos[0, 1] = m * (k // 2) + 1          # fewer than k visible
    pos[-1, -1] = 1                       # none visible
    ws = torch.empty(api.csa_indexer_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    fused = torch.full((B, n_q, k), -7, dtype=torch.int32, device=DEV)
    api.csa_indexer_topk(p, dev(q), dev(w), dev(keys), dev(pos), fused, ws)
    assert api.lca_device_error() == 0
    stride = (rows + 3) // 4 * 4
    scores = torch.empty((B, n_q, stride), device=DEV)
    api.csa_indexer_scores(p, dev(q), dev(w), dev(keys), dev(pos), scores)
    plain = torch.empty_like(fused)
    api.lca_topk(p, scores, dev(pos), rows, plain)
    assert api.lca_device_error() == 0
    assert torch.equal(fused, plain)
    # the selection's warp groups synchronise among themselves: repeated calls give the same lists
    for _ in range(6):
        again = torch.full_like(fused, -7)
        api.csa_indexer_topk(p, dev(q), dev(w), dev(keys), dev(pos), again, ws)
        assert torch.equal(again, fused)
    assert api.lca_device_error() == 0
    got = fused.cpu().numpy()
    qb, wf, kb = u16(q), f32(w), u16(keys)
    for b in range(B):
        for i in range(n_q):
            n_vis = oracle.visible_entries(int(pos[b, i]), m)
            ref = oracle.indexer_scores(qb[b, i], wf[b, i], kb[b], n_vis)
            check_topk(got[b, i], ref, k, "b=%d i=%d" % (b, i))
