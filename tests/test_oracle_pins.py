"""Pins for the CPU oracle: closed forms, invariants, special cases and brute force.

Each test checks the oracle against something other than itself -- a value fixed by
the definition of the step in closed form, a textbook computation written another
way (numpy), or a hand derivation -- so that a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle fails at least one of them.
The definitions follow the DeepSeek-V4 hybrid-attention write-ups: CSA steps one to
four and the HCA paragraph (gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制) and
the Flash hyper-parameters (zhinnengdao.top, section 3.1 "Hybrid Attention: CSA + HCA").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_bits(x) -> np.ndarray:
    """Round float values to bf16 and return the bit patterns (exact for small integers)."""
    return bf16_bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def from_bits(b) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def rand_bits(rng, shape, std=1.0):
    return to_bits(rng.standard_normal(shape) * std)


# ---------------------------------------------------------------- compressor ----

def test_compress_uniform_weights_give_window_means():
    """z = 0 and b = 0: every entry is the plain mean of the tokens its window covers."""
    rng = np.random.default_rng(1)
    v = rand_bits(rng, (16, 8))
    vf = from_bits(v)
    z = np.zeros(16, np.float32)
    # CSA, m = 4: windows [4(j-1), 4(j+1)) clipped at 0.
    out = oracle.compress(v, z, 0, np.zeros(8, np.float32), None, 0.0, 0, 10000.0,
                          span=8, stride=4, first_entry=0, n_new=4)
    expect = [vf[0:4].mean(0), vf[0:8].mean(0), vf[4:12].mean(0), vf[8:16].mean(0)]
    np.testing.assert_allclose(out, np.stack(expect), rtol=0, atol=1e-14)
    # HCA, m' = 4: windows [4j, 4(j+1)), no overlap.
    out = oracle.compress(v, z, 0, np.zeros(4, np.float32), None, 0.0, 0, 10000.0,
                          span=4, stride=4, first_entry=0, n_new=4)
    expect = [vf[4 * j:4 * j + 4].mean(0) for j in range(4)]
    np.testing.assert_allclose(out, np.stack(expect), rtol=0, atol=1e-14)


def test_compress_dominant_logit_copies_its_token():
    """One token's logit 60 above the others: the entry is that token (weights e^-60 elsewhere)."""
    rng = np.random.default_rng(2)
    v = rand_bits(rng, (12, 16))
    for hot in range(4, 12):
        z = np.zeros(12, np.float32)
        z[hot] = 60.0
        out = oracle.compress(v, z, 0, np.zeros(8, np.float32), None, 0.0, 0, 10000.0,
                              span=8, stride=4, first_entry=2, n_new=1)
        np.testing.assert_allclose(out[0], from_bits(v[hot]), rtol=0, atol=1e-20)


def test_compress_position_bias_uses_offsets_in_the_nominal_window():
    """b_r = log(r+1), z = 0: weights proportional to r+1 over the offsets that survive.

    Entry 0 of CSA covers tokens 0..3, which sit at offsets 4..7 of its nominal window
    [-4, 4); entry 1 covers tokens 0..7 at offsets 0..7.
    """
    v = to_bits(np.arange(8, dtype=np.float32)[:, None] * np.ones((1, 2)))  # token t = (t, t)
    b = np.log(np.arange(1, 9, dtype=np.float64)).astype(np.float32)
    z = np.zeros(8, np.float32)
    out = oracle.compress(v, z, 0, b, None, 0.0, 0, 10000.0, span=8, stride=4, first_entry=0, n_new=2)
    bw = np.exp(b.astype(np.float64))  # the fp32-rounded logs, exponentiated
    w0 = bw[4:8] / bw[4:8].sum()
    w1 = bw / bw.sum()
    assert out[0, 0] == pytest.approx(float((w0 * np.arange(4)).sum()), abs=1e-13)
    assert out[1, 0] == pytest.approx(float((w1 * np.arange(8)).sum()), abs=1e-13)
    # close to the exact-weight values 5..8 / 26 and 1..8 / 36
    assert out[0, 0] == pytest.approx((0 * 5 + 1 * 6 + 2 * 7 + 3 * 8) / 26.0, rel=1e-6)
    assert out[1, 0] == pytest.approx(sum(t * (t + 1) for t in range(8)) / 36.0, rel=1e-6)


def test_compress_logit_and_bias_add():
    """z_t and b_r enter the softmax as a sum: z = log 3 on one token equals b = log 3 on its offset."""
    rng = np.random.default_rng(3)
    v = rand_bits(rng, (8, 4))
    z = np.zeros(8, np.float32)
    z[5] = math.log(3.0)
    b = np.zeros(8, np.float32)
    b[5] = math.log(3.0)
    a = oracle.compress(v, z, 0, np.zeros(8, np.float32), None, 0.0, 0, 1e4, 8, 4, 1, 1)
    c = oracle.compress(v, np.zeros(8, np.float32), 0, b, None, 0.0, 0, 1e4, 8, 4, 1, 1)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-15)
    vf = from_bits(v)
    expect = (vf.sum(0) + 2 * vf[5]) / 10.0   # weights 1,1,1,1,1,3,1,1 over 10
    np.testing.assert_allclose(a[0], expect, rtol=1e-6, atol=1e-7)


def test_compress_missing_tokens_rejected():
    v = to_bits(np.ones((4, 2)))
    with pytest.raises(ValueError):
        oracle.compress(v, np.zeros(4, np.float32), 4, np.zeros(8, np.float32), None, 0.0, 0, 1e4,
                        8, 4, 1, 1)   # entry 1 needs tokens 0..7, only 4..7 given


# ----------------------------------------------------------------- RMSNorm -----

def _single(v_row, gamma, eps, rope_dims=0, base=10000.0, pos=0):
    """Compress a single token alone (span = stride = 1): the entry is the token, at `pos`."""
    v = np.asarray(v_row, np.uint16)[None, :]
    return oracle.compress(v, np.zeros(1, np.float32), pos, np.zeros(1, np.float32), gamma, eps,
                           rope_dims, base, span=1, stride=1, first_entry=pos, n_new=1)[0]


def test_rmsnorm_unit_rms_scale_invariance_gamma_and_eps():
    rng = np.random.default_rng(4)
    v = rand_bits(rng, (64,))
    ones = np.ones(64, np.float32)
    y = _single(v, ones, 0.0)
    assert np.mean(y * y) == pytest.approx(1.0, abs=1e-14)
    # scale invariance: 2x is exact in bf16
    y2 = _single(to_bits(2.0 * from_bits(v)), ones, 0.0)
    np.testing.assert_allclose(y2, y, rtol=0, atol=1e-14)
    # y / gamma has unit RMS
    gam = (0.5 + rng.random(64)).astype(np.float32)
    yg = _single(v, gam, 0.0)
    assert np.mean((yg / gam) ** 2) == pytest.approx(1.0, abs=1e-12)
    # eps enters under the root next to the mean square: all-ones row, eps = 3 -> 1/2
    yo = _single(to_bits(np.ones(64)), ones, 3.0)
    np.testing.assert_allclose(yo, 0.5, rtol=0, atol=1e-15)


# -------------------------------------------------------------------- RoPE -----

def test_rope_rotates_trailing_dims_half_split_pairs():
    """c=8, R=4, base=100: pairs (4,6) at theta=1 and (5,7) at theta=100^(-1/2); dims 0..3 fixed."""
    c, R, base = 8, 4, 100.0
    for pos in (0, 1, 3, 7, 1000):
        for src, partner, theta in ((4, 6, 1.0), (5, 7, 0.1)):
            e = np.zeros(c)
            e[src] = 1.0
            y = _single(to_bits(e), None, 0.0, R, base, pos)
            expect = np.zeros(c)
            expect[src] = math.cos(pos * theta)
            expect[partner] = math.sin(pos * theta)
            np.testing.assert_allclose(y, expect, rtol=0, atol=1e-12)
            # the partner goes to (-sin, cos)
            e = np.zeros(c)
            e[partner] = 1.0
            y = _single(to_bits(e), None, 0.0, R, base, pos)
            expect = np.zeros(c)
            expect[src] = -math.sin(pos * theta)
            expect[partner] = math.cos(pos * theta)
            np.testing.assert_allclose(y, expect, rtol=0, atol=1e-12)
        for i in range(c - R):
            e = np.zeros(c)
            e[i] = 1.0
            np.testing.assert_array_equal(_single(to_bits(e), None, 0.0, R, base, pos), e)


def test_entry_position_is_its_last_token():
    """CSA entry j is rotated at m(j+1)-1, HCA entry j at m'(j+1)-1 (R=2, theta=1)."""
    c = 4
    e = np.zeros((16, c))
    e[:, 2] = 1.0
    v = to_bits(e)
    z = np.zeros(16, np.float32)
    csa = oracle.compress(v, z, 0, np.zeros(8, np.float32), None, 0.0, 2, 1e4, 8, 4, 0, 4)
    hca = oracle.compress(v, z, 0, np.zeros(8, np.float32), None, 0.0, 2, 1e4, 8, 8, 0, 2)
    for j in range(4):
        p = 4 * (j + 1) - 1
        np.testing.assert_allclose(csa[j, 2:], [math.cos(p), math.sin(p)], atol=1e-12)
    for j in range(2):
        p = 8 * (j + 1) - 1
        np.testing.assert_allclose(hca[j, 2:], [math.cos(p), math.sin(p)], atol=1e-12)


def test_visible_entries_strictly_causal():
    # m = 4: the block [4j, 4j+4) becomes visible at position 4j+3
    assert [oracle.visible_entries(p, 4) for p in range(10)] == [0, 0, 0, 1, 1, 1, 1, 2, 2, 2]
    assert oracle.visible_entries(131071, 4) == 32768
    assert oracle.visible_entries(1048575, 128) == 8192
    assert oracle.visible_entries(1048574, 128) == 8191


# ----------------------------------------------------------------- indexer -----

def test_indexer_single_head_is_relu_dot():
    rng = np.random.default_rng(5)
    q = rand_bits(rng, (1, 32))
    k = rand_bits(rng, (50, 32))
    s = oracle.indexer_scores(q, np.ones(1, np.float32), k, 50)
    np.testing.assert_allclose(s, np.maximum(from_bits(k) @ from_bits(q)[0], 0.0), rtol=1e-14, atol=1e-13)
    assert (s == 0).any() and (s > 0).any()


def test_indexer_head_permutation_and_linearity_in_w():
    rng = np.random.default_rng(6)
    q = rand_bits(rng, (8, 16))
    k = rand_bits(rng, (40, 16))
    w1 = rng.standard_normal(8).astype(np.float32)
    w2 = rng.standard_normal(8).astype(np.float32)
    s1 = oracle.indexer_scores(q, w1, k, 40)
    s2 = oracle.indexer_scores(q, w2, k, 40)
    s12 = oracle.indexer_scores(q, (w1.astype(np.float64) + w2).astype(np.float32), k, 40)
    np.testing.assert_allclose(s12, s1 + s2, rtol=1e-6, atol=1e-6)
    perm = rng.permutation(8)
    np.testing.assert_allclose(oracle.indexer_scores(q[perm], w1[perm], k, 40), s1, rtol=1e-13, atol=1e-12)
    # a head contributes w_h * relu(dot): brute force per head
    dots = from_bits(k) @ from_bits(q).T
    np.testing.assert_allclose(s1, (np.maximum(dots, 0) * w1.astype(np.float64)).sum(1), rtol=1e-12, atol=1e-11)
    # only the first n_vis entries are scored
    np.testing.assert_array_equal(oracle.indexer_scores(q, w1, k, 7), s1[:7])


# ------------------------------------------------------------------- top-k -----

def _brute_topk(scores, k):
    order = np.lexsort((np.arange(len(scores)), -np.asarray(scores)))
    take = np.sort(order[:min(k, len(scores))])
    return np.concatenate([take, -np.ones(k - len(take), np.int64)]).astype(np.int32)


def test_topk_matches_full_sort_with_ties():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, 64))
        s = rng.integers(-5, 6, n).astype(np.float64)   # many ties
        np.testing.assert_array_equal(oracle.topk(s, k), _brute_topk(s, k))
        s = rng.standard_normal(n)
        np.testing.assert_array_equal(oracle.topk(s, k), _brute_topk(s, k))


def test_topk_ties_go_to_lower_index_and_short_lists_pad():
    np.testing.assert_array_equal(oracle.topk(np.zeros(10), 4), [0, 1, 2, 3])
    np.testing.assert_array_equal(oracle.topk(np.array([1.0, 2.0, 2.0, 0.0, 2.0]), 2), [1, 2])
    np.testing.assert_array_equal(oracle.topk(np.array([3.0, 1.0]), 4), [0, 1, -1, -1])
    np.testing.assert_array_equal(oracle.topk(np.zeros(0), 3), [-1, -1, -1])


def test_topk_local_then_merge_equals_global():
    """Top-k of the union of per-chunk top-k lists equals the global top-k."""
    rng = np.random.default_rng(8)
    s = np.round(rng.standard_normal(1000), 1)   # ties across chunks
    k = 37
    cand = []
    for lo in range(0, 1000, 128):
        local = oracle.topk(s[lo:lo + 128], k)
        cand += [lo + i for i in local if i >= 0]
    cand = np.array(sorted(cand))
    merged = cand[oracle.topk(s[cand], k)]
    np.testing.assert_array_equal(merged, oracle.topk(s, k))


# --------------------------------------------------------------- attention -----

def _textbook(qf, gamma, rows, sink, scale):
    """Softmax attention with a sink column written with numpy (no RoPE: R = 0)."""
    qh = qf / np.sqrt((qf * qf).mean(1, keepdims=True)) * gamma
    logits = scale * qh @ rows.T
    full = np.concatenate([sink[:, None], logits], 1)
    mx = full.max(1, keepdims=True)
    e = np.exp(full - mx)
    p = e / e.sum(1, keepdims=True)
    return p[:, 1:] @ rows, (mx[:, 0] + np.log(e.sum(1)))


def test_attend_full_selection_equals_textbook_attention():
    """k >= visible entries and W >= pos+1: CSA is softmax attention over all visible
    entries plus all tokens up to the query (no RoPE, sink in the denominator)."""
    rng = np.random.default_rng(9)
    H, c, pos = 3, 16, 13
    comp = rand_bits(rng, (20, c))
    win = rand_bits(rng, (32, c))
    q = rand_bits(rng, (H, c))
    gamma = (0.5 + rng.random(c)).astype(np.float32)
    sink = rng.standard_normal(H).astype(np.float32)
    n_vis = oracle.visible_entries(pos, 4)          # 3
    idx = np.array(list(range(n_vis)) + [-1] * 5, np.int32)
    out, lse = oracle.attend(q, gamma, pos, comp, sink, win, 32, 32, 0, 1e4, 0.0, 0.25, idx=idx)
    rows = np.concatenate([from_bits(comp[:n_vis]), from_bits(win[:pos + 1])])
    e_out, e_lse = _textbook(from_bits(q), gamma.astype(np.float64), rows, sink.astype(np.float64), 0.25)
    np.testing.assert_allclose(out, e_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, e_lse, rtol=1e-12, atol=1e-13)
    # HCA with the same rows: dense over the first n_dense entries
    out, lse = oracle.attend(q, gamma, pos, comp, sink, win, 32, 32, 0, 1e4, 0.0, 0.25, n_dense=n_vis)
    np.testing.assert_allclose(out, e_out, rtol=1e-12, atol=1e-13)


def test_attend_window_reads_ring_slots():
    """W = 3 at pos 12 with a ring of 5 rows: tokens 10, 11, 12 -> slots 0, 1, 2."""
    rng = np.random.default_rng(10)
    H, c = 2, 8
    win = rand_bits(rng, (5, c))
    win[3:] = to_bits(np.full((2, c), 50.0))   # slots not in the window: would dominate if read
    q = rand_bits(rng, (H, c))
    gamma = np.ones(c, np.float32)
    sink = np.zeros(H, np.float32)
    comp = rand_bits(rng, (4, c))
    out, _ = oracle.attend(q, gamma, 12, comp, sink, win, 5, 3, 0, 1e4, 0.0, 0.3, n_dense=0)
    e_out, _ = _textbook(from_bits(q), 1.0, from_bits(win[[0, 1, 2]]), sink.astype(np.float64), 0.3)
    np.testing.assert_allclose(out, e_out, rtol=1e-12, atol=1e-13)
    # pos 1 with W = 3: only tokens 0, 1
    out, _ = oracle.attend(q, gamma, 1, comp, sink, win, 5, 3, 0, 1e4, 0.0, 0.3, n_dense=0)
    e_out, _ = _textbook(from_bits(q), 1.0, from_bits(win[[0, 1]]), sink.astype(np.float64), 0.3)
    np.testing.assert_allclose(out, e_out, rtol=1e-12, atol=1e-13)


def test_attend_probabilities_plus_sink_sum_to_one():
    """One-hot rows e_r (R = 0): o_r = p_r, so sum(o) + exp(sink - lse) = 1 per head."""
    rng = np.random.default_rng(11)
    H, c = 4, 16
    comp = to_bits(np.eye(c)[:10])
    win = to_bits(np.eye(c)[10:14])
    q = rand_bits(rng, (H, c))
    sink = rng.standard_normal(H).astype(np.float32)
    out, lse = oracle.attend(q, np.ones(c, np.float32), 3, comp, sink, win, 4, 4, 0, 1e4, 0.0, 0.7,
                             idx=np.arange(10, dtype=np.int32))
    mass = out.sum(1) + np.exp(sink.astype(np.float64) - lse)
    np.testing.assert_allclose(mass, 1.0, rtol=0, atol=1e-14)
    assert (out[:, 14:] == 0).all()


def test_attend_sink_limits_and_identical_rows():
    rng = np.random.default_rng(12)
    H, c = 2, 8
    q = rand_bits(rng, (H, c))
    comp = rand_bits(rng, (6, c))
    win = rand_bits(rng, (4, c))
    g = np.ones(c, np.float32)
    idx = np.arange(6, dtype=np.int32)
    # sink -> -inf: plain softmax
    out, _ = oracle.attend(q, g, 3, comp, np.full(H, -1e4, np.float32), win, 4, 4, 0, 1e4, 0.0, 0.5, idx=idx)
    rows = np.concatenate([from_bits(comp), from_bits(win)])
    qh = from_bits(q) / np.sqrt((from_bits(q) ** 2).mean(1, keepdims=True))
    lg = 0.5 * qh @ rows.T
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(out, p @ rows, rtol=1e-12, atol=1e-13)
    # sink -> +inf: all mass on the sink, output vanishes, lse -> sink
    out, lse = oracle.attend(q, g, 3, comp, np.full(H, 1e4, np.float32), win, 4, 4, 0, 1e4, 0.0, 0.5, idx=idx)
    assert np.abs(out).max() < 1e-300
    np.testing.assert_allclose(lse, 1e4, rtol=1e-15)
    # identical rows v: o = (1 - p_sink) v with p_sink = e^s / (e^s + n e^l)
    v = rand_bits(rng, (c,))
    same = np.tile(v, (6, 1))
    wsame = np.tile(v, (4, 1))
    s = np.array([0.3, -1.2], np.float32)
    out, _ = oracle.attend(q, g, 3, same, s, wsame, 4, 4, 0, 1e4, 0.0, 0.5, idx=idx)
    vf = from_bits(v)
    l = 0.5 * qh @ vf
    n = 6 + 4
    psink = np.exp(s.astype(np.float64)) / (np.exp(s.astype(np.float64)) + n * np.exp(l))
    np.testing.assert_allclose(out, (1 - psink)[:, None] * vf[None, :], rtol=1e-12, atol=1e-13)


def test_hca_ratio_one_is_causal_attention_with_window_counted_twice():
    """HCA with m' = 1, b = 0: entries are the normalised tokens themselves; attention is
    causal over all tokens 0..i plus the last W tokens again (no de-duplication)."""
    rng = np.random.default_rng(13)
    H, c, n, W = 2, 8, 10, 3
    v = rand_bits(rng, (n, c))
    gamma = np.ones(c, np.float32)
    ent = oracle.compress(v, rng.standard_normal(n).astype(np.float32), 0, np.zeros(1, np.float32),
                          gamma, 1e-6, 0, 1e4, 1, 1, 0, n)
    np.testing.assert_allclose(ent, from_bits(v) / np.sqrt((from_bits(v) ** 2).mean(1, keepdims=True) + 1e-6),
                               rtol=1e-13, atol=1e-14)
    comp = to_bits(ent)
    win = comp.copy()          # window rows of token t are the same normalised vectors
    q = rand_bits(rng, (H, c))
    sink = rng.standard_normal(H).astype(np.float32)
    i = 7
    n_vis = oracle.visible_entries(i, 1)
    assert n_vis == i + 1
    out, _ = oracle.attend(q, gamma, i, comp, sink, win, n, W, 0, 1e4, 0.0, 0.4, n_dense=n_vis)
    rows = np.concatenate([from_bits(comp[:i + 1]), from_bits(win[i - W + 1:i + 1])])
    e_out, _ = _textbook(from_bits(q), 1.0, rows, sink.astype(np.float64), 0.4)
    np.testing.assert_allclose(out, e_out, rtol=1e-12, atol=1e-13)


def _rotate_rows(x, positions, R, base):
    """RoPE written as complex multiplication (a + ib) e^{i p theta}: an independent restatement."""
    x = np.array(x, dtype=np.float64, copy=True)
    c = x.shape[-1]
    half = R // 2
    theta = base ** (-2.0 * np.arange(half) / R)
    z = x[..., c - R:c - half] + 1j * x[..., c - half:]
    z = z * np.exp(1j * np.asarray(positions, dtype=np.float64)[..., None] * theta)
    x[..., c - R:c - half] = z.real
    x[..., c - half:] = z.imag
    return x


def test_relative_position_invariance_under_a_global_shift():
    """Shifting every position (query, entries, window rows) by D leaves the output unchanged:
    q is rotated by +i, rows by their positions and the output by -i, so only differences remain.
    Rows are stored in bf16 at their absolute angles, so the two runs agree to bf16 rounding."""
    rng = np.random.default_rng(14)
    H, c, R, base, m, W = 4, 32, 16, 10000.0, 4, 6
    raw_e = rng.standard_normal((8, c))
    raw_w = rng.standard_normal((W, c))
    q = rand_bits(rng, (H, c))
    g = np.ones(c, np.float32)
    sink = rng.standard_normal(H).astype(np.float32)
    outs = []
    for shift_blocks in (0, 25, 1000):
        D = m * shift_blocks
        pos = 40 + D
        ent_pos = [m * (j + shift_blocks + 1) - 1 for j in range(8)]
        comp = np.zeros((8 + shift_blocks, c), np.uint16)
        comp[shift_blocks:] = to_bits(_rotate_rows(raw_e, ent_pos, R, base))
        win = np.zeros((W, c), np.uint16)
        for t in range(pos - W + 1, pos + 1):
            win[t % W] = to_bits(_rotate_rows(raw_w[t - (pos - W + 1)], t, R, base))
        idx = np.arange(shift_blocks, shift_blocks + 8, dtype=np.int32)
        out, _ = oracle.attend(q, g, pos, comp, sink, win, W, W, R, base, 0.0, c ** -0.5, idx=idx)
        outs.append(out)
    rms = np.sqrt(np.mean(outs[0] ** 2))
    for o in outs[1:]:
        # bf16 rounding of rows stored at different absolute angles: ~2^-9 per element
        assert np.abs(o - outs[0]).max() < 3e-2 * rms
    # and with the output rotation compared against the complex restatement directly
    pos = 40
    comp = to_bits(_rotate_rows(raw_e, [m * (j + 1) - 1 for j in range(8)], R, base))
    win = np.zeros((W, c), np.uint16)
    for t in range(pos - W + 1, pos + 1):
        win[t % W] = to_bits(_rotate_rows(raw_w[t - (pos - W + 1)], t, R, base))
    out, _ = oracle.attend(q, g, pos, comp, sink, win, W, W, R, base, 0.0, c ** -0.5,
                           idx=np.arange(8, dtype=np.int32))
    rows = np.concatenate([from_bits(comp), from_bits(win[[t % W for t in range(pos - W + 1, pos + 1)]])])
    qf = from_bits(q)
    qh = _rotate_rows(qf / np.sqrt((qf ** 2).mean(1, keepdims=True)), pos, R, base)
    lg = np.concatenate([sink[:, None].astype(np.float64), c ** -0.5 * qh @ rows.T], 1)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    expect = _rotate_rows(p[:, 1:] @ rows, -pos, R, base)
    np.testing.assert_allclose(out, expect, rtol=1e-11, atol=1e-12)


def test_attend_rejects_indices_outside_the_cache():
    g = np.ones(4, np.float32)
    z = np.zeros((2, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.attend(z[:1], g, 3, z, np.zeros(1, np.float32), z, 2, 2, 0, 1e4, 0.0, 0.5,
                      idx=np.array([2], np.int32))


# ------------------------------------------------------- hand-worked example ---

def test_hand_worked_8_token_example():
    """Eight tokens, m = 4, c = 4, R = 2, H = H_I = 1, d_I = 2, k = 1, W = 2, query at 7.

    Derivation (eps = 0, gamma = 1, z = b = 0, so every compressor weight is uniform):
      Compression.  Entry 0 pools tokens 0..3 = (1,1,1,-1): u0 = (1,1,1,-1), mean square 1,
        so RMSNorm leaves it; RoPE at position 3 rotates (1,-1) by 3 rad:
        (cos3 + sin3, sin3 - cos3).
        Entry 1 pools tokens 0..7: u1 = (1,0,1,0), mean square 1/2, RMSNorm -> (r2,0,r2,0)
        with r2 = sqrt 2; RoPE at 7 rotates (r2, 0) to (r2 cos7, r2 sin7).
        Indexer keys (no norm, no RoPE): k0 = (1,0), k1 = mean of 4x(1,0) and 4x(-1,2) = (0,1).
      Indexer at pos 7: both entries visible (floor(8/4) = 2).
        s0 = 0.5 ReLU(2*1 - 1*0) = 1,  s1 = 0.5 ReLU(2*0 - 1*1) = 0  ->  top-1 = [0].
      Window rows: tokens 6 and 7 = (1,-1,1,1) (mean square 1), RoPE (1,1) at 6 and 7.
      Query: (1,1,1,1) has mean square 1; RoPE at 7.
        Logit with a row at position p (scale 1/2): q.row = q01.row01 + [cos(p-7)(q2r2+q3r3)
        + sin(p-7)(q3 r2 - q2 r3)] over the raw rotated pairs:
          entry 0 (p=3, raw pair (1,-1)): (1+1) + cos4*0 + sin(-4)*(1+1)  -> l = 1 - sin 4
          token 6 (p=6, raw pair (1,1)):  (1-1) + cos1*2 + sin(-1)*0       -> l = cos 1
          token 7 (p=7):                  (1-1) + 2                         -> l = 1
      Softmax with sink 1: den = e^1 + e^(1-sin4) + e^(cos1) + e^1; p_r = e^(l_r) / den.
      Output: o = RoPE(sum p_r row_r, -7), i.e. each row's rotated pair ends up rotated by
        (p_r - 7):  R(-4)(1,-1) = (cos4 - sin4, -sin4 - cos4),  R(-1)(1,1) = (cos1 + sin1,
        cos1 - sin1),  R(0)(1,1) = (1,1); unrotated dims: entry 0 (1,1), tokens 6,7 (1,-1).
    """
    with open(os.path.join(GOLDEN, "hand_example_8tok.json")) as f:
        ex = json.load(f)
    m, c, R, base, eps = ex["m"], ex["c"], ex["rope_dims"], ex["rope_base"], ex["rms_eps"]
    v = to_bits(ex["tok_v"])
    vi = to_bits(ex["tok_vi"])
    z = np.array(ex["tok_z"], np.float32)
    ones = np.ones(c, np.float32)
    kv = oracle.compress(v, z, 0, np.zeros(2 * m, np.float32), ones, eps, R, base, 2 * m, m, 0, 2)
    ki = oracle.compress(vi, z, 0, np.zeros(2 * m, np.float32), None, eps, 0, base, 2 * m, m, 0, 2)
    c3, s3, c7, s7, c6, s6 = math.cos(3), math.sin(3), math.cos(7), math.sin(7), math.cos(6), math.sin(6)
    r2 = math.sqrt(2.0)
    np.testing.assert_allclose(kv[0], [1, 1, c3 + s3, s3 - c3], atol=1e-14)
    np.testing.assert_allclose(kv[1], [r2, 0, r2 * c7, r2 * s7], atol=1e-14)
    np.testing.assert_allclose(ki, [[1, 0], [0, 1]], atol=1e-15)

    pos = ex["query_pos"]
    n_vis = oracle.visible_entries(pos, m)
    assert n_vis == 2
    s = oracle.indexer_scores(to_bits(ex["q_idx"]), np.array(ex["idx_w"], np.float32), to_bits(ki), n_vis)
    np.testing.assert_allclose(s, [1.0, 0.0], atol=1e-15)
    idx = oracle.topk(s, ex["topk"])
    np.testing.assert_array_equal(idx, [0])

    win = np.zeros((ex["win_cap"], c), np.uint16)
    for t in (6, 7):
        row = oracle.window_row(v[t], ones, eps, R, base, t)
        np.testing.assert_allclose(row, [1, -1, math.cos(t) - math.sin(t), math.sin(t) + math.cos(t)], atol=1e-14)
        win[t % ex["win_cap"]] = to_bits(row)
    comp = to_bits(kv)
    out, lse = oracle.attend(to_bits(ex["q"]), ones, pos, comp, np.array(ex["sink"], np.float32), win,
                             ex["win_cap"], ex["window"], R, base, eps, c ** -0.5, idx=idx)
    # The stored rows are bf16-rounded; the closed form below uses the exact rows, so the
    # comparison allows bf16 rounding of the row values (relative 2^-8).
    l = np.array([1 - math.sin(4), math.cos(1), 1.0])
    den = math.e + np.exp(l).sum()
    p = np.exp(l) / den
    c4, s4, c1, s1 = math.cos(4), math.sin(4), math.cos(1), math.sin(1)
    expect = np.array([
        p[0] * 1 + p[1] * 1 + p[2] * 1,
        p[0] * 1 + p[1] * -1 + p[2] * -1,
        p[0] * (c4 - s4) + p[1] * (c1 + s1) + p[2] * 1,
        p[0] * (-s4 - c4) + p[1] * (c1 - s1) + p[2] * 1,
    ])
    np.testing.assert_allclose(out[0], expect, rtol=0, atol=1.5e-2)
    assert lse[0] == pytest.approx(math.log(den), abs=1.5e-2)
    # exact agreement once the same bf16 rows are used in the closed form
    rows = np.stack([from_bits(comp[0]), from_bits(win[6]), from_bits(win[7])])
    qh = np.array([1.0, 1.0, c7 - s7, s7 + c7])
    l_exact = 0.5 * rows @ qh
    den = math.e + np.exp(l_exact).sum()
    o = (np.exp(l_exact) / den) @ rows
    a, b = o[2], o[3]
    o_rot = [o[0], o[1], a * c7 + b * s7, -a * s7 + b * c7]   # rotation by -7
    np.testing.assert_allclose(out[0], o_rot, rtol=0, atol=1e-13)
    assert lse[0] == pytest.approx(math.log(den), abs=1e-13)


# ------------------------------------------------------- output projection -----

def test_grouped_projection_is_block_diagonal_matmul():
    rng = np.random.default_rng(15)
    H, c, G, d_g, d = 8, 16, 4, 6, 10
    o = rand_bits(rng, (H, c))
    Wg = rand_bits(rng, (G * d_g, (H // G) * c), 0.1)
    Wm = rand_bits(rng, (d, G * d_g), 0.1)
    y = oracle.grouped_oproj(o, Wg, Wm, G)
    blk = np.zeros((G * d_g, H * c))
    in_g = (H // G) * c
    Wgf = from_bits(Wg)
    for g in range(G):
        blk[g * d_g:(g + 1) * d_g, g * in_g:(g + 1) * in_g] = Wgf[g * d_g:(g + 1) * d_g]
    np.testing.assert_allclose(y, from_bits(Wm) @ (blk @ from_bits(o).reshape(-1)), rtol=1e-12, atol=1e-13)


def test_gemm_matches_numpy():
    rng = np.random.default_rng(16)
    A = rand_bits(rng, (7, 33))
    B = rand_bits(rng, (5, 33))
    np.testing.assert_allclose(oracle.gemm_bf16(A, B), from_bits(A) @ from_bits(B).T, rtol=1e-13, atol=1e-13)


# ------------------------------------------- manifold-constrained hyper-connections ----
# The mHC section of the first page (and [P4] 3.2): a, c through a sigmoid, B projected onto the
# doubly stochastic matrices by Sinkhorn-Knopp (row and column normalisations in turn).

def _mhc_inputs(rng, n, d, z_target=None):
    """x and phi chosen so that z = flatten(x) . phi^T + bias is known: phi = 0 gives z = bias."""
    x = rand_bits(rng, (n, d))
    phi = np.zeros((2 * n + n * n, n * d), np.uint16)
    bias = np.asarray(z_target, np.float32) if z_target is not None else rng.standard_normal(2 * n + n * n).astype(
        np.float32)
    return x, phi, bias


def test_mhc_generated_logits_and_sigmoids_match_numpy():
    rng = np.random.default_rng(60)
    n, d = 4, 48
    x = rand_bits(rng, (n, d))
    phi = rand_bits(rng, (2 * n + n * n, n * d), 0.1)
    bias = rng.standard_normal(2 * n + n * n).astype(np.float32)
    a, c, B = oracle.mhc_coeffs(x, phi, bias, iters=0)
    z = from_bits(phi) @ from_bits(x).reshape(-1) + bias.astype(np.float64)
    np.testing.assert_allclose(a, 1.0 / (1.0 + np.exp(-z[:n])), rtol=1e-13)
    np.testing.assert_allclose(c, 1.0 / (1.0 + np.exp(-z[n:2 * n])), rtol=1e-13)
    # with no iteration B is exp(z) of the last n*n values, row-major
    np.testing.assert_allclose(B, np.exp(z[2 * n:]).reshape(n, n), rtol=1e-13)


def test_sinkhorn_equal_logits_give_uniform_matrix():
    rng = np.random.default_rng(61)
    n = 4
    x, phi, bias = _mhc_inputs(rng, n, 16, np.full(2 * n + n * n, 0.7))
    _, _, B = oracle.mhc_coeffs(x, phi, bias, iters=1)
    np.testing.assert_allclose(B, np.full((n, n), 1.0 / n), rtol=1e-15)


def test_sinkhorn_columns_exact_rows_converge():
    rng = np.random.default_rng(62)
    n = 4
    x, phi, bias = _mhc_inputs(rng, n, 16)
    _, _, B = oracle.mhc_coeffs(x, phi, bias, iters=20)
    np.testing.assert_allclose(B.sum(0), 1.0, atol=1e-14)          # the last pass normalises columns
    assert np.abs(B.sum(1) - 1.0).max() < 1e-6                     # rows have converged
    assert (B > 0).all()
    # one row pass alone leaves rows summing to one; more passes keep B doubly stochastic
    _, _, B1 = oracle.mhc_coeffs(x, phi, bias, iters=60)
    np.testing.assert_allclose(B1.sum(1), 1.0, atol=1e-13)


def test_sinkhorn_2x2_limit_closed_form():
    """For a positive 2 x 2 matrix [[p, q], [r, s]] the Sinkhorn-Knopp limit is [[t, 1-t], [1-t, t]]
    with t / (1 - t) = sqrt(p s / (q r))."""
    rng = np.random.default_rng(63)
    n = 2
    zB = np.array([0.3, -1.1, 0.8, 0.2])
    x, phi, bias = _mhc_inputs(rng, n, 8, np.concatenate([np.zeros(4), zB]))
    _, _, B = oracle.mhc_coeffs(x, phi, bias, iters=200)
    p, q, r, s = np.exp(zB)
    ratio = math.sqrt(p * s / (q * r))
    t = ratio / (1.0 + ratio)
    np.testing.assert_allclose(B, [[t, 1 - t], [1 - t, t]], atol=1e-12)


def test_sinkhorn_ignores_a_row_scaling_of_its_input():
    """Adding a constant to one row of logits multiplies that row of exp(z) by a constant, which
    the first row normalisation removes: the result is the same for any iteration count."""
    rng = np.random.default_rng(64)
    n = 4
    x, phi, bias = _mhc_inputs(rng, n, 16)
    shifted = bias.copy()
    shifted[2 * n + 2 * n: 2 * n + 3 * n] += 1.5                     # row 2 of B
    for iters in (1, 3, 20):
        _, _, B0 = oracle.mhc_coeffs(x, phi, bias, iters=iters)
        _, _, B1 = oracle.mhc_coeffs(x, phi, shifted, iters=iters)
        np.testing.assert_allclose(B0, B1, rtol=1e-6)
    # a column shift is not removed after one pass (rows first), so the test can tell them apart
    col = bias.copy()
    col[2 * n + 1::n] += 1.5
    _, _, Bc = oracle.mhc_coeffs(x, phi, col, iters=1)
    _, _, B0 = oracle.mhc_coeffs(x, phi, bias, iters=1)
    assert np.abs(Bc - B0).max() > 1e-3


def test_mhc_pre_selects_a_stream_and_post_preserves_the_stream_sum():
    rng = np.random.default_rng(65)
    n, d = 4, 32
    x = rand_bits(rng, (n, d))
    # a: stream 1 fully on, the others off (sigmoid at +-60)
    a = 1.0 / (1.0 + np.exp(-np.array([-60.0, 60.0, -60.0, -60.0])))
    np.testing.assert_allclose(oracle.mhc_pre(x, a), from_bits(x[1]), atol=1e-20)
    # post: with B doubly stochastic (columns summing to one), the sum over streams is the input
    # streams' sum plus (sum of c) * y
    _, c, B = oracle.mhc_coeffs(*_mhc_inputs(rng, n, d), iters=20)
    y = rand_bits(rng, (d,))
    xo = oracle.mhc_post(x, B, c, y)
    np.testing.assert_allclose(xo.sum(0), from_bits(x).sum(0) + c.sum() * from_bits(y), atol=1e-12)
    # and each stream is the textbook mixing
    np.testing.assert_allclose(xo, B @ from_bits(x) + np.outer(c, from_bits(y)), atol=1e-12)


# ------------------------------------------------------- FP8 (e4m3) caches ----
# e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities, S.1111.111 NaN,
# largest finite 448; the conversion rounds to nearest even and saturates.

def test_e4m3_codes_fixed_by_the_format():
    assert oracle.e4m3_decode(0x00) == 0.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9            # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6            # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x30) == 0.5
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    # ties go to the even mantissa; beyond 448 saturates
    assert oracle.e4m3_encode(1.0625) == 0x38               # between 1 (m=0) and 1.125 (m=1)
    assert oracle.e4m3_encode(1.1875) == 0x3A               # between 1.125 (m=1) and 1.25 (m=2)
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00           # half the smallest subnormal
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02       # between 2^-9 (m=1) and 2^-8 (m=2)
    assert oracle.e4m3_encode(460.0) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80


def test_e4m3_every_finite_code_round_trips():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


def test_e4m3_encode_matches_torch_float8_conversion():
    """In range, the oracle's code is the one torch's float8_e4m3fn cast gives (a library
    routine for the same rounding)."""
    g = np.random.default_rng(5)
    x = (g.standard_normal(4000) * np.exp(g.uniform(-9, 6, 4000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_quantize_rows_scale_codes_and_round_trip():
    g = np.random.default_rng(6)
    x = rand_bits(g, (7, 64), std=3.0)
    x[3] = to_bits(np.zeros(64))
    q, sc = oracle.quantize_rows_e4m3(x)
    xf = from_bits(x)
    for r in range(7):
        amax = np.float32(np.abs(xf[r]).max())
        assert sc[r] == np.float32(amax / np.float32(448.0))
        if amax == 0:
            assert (q[r] == 0).all()
            continue
        # the largest magnitude maps to +-448; the codes are torch's cast of x / scale in fp32
        i = int(np.abs(xf[r]).argmax())
        assert q[r, i] & 0x7F == 0x7E
        y = (xf[r].astype(np.float32) / sc[r]).astype(np.float32)
        np.testing.assert_array_equal(q[r], torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    back = oracle.dequantize_rows_e4m3(q, sc)
    # three mantissa bits: normal values come back within 2^-4 relative
    big = np.abs(xf) >= 2.0 ** -6 * sc[:, None].astype(np.float64)
    assert np.all(np.abs(back - xf)[big] <= 2.0 ** -4 * np.abs(xf)[big] + 1e-30)


def test_compress_per_channel_equal_channels_is_the_scalar_compressor():
    g = np.random.default_rng(7)
    m, width, n_tok = 4, 16, 12
    v = rand_bits(g, (n_tok, width))
    z1 = g.standard_normal(n_tok).astype(np.float32)
    b1 = (0.3 * g.standard_normal(2 * m)).astype(np.float32)
    gamma = (1 + 0.1 * g.standard_normal(width)).astype(np.float32)
    ref = oracle.compress(v, z1, 0, b1, gamma, 1e-6, 8, 10000.0, 2 * m, m, 0, n_tok // m)
    got = oracle.compress_pc(v, np.repeat(z1[:, None], width, 1), 0, np.repeat(b1[:, None], width, 1), gamma, 1e-6,
                             8, 10000.0, 2 * m, m, 0, n_tok // m)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_compress_per_channel_weights_act_per_channel():
    """A logit far above the others in one channel picks that token's value in that channel
    only; a channel with equal logits averages the window (closed forms, no norm or RoPE)."""
    m, width, n_tok = 4, 8, 8
    g = np.random.default_rng(8)
    v = rand_bits(g, (n_tok, width))
    z = np.zeros((n_tok, width), dtype=np.float32)
    z[5, 2] = 80.0                          # entry 1 covers tokens 0..7; channel 2 picks token 5
    bias = np.zeros((2 * m, width), dtype=np.float32)
    out = oracle.compress_pc(v, z, 0, bias, None, 1e-6, 0, 10000.0, 2 * m, m, 1, 1)[0]
    vf = from_bits(v)
    assert abs(out[2] - vf[5, 2]) < 1e-12 * max(1.0, abs(vf[5, 2]))
    np.testing.assert_allclose(out[[0, 1, 3, 4, 5, 6, 7]], vf[:, [0, 1, 3, 4, 5, 6, 7]].mean(0), rtol=1e-13, atol=1e-13)


def test_indexer_e4m3_is_the_bf16_indexer_on_the_decoded_values():
    """With power-of-two scales the decoded rows are exact bf16 values: the e4m3 score equals
    the bf16 indexer's on those rows."""
    g = np.random.default_rng(9)
    H, d, n = 4, 32, 50
    q8 = g.integers(0, 256, (H, d)).astype(np.uint8)
    k8 = g.integers(0, 256, (n, d)).astype(np.uint8)
    q8[(q8 & 0x7F) == 0x7F] = 0x11
    k8[(k8 & 0x7F) == 0x7F] = 0x22
    qs = (2.0 ** g.integers(-3, 3, H)).astype(np.float32)
    ks = (2.0 ** g.integers(-3, 3, n)).astype(np.float32)
    w = g.standard_normal(H).astype(np.float32)
    got = oracle.indexer_scores_e4m3(q8, qs, w, k8, ks, n)
    qv = oracle.dequantize_rows_e4m3(q8, qs)
    kv = oracle.dequantize_rows_e4m3(k8, ks)
    ref = oracle.indexer_scores(to_bits(qv), w, to_bits(kv), n)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-9)


def test_attend_e4m3_is_the_attention_over_the_decoded_rows():
    """With power-of-two row scales the decoded e4m3 rows are exact bf16 values: the e4m3
    attention equals the bf16 attention over those rows (CSA selection and HCA dense)."""
    g = np.random.default_rng(11)
    H, c, rows, W, cap = 4, 64, 40, 8, 16
    q = rand_bits(g, (H, c))
    comp8 = g.integers(0, 256, (rows, c)).astype(np.uint8)
    comp8[(comp8 & 0x7F) >= 0x78] = 0x30               # keep magnitudes moderate, no NaN codes
    cs = (2.0 ** g.integers(-4, 2, rows)).astype(np.float32)
    win = rand_bits(g, (cap, c))
    sink = g.standard_normal(H).astype(np.float32)
    gam = np.ones(c, np.float32)
    comp_bf = to_bits(oracle.dequantize_rows_e4m3(comp8, cs))
    idx = np.array([3, -1, 17, 0, 39, 5], dtype=np.int32)
    for kw in (dict(idx=idx), dict(n_dense=rows)):
        o8, l8 = oracle.attend_e4m3(q, gam, 100, comp8, cs, sink, win, cap, W, 16, 10000.0, 1e-6, 0.125, **kw)
        o16, l16 = oracle.attend(q, gam, 100, comp_bf, sink, win, cap, W, 16, 10000.0, 1e-6, 0.125, **kw)
        np.testing.assert_allclose(o8, o16, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l8, l16, rtol=1e-12, atol=1e-12)
