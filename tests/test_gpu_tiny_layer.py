"""The tiny CSA layer end to end: a full prefill of 2048 tokens from hidden states.

Hidden states x [2048, 256] and projection weights (N(0, 0.02)) give the per-token inputs of
the layer (queries, KV vectors, compressor logits, indexer queries, keys, logits and head
weights).  The pages describe no projections, so they are plain linear maps; the oracle
computes them (fp64, then bf16 / fp32 storage) and the GPU path is fed those same inputs,
so every later comparison isolates the attention path.  `lca_gemm_bf16` is checked on the
same projections separately.

Compared against the oracle: the 512 compressed entries and keys and the 2048 window rows
(bf16 rounding), the top-k list of every query (near-ties only), and every query's
attention output (2e-2 x RMS), both with the oracle's caches and indices injected and end to
end through the GPU's own caches and selection.  A second run with k = 512 (every entry) and
W = 2048 (every token) makes the layer plain causal attention over entries and tokens with
a sink, and is compared on a sample of queries.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close_rms, assert_rows_close, check_topk, round_bf16_bits
from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.layers import CsaLayer, LayerWeights
from workloads import TINY_CSA_PREFILL, Rng, bf16_bits, bits_to_bf16, tiny_prefill_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield


@pytest.fixture(scope="module")
def tiny():
    """Inputs and the oracle's projections of the tiny layer (seed 0)."""
    inp = tiny_prefill_inputs(Rng(0))
    x = bf16_bits(inp["x"])
    proj = {k: oracle.gemm_bf16(x, bf16_bits(inp[w])) for k, w in
            (("q", "W_q"), ("v", "W_kv"), ("z", "W_z"), ("qi", "W_qi"), ("vi", "W_ki"), ("zi", "W_zi"),
             ("w", "W_w"))}
    return inp, proj


def _layer_inputs(s, n, proj):
    """The projections as the layer's tensors: bf16 vectors rounded from the oracle's fp64."""
    bf = lambda a, shape: bits_to_bf16(round_bf16_bits(a)).view(shape)
    return dict(
        q=bf(proj["q"], (1, n, s.heads, s.head_dim)),
        v=bf(proj["v"], (1, n, s.head_dim)),
        z=torch.from_numpy(proj["z"][:, 0].astype(np.float32)).view(1, n),
        qi=bf(proj["qi"], (1, n, s.idx_heads, s.idx_dim)),
        vi=bf(proj["vi"], (1, n, s.idx_dim)),
        zi=torch.from_numpy(proj["zi"][:, 0].astype(np.float32)).view(1, n),
        w=torch.from_numpy(proj["w"].astype(np.float32)).view(1, n, s.idx_heads),
    )


def _oracle_layer(p, s, n, t, inp, k, W, cap, queries):
    """The oracle's layer: caches, window ring, per-query scores, top-k and outputs."""
    g = inp["gamma_kv"].numpy()
    m = s.ratio
    kv = oracle.compress(bf16_bits(t["v"][0]), t["z"][0].numpy(), 0, inp["bias_kv"].numpy(), g, s.rms_eps,
                         s.rope_dims, s.rope_base, 2 * m, m, 0, n // m)
    keys = oracle.compress(bf16_bits(t["vi"][0]), t["zi"][0].numpy(), 0, inp["bias_idx"].numpy(), None, s.rms_eps,
                           0, s.rope_base, 2 * m, m, 0, n // m)
    vb = bf16_bits(t["v"][0])
    win = np.stack([oracle.window_row(vb[i], g, s.rms_eps, s.rope_dims, s.rope_base, i) for i in range(n)])
    kvb, keyb = round_bf16_bits(kv), round_bf16_bits(keys)
    ring = np.zeros((cap, s.head_dim), np.uint16)
    for i in range(n):
        ring[i % cap] = round_bf16_bits(win[i])
    res = {}
    for i in queries:
        n_vis = oracle.visible_entries(i, m)
        sc = oracle.indexer_scores(bf16_bits(t["qi"][0, i]), t["w"][0, i].numpy(), keyb, n_vis)
        idx = oracle.topk(sc, k)
        out, lse = oracle.attend(bf16_bits(t["q"][0, i]), inp["gamma_q"].numpy(), i, kvb, inp["sink"].numpy(), ring,
                                 cap, W, s.rope_dims, s.rope_base, s.rms_eps, p.scale, idx=idx)
        res[i] = (sc, idx, out, lse)
    return kv, keys, win, kvb, keyb, ring, res


def _run_layer(p, s, n, t, inp, cap):
    w = LayerWeights(inp["gamma_kv"].to(DEV), inp["gamma_q"].to(DEV), inp["bias_kv"].to(DEV), inp["sink"].to(DEV),
                     inp["bias_idx"].to(DEV))
    kv = torch.zeros((1, n // s.ratio, s.head_dim), dtype=torch.bfloat16, device=DEV)
    keys = torch.zeros((1, n // s.ratio, s.idx_dim), dtype=torch.bfloat16, device=DEV)
    ring = torch.zeros((1, cap, s.head_dim), dtype=torch.bfloat16, device=DEV)
    L = CsaLayer(p, w, kv, keys, ring, n_q=n)
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_pos = torch.arange(n, dtype=torch.int32, device=DEV).view(1, n)
    out = torch.empty((1, n, s.heads, s.head_dim), dtype=torch.bfloat16, device=DEV)
    td = {k: v.to(DEV) for k, v in t.items()}
    L.step(td["v"], td["z"], td["vi"], td["zi"], zero, zero, n // s.ratio, td["v"], zero, td["q"], td["qi"], td["w"],
           q_pos, out)
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    return L, out, q_pos, w


def test_projections_through_lca_gemm(tiny):
    inp, proj = tiny
    x = inp["x"].to(DEV)
    for name, wname in (("q", "W_q"), ("v", "W_kv"), ("qi", "W_qi"), ("w", "W_w")):
        Wt = inp[wname].to(DEV)
        for r0 in (0, 1000, 2032):
            C = torch.empty((16, Wt.shape[0]), dtype=torch.bfloat16, device=DEV)
            api.lca_gemm_bf16(x[r0:r0 + 16], Wt, C)
            got = C.cpu().float().numpy().astype(np.float64)
            ref = proj[name][r0:r0 + 16]
            # fp32 accumulation rounded to bf16 vs fp64 rounded to bf16: equal up to one bf16 step
            bound = 2.0 ** -7 * np.abs(ref) + 1e-6
            assert (np.abs(got - ref) <= bound).all(), name


def test_tiny_layer_end_to_end(tiny):
    inp, proj = tiny
    cfg = TINY_CSA_PREFILL
    s, n = cfg["shape"], cfg["n_tok"]
    p = api.params_from(s)
    cap = n                                    # the ring keeps every token of the prefill
    t = _layer_inputs(s, n, proj)
    L, out, q_pos, w = _run_layer(p, s, n, t, inp, cap)
    queries = list(range(n))
    kv, keys, win, kvb, keyb, ring, ref = _oracle_layer(p, s, n, t, inp, s.topk, s.window, cap, queries)
    # written rows
    for j in range(n // s.ratio):
        assert_rows_close(L.kv_cache[0, j], kv[j], "kv entry %d" % j)
        assert_rows_close(L.idx_cache[0, j], keys[j], "key %d" % j)
    for i in range(n):
        assert_rows_close(L.win_kv[0, i], win[i], "window row %d" % i)
    # selection and outputs end to end (GPU caches and GPU selection)
    gpu_idx = L.idx[0].cpu().numpy()
    o = out[0].cpu().float().numpy()
    swapped = 0
    for i in queries:
        sc, idx, ro, _ = ref[i]
        if check_topk(gpu_idx[i], sc, s.topk, what="topk query %d" % i):
            swapped += 1
            continue
        assert_close_rms(o[i], ro, what="end-to-end query %d" % i)
    assert swapped <= n // 100
    # the oracle's caches and indices injected: selection and attention alone
    keys_d = bits_to_bf16(keyb).view(1, -1, s.idx_dim).to(DEV)
    idx_d = torch.empty_like(L.idx)
    ws = torch.empty(api.csa_indexer_workspace(p, 1, n, keyb.shape[0]), dtype=torch.uint8, device=DEV)
    api.csa_indexer_topk(p, t["qi"].to(DEV), t["w"].to(DEV), keys_d, q_pos, idx_d, ws)
    got_idx = idx_d[0].cpu().numpy()
    for i in queries:
        check_topk(got_idx[i], ref[i][0], s.topk, what="injected-keys topk query %d" % i)
    kv_d = bits_to_bf16(kvb).view(1, -1, s.head_dim).to(DEV)
    ring_d = bits_to_bf16(ring).view(1, cap, s.head_dim).to(DEV)
    idx_ref = torch.from_numpy(np.stack([ref[i][1] for i in queries])).view(1, n, s.topk).to(DEV)
    out2 = torch.empty_like(out)
    lse2 = torch.empty((1, n, s.heads), dtype=torch.float32, device=DEV)
    ws2 = torch.empty(api.csa_attend_workspace(p, 1, n), dtype=torch.uint8, device=DEV)
    api.csa_attend(p, t["q"].to(DEV), w.gamma_q, q_pos, kv_d, idx_ref, ring_d, w.sink, out2, ws2, lse2)
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    o2 = out2[0].cpu().float().numpy()
    l2 = lse2[0].cpu().numpy()
    for i in queries:
        assert_close_rms(o2[i], ref[i][2], what="injected query %d" % i)
        np.testing.assert_allclose(l2[i], ref[i][3], rtol=0, atol=2e-3 * max(1.0, np.abs(ref[i][3]).max()))


def test_tiny_layer_every_entry_and_token_is_causal_attention(tiny):
    inp, proj = tiny
    cfg = TINY_CSA_PREFILL
    base, n = cfg["shape"], cfg["n_tok"]
    k, W = n // base.ratio, n                 # k >= n/m and the window covers every token
    p = api.params_from(base, window=W, topk=k)
    cap = n
    t = _layer_inputs(base, n, proj)
    L, out, _, _ = _run_layer(p, base, n, t, inp, cap)
    queries = sorted(set(list(range(0, n, 97)) + [1, 2, 3, 4, 5, 7, 8, n - 1]))
    _, _, _, _, _, _, ref = _oracle_layer(p, base, n, t, inp, k, W, cap, queries)
    gpu_idx = L.idx[0].cpu().numpy()
    o = out[0].cpu().float().numpy()
    for i in queries:
        sc, idx, ro, _ = ref[i]
        n_vis = oracle.visible_entries(i, base.ratio)
        assert (gpu_idx[i][:n_vis] == np.arange(n_vis)).all() and (gpu_idx[i][n_vis:] == -1).all()
        assert_close_rms(o[i], ro, what="k=all W=all query %d" % i)
