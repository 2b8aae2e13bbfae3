"""Parity at the benchmark's full sizes, in the launch configuration bench.py times.

Each test builds a bench workload (same batch, caches, split plan and kernels), runs one
step of the whole path on the GPU, and compares sampled outputs with the oracle computed
one by one on the host from the same seeded inputs:
  * the rows the step writes (the new compressed entries and window rows) within bf16 rounding;
  * the top-k lists (sets equal except at near-ties of the k-th score);
  * the attention outputs within 2e-2 x RMS wherever the top-k set equals the oracle's
    (a near-tie swap changes which rows are attended, so that output is not comparable).
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import assert_close_bf16_out, assert_close_rms, assert_rows_close, check_topk, round_bf16_bits
from long_context_attention_04_b300 import api, build as lca_build
from workloads import WORKLOADS, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield


def _host(t):
    return t.detach().cpu()


def _csa_before(wk, samples):
    d = wk.d
    return {b: (bf16_bits(_host(d["kv_cache"][b])), bf16_bits(_host(d["idx_cache"][b])),
                bf16_bits(_host(d["win_kv"][b]))) for b in samples}


def _csa_check(wk, before, what):
    """Rows written, top-k and outputs of a CSA decode step for the sampled sequences; returns the
    oracle outputs {b: out} of the sequences whose top-k equals the oracle's."""
    s, d, pos, E = wk.s, wk.d, wk.pos, wk.entries
    cap = d["win_kv"].shape[1]
    g = d["gamma_kv"].cpu().numpy()
    outs = {}
    for b, (kvb, ixb, winb) in before.items():
        tv, tz = bf16_bits(_host(d["tok_v"][b])), _host(d["tok_z"][b]).numpy()
        tvi, tzi = bf16_bits(_host(d["tok_vi"][b])), _host(d["tok_zi"][b]).numpy()
        kv_new = oracle.compress(tv, tz, d["tok_pos0"], d["bias_kv"].cpu().numpy(), g, s.rms_eps, s.rope_dims,
                                 s.rope_base, 2 * s.ratio, s.ratio, E - 1, 1)[0]
        k_new = oracle.compress(tvi, tzi, d["tok_pos0"], d["bias_idx"].cpu().numpy(), None, s.rms_eps, 0,
                                s.rope_base, 2 * s.ratio, s.ratio, E - 1, 1)[0]
        w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, pos)
        assert_rows_close(wk.layer.kv_cache[b, E - 1], kv_new, "%s kv entry b=%d" % (what, b))
        assert_rows_close(wk.layer.idx_cache[b, E - 1], k_new, "%s key entry b=%d" % (what, b))
        assert_rows_close(wk.layer.win_kv[b, pos % cap], w_new, "%s window row b=%d" % (what, b))
        kvb[E - 1] = round_bf16_bits(kv_new)
        ixb[E - 1] = round_bf16_bits(k_new)
        winb[pos % cap] = round_bf16_bits(w_new)
        n_vis = oracle.visible_entries(pos, s.ratio)
        sc = oracle.indexer_scores(bf16_bits(_host(d["q_idx"][b, 0])), _host(d["w_idx"][b, 0]).numpy(), ixb, n_vis)
        ref_idx = oracle.topk(sc, s.topk)
        gpu_idx = _host(wk.layer.idx[b, 0]).numpy()
        if check_topk(gpu_idx, sc, s.topk, what="%s topk b=%d" % (what, b)) == 0:
            ro, _ = oracle.attend(bf16_bits(_host(d["q"][b, 0])), d["gamma_q"].cpu().numpy(), pos, kvb,
                                  d["sink"].cpu().numpy(), winb, cap, s.window, s.rope_dims, s.rope_base, s.rms_eps,
                                  wk.p.scale, idx=ref_idx)
            assert_close_rms(_host(wk.out[b, 0]).float().numpy(), ro, what="%s out b=%d" % (what, b))
            outs[b] = ro
    assert len(outs) >= len(before) - 1
    return outs


def test_csa_decode_128k_sampled_sequences():
    wk = bench.CsaDecode(WORKLOADS["csa_decode_128k"], seed=0)
    before = _csa_before(wk, [0, 17, wk.B - 1])
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    _csa_check(wk, before, "csa")


def _hca_before(wk, samples):
    d = wk.d
    return {b: (bf16_bits(_host(d["kv_cache"][b])), bf16_bits(_host(d["win_kv"][b]))) for b in samples}


def _hca_check(wk, before, what):
    s, d, pos, E = wk.s, wk.d, wk.pos, wk.entries
    cap = d["win_kv"].shape[1]
    g = d["gamma_kv"].cpu().numpy()
    outs = {}
    for b, (kvb, winb) in before.items():
        tv, tz = bf16_bits(_host(d["tok_v"][b])), _host(d["tok_z"][b]).numpy()
        kv_new = oracle.compress(tv, tz, d["tok_pos0"], d["bias_kv"].cpu().numpy(), g, s.rms_eps, s.rope_dims,
                                 s.rope_base, s.ratio, s.ratio, E - 1, 1)[0]
        w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, pos)
        assert_rows_close(wk.layer.kv_cache[b, E - 1], kv_new, "%s kv entry b=%d" % (what, b))
        assert_rows_close(wk.layer.win_kv[b, pos % cap], w_new, "%s window row b=%d" % (what, b))
        kvb[E - 1] = round_bf16_bits(kv_new)
        winb[pos % cap] = round_bf16_bits(w_new)
        ro, _ = oracle.attend(bf16_bits(_host(d["q"][b, 0])), d["gamma_q"].cpu().numpy(), pos, kvb,
                              d["sink"].cpu().numpy(), winb, cap, s.window, s.rope_dims, s.rope_base, s.rms_eps,
                              wk.p.scale, n_dense=oracle.visible_entries(pos, s.ratio))
        assert_close_rms(_host(wk.out[b, 0]).float().numpy(), ro, what="%s out b=%d" % (what, b))
        outs[b] = ro
    return outs


def test_hca_decode_1m_sampled_sequences():
    wk = bench.HcaDecode(WORKLOADS["hca_decode_1m"], seed=0)
    before = _hca_before(wk, [0, 9, wk.B - 1])
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    _hca_check(wk, before, "hca")


def test_block_decode_1m_sampled():
    """The 16-layer block (8 CSA at 262144 entries, 8 HCA at 8192, batch 4) in one step: a CSA and
    an HCA layer checked on a sampled sequence, with their grouped output projections applied by
    the oracle to the oracle's attention output (rounded to bf16, as the kernel's input is)."""
    wk = bench.BlockDecode(WORKLOADS["block_decode_1m"], seed=0)
    csa, hca = wk.layers[0], wk.layers[1]
    b = 2
    bc, bh = _csa_before(csa, [b]), _hca_before(hca, [b])
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    outs = [_csa_check(csa, bc, "block csa"), _hca_check(hca, bh, "block hca")]
    for i, o in enumerate(outs):
        if b not in o:
            continue                                  # a near-tie swap changed that layer's rows
        ref = oracle.grouped_oproj(round_bf16_bits(o[b]), bf16_bits(_host(wk.W[i]["Wg"])),
                                   bf16_bits(_host(wk.W[i]["Wm"])), wk.G)
        assert_close_rms(_host(wk.y[i][b]).float().numpy(), ref, what="block layer %d projection" % i)


def test_csa_prefill_1m_sampled_queries():
    wk = bench.CsaPrefill(WORKLOADS["csa_prefill_1m"], seed=0)
    s, d = wk.s, wk.d
    Tq, E, q0, m = wk.Tq, wk.entries, wk.q_begin, s.ratio
    kvb = bf16_bits(_host(d["kv_cache"][0]))
    ixb = bf16_bits(_host(d["idx_cache"][0]))
    winb = bf16_bits(_host(d["win_kv"][0]))
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    cap = winb.shape[0]
    g = d["gamma_kv"].cpu().numpy()
    tv, tz = bf16_bits(_host(d["tok_v"][0])), _host(d["tok_z"][0]).numpy()
    tvi, tzi = bf16_bits(_host(d["tok_vi"][0])), _host(d["tok_zi"][0]).numpy()
    first, n_new = d["first_entry"], Tq // m
    kv_new = oracle.compress(tv, tz, d["tok_pos0"], d["bias_kv"].cpu().numpy(), g, s.rms_eps, s.rope_dims,
                             s.rope_base, 2 * m, m, first, n_new)
    k_new = oracle.compress(tvi, tzi, d["tok_pos0"], d["bias_idx"].cpu().numpy(), None, s.rms_eps, 0, s.rope_base,
                            2 * m, m, first, n_new)
    for j in (0, 1, n_new // 2, n_new - 1):
        assert_rows_close(wk.layer.kv_cache[0, first + j], kv_new[j], "kv entry %d" % (first + j))
        assert_rows_close(wk.layer.idx_cache[0, first + j], k_new[j], "key entry %d" % (first + j))
    kvb[first:first + n_new] = round_bf16_bits(kv_new)
    ixb[first:first + n_new] = round_bf16_bits(k_new)
    # window rows of the chunk's tokens (the staging rows start m tokens before the chunk)
    for i in range(Tq):
        t = q0 + i
        row = oracle.window_row(tv[m + i], g, s.rms_eps, s.rope_dims, s.rope_base, t)
        if i in (0, Tq // 2, Tq - 1):
            assert_rows_close(wk.layer.win_kv[0, t % cap], row, "window row %d" % t)
        winb[t % cap] = round_bf16_bits(row)
    compared = 0
    samples = [0, Tq // 2 + 3, Tq - 1]
    for i in samples:
        t = q0 + i
        n_vis = oracle.visible_entries(t, m)
        sc = oracle.indexer_scores(bf16_bits(_host(d["q_idx"][0, i])), _host(d["w_idx"][0, i]).numpy(), ixb, n_vis)
        ref_idx = oracle.topk(sc, s.topk)
        gpu_idx = _host(wk.layer.idx[0, i]).numpy()
        if check_topk(gpu_idx, sc, s.topk, what="topk query %d" % t) == 0:
            ro, _ = oracle.attend(bf16_bits(_host(d["q"][0, i])), d["gamma_q"].cpu().numpy(), t, kvb,
                                  d["sink"].cpu().numpy(), winb, cap, s.window, s.rope_dims, s.rope_base, s.rms_eps,
                                  wk.p.scale, idx=ref_idx)
            assert_close_rms(_host(wk.out[0, i]).float().numpy(), ro, what="prefill out query %d" % t)
            compared += 1
    assert compared >= len(samples) - 1


def test_prefill_input_projections_sampled_rows():
    """The 1M prefill chunk's input projections (tensor-core products of the 8192 + m staging
    tokens' hidden states, width 4096) at the benchmark's shapes: sampled rows of every projected
    tensor against the oracle's product of the same rows."""
    wk = bench.CsaPrefillProj(WORKLOADS["csa_prefill_1m_proj"], seed=0)
    wk.project()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    x = bf16_bits(_host(wk.x))
    m = wk.s.ratio
    for A, Wm, C in wk.proj:
        row0 = 0 if A.data_ptr() == wk.x.data_ptr() else m
        got = _host(C).float().numpy()
        Wb = bf16_bits(_host(Wm))
        for r in (0, 1, 4097, C.shape[0] - 1):
            ref = oracle.gemm_bf16(x[row0 + r:row0 + r + 1], Wb)[0]
            if C.dtype == torch.float32:
                np.testing.assert_allclose(got[r], ref, rtol=1e-5, atol=1e-4 * max(1e-30, float(np.abs(ref).max())))
            else:
                assert_close_bf16_out(got[r], ref, what="projection row %d" % r)


# ------------------------------------------------------------- FP8 (e4m3) caches ----
# The oracle quantises the same seeded bf16 caches with its own quantiser (bit-exact with the
# library's, tests/test_gpu_fp8.py), so every oracle input comes from the generator.

def _e4m3_row_close(codes, scale, ref, what):
    """A stored e4m3 row against the oracle's fp64 row: 2^-4 relative (three mantissa bits), half
    the smallest step of the row's scale, and the bf16 rounding before the quantisation."""
    back = oracle.dequantize_rows_e4m3(np.asarray(codes)[None], np.asarray([scale], np.float32))[0]
    ref = np.asarray(ref, np.float64)
    bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -9 * float(scale) + 2e-3 * np.sqrt(np.mean(ref * ref))
    assert (np.abs(back - ref) <= bound).all(), what


def test_csa_decode_128k_fp8_sampled_sequence():
    """The CSA decode step with e4m3 keys and KV rows: the new entries (e4m3), the top-k of the e4m3
    indexer and the attention over e4m3 rows, against the oracle on its own quantised caches."""
    wk = bench.CsaDecode(WORKLOADS["csa_decode_128k_fp8"], seed=0)
    s, d, pos, E = wk.s, wk.d, wk.pos, wk.entries
    b = 5
    kvb, ixb, winb = (bf16_bits(_host(d[k][b])) for k in ("kv_cache", "idx_cache", "win_kv"))
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    cap = d["win_kv"].shape[1]
    g = d["gamma_kv"].cpu().numpy()
    tv, tz = bf16_bits(_host(d["tok_v"][b])), _host(d["tok_z"][b]).numpy()
    tvi, tzi = bf16_bits(_host(d["tok_vi"][b])), _host(d["tok_zi"][b]).numpy()
    kv_new = oracle.compress(tv, tz, d["tok_pos0"], d["bias_kv"].cpu().numpy(), g, s.rms_eps, s.rope_dims,
                             s.rope_base, 2 * s.ratio, s.ratio, E - 1, 1)[0]
    k_new = oracle.compress(tvi, tzi, d["tok_pos0"], d["bias_idx"].cpu().numpy(), None, s.rms_eps, 0, s.rope_base,
                            2 * s.ratio, s.ratio, E - 1, 1)[0]
    w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, pos)
    L = wk.layer
    _e4m3_row_close(_host(L.kv_cache[b, E - 1]).numpy(), float(L.kv_scale[b, E - 1]), kv_new, "kv entry")
    _e4m3_row_close(_host(L.idx_cache[b, E - 1]).numpy(), float(L.idx_scale[b, E - 1]), k_new, "key entry")
    assert_rows_close(L.win_kv[b, pos % cap], w_new, "window row")
    kvb[E - 1] = round_bf16_bits(kv_new)
    ixb[E - 1] = round_bf16_bits(k_new)
    winb[pos % cap] = round_bf16_bits(w_new)
    kv8, kvs = oracle.quantize_rows_e4m3(kvb)
    ix8, ixs = oracle.quantize_rows_e4m3(ixb)
    q8, qs = oracle.quantize_rows_e4m3(bf16_bits(_host(d["q_idx"][b, 0])))
    n_vis = oracle.visible_entries(pos, s.ratio)
    sc = oracle.indexer_scores_e4m3(q8, qs, _host(d["w_idx"][b, 0]).numpy(), ix8, ixs, n_vis)
    gpu_idx = _host(L.idx[b, 0]).numpy()
    if check_topk(gpu_idx, sc, s.topk, what="fp8 topk") == 0:
        ro, _ = oracle.attend_e4m3(bf16_bits(_host(d["q"][b, 0])), d["gamma_q"].cpu().numpy(), pos, kv8, kvs,
                                   d["sink"].cpu().numpy(), winb, cap, s.window, s.rope_dims, s.rope_base, s.rms_eps,
                                   wk.p.scale, idx=oracle.topk(sc, s.topk))
        assert_close_rms(_host(wk.out[b, 0]).float().numpy(), ro, what="fp8 csa out")


def test_hca_decode_1m_fp8_sampled_sequence():
    """The HCA decode step over an e4m3 KV cache: the new entry and the attention against the oracle
    on its own quantised cache."""
    wk = bench.HcaDecode(WORKLOADS["hca_decode_1m_fp8"], seed=0)
    s, d, pos, E = wk.s, wk.d, wk.pos, wk.entries
    b = 11
    kvb, winb = bf16_bits(_host(d["kv_cache"][b])), bf16_bits(_host(d["win_kv"][b]))
    wk.step()
    torch.cuda.synchronize()
    assert api.lca_device_error() == 0
    cap = d["win_kv"].shape[1]
    g = d["gamma_kv"].cpu().numpy()
    tv, tz = bf16_bits(_host(d["tok_v"][b])), _host(d["tok_z"][b]).numpy()
    kv_new = oracle.compress(tv, tz, d["tok_pos0"], d["bias_kv"].cpu().numpy(), g, s.rms_eps, s.rope_dims,
                             s.rope_base, s.ratio, s.ratio, E - 1, 1)[0]
    w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, pos)
    L = wk.layer
    _e4m3_row_close(_host(L.kv_cache[b, E - 1]).numpy(), float(L.kv_scale[b, E - 1]), kv_new, "kv entry")
    assert_rows_close(L.win_kv[b, pos % cap], w_new, "window row")
    kvb[E - 1] = round_bf16_bits(kv_new)
    winb[pos % cap] = round_bf16_bits(w_new)
    kv8, kvs = oracle.quantize_rows_e4m3(kvb)
    ro, _ = oracle.attend_e4m3(bf16_bits(_host(d["q"][b, 0])), d["gamma_q"].cpu().numpy(), pos, kv8, kvs,
                               d["sink"].cpu().numpy(), winb, cap, s.window, s.rope_dims, s.rope_base, s.rms_eps,
                               wk.p.scale, n_dense=oracle.visible_entries(pos, s.ratio))
    assert_close_rms(_host(wk.out[b, 0]).float().numpy(), ro, what="fp8 hca out")
