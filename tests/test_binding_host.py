"""The Python binding's argument checks, on CPU tensors: the library indexes every buffer as
a flat array of the size the call implies and cannot see torch's shapes or strides, so the
binding rejects a buffer of the wrong size or layout before passing its pointer.  Buffers of
the right shapes get past every shape check and stop only at the device check (these
tensors are not on a GPU), which no GPU is needed to see."""
import pytest
import torch

from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.api import AttnParams

bf16, f32, i32 = torch.bfloat16, torch.float32, torch.int32


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()


def _reaches_device_check(fn, *args, **kw):
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        fn(*args, **kw)


def _rejected(fn, name, *args, **kw):
    with pytest.raises(ValueError, match=name):
        fn(*args, **kw)


def _attend_args(B=2, n_q=3, H=8, c=128, rows=50, cap=24):
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=16, ratio=4, topk=8)
    a = dict(q=torch.zeros(B, n_q, H, c, dtype=bf16), gamma_q=torch.ones(c), q_pos=torch.zeros(B, n_q, dtype=i32),
             kv_cache=torch.zeros(B, rows, c, dtype=bf16), idx=torch.zeros(B, n_q, 8, dtype=i32),
             win_kv=torch.zeros(B, cap, c, dtype=bf16), sink=torch.zeros(H), out=torch.empty(B, n_q, H, c, dtype=bf16),
             workspace=torch.empty(16, dtype=torch.uint8), lse=torch.empty(B, n_q, H))
    return p, a


def test_attention_buffers_of_the_right_size_pass():
    p, a = _attend_args()
    _reaches_device_check(api.csa_attend, p, **a)
    a.pop("idx")
    _reaches_device_check(api.hca_attend, p, **a)
    a.pop("workspace")
    _reaches_device_check(api.hca_attend_noalloc, p, **a)
    # out as a differently shaped dense view of the same size, lse omitted
    p, a = _attend_args()
    a["out"] = a["out"].view(2 * 3, 8 * 128)
    a["lse"] = None
    _reaches_device_check(api.csa_attend, p, **a)


@pytest.mark.parametrize("name,bad", [
    ("out", torch.empty(2, 3, 8, 127, dtype=bf16)),
    ("out", torch.empty(2, 3, 16, 128, dtype=bf16)[:, :, ::2]),
    ("lse", torch.empty(2, 3, 7)),
    ("q_pos", torch.zeros(2, 2, dtype=i32)),
    ("sink", torch.zeros(7)),
    ("gamma_q", torch.ones(64)),
])
def test_attention_rejects_wrong_sizes(name, bad):
    for fn in (api.csa_attend, api.hca_attend):
        p, a = _attend_args()
        if fn is api.hca_attend:
            a.pop("idx")
        a[name] = bad
        _rejected(fn, name, p, **a)


def test_indexer_and_topk_buffers():
    p = AttnParams(idx_heads=4, idx_dim=32, ratio=4, topk=8)
    B, n_q, rows = 2, 3, 40
    q = torch.zeros(B, n_q, 4, 32, dtype=bf16)
    w = torch.zeros(B, n_q, 4)
    keys = torch.zeros(B, rows, 32, dtype=bf16)
    pos = torch.zeros(B, n_q, dtype=i32)
    out = torch.zeros(B, n_q, 8, dtype=i32)
    ws = torch.empty(16, dtype=torch.uint8)
    scores = torch.zeros(B, n_q, 40)
    _reaches_device_check(api.csa_indexer_topk, p, q, w, keys, pos, out, ws)
    _reaches_device_check(api.csa_indexer_scores, p, q, w, keys, pos, scores)
    _reaches_device_check(api.lca_topk, p, scores, pos, rows, out)
    _rejected(api.csa_indexer_topk, "out_idx", p, q, w, keys, pos, torch.zeros(B, n_q, 7, dtype=i32), ws)
    _rejected(api.csa_indexer_topk, "q_pos", p, q, w, keys, torch.zeros(B, dtype=i32), out, ws)
    _rejected(api.csa_indexer_scores, "q_pos", p, q, w, keys, torch.zeros(B, n_q + 1, dtype=i32), scores)
    _rejected(api.lca_topk, "scores", p, torch.zeros(B, n_q, 80)[:, :, ::2], pos, rows, out)


@pytest.mark.parametrize("csa", [True, False])
def test_compression_and_window_buffers(csa):
    ratio = 4 if csa else 128
    span = 2 * ratio if csa else ratio
    p = AttnParams(head_dim=128, ratio=ratio)
    fn = api.csa_compress_kv if csa else api.hca_compress_kv
    B, n_tok = 2, 2 * span
    args = dict(tok_v=torch.zeros(B, n_tok, 128, dtype=bf16), tok_z=torch.zeros(B, n_tok),
                tok_pos0=torch.zeros(B, dtype=i32), pos_bias=torch.zeros(span), gamma=torch.ones(128), apply_rope=1,
                first_entry=torch.zeros(B, dtype=i32), n_new=1, cache=torch.zeros(B, 10, 128, dtype=bf16))
    _reaches_device_check(fn, p, **args)
    for name, bad in (("pos_bias", torch.zeros(span - 1)), ("gamma", torch.ones(64)),
                      ("tok_pos0", torch.zeros(1, dtype=i32)), ("first_entry", torch.zeros(1, dtype=i32))):
        _rejected(fn, name, p, **dict(args, **{name: bad}))
    win = torch.zeros(B, 8, 128, dtype=bf16)
    _reaches_device_check(api.lca_window_update, p, args["tok_v"], args["tok_pos0"], args["gamma"], win)
    _rejected(api.lca_window_update, "gamma", p, args["tok_v"], args["tok_pos0"], torch.ones(127), win)


def test_projection_buffers():
    B, H, c, G, d_g, d = 2, 8, 64, 4, 32, 48
    o = torch.zeros(B, H, c, dtype=bf16)
    Wg = torch.zeros(G * d_g, (H // G) * c, dtype=bf16)
    Wm = torch.zeros(d, G * d_g, dtype=bf16)
    mid = torch.zeros(B, G * d_g, dtype=bf16)
    y = torch.zeros(B, d, dtype=bf16)
    _reaches_device_check(api.lca_grouped_oproj, o, Wg, Wm, G, mid, y)
    _rejected(api.lca_grouped_oproj, "groups", o, Wg, Wm, 3, mid, y)
    _rejected(api.lca_grouped_oproj, "Wg", o, torch.zeros(G * d_g, (H // G) * c - 8, dtype=bf16), Wm, G, mid, y)
    _rejected(api.lca_grouped_oproj, "Wm", o, Wg, torch.zeros(d, G * d_g + 8, dtype=bf16), G, mid, y)
    _rejected(api.lca_grouped_oproj, "mid", o, Wg, Wm, G, torch.zeros(B, G * d_g - 1, dtype=bf16), y)
    _rejected(api.lca_grouped_oproj, "y", o, Wg, Wm, G, mid, torch.zeros(B, d - 1, dtype=bf16))
    A = torch.zeros(4, 64, dtype=bf16)
    Wt = torch.zeros(24, 64, dtype=bf16)
    _reaches_device_check(api.lca_gemm_bf16, A, Wt, torch.zeros(4, 24, dtype=bf16))
    _rejected(api.lca_gemm_bf16, "B must", A, torch.zeros(24, 32, dtype=bf16), torch.zeros(4, 24, dtype=bf16))
    _rejected(api.lca_gemm_bf16, "C must", A, Wt, torch.zeros(4, 23, dtype=bf16))
    _rejected(api.lca_gemm_bf16, "A must", torch.zeros(64, 4, dtype=bf16).t(), Wt, torch.zeros(4, 24, dtype=bf16))
