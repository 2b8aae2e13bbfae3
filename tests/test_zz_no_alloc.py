"""hca_attend_noalloc, the entry point for callers that cannot allocate device memory (its
scratch is the library's static device array), against hca_attend with a caller workspace,
through the C ABI, on two consecutive calls.

The two calls differ in inputs and in batch x queries, so the split count and the layout of
the partials in the shared array change between them: the second call cannot pass by reading
what the first one left there.  Each call must equal hca_attend on the same inputs bit for bit
(same kernels, same split plan), and one is also compared with the oracle.

Named so that it is collected last: it must pass both alone in a fresh process (where its
first call looks the array up on the device) and after every other test has run.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_rms, oracle_attend_batch
from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.api import AttnParams, LcaError
from workloads import Rng

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield


def _case(seed, B, n_q, H, c, rows, W, m):
    rng = Rng(seed)
    cap = W + 8
    d = dict(q=rng.normal_bf16((B, n_q, H, c)), kv=rng.normal_bf16((B, rows, c)), win=rng.normal_bf16((B, cap, c)),
             gamma=(0.5 + torch.rand(c, generator=rng.g)).float(), sink=rng.normal_f32((H,)))
    g = np.random.default_rng(seed)
    pos = torch.from_numpy(g.integers(0, m * rows, size=(B, n_q), dtype=np.int32))
    pos[0, 0] = m * rows - 1            # every entry visible
    return d, pos


def _run(fn, p, d, pos, ws=None):
    B, n_q = pos.shape
    out = torch.full((B, n_q, p.heads, p.head_dim), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, n_q, p.heads), float("nan"), dtype=torch.float32, device=DEV)
    args = [d[k].to(DEV) for k in ("q", "gamma")] + [pos.to(DEV)] + [d[k].to(DEV) for k in ("kv", "win", "sink")]
    if ws is None:
        fn(p, *args, out, lse)
    else:
        fn(p, *args, out, ws, lse)
    assert api.lca_device_error() == 0
    return out.cpu(), lse.cpu()


def test_noalloc_matches_workspace_entry_twice():
    H, c, R, W, m, rows = 64, 512, 64, 128, 128, 1500
    p = AttnParams(heads=H, head_dim=c, rope_dims=R, window=W, ratio=m)
    # call 1: 8 queries, 13 splits each (one per tile); call 2: other inputs, 15 queries, 9 splits each
    for call, (seed, B, n_q) in enumerate(((41, 4, 2), (43, 5, 3))):
        d, pos = _case(seed, B, n_q, H, c, rows, W, m)
        ws = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
        ref_o, ref_l = _run(api.hca_attend, p, d, pos, ws)
        o, l = _run(api.hca_attend_noalloc, p, d, pos)
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)), "call %d: outputs differ" % call
        assert torch.equal(l, ref_l), "call %d: lse differs" % call
        if call == 1:
            ref = oracle_attend_batch(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"])
            for (b, i), (ro, rl) in ref.items():
                assert_close_rms(o[b, i].float().numpy(), ro, what="noalloc vs oracle b=%d i=%d" % (b, i))
                np.testing.assert_allclose(l[b, i].numpy(), rl, rtol=0, atol=2e-3 * max(1.0, np.abs(rl).max()))


def test_noalloc_rejects_calls_beyond_the_array():
    H, c, W, m = 64, 512, 128, 128
    B, rows = 160, 16                   # 160 queries need more than 32 MiB of partials + query images
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m)
    assert api.hca_attend_workspace(p, B, 1, rows) > 32 << 20
    d, pos = _case(42, B, 1, H, c, rows, W, m)
    out = torch.empty((B, 1, H, c), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(LcaError) as e:
        api.hca_attend_noalloc(p, *[d[k].to(DEV) for k in ("q", "gamma")], pos.to(DEV),
                               *[d[k].to(DEV) for k in ("kv", "win", "sink")], out)
    assert e.value.status == 3 and "static array" in str(e.value)
    assert api.lca_device_error() == 0
