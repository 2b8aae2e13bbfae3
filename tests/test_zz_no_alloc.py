"""hca_attend_noalloc (scratch in the library's static device array) against hca_attend
(caller workspace), through the C ABI, on two consecutive calls.

Named so that it is collected last: it must pass both alone in a fresh process (where its
first call does the per-device set-up) and after every other test has run.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_rms
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
    return {k: v.to(DEV) for k, v in d.items()}, pos.to(DEV)


def test_noalloc_matches_workspace_entry_twice():
    H, c, R, W, m = 64, 512, 64, 128, 128
    B, n_q, rows = 4, 2, 1500
    p = AttnParams(heads=H, head_dim=c, rope_dims=R, window=W, ratio=m)
    d, pos = _case(41, B, n_q, H, c, rows, W, m)
    out_ws = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse_ws = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    api.hca_attend(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"], out_ws, ws, lse_ws)
    ref_o = out_ws.float().cpu().numpy()
    ref_l = lse_ws.cpu().numpy()
    # two consecutive calls into the shared array, each compared with the workspace entry
    for call in range(2):
        out = torch.full((B, n_q, H, c), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, n_q, H), float("nan"), dtype=torch.float32, device=DEV)
        api.hca_attend_noalloc(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"], out, lse)
        assert api.lca_device_error() == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        for b in range(B):
            for i in range(n_q):
                assert_close_rms(o[b, i], ref_o[b, i], what="noalloc call %d b=%d i=%d" % (call, b, i))
        np.testing.assert_allclose(l, ref_l, rtol=0, atol=2e-3 * max(1.0, float(np.abs(ref_l).max())))


def test_noalloc_rejects_calls_beyond_the_array():
    H, c, W, m = 64, 512, 128, 128
    B, rows = 160, 16                   # 160 queries need more than 32 MiB of partials + query images
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m)
    assert api.hca_attend_workspace(p, B, 1, rows) > 32 << 20
    d, pos = _case(42, B, 1, H, c, rows, W, m)
    out = torch.empty((B, 1, H, c), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(LcaError) as e:
        api.hca_attend_noalloc(p, d["q"], d["gamma"], pos, d["kv"], d["win"], d["sink"], out)
    assert e.value.status == 3 and "static array" in str(e.value)
    assert api.lca_device_error() == 0
