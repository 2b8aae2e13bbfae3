"""Failure path of the kernels' bounded waits, in the form that leaves the GPU usable: a wait
that nothing will ever complete runs out, the kernel stops and frees what it holds, the host
reads LCA_ERR_TIMEOUT, and the next call on the same context is correct.

The wait has nothing to wait for because the attention kernel's producer is told (through
lca_test_hooks) to leave one tile unloaded; no copy is in flight for it, and the wait bound is
shortened to 1e6 cycles (~0.5 ms) so the test is quick.  The hooks are reset afterwards.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_rms, oracle_attend_batch
from long_context_attention_04_b300 import api, build as lca_build
from long_context_attention_04_b300.api import AttnParams
from workloads import Rng

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield
    api.lca_test_hooks(0, -1)


def test_attention_wait_runs_out_then_next_call_is_correct():
    rng = Rng(31)
    H, c, W, m, rows = 64, 512, 128, 4, 700
    B, n_q = 40, 2                     # 80 queries: one split each, so every CTA walks 7 tiles
    p = AttnParams(heads=H, head_dim=c, rope_dims=64, window=W, ratio=m)
    q = rng.normal_bf16((B, n_q, H, c))
    kv = rng.normal_bf16((B, rows, c))
    win = rng.normal_bf16((B, W, c))
    gamma = torch.ones(c)
    sink = rng.normal_f32((H,))
    pos = torch.full((B, n_q), m * rows - 1, dtype=torch.int32)
    args = [t.to(DEV) for t in (q, gamma, pos, kv, win, sink)]
    out = torch.empty((B, n_q, H, c), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, n_q, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.hca_attend_workspace(p, B, n_q, rows), dtype=torch.uint8, device=DEV)
    try:
        api.lca_test_hooks(1_000_000, 1)       # tile 1 of every CTA is never loaded
        api.hca_attend(p, *args, out, ws, lse)
        torch.cuda.synchronize()
        word = api.lca_device_error()
    finally:
        api.lca_test_hooks(0, -1)
    assert word & 0x100, "the wait on the unloaded tile did not report a timeout (word 0x%x)" % word
    assert word & ~0x100 == 0, hex(word)
    # the context is intact and the kernel's tensor memory was released: the same call now
    # runs to completion and matches the oracle
    out.fill_(float("nan"))
    api.hca_attend(p, *args, out, ws, lse)
    assert api.lca_device_error() == 0
    o = out.float().cpu().numpy()
    units = [(0, 0), (17, 1), (B - 1, 1)]
    ref = oracle_attend_batch(p, q, gamma, pos, kv, win, sink, units=units)
    for (b, i), (ro, _) in ref.items():
        assert_close_rms(o[b, i], ro, what="after the timeout b=%d i=%d" % (b, i))
    assert np.isfinite(o).all()
