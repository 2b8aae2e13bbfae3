"""GPU parity of the manifold-constrained hyper-connection kernels (lca_mhc_pre, lca_mhc_post)
against the oracle, through the C ABI: the generated coefficients (sigmoid pre and post weights,
the Sinkhorn-Knopp matrix), the layer input and the mixed streams, on small shapes with every
supported stream count and at the benchmark's size on sampled tokens.

Tolerances: the coefficients come from fp32 logits (a tensor-core product of n d terms accumulated
in fp32: a rounding error that grows like sqrt(n d) ulps of the partial sums, which are of order 1
here) and fp32 iterations, so a, c and B sit within 4e-7 x sqrt(n d) of the oracle's fp64 values
(5e-5 at n d = 16384; the sigmoid and the Sinkhorn-Knopp map have slopes below 1); the bf16
outputs within half a bf16 ulp of each value plus 1e-3 of the output RMS.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close_bf16_out, u16
from long_context_attention_04_b300 import api, build as lca_build
from workloads import Rng

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    lca_build.build()
    api.lca_device_error()
    yield


def _inputs(seed, T, n, d):
    rng = Rng(seed)
    K = 2 * n + n * n
    return dict(x=rng.normal_bf16((T, n, d)), phi=rng.normal_bf16((K, n * d), 1.0 / math.sqrt(n * d)),
                bias=rng.normal_f32((K,)), y=rng.normal_bf16((T, d)))


def _run(d_in, iters):
    T, n, d = d_in["x"].shape
    g = {k: v.to(DEV) for k, v in d_in.items()}
    h = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    a = torch.empty((T, n), dtype=torch.float32, device=DEV)
    c = torch.empty((T, n), dtype=torch.float32, device=DEV)
    B = torch.empty((T, n, n), dtype=torch.float32, device=DEV)
    ws = torch.empty(api.lca_mhc_workspace(T, n), dtype=torch.uint8, device=DEV)
    api.lca_mhc_pre(g["x"], g["phi"], g["bias"], h, a, c, B, ws, iters=iters)
    xo = torch.empty_like(g["x"])
    api.lca_mhc_post(g["x"], B, c, g["y"], xo)
    assert api.lca_device_error() == 0
    return {k: v.cpu() for k, v in dict(h=h, a=a, c=c, B=B, xo=xo).items()}


def _check_token(d_in, got, t, iters):
    x = u16(d_in["x"][t])
    n, d = x.shape
    tol = 4e-7 * math.sqrt(n * d)
    a, c, B = oracle.mhc_coeffs(x, u16(d_in["phi"]), d_in["bias"].numpy(), iters=iters)
    np.testing.assert_allclose(got["a"][t].numpy(), a, atol=tol, err_msg="a t=%d" % t)
    np.testing.assert_allclose(got["c"][t].numpy(), c, atol=tol, err_msg="c t=%d" % t)
    np.testing.assert_allclose(got["B"][t].numpy(), B, atol=tol, err_msg="B t=%d" % t)
    assert_close_bf16_out(got["h"][t].float().numpy(), oracle.mhc_pre(x, a), what="h t=%d" % t)
    ref = oracle.mhc_post(x, B, c, u16(d_in["y"][t]))
    assert_close_bf16_out(got["xo"][t].float().numpy(), ref, what="x_out t=%d" % t)


@pytest.mark.parametrize("T,n,d,iters", [(37, 4, 512, 20), (5, 2, 256, 20), (3, 1, 64, 20), (130, 4, 4096, 20),
                                         (9, 4, 1000, 3)])
def test_mhc_matches_oracle(T, n, d, iters):
    d_in = _inputs(70 + T, T, n, d)
    got = _run(d_in, iters)
    for t in range(T):
        _check_token(d_in, got, t, iters)
    # the kernel's B is doubly stochastic to fp32 rounding: columns exactly normalised last
    np.testing.assert_allclose(got["B"].sum(1).numpy(), 1.0, atol=2e-6)


def test_mhc_benchmark_size_sampled_tokens():
    """The benchmark's chunk (8192 tokens, 4 streams of 4096): sampled tokens against the oracle."""
    T, n, d = 8192, 4, 4096
    d_in = _inputs(77, T, n, d)
    got = _run(d_in, 20)
    for t in (0, 1, 777, 4096, T - 1):
        _check_token(d_in, got, t, 20)


def test_mhc_rejects_unsupported_shapes():
    x = torch.zeros((2, 3, 64), dtype=torch.bfloat16, device=DEV)      # 3 streams
    K = 15
    with pytest.raises(api.LcaError) as e:
        api.lca_mhc_pre(x, torch.zeros((K, 192), dtype=torch.bfloat16, device=DEV),
                        torch.zeros(K, device=DEV), torch.empty((2, 64), dtype=torch.bfloat16, device=DEV),
                        torch.empty((2, 3), device=DEV), torch.empty((2, 3), device=DEV),
                        torch.empty((2, 3, 3), device=DEV), torch.empty(1024, dtype=torch.uint8, device=DEV))
    assert e.value.status == 2
