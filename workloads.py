"""Seeded synthetic inputs for the CSA/HCA attention path.

This module is the one thing the CUDA path and the CPU oracle share: it draws
random numbers into tensors of the workload shapes and does none of the method's
arithmetic (no pooling, normalisation, rotation, scoring or selection).

Distributions (the pages publish no data; these follow the workload statements):
  * activations, per-token KV vectors, queries, indexer queries and keys: N(0, 1), bf16;
  * compressed cache rows: N(0, 1), bf16.  A row of N(0,1) draws has RMS 1 to within
    sampling error and is rotation invariant in law, so it is distributed like a
    RMS-normalised, RoPE-rotated row with gamma = 1;
  * compressor logits z: N(0, 1) fp32; learned position biases: N(0, 0.02) fp32;
  * indexer head weights w: N(0, 1) / sqrt(H_I) fp32;
  * per-head sink logits: N(0, 1) fp32;
  * projection weights: N(0, 0.02) bf16;  norm gammas: 1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a (CPU) bf16 tensor as a numpy uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


class Rng:
    """A seeded torch generator (CPU by default) with the draws the workloads use."""

    def __init__(self, seed: int = 0, device: str = "cpu"):
        self.device = device
        self.g = torch.Generator(device=device)
        self.g.manual_seed(seed)

    def normal_bf16(self, shape, std: float = 1.0) -> torch.Tensor:
        x = torch.randn(shape, generator=self.g, device=self.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    def normal_f32(self, shape, std: float = 1.0) -> torch.Tensor:
        x = torch.randn(shape, generator=self.g, device=self.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x

    def ints(self, low: int, high: int, shape) -> torch.Tensor:
        return torch.randint(low, high, shape, generator=self.g, device=self.device, dtype=torch.int32)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Sizes of one attention layer (names follow the pages' notation)."""
    heads: int = 64          # H, query heads (Multi-Query: one KV for all)
    head_dim: int = 512      # c
    rope_dims: int = 64      # R, rotated trailing dims
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    window: int = 128        # W, sliding-window tokens
    ratio: int = 4           # m (CSA) or m' (HCA)
    topk: int = 512          # k (CSA)
    idx_heads: int = 64      # H_I
    idx_dim: int = 128       # d_I

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The workloads.  Names say what each is and at which sizes.
TINY_CSA_PREFILL = dict(
    name="tiny CSA prefill, 2048 tokens, hidden 256, H=8 c=128, H_I=4 d_I=32, k=64, W=16",
    kind="csa_prefill", B=1, n_tok=2048, hidden=256,
    shape=LayerShape(heads=8, head_dim=128, rope_dims=64, window=16, ratio=4, topk=64,
                     idx_heads=4, idx_dim=32))

CSA_DECODE_128K = dict(
    name="CSA decode, batch 32, 128K context (32768 entries x 512), k=512, W=128, H=64",
    kind="csa_decode", B=32, pos=131071, entries=32768,
    shape=LayerShape(ratio=4, topk=512))

# The same decode step with FP8 caches: the indexer keys and the KV entries in e4m3 (one fp32
# scale per row); the step compresses into e4m3, quantises its indexer queries, and attends over
# the e4m3 rows (the window rows stay bf16).
CSA_DECODE_128K_FP8 = dict(CSA_DECODE_128K, idx_e4m3=True, kv_e4m3=True,
                           name="CSA decode with e4m3 caches (keys and KV), batch 32, 128K context "
                                "(32768 entries x 512), k=512, W=128, H=64")

HCA_DECODE_1M = dict(
    name="HCA decode, batch 16, 1M context (8192 entries x 512), W=128, H=64",
    kind="hca_decode", B=16, pos=1048575, entries=8192,
    shape=LayerShape(ratio=128))

CSA_PREFILL_1M = dict(
    name="CSA chunked prefill, 8192 queries at 1M context (262144 entries), k=1024, W=128, H=64",
    kind="csa_prefill_chunk", B=1, q_begin=1040384, Tq=8192, entries=262144,
    shape=LayerShape(ratio=4, topk=1024))

# The same chunked prefill at 128K context: the 1M chunk's kernels at a size (0.4 GB on the
# device) that a profiler can replay many times.
CSA_PREFILL_128K = dict(
    name="CSA chunked prefill, 2048 queries at 128K context (32768 entries), k=1024, W=128, H=64",
    kind="csa_prefill_chunk", B=1, q_begin=129024, Tq=2048, entries=32768,
    shape=LayerShape(ratio=4, topk=1024))

# The HCA decode step over an e4m3 KV cache (one fp32 scale per row).
HCA_DECODE_1M_FP8 = dict(HCA_DECODE_1M, kv_e4m3=True,
                         name="HCA decode with an e4m3 KV cache, batch 16, 1M context (8192 entries x 512), W=128, "
                              "H=64")

BLOCK_DECODE_1M = dict(
    name="V4-Flash-style block decode, batch 4, 1M context, 8 CSA (k=512) + 8 HCA layers, "
         "grouped O-proj 64 heads -> 8 x 1024 -> 4096",
    kind="block_decode", B=4, pos=1048575, csa_entries=262144, hca_entries=8192,
    n_csa=8, n_hca=8, groups=8, d_g=1024, d_model=4096,
    csa=LayerShape(ratio=4, topk=512), hca=LayerShape(ratio=128))

# The whole V4-Flash attention stack at decode: 43 layers, CSA and HCA alternating (CSA first:
# 22 CSA + 21 HCA), each with its grouped output projection, batch 4 at 1M context.
V4FLASH_DECODE_1M = dict(
    name="V4-Flash attention stack decode, batch 4, 1M context, 43 layers (22 CSA k=512 + 21 HCA alternating), "
         "grouped O-proj 64 heads -> 8 x 1024 -> 4096",
    kind="block_decode", B=4, pos=1048575, csa_entries=262144, hca_entries=8192,
    n_csa=22, n_hca=21, groups=8, d_g=1024, d_model=4096,
    csa=LayerShape(ratio=4, topk=512), hca=LayerShape(ratio=128))

# The 1M-context CSA prefill chunk with its input projections: the chunk's hidden states
# (V4-Flash width 4096) mapped to the queries, indexer queries and weights, and the KV and
# indexer-key token vectors and compressor logits by plain linear maps (the pages do not give
# the projections; the tiny configuration's reading) on the tensor cores, then the layer.
CSA_PREFILL_1M_PROJ = dict(CSA_PREFILL_1M, hidden=4096,
                           name="CSA chunked prefill with input projections from hidden 4096, 8192 queries at 1M "
                                "context (262144 entries), k=1024, W=128, H=64")

# The same chunk with the indexer's scores written out (8192 x 262144 fp32) and selected by a
# separate top-k pass: the path the fused selection replaces, timed beside it.
CSA_PREFILL_1M_SCORED = dict(CSA_PREFILL_1M, materialise=True,
                             name="CSA chunked prefill, scores materialised then top-k, 8192 queries at 1M "
                                  "context (262144 entries), k=1024, W=128, H=64")

# Manifold-constrained hyper-connections around one layer, for a prefill chunk: 4 residual
# streams of the V4-Flash hidden size (4096), the generated coefficients (Sinkhorn-Knopp, 20
# passes), the layer input and, given the layer's output, the new streams.
MHC_PREFILL_8192 = dict(
    name="mHC around one layer, 8192 tokens, 4 streams x 4096, Sinkhorn-Knopp 20 passes",
    kind="mhc", T=8192, n=4, d=4096, iters=20)

WORKLOADS = {
    "tiny_csa_prefill": TINY_CSA_PREFILL,
    "csa_decode_128k": CSA_DECODE_128K,
    "hca_decode_1m": HCA_DECODE_1M,
    "csa_prefill_1m": CSA_PREFILL_1M,
    "csa_prefill_128k": CSA_PREFILL_128K,
    "block_decode_1m": BLOCK_DECODE_1M,
    "mhc_prefill_8192": MHC_PREFILL_8192,
    "v4flash_decode_1m": V4FLASH_DECODE_1M,
    "csa_prefill_1m_proj": CSA_PREFILL_1M_PROJ,
    "csa_prefill_1m_scored": CSA_PREFILL_1M_SCORED,
    "csa_decode_128k_fp8": CSA_DECODE_128K_FP8,
    "hca_decode_1m_fp8": HCA_DECODE_1M_FP8,
}


def layer_weights(rng: Rng, s: LayerShape, csa: bool) -> dict:
    """Learned per-layer parameters that the path reads (norm gammas, biases, sinks)."""
    span = 2 * s.ratio if csa else s.ratio
    w = dict(
        gamma_kv=torch.ones(s.head_dim, dtype=torch.float32, device=rng.device),
        gamma_q=torch.ones(s.head_dim, dtype=torch.float32, device=rng.device),
        bias_kv=rng.normal_f32((span,), 0.02),
        sink=rng.normal_f32((s.heads,)),
    )
    if csa:
        w["bias_idx"] = rng.normal_f32((span,), 0.02)
    return w


def decode_inputs(rng: Rng, s: LayerShape, B: int, pos: int, entries: int, csa: bool,
                  win_cap: int | None = None) -> dict:
    """State and per-step inputs of one decode step at position `pos` for B sequences.

    The step's new token at `pos` completes block entries-1, so the caches hold
    entries-1 rows before the step (row entries-1 is drawn too and is overwritten by
    the step's compression).  The staging rows hold the tokens that block's
    compressor window covers: 2m for CSA, m' for HCA, the last one being `pos`.
    """
    m = s.ratio
    span = 2 * m if csa else m
    win_cap = win_cap or s.window
    d = dict(
        pos=pos, entries=entries, win_cap=win_cap, tok_pos0=pos + 1 - span,
        kv_cache=rng.normal_bf16((B, entries, s.head_dim)),
        win_kv=rng.normal_bf16((B, win_cap, s.head_dim)),
        tok_v=rng.normal_bf16((B, span, s.head_dim)),
        tok_z=rng.normal_f32((B, span)),
        q=rng.normal_bf16((B, 1, s.heads, s.head_dim)),
    )
    if csa:
        d.update(
            idx_cache=rng.normal_bf16((B, entries, s.idx_dim)),
            tok_vi=rng.normal_bf16((B, span, s.idx_dim)),
            tok_zi=rng.normal_f32((B, span)),
            q_idx=rng.normal_bf16((B, 1, s.idx_heads, s.idx_dim)),
            w_idx=rng.normal_f32((B, 1, s.idx_heads), 1.0 / math.sqrt(s.idx_heads)),
        )
    d.update(layer_weights(rng, s, csa))
    return d


def prefill_chunk_inputs(rng: Rng, s: LayerShape, q_begin: int, Tq: int, entries: int,
                         win_cap: int) -> dict:
    """State and inputs of one CSA prefill chunk of Tq query tokens at [q_begin, q_begin+Tq).

    The caches hold entries - Tq/m rows before the chunk; the chunk compresses the
    remaining Tq/m.  The staging rows start m tokens before the chunk (the first new
    entry's window reaches back one block).  The window ring holds the W-1 tokens
    before the chunk; the chunk's own rows are written by the window update.
    """
    m = s.ratio
    tok_pos0 = q_begin - m
    n_tok = Tq + m
    return dict(
        q_begin=q_begin, Tq=Tq, entries=entries, first_entry=entries - Tq // m,
        tok_pos0=tok_pos0, win_cap=win_cap,
        kv_cache=rng.normal_bf16((1, entries, s.head_dim)),
        idx_cache=rng.normal_bf16((1, entries, s.idx_dim)),
        win_kv=rng.normal_bf16((1, win_cap, s.head_dim)),
        tok_v=rng.normal_bf16((1, n_tok, s.head_dim)),
        tok_z=rng.normal_f32((1, n_tok)),
        tok_vi=rng.normal_bf16((1, n_tok, s.idx_dim)),
        tok_zi=rng.normal_f32((1, n_tok)),
        q=rng.normal_bf16((1, Tq, s.heads, s.head_dim)),
        q_idx=rng.normal_bf16((1, Tq, s.idx_heads, s.idx_dim)),
        w_idx=rng.normal_f32((1, Tq, s.idx_heads), 1.0 / math.sqrt(s.idx_heads)),
        **layer_weights(rng, s, True),
    )


def tiny_prefill_inputs(rng: Rng, cfg: dict = TINY_CSA_PREFILL) -> dict:
    """Hidden states and projection weights of the tiny CSA layer (full prefill from 0).

    The per-token projections are not described on the pages; the tiny layer uses
    plain linear maps from the hidden state: q (H*c), KV vector (c), compressor logit
    (1), indexer query (H_I*d_I), indexer key vector (d_I), indexer logit (1) and the
    indexer head weights (H_I).
    """
    s = cfg["shape"]
    n, hid = cfg["n_tok"], cfg["hidden"]
    std = 0.02
    return dict(
        x=rng.normal_bf16((n, hid)),
        W_q=rng.normal_bf16((s.heads * s.head_dim, hid), std),
        W_kv=rng.normal_bf16((s.head_dim, hid), std),
        W_z=rng.normal_bf16((1, hid), std),
        W_qi=rng.normal_bf16((s.idx_heads * s.idx_dim, hid), std),
        W_ki=rng.normal_bf16((s.idx_dim, hid), std),
        W_zi=rng.normal_bf16((1, hid), std),
        W_w=rng.normal_bf16((s.idx_heads, hid), std),
        **layer_weights(rng, s, True),
    )


def oproj_weights(rng: Rng, heads: int, head_dim: int, groups: int, d_g: int, d_model: int) -> dict:
    return dict(
        Wg=rng.normal_bf16((groups * d_g, (heads // groups) * head_dim), 0.02),
        Wm=rng.normal_bf16((d_model, groups * d_g), 0.02),
    )


def mhc_inputs(rng: Rng, T: int, n: int, d: int) -> dict:
    """Residual streams x [T, n, d] and the layer's output y [T, d] (N(0, 1), bf16); the generating
    weights phi [2n + n^2, n d] (N(0, 1/(n d)), bf16: unit-scale generated logits) and bias
    [2n + n^2] (N(0, 1), fp32)."""
    K = 2 * n + n * n
    return dict(x=rng.normal_bf16((T, n, d)), y=rng.normal_bf16((T, d)),
                phi=rng.normal_bf16((K, n * d), 1.0 / math.sqrt(n * d)), bias=rng.normal_f32((K,)))


def prefill_projection_weights(rng: Rng, s: LayerShape, hidden: int) -> dict:
    """Plain linear maps from the hidden state (N(0, 0.02), bf16), one weight row per output:
    queries (H c), KV token vector (c), compressor logit (1), indexer queries (H_I d_I), indexer
    key vector (d_I), its compressor logit (1), indexer head weights (H_I)."""
    std = 0.02
    return dict(
        W_q=rng.normal_bf16((s.heads * s.head_dim, hidden), std),
        W_kv=rng.normal_bf16((s.head_dim, hidden), std),
        W_z=rng.normal_bf16((1, hidden), std),
        W_qi=rng.normal_bf16((s.idx_heads * s.idx_dim, hidden), std),
        W_ki=rng.normal_bf16((s.idx_dim, hidden), std),
        W_zi=rng.normal_bf16((1, hidden), std),
        W_w=rng.normal_bf16((s.idx_heads, hidden), std),
    )
