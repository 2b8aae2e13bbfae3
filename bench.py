"""Benchmark of the CSA/HCA attention path on B300 (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of a layer's whole path over one batch: compression of the block the new
tokens complete, the window rows of the new tokens, (CSA) indexer scores and top-k, core
attention with split-K combine.  Workloads (sizes of the pages' V4-Flash configuration):
  csa_decode_128k (default)  batch 32, 128K context, one query per sequence
  hca_decode_1m              batch 16, 1M context, one query per sequence
  csa_prefill_1m             one 8192-query chunk at 1M context
  csa_prefill_128k           one 2048-query chunk at 128K context (the same kernels, profiler-sized)
  csa_prefill_1m_scored      the 1M chunk with its scores written out and selected by a separate top-k
  csa_decode_128k_fp8        csa_decode_128k with e4m3 caches: indexer keys (and queries) and KV rows
  hca_decode_1m_fp8          hca_decode_1m over an e4m3 KV cache (per-row scales)
Inputs are seeded synthetic tensors (workloads.py); the caches are larger than L2 and L2 is
also flushed between timed steps.  Under torchrun each rank runs the workload on its own
GPU (sequences shard with no exchange: weak scaling); the value is all ranks' tokens over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "CSA/HCA attention tokens/s per layer at 128K–1M ctx; % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "csa_decode_128k"
L2_FLUSH_BYTES = 512 << 20


def source_hash() -> str:
    """sha1 over the library sources (csrc/* and include/lca.h), first 16 hex digits."""
    import glob
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    files = sorted(glob.glob(os.path.join(root, "long_context_attention_04_b300", "csrc", "*")))
    files.append(os.path.join(root, "include", "lca.h"))
    h = hashlib.sha1()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per dominant call from profiles/dram_traffic.md, if taken with these sources."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    h = source_hash()
    for line in lines:
        cols = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cols) == 7 and cols[0] == workload and cols[6] == h:
            return int(cols[4])
    return None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


# ------------------------------------------------------------------------- clocks -----

class _Nvml:
    """The few read-only NVML queries the clock sampler needs, through ctypes on the driver's
    libnvidia-ml (no Python NVML package is required)."""
    CLOCK_SM = 0

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._check(self.lib.nvmlInit_v2())
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _check(self, rc):
        if rc != 0:
            raise RuntimeError("NVML error %d" % rc)

    def handle(self, bus_id: str, index: int):
        h = self.ct.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), self.ct.byref(h)) != 0:
            self._check(self.lib.nvmlDeviceGetHandleByIndex_v2(self.ct.c_uint(index), self.ct.byref(h)))
        return h

    def sm_clock(self, h) -> int:
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, self.ct.byref(v)))
        return v.value

    def sm_max_clock(self, h) -> int:
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, self.ct.byref(v)))
        return v.value

    def reasons(self, h) -> int:
        v = self.ct.c_ulonglong()
        self._check(self.reasons_fn(h, self.ct.byref(v)))
        return v.value

    def shutdown(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event (throttle) reasons, read through NVML about every millisecond
    on a background thread while the timed region runs (a 200 ms nvidia-smi loop would miss
    a timed region of a few milliseconds).  Read-only: no clock or other setting is touched."""

    # NVML clock-event reason bits
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.device_index = device_index
        self.period = period_s
        self.samples = []          # (sm_mhz, reason bits)
        self.max_mhz = None
        self.nv = None
        self.handle = None
        self.stop = threading.Event()
        self.thread = None
        self.error = None

    def __enter__(self):
        try:
            self.nv = _Nvml()
            pr = torch.cuda.get_device_properties(self.device_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip().isdigit()]
            idx = int(vis[self.device_index]) if self.device_index < len(vis) else self.device_index
            self.handle = self.nv.handle(bus, idx)
            self.max_mhz = float(self.nv.sm_max_clock(self.handle))
            self._sample()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        except Exception as e:     # no NVML: the line reports zero samples and why
            self.handle = None
            self.error = "%s: %s" % (type(e).__name__, e)
        return self

    def _sample(self):
        self.samples.append((float(self.nv.sm_clock(self.handle)), int(self.nv.reasons(self.handle))))

    def _loop(self):
        while not self.stop.is_set():
            try:
                self._sample()
            except Exception as e:
                self.error = "%s: %s" % (type(e).__name__, e)
                return
            time.sleep(self.period)

    def __exit__(self, *exc):
        self.stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
        if self.nv is not None:
            try:
                self.nv.shutdown()
            except Exception:
                pass

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "nvml",
                    "error": self.error}
        reasons = set()
        for _, bits in self.samples:
            for name, bit in self.REASONS:
                if bits & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([m for m, _ in self.samples])), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


# ---------------------------------------------------------------------- workloads -----

def csa_layer_work(s, B: int, n_vis, Tq: int, entries: int = 0):
    """Algorithmic bytes and FLOPs of one CSA layer step: inputs read once, outputs written once,
    workspace round trips (scores, split-K partials) left out.  Decode (Tq = 1): per sequence the
    keys of the visible entries, the selected and window rows, the query and the output, the
    tokens compressed into the new KV and key entries.  Prefill (one chunk): the keys of all
    entries once (`entries`), each query's selected and window rows."""
    m, c, dI, HI, H, k, W = s.ratio, s.head_dim, s.idx_dim, s.idx_heads, s.heads, s.topk, s.window
    n_vis_sum = float(np.sum(n_vis)) * (B if np.ndim(n_vis) == 0 else 1)
    n_new = max(1, Tq // m)
    compress = B * n_new * ((2 * m) * (2 * c + 4) + 2 * c + (2 * m) * (2 * dI + 4) + 2 * dI)
    window = B * Tq * 4 * c
    keys = B * entries * 2 * dI if entries else n_vis_sum * 2 * dI
    indexer = keys + B * Tq * HI * (2 * dI + 4)
    attention = B * Tq * ((k + W) * 2 * c + 2 * H * c * 2 + 4 * k)
    flops = 2.0 * n_vis_sum * HI * dI + 4.0 * B * Tq * (k + W) * H * c
    return float(compress + window + indexer + attention), flops


def hca_layer_work(s, B: int, n_vis: int):
    """Algorithmic bytes and FLOPs of one HCA decode step: the block of m' tokens compressed into
    the new entry, the window row, every visible entry and the window rows once, query and output."""
    m, c, H, W = s.ratio, s.head_dim, s.heads, s.window
    compress = B * (m * (2 * c + 4) + 2 * c)
    window = B * 4 * c
    attention = B * ((n_vis + W) * 2 * c + 2 * H * c * 2)
    return float(compress + window + attention), 4.0 * B * (n_vis + W) * H * c


class Workload:
    """Common shape of a benchmark workload (device state + per-step inputs)."""

    def _stage_inputs(self, keys, stage: bool, groups: dict = None):
        """The per-step inputs as views of one packed device buffer with a pinned host mirror
        (host_in), uploaded group by group; without `stage`, plain pinned host copies."""
        from long_context_attention_04_b300.layers import StagingBuffer
        if stage:
            sub = {k: self.d[k] for k in keys}
            self.stage = StagingBuffer(sub, groups)
            self.d.update(sub)
            self.host_in = self.stage.host
        else:
            self.stage = None
            self.host_in = {k: self.d[k].cpu().pin_memory() for k in keys}
    name = ""
    tokens = 0                 # tokens processed per step (per rank)
    launches = 0               # our kernel launches per step
    dominant = ""              # name of the dominant kernel
    bound = "hbm"

    def step(self):
        raise NotImplementedError

    def dominant_call(self):   # the dominant kernel's launch alone
        raise NotImplementedError

    def e2e_step(self):
        raise NotImplementedError


def _quantized(api, x):
    """e4m3 codes and per-row scales of a bf16 cache [B, rows, width] (the library's quantiser)."""
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty(x.shape[:2], dtype=torch.float32, device="cuda")
    api.lca_quantize_rows_e4m3(x, q, sc)
    return q, sc


class CsaDecode(Workload):
    def __init__(self, cfg: dict, seed: int = 0, stage: bool = True):
        from long_context_attention_04_b300 import api
        from long_context_attention_04_b300.layers import CsaLayer, LayerWeights
        self.api = api
        s = cfg["shape"]
        self.cfg = cfg
        B, pos, entries = cfg["B"], cfg["pos"], cfg["entries"]
        self.B, self.pos, self.entries = B, pos, entries
        self.p = api.params_from(s)
        self.s = s
        rng = wl.Rng(seed, device="cuda")
        d = wl.decode_inputs(rng, s, B, pos, entries, csa=True)
        self.d = d
        w = LayerWeights(d["gamma_kv"], d["gamma_q"], d["bias_kv"], d["sink"], d["bias_idx"])
        # e4m3 indexer keys: the synthetic bf16 key cache quantised once (per-row scales)
        self.e4m3 = bool(cfg.get("idx_e4m3"))
        self.kv8 = bool(cfg.get("kv_e4m3"))
        kv, kv_scale, keys, key_scale = d["kv_cache"], None, d["idx_cache"], None
        if self.kv8:     # the synthetic bf16 KV cache quantised once (per-row scales)
            kv, kv_scale = _quantized(api, d["kv_cache"])
        if self.e4m3:
            keys, key_scale = _quantized(api, d["idx_cache"])
        self.layer = CsaLayer(self.p, w, kv, keys, d["win_kv"], n_q=1, idx_scale=key_scale, kv_scale=kv_scale)
        if self.e4m3:
            api.lca_quantize_rows_e4m3(d["q_idx"], self.layer.q8, self.layer.q8_scale)
        i32 = dict(dtype=torch.int32, device="cuda")
        self.tok_pos0 = torch.full((B,), d["tok_pos0"], **i32)
        self.first = torch.full((B,), entries - 1, **i32)
        self.new_pos = torch.full((B,), pos, **i32)
        self.q_pos = torch.full((B, 1), pos, **i32)
        self.out = torch.empty((B, 1, s.heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        self.scores = self.layer.ws_idx.view(torch.float32).view(B, 1, -1)
        self.tokens = B
        # 2 compress, window, q prep, (query quantisation,) indexer, top-k, attention, combine
        self.launches = 9 if self.e4m3 else 8
        self.dominant = "indexer"
        # per-step inputs, pinned on the host for the end-to-end leg
        # (the selection's inputs first; the rest goes up on the side stream during the selection)
        self.groups = {"main": ["tok_vi", "tok_zi", "q_idx", "w_idx"], "side": ["tok_v", "tok_z", "q"]}
        self._stage_inputs(("tok_v", "tok_z", "tok_vi", "tok_zi", "q", "q_idx", "w_idx"), stage, self.groups)
        self.host_out = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host_in.values())
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        # algorithmic bytes of one indexer launch: keys of the visible entries, queries, weights (the
        # scores it writes are a workspace round trip to the top-k, so they are not counted)
        n_vis = (pos + 1) // s.ratio
        if self.e4m3:   # one byte per key element plus the row's scale; the query's codes and scales
            self.dom_bytes = B * (n_vis * (s.idx_dim + 4) + s.idx_heads * s.idx_dim + s.idx_heads * 8)
        else:
            self.dom_bytes = B * (n_vis * s.idx_dim * 2 + s.idx_heads * s.idx_dim * 2 + s.idx_heads * 4)
        self.dom_flops = 2.0 * B * n_vis * s.idx_heads * s.idx_dim
        self.step_bytes, self.step_flops = csa_layer_work(s, B, n_vis, 1)
        if self.e4m3:   # a key row is d_I bytes + its scale instead of 2 d_I
            self.step_bytes -= B * n_vis * (s.idx_dim - 4)
        if self.kv8:    # a selected KV row is c bytes + its scale instead of 2 c
            self.step_bytes -= B * s.topk * (s.head_dim - 4)

    def dominant_call(self):
        d, L = self.d, self.layer
        if self.e4m3:
            self.api.csa_indexer_scores_e4m3(self.p, L.q8, L.q8_scale, d["w_idx"], L.idx_cache, L.idx_scale,
                                             self.q_pos, self.scores)
        else:
            self.api.csa_indexer_scores(self.p, d["q_idx"], d["w_idx"], L.idx_cache, self.q_pos, self.scores)

    def step(self, side_prologue=None):
        d = self.d
        self.layer.step_overlapped(d["tok_v"], d["tok_z"], d["tok_vi"], d["tok_zi"], self.tok_pos0, self.first, 1,
                                   d["tok_v"][:, -1:], self.new_pos, d["q"], d["q_idx"], d["w_idx"], self.q_pos,
                                   self.out, side_prologue)

    def e2e_step(self):
        self.stage.upload(group="main")
        self.step(lambda side: self.stage.upload(side, "side"))
        self.host_out.copy_(self.out, non_blocking=True)

    def cpu_sample(self, budget_s: float) -> dict:
        """The oracle on whole sequences of this step until the budget is spent."""
        import oracle
        from workloads import bf16_bits
        s = self.s
        t_total, n_done = 0.0, 0
        for b in range(self.B):
            kvb = bf16_bits(self.kv_host[b])
            ixb = bf16_bits(self.idx_host[b])
            winb = bf16_bits(self.win_host[b])
            tv, tz = bf16_bits(self.host_in["tok_v"][b]), self.host_in["tok_z"][b].numpy()
            tvi, tzi = bf16_bits(self.host_in["tok_vi"][b]), self.host_in["tok_zi"][b].numpy()
            q = bf16_bits(self.host_in["q"][b, 0])
            qi = bf16_bits(self.host_in["q_idx"][b, 0])
            wi = self.host_in["w_idx"][b, 0].numpy()
            g = self.w_host["gamma_kv"]
            t0 = time.perf_counter()
            kv_new = oracle.compress(tv, tz, self.d["tok_pos0"], self.w_host["bias_kv"], g, s.rms_eps, s.rope_dims,
                                     s.rope_base, 2 * s.ratio, s.ratio, self.entries - 1, 1)
            k_new = oracle.compress(tvi, tzi, self.d["tok_pos0"], self.w_host["bias_idx"], None, s.rms_eps, 0,
                                    s.rope_base, 2 * s.ratio, s.ratio, self.entries - 1, 1)
            w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, self.pos)
            t1 = time.perf_counter()
            kvb[-1] = _round_bits(kv_new[0])
            ixb[-1] = _round_bits(k_new[0])
            winb[self.pos % winb.shape[0]] = _round_bits(w_new)
            t2 = time.perf_counter()
            n_vis = oracle.visible_entries(self.pos, s.ratio)
            t_fp8 = 0.0
            if self.e4m3:
                # the e4m3 key cache of the sequence (state before the step, not timed), then the
                # step's own quantisations: the new key row and the queries
                t4 = time.perf_counter()
                k8, ks = oracle.quantize_rows_e4m3(ixb[:-1])
                t5 = time.perf_counter()
                kn8, kns = oracle.quantize_rows_e4m3(ixb[-1:])
                q8, qs = oracle.quantize_rows_e4m3(qi)
                sc = oracle.indexer_scores_e4m3(q8, qs, wi, np.concatenate([k8, kn8]), np.concatenate([ks, kns]),
                                                n_vis)
                t_fp8 = t5 - t4
            else:
                sc = oracle.indexer_scores(qi, wi, ixb, n_vis)
            idx = oracle.topk(sc, s.topk)
            if self.kv8:
                t6 = time.perf_counter()
                kv8, kvs = oracle.quantize_rows_e4m3(kvb[:-1])             # the cache before the step, not timed
                t7 = time.perf_counter()
                t_fp8 += t7 - t6
                kn8, kns = oracle.quantize_rows_e4m3(kvb[-1:])
                oracle.attend_e4m3(q, self.w_host["gamma_q"], self.pos, np.concatenate([kv8, kn8]),
                                   np.concatenate([kvs, kns]), self.w_host["sink"], winb, winb.shape[0], s.window,
                                   s.rope_dims, s.rope_base, s.rms_eps, self.p.scale, idx=idx)
            else:
                oracle.attend(q, self.w_host["gamma_q"], self.pos, kvb, self.w_host["sink"], winb, winb.shape[0],
                              s.window, s.rope_dims, s.rope_base, s.rms_eps, self.p.scale, idx=idx)
            t3 = time.perf_counter()
            t_total += (t1 - t0) + (t3 - t2) - t_fp8
            n_done += 1
            if t_total >= budget_s:
                break
        return dict(value=n_done / t_total, unit="tokens/s", cores=1, kind="oracle",
                    sample="%d of %d sequences of the step (compression, window row, indexer over %d entries, "
                           "top-%d, attention), single-threaded fp64" % (n_done, self.B, self.entries, s.topk))

    def snapshot_host(self):
        """Host copies of the state the oracle needs, taken before any GPU step touches it."""
        n = min(self.B, 64)
        self.kv_host = self.d["kv_cache"][:n].cpu()
        self.idx_host = self.d["idx_cache"][:n].cpu()
        self.win_host = self.d["win_kv"][:n].cpu()
        self.w_host = {k: self.d[k].cpu().numpy() for k in ("gamma_kv", "gamma_q", "bias_kv", "bias_idx", "sink")}


class HcaDecode(Workload):
    def __init__(self, cfg: dict, seed: int = 0, stage: bool = True):
        from long_context_attention_04_b300 import api
        from long_context_attention_04_b300.layers import HcaLayer, LayerWeights
        self.api = api
        s = cfg["shape"]
        self.cfg, self.s = cfg, s
        B, pos, entries = cfg["B"], cfg["pos"], cfg["entries"]
        self.B, self.pos, self.entries = B, pos, entries
        self.p = api.params_from(s)
        rng = wl.Rng(seed, device="cuda")
        d = wl.decode_inputs(rng, s, B, pos, entries, csa=False)
        self.d = d
        w = LayerWeights(d["gamma_kv"], d["gamma_q"], d["bias_kv"], d["sink"])
        self.kv8 = bool(cfg.get("kv_e4m3"))
        if self.kv8:     # the synthetic bf16 KV cache quantised once (per-row scales)
            kv8, kv8_scale = _quantized(api, d["kv_cache"])
            self.layer = HcaLayer(self.p, w, kv8, d["win_kv"], n_q=1, kv_scale=kv8_scale)
        else:
            self.layer = HcaLayer(self.p, w, d["kv_cache"], d["win_kv"], n_q=1)
        i32 = dict(dtype=torch.int32, device="cuda")
        self.tok_pos0 = torch.full((B,), d["tok_pos0"], **i32)
        self.first = torch.full((B,), entries - 1, **i32)
        self.new_pos = torch.full((B,), pos, **i32)
        self.q_pos = torch.full((B, 1), pos, **i32)
        self.out = torch.empty((B, 1, s.heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        self.tokens = B
        self.launches = 5          # compress, window, q prep, attention, combine
        self.dominant = "attend e4m3" if self.kv8 else "attend"
        # (the compression's inputs first; the query goes up on the side stream meanwhile)
        self.groups = {"main": ["tok_v", "tok_z"], "side": ["q"]}
        self._stage_inputs(("tok_v", "tok_z", "q"), stage, self.groups)
        self.host_out = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host_in.values())
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        n_vis = (pos + 1) // s.ratio
        rows = n_vis + s.window
        # e4m3 compressed rows: c bytes + the row's scale instead of 2 c
        comp_row = (s.head_dim + 4) if self.kv8 else 2 * s.head_dim
        self.dom_bytes = B * (n_vis * comp_row + s.window * s.head_dim * 2 + 2 * s.heads * s.head_dim * 2)
        self.dom_flops = 4.0 * B * rows * s.heads * s.head_dim
        self.step_bytes, self.step_flops = hca_layer_work(s, B, n_vis)
        if self.kv8:
            self.step_bytes -= B * n_vis * (2 * s.head_dim - comp_row)

    def dominant_call(self):
        # the attention kernel and its split-K combine
        self.layer.attend(self.d["q"], self.q_pos, self.out)

    def step(self, side_prologue=None):
        d = self.d
        self.layer.step_overlapped(d["tok_v"], d["tok_z"], self.tok_pos0, self.first, 1, d["tok_v"][:, -1:],
                                   self.new_pos, d["q"], self.q_pos, self.out, side_prologue)

    def e2e_step(self):
        self.stage.upload(group="main")
        self.step(lambda side: self.stage.upload(side, "side"))
        self.host_out.copy_(self.out, non_blocking=True)

    def snapshot_host(self):
        n = min(self.B, 64)
        self.kv_host = self.d["kv_cache"][:n].cpu()
        self.win_host = self.d["win_kv"][:n].cpu()
        self.w_host = {k: self.d[k].cpu().numpy() for k in ("gamma_kv", "gamma_q", "bias_kv", "sink")}

    def cpu_sample(self, budget_s: float) -> dict:
        import oracle
        from workloads import bf16_bits
        s = self.s
        t_total, n_done = 0.0, 0
        for b in range(self.B):
            kvb = bf16_bits(self.kv_host[b])
            winb = bf16_bits(self.win_host[b])
            tv, tz = bf16_bits(self.host_in["tok_v"][b]), self.host_in["tok_z"][b].numpy()
            q = bf16_bits(self.host_in["q"][b, 0])
            g = self.w_host["gamma_kv"]
            t0 = time.perf_counter()
            kv_new = oracle.compress(tv, tz, self.d["tok_pos0"], self.w_host["bias_kv"], g, s.rms_eps, s.rope_dims,
                                     s.rope_base, s.ratio, s.ratio, self.entries - 1, 1)
            w_new = oracle.window_row(tv[-1], g, s.rms_eps, s.rope_dims, s.rope_base, self.pos)
            t1 = time.perf_counter()
            kvb[-1] = _round_bits(kv_new[0])
            winb[self.pos % winb.shape[0]] = _round_bits(w_new)
            t_fp8 = 0.0
            if self.kv8:
                t4 = time.perf_counter()
                kv8, kvs = oracle.quantize_rows_e4m3(kvb[:-1])             # the cache before the step, not timed
                t_fp8 = time.perf_counter() - t4
            t2 = time.perf_counter()
            if self.kv8:
                kn8, kns = oracle.quantize_rows_e4m3(kvb[-1:])
                oracle.attend_e4m3(q, self.w_host["gamma_q"], self.pos, np.concatenate([kv8, kn8]),
                                   np.concatenate([kvs, kns]), self.w_host["sink"], winb, winb.shape[0], s.window,
                                   s.rope_dims, s.rope_base, s.rms_eps, self.p.scale,
                                   n_dense=oracle.visible_entries(self.pos, s.ratio))
            else:
                oracle.attend(q, self.w_host["gamma_q"], self.pos, kvb, self.w_host["sink"], winb, winb.shape[0],
                              s.window, s.rope_dims, s.rope_base, s.rms_eps, self.p.scale,
                              n_dense=oracle.visible_entries(self.pos, s.ratio))
            t3 = time.perf_counter()
            t_total += (t1 - t0) + (t3 - t2)
            n_done += 1
            if t_total >= budget_s:
                break
        return dict(value=n_done / t_total, unit="tokens/s", cores=1, kind="oracle",
                    sample="%d of %d sequences of the step (compression of the 128-token block, window row, "
                           "attention over %d entries + %d window rows), single-threaded fp64"
                           % (n_done, self.B, self.entries, s.window))


class CsaPrefill(Workload):
    def __init__(self, cfg: dict, seed: int = 0, stage: bool = True):
        from long_context_attention_04_b300 import api
        from long_context_attention_04_b300.layers import CsaLayer, LayerWeights
        self.api = api
        s = cfg["shape"]
        self.cfg, self.s = cfg, s
        Tq, entries, q_begin = cfg["Tq"], cfg["entries"], cfg["q_begin"]
        self.Tq, self.entries, self.q_begin = Tq, entries, q_begin
        self.p = api.params_from(s)
        win_cap = Tq + s.window
        rng = wl.Rng(seed, device="cuda")
        d = wl.prefill_chunk_inputs(rng, s, q_begin, Tq, entries, win_cap)
        self.d = d
        w = LayerWeights(d["gamma_kv"], d["gamma_q"], d["bias_kv"], d["sink"], d["bias_idx"])
        self.layer = CsaLayer(self.p, w, d["kv_cache"], d["idx_cache"], d["win_kv"], n_q=Tq)
        i32 = dict(dtype=torch.int32, device="cuda")
        self.tok_pos0 = torch.tensor([d["tok_pos0"]], **i32)
        self.first = torch.tensor([d["first_entry"]], **i32)
        self.new_pos = torch.tensor([q_begin], **i32)
        self.q_pos = torch.arange(q_begin, q_begin + Tq, **i32).view(1, Tq)
        self.out = torch.empty((1, Tq, s.heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        self.tokens = Tq
        # the fused indexer selects the top k as its scores stream; the materialised variant
        # writes the scores and selects them in a separate pass
        self.materialise = bool(cfg.get("materialise"))
        if self.materialise:
            self.scores = torch.empty((1, Tq, entries), dtype=torch.float32, device="cuda")
            self.launches = 8      # 2 compress, window, indexer, top-k, q prep, attention, combine
            self.dominant = "indexer"
        else:
            self.launches = 7      # 2 compress, window, indexer with its top-k, q prep, attention, combine
            self.dominant = "indexer with top-k"
        self.bound = "tensor"
        self._stage_inputs(("tok_v", "tok_z", "tok_vi", "tok_zi", "q", "q_idx", "w_idx"), stage)
        self.host_out = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host_in.values())
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        n_vis = np.array([(q_begin + i + 1) // s.ratio for i in range(Tq)], dtype=np.float64)
        self.dom_flops = float(2.0 * n_vis.sum() * s.idx_heads * s.idx_dim)
        self.dom_bytes = entries * s.idx_dim * 2 + Tq * s.idx_heads * (s.idx_dim * 2 + 4)
        self.step_bytes, self.step_flops = csa_layer_work(s, 1, n_vis, Tq, entries=entries)

    def _select(self):
        L, d = self.layer, self.d
        if self.materialise:
            self.api.csa_indexer_scores(self.p, d["q_idx"], d["w_idx"], L.idx_cache, self.q_pos, self.scores)
            self.api.lca_topk(self.p, self.scores, self.q_pos, self.entries, L.idx)
        else:
            L.select(d["q_idx"], d["w_idx"], self.q_pos)

    def dominant_call(self):
        # the indexer: with its top-k (fused), or writing the scores (materialised)
        if self.materialise:
            d = self.d
            self.api.csa_indexer_scores(self.p, d["q_idx"], d["w_idx"], self.layer.idx_cache, self.q_pos, self.scores)
        else:
            self._select()

    def step(self):
        L, d = self.layer, self.d
        L.compress(d["tok_v"], d["tok_z"], d["tok_vi"], d["tok_zi"], self.tok_pos0, self.first, self.Tq // self.s.ratio)
        L.window(d["tok_v"][:, self.s.ratio:], self.new_pos)
        self._select()
        L.attend(d["q"], self.q_pos, self.out)

    def e2e_step(self):
        self.stage.upload()
        self.step()
        self.host_out.copy_(self.out, non_blocking=True)

    def snapshot_host(self):
        self.kv_host = self.d["kv_cache"][0].cpu()
        self.idx_host = self.d["idx_cache"][0].cpu()
        self.win_host = self.d["win_kv"][0].cpu()
        self.w_host = {k: self.d[k].cpu().numpy() for k in ("gamma_kv", "gamma_q", "bias_kv", "bias_idx", "sink")}

    def cpu_sample(self, budget_s: float) -> dict:
        """Oracle on evenly spaced queries of the chunk (their indexer over ~262K entries dominates),
        with the compression and window rows those queries need."""
        import oracle
        from workloads import bf16_bits
        s = self.s
        kvb = bf16_bits(self.kv_host)
        ixb = bf16_bits(self.idx_host)
        winb = bf16_bits(self.win_host)
        tv, tz = bf16_bits(self.host_in["tok_v"][0]), self.host_in["tok_z"][0].numpy()
        tvi, tzi = bf16_bits(self.host_in["tok_vi"][0]), self.host_in["tok_zi"][0].numpy()
        g = self.w_host["gamma_kv"]
        t_total = 0.0
        # compression of the chunk's entries and its window rows, timed once and charged per query
        t0 = time.perf_counter()
        n_new = self.Tq // s.ratio
        kv_new = oracle.compress(tv, tz, self.d["tok_pos0"], self.w_host["bias_kv"], g, s.rms_eps, s.rope_dims,
                                 s.rope_base, 2 * s.ratio, s.ratio, self.d["first_entry"], n_new)
        k_new = oracle.compress(tvi, tzi, self.d["tok_pos0"], self.w_host["bias_idx"], None, s.rms_eps, 0,
                                s.rope_base, 2 * s.ratio, s.ratio, self.d["first_entry"], n_new)
        rows = [oracle.window_row(tv[s.ratio + t], g, s.rms_eps, s.rope_dims, s.rope_base, self.q_begin + t)
                for t in range(self.Tq)]
        t_shared = time.perf_counter() - t0
        fe = self.d["first_entry"]
        kvb[fe:fe + n_new] = _round_bits(kv_new)
        ixb[fe:fe + n_new] = _round_bits(k_new)
        for t in range(self.Tq):
            winb[(self.q_begin + t) % winb.shape[0]] = _round_bits(rows[t])
        n_done = 0
        for i in np.linspace(0, self.Tq - 1, 32).astype(int):
            pos = self.q_begin + int(i)
            qi = bf16_bits(self.host_in["q_idx"][0, i])
            wi = self.host_in["w_idx"][0, i].numpy()
            q = bf16_bits(self.host_in["q"][0, i])
            t0 = time.perf_counter()
            n_vis = oracle.visible_entries(pos, s.ratio)
            sc = oracle.indexer_scores(qi, wi, ixb, n_vis)
            idx = oracle.topk(sc, s.topk)
            oracle.attend(q, self.w_host["gamma_q"], pos, kvb, self.w_host["sink"], winb, winb.shape[0], s.window,
                          s.rope_dims, s.rope_base, s.rms_eps, self.p.scale, idx=idx)
            t_total += time.perf_counter() - t0
            n_done += 1
            if t_total >= budget_s:
                break
        per_query = t_total / n_done + t_shared / self.Tq
        return dict(value=1.0 / per_query, unit="tokens/s", cores=1, kind="oracle",
                    sample="%d evenly spaced queries of the 8192-query chunk (indexer over ~262K entries, top-%d, "
                           "attention) plus the chunk's compression and window rows charged per query; "
                           "single-threaded fp64, extrapolated per query" % (n_done, s.topk))


def _round_bits(x: np.ndarray) -> np.ndarray:
    from workloads import bf16_bits
    return bf16_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


class BlockDecode(Workload):
    """A V4-Flash-style attention block at decode: alternating CSA and HCA layers, each with its
    own caches, followed by the grouped output projection of its heads.  Layers start from the
    projected per-token inputs (the input projections are not part of the path)."""

    def __init__(self, cfg: dict, seed: int = 0):
        from long_context_attention_04_b300 import api
        self.api = api
        self.cfg = cfg
        B, pos = cfg["B"], cfg["pos"]
        self.B, self.pos = B, pos
        self.layers = []
        n_csa = n_hca = 0
        for i in range(cfg["n_csa"] + cfg["n_hca"]):
            # alternate CSA and HCA layers, CSA first, while both kinds remain
            csa = n_hca >= cfg["n_hca"] or (n_csa < cfg["n_csa"] and n_csa <= n_hca)
            n_csa, n_hca = n_csa + csa, n_hca + (not csa)
            if csa:
                sub = dict(name="CSA layer", B=B, pos=pos, entries=cfg["csa_entries"], shape=cfg["csa"])
                self.layers.append(CsaDecode(sub, seed=seed * 1000 + i, stage=False))
            else:
                sub = dict(name="HCA layer", B=B, pos=pos, entries=cfg["hca_entries"], shape=cfg["hca"])
                self.layers.append(HcaDecode(sub, seed=seed * 1000 + i, stage=False))
        # every layer's per-step inputs in one staging buffer, one group per layer: a copy stream
        # uploads the groups in layer order while the earlier layers compute
        from long_context_attention_04_b300.layers import StagingBuffer
        packed = {(i, k): L.d[k] for i, L in enumerate(self.layers) for k in L.host_in}
        self.stage = StagingBuffer(packed, {i: [(i, k) for k in L.host_in] for i, L in enumerate(self.layers)})
        self.copy_stream = torch.cuda.Stream()
        for (i, k), t in packed.items():
            self.layers[i].d[k] = t
            self.layers[i].host_in[k] = self.stage.host[(i, k)]
        s = cfg["csa"]
        G, d_g, d_model = cfg["groups"], cfg["d_g"], cfg["d_model"]
        self.G = G
        rng = wl.Rng(seed * 1000 + 999, device="cuda")
        self.W = [wl.oproj_weights(rng, s.heads, s.head_dim, G, d_g, d_model) for _ in self.layers]
        self.mid = torch.empty((B, G * d_g), dtype=torch.bfloat16, device="cuda")
        self.y = [torch.empty((B, d_model), dtype=torch.bfloat16, device="cuda") for _ in self.layers]
        self.tokens = B
        self.launches = sum(L.launches for L in self.layers) + 2 * len(self.layers)
        self.dominant = "indexer"
        csa0 = self.layers[0]
        self.dom_bytes, self.dom_flops = csa0.dom_bytes, csa0.dom_flops
        # the layers' own work plus each layer's two projection weight matrices and activations
        w_params = sum(int(W["Wg"].numel() + W["Wm"].numel()) for W in self.W)
        self.step_bytes = sum(L.step_bytes for L in self.layers) + 2 * w_params + \
            len(self.layers) * B * (s.heads * s.head_dim + d_model) * 2
        self.step_flops = sum(L.step_flops for L in self.layers) + 2.0 * B * w_params
        self.host_out = [torch.empty(y.shape, dtype=torch.bfloat16).pin_memory() for y in self.y]
        self.h2d_bytes = sum(L.h2d_bytes for L in self.layers)
        self.d2h_bytes = sum(y.numel() * y.element_size() for y in self.y)

    def dominant_call(self):
        # the indexer of one CSA layer (the largest single read of the block)
        self.layers[0].dominant_call()

    def _oproj(self, i):
        L = self.layers[i]
        self.api.lca_grouped_oproj(L.out.view(self.B, L.s.heads, L.s.head_dim), self.W[i]["Wg"], self.W[i]["Wm"],
                                   self.G, self.mid, self.y[i])

    def step(self):
        for i, L in enumerate(self.layers):
            L.step()
            self._oproj(i)

    def e2e_step(self):
        main, cs = torch.cuda.current_stream(), self.copy_stream
        cs.wait_stream(main)
        ready = []
        for i in range(len(self.layers)):
            self.stage.upload(cs, i)
            ev = torch.cuda.Event()
            ev.record(cs)
            ready.append(ev)
        for i, L in enumerate(self.layers):
            main.wait_event(ready[i])
            L.step()
            self._oproj(i)
            self.host_out[i].copy_(self.y[i], non_blocking=True)
        main.wait_stream(cs)

    def snapshot_host(self):
        self.layers[0].snapshot_host()
        self.layers[1].snapshot_host()
        self.W_host = [{k: v.cpu() for k, v in W.items()} for W in self.W[:2]]

    def cpu_sample(self, budget_s: float) -> dict:
        """The oracle on one sequence of the first CSA and the first HCA layer (with their output
        projections), extrapolated to the whole block: every CSA layer costs the same, and so does
        every HCA layer."""
        import oracle
        from workloads import bf16_bits
        t0 = time.perf_counter()
        c = self.layers[0].cpu_sample(0.0)          # one sequence each (a zero budget stops after one)
        h = self.layers[1].cpu_sample(0.0)
        t1 = time.perf_counter()
        o = np.zeros((64, 512), np.uint16)
        for i in range(2):
            oracle.grouped_oproj(o, bf16_bits(self.W_host[i]["Wg"]), bf16_bits(self.W_host[i]["Wm"]), self.G)
        t2 = time.perf_counter()
        n_csa, n_hca = self.cfg["n_csa"], self.cfg["n_hca"]
        per_token = n_csa / c["value"] + n_hca / h["value"] + (n_csa + n_hca) * (t2 - t1) / 2
        return dict(value=1.0 / per_token, unit="tokens/s", cores=1, kind="oracle",
                    sample="one sequence through the first CSA and the first HCA layer and two output projections "
                           "(%.1f s), extrapolated to %d CSA + %d HCA layers; single-threaded fp64"
                           % (t2 - t0, n_csa, n_hca))


class CsaPrefillProj(CsaPrefill):
    """The CSA prefill chunk preceded by its input projections: the hidden states of the chunk's
    staging tokens (m before the chunk, then the chunk) mapped on the tensor cores to the KV and
    indexer-key token vectors and compressor logits, and those of the chunk's queries to the
    queries, indexer queries and indexer head weights; then the layer as in CsaPrefill."""

    def __init__(self, cfg: dict, seed: int = 0, stage: bool = True):
        super().__init__(cfg, seed, stage=False)
        s, hid, m = self.s, cfg["hidden"], self.s.ratio
        rng = wl.Rng(seed + 7919, device="cuda")
        n_tok = self.Tq + m
        self.hid = hid
        self.x = rng.normal_bf16((n_tok, hid))
        self.W = wl.prefill_projection_weights(rng, s, hid)
        d = self.d
        # the projections write straight into the layer's per-step input buffers
        self.proj = [
            (self.x, self.W["W_kv"], d["tok_v"].view(n_tok, s.head_dim)),
            (self.x, self.W["W_z"], d["tok_z"].view(n_tok, 1)),
            (self.x, self.W["W_ki"], d["tok_vi"].view(n_tok, s.idx_dim)),
            (self.x, self.W["W_zi"], d["tok_zi"].view(n_tok, 1)),
            (self.x[m:], self.W["W_q"], d["q"].view(self.Tq, s.heads * s.head_dim)),
            (self.x[m:], self.W["W_qi"], d["q_idx"].view(self.Tq, s.idx_heads * s.idx_dim)),
            (self.x[m:], self.W["W_w"], d["w_idx"].view(self.Tq, s.idx_heads)),
        ]
        self.launches += len(self.proj)
        self.stage = None
        self.host_in = {"x": self.x.cpu().pin_memory()}
        self.h2d_bytes = self.x.numel() * self.x.element_size()
        proj_flops = 2.0 * hid * (n_tok * (s.head_dim + 1 + s.idx_dim + 1) +
                                  self.Tq * (s.heads * s.head_dim + s.idx_heads * s.idx_dim + s.idx_heads))
        self.step_flops += proj_flops
        self.step_bytes += float(self.x.numel() * 2 + sum(w.numel() * 2 for w in self.W.values()))

    def project(self):
        for A, Wm, C in self.proj:
            self.api.lca_gemm_bf16(A, Wm, C)

    def step(self):
        self.project()
        super().step()

    def e2e_step(self):
        self.x.copy_(self.host_in["x"], non_blocking=True)
        self.step()
        self.host_out.copy_(self.out, non_blocking=True)


class MhcLayer(Workload):
    """Manifold-constrained hyper-connections around one layer: the coefficients and layer input
    (lca_mhc_pre), then, given the layer's output, the new residual streams (lca_mhc_post)."""

    def __init__(self, cfg: dict, seed: int = 0, stage: bool = True):
        from long_context_attention_04_b300 import api
        self.api = api
        self.cfg = cfg
        T, n, d = cfg["T"], cfg["n"], cfg["d"]
        self.T, self.n, self.dim, self.iters = T, n, d, cfg["iters"]
        rng = wl.Rng(seed, device="cuda")
        self.d = wl.mhc_inputs(rng, T, n, d)
        dv = dict(device="cuda")
        self.h = torch.empty((T, d), dtype=torch.bfloat16, **dv)
        self.a = torch.empty((T, n), dtype=torch.float32, **dv)
        self.c = torch.empty((T, n), dtype=torch.float32, **dv)
        self.B = torch.empty((T, n, n), dtype=torch.float32, **dv)
        self.x_out = torch.empty((T, n, d), dtype=torch.bfloat16, **dv)
        self.ws = torch.empty(api.lca_mhc_workspace(T, n), dtype=torch.uint8, **dv)
        self.tokens = T
        self.launches = 3          # generated-logit product, pre mixing (with Sinkhorn-Knopp), post mixing
        self.dominant = "mhc pre + post"
        self._stage_inputs(("x", "y"), stage)
        self.host_out = torch.empty(self.x_out.shape, dtype=torch.bfloat16).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host_in.values())
        self.d2h_bytes = self.x_out.numel() * self.x_out.element_size()
        K = 2 * n + n * n
        # algorithmic bytes: each of the two calls reads the streams once (the layer runs in
        # between), the generating weights once, the layer output once; h and the new streams
        # are written once (the generated logits are a workspace round trip)
        self.step_bytes = float(T * (2 * n * d * 2 + d * 2 + d * 2 + n * d * 2 + (2 * n + n * n) * 4)
                                + K * n * d * 2)
        self.step_flops = 2.0 * T * K * n * d
        self.dom_bytes, self.dom_flops = self.step_bytes, self.step_flops

    def step(self):
        d, api = self.d, self.api
        api.lca_mhc_pre(d["x"], d["phi"], d["bias"], self.h, self.a, self.c, self.B, self.ws, iters=self.iters)
        api.lca_mhc_post(d["x"], self.B, self.c, d["y"], self.x_out)

    def dominant_call(self):
        self.step()

    def e2e_step(self):
        self.stage.upload()
        self.step()
        self.host_out.copy_(self.x_out, non_blocking=True)

    def snapshot_host(self):
        self.host = {k: self.d[k].cpu() for k in ("phi", "bias")}

    def cpu_sample(self, budget_s: float) -> dict:
        import oracle
        from workloads import bf16_bits
        phi = bf16_bits(self.host["phi"])
        bias = self.host["bias"].numpy()
        t_total, n_done = 0.0, 0
        for t in range(self.T):
            x = bf16_bits(self.host_in["x"][t])
            y = bf16_bits(self.host_in["y"][t])
            t0 = time.perf_counter()
            a, c, B = oracle.mhc_coeffs(x, phi, bias, iters=self.iters)
            oracle.mhc_pre(x, a)
            oracle.mhc_post(x, B, c, y)
            t_total += time.perf_counter() - t0
            n_done += 1
            if t_total >= budget_s:
                break
        return dict(value=n_done / t_total, unit="tokens/s", cores=1, kind="oracle",
                    sample="%d of %d tokens (coefficients, layer input, new streams), single-threaded fp64"
                           % (n_done, self.T))


WORKLOADS = {"csa_decode_128k": CsaDecode, "hca_decode_1m": HcaDecode, "csa_prefill_1m": CsaPrefill,
             "csa_prefill_128k": CsaPrefill, "block_decode_1m": BlockDecode, "mhc_prefill_8192": MhcLayer,
             "v4flash_decode_1m": BlockDecode, "csa_prefill_1m_proj": CsaPrefillProj,
             "csa_prefill_1m_scored": CsaPrefill, "csa_decode_128k_fp8": CsaDecode, "hca_decode_1m_fp8": HcaDecode}


# ------------------------------------------------------------------- distributed -----

def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest value over all ranks (the slowest rank's time); identity on one process."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- main -----

def capture(fn) -> torch.cuda.CUDAGraph:
    """Capture fn()'s launches (all on the current stream) into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2, then reads a second one,
    so that the first buffer's dirty lines are written back here, outside the timed span, and
    the step starts on a clean cache holding none of its inputs."""

    def __init__(self, device):
        n = L2_FLUSH_BYTES // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.ones(n, dtype=torch.float32, device=device)
        self.s = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.s)


def time_replays(graph: torch.cuda.CUDAGraph, steps: int, flush: L2Flush, world: int):
    """Device time (ms) of each of `steps` replays, L2 flushed (outside the timed span) before each."""
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_eager(fn, steps: int, flush: L2Flush, world: int):
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def roofline_of(wk, dom_ms: float, peaks: dict, workload: str) -> dict:
    """The dominant call against its roofline (algorithmic bytes or FLOPs per launch / CUDA-event
    time), with the DRAM traffic measured for it while the sources are unchanged."""
    if wk.bound == "hbm":
        achieved = wk.dom_bytes / (dom_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": measured_traffic(workload),
                "kernel": wk.dominant, "algorithmic_bytes": int(wk.dom_bytes), "kernel_ms": round(dom_ms, 4),
                "peak_source": peaks["source"]}
    achieved = wk.dom_flops / (dom_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": measured_traffic(workload),
            "kernel": wk.dominant, "algorithmic_flops": wk.dom_flops, "kernel_ms": round(dom_ms, 4),
            "peak_source": peaks["source"],
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}


def step_roofline_of(wk, step_ms: float, peaks: dict) -> dict:
    """The whole step against its own roofline: all of its algorithmic bytes (or FLOPs, for a
    tensor-bound step) at the measured peak, over the measured step time."""
    if wk.bound == "hbm":
        t = wk.step_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
        return {"bound": "hbm", "algorithmic_bytes": int(wk.step_bytes), "roofline_ms": round(t, 4),
                "frac": round(t / step_ms, 4)}
    t = wk.step_flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    return {"bound": "tensor", "algorithmic_flops": wk.step_flops, "roofline_ms": round(t, 4),
            "frac": round(t / step_ms, 4)}


def measure(name: str, args, flush, world: int, device, rank: int, seed: int, snapshot: bool = False) -> tuple:
    """Builds workload `name`, warms it up and times its step, its dominant call and its end-to-end
    step (CUDA events, L2 flushed before each step); returns (workload, result dict).  With
    `snapshot`, host copies of the state the oracle needs are taken before the first step."""
    cfg = wl.WORKLOADS[name]
    wk = WORKLOADS[name](cfg, seed=seed)
    if snapshot:
        wk.snapshot_host()
    for _ in range(args.warmup):
        wk.step()
    torch.cuda.synchronize()
    step_graph = capture(wk.step)            # the whole step: every launch of the layer
    dom_graph = capture(wk.dominant_call)    # the dominant kernel alone
    step_graph.replay()
    dom_graph.replay()
    with ClockSampler(torch.cuda.current_device()) as clk:
        step_ms = time_replays(step_graph, args.steps, flush, world)
        dom_ms = time_replays(dom_graph, args.steps, flush, world)
    # end to end through the public API: the step with its input copies (pinned host -> device)
    # and its result copy (device -> pinned host), captured once and replayed per step
    from long_context_attention_04_b300.layers import StepGraph
    e2e = StepGraph(wk.e2e_step, warmup=max(1, args.warmup // 2))
    e2e_ms = time_eager(e2e, args.steps, flush, world)
    ms_all = max_over_ranks(float(np.mean(step_ms)), world, device)
    e2e_all = max_over_ranks(float(np.mean(e2e_ms)), world, device)
    dom = float(np.mean(dom_ms))
    from long_context_attention_04_b300 import api
    peaks = measured_peaks()
    res = {
        "workload": cfg["name"],
        "value": round(world * wk.tokens / (ms_all * 1e-3), 1), "unit": "tokens/s",
        "ms_per_step": round(ms_all, 4),
        "roofline": roofline_of(wk, dom, peaks, name),
        "step_roofline": step_roofline_of(wk, ms_all, peaks),
        "e2e": {"value": round(world * wk.tokens / (e2e_all * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": wk.h2d_bytes, "d2h_bytes_per_step": wk.d2h_bytes},
        "gpu_launches": wk.launches * args.steps,
        "clocks": clk.summary(),
        "device_error_word": api.lca_device_error(),
    }
    del step_graph, dom_graph, e2e
    return wk, res


# Target configurations timed beside the headline workload (one process, one GPU): HCA decode at
# 1M context (HBM-bound), the 8192-query CSA prefill chunk at 1M (tensor-bound), the block of
# 8 CSA + 8 HCA layers with output projections at 1M (HBM-bound), the hyper-connection
# mixing around a layer for an 8192-token chunk (HBM-bound), the 43-layer V4-Flash attention
# stack at decode (HBM-bound), and the prefill chunk with its input projections (tensor-bound).
EXTRA_WORKLOADS = ("csa_decode_128k_fp8", "hca_decode_1m", "hca_decode_1m_fp8", "csa_prefill_1m", "csa_prefill_1m_scored",
                   "block_decode_1m", "mhc_prefill_8192", "v4flash_decode_1m", "csa_prefill_1m_proj")


def run_ours(args):
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    from long_context_attention_04_b300 import build as lca_build
    if rank == 0:
        lca_build.build()
    barrier(world)
    cfg = wl.WORKLOADS[args.workload]
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    flush = L2Flush(device)
    wk, res = measure(args.workload, args, flush, world, device, rank, args.seed + rank, snapshot=do_cpu)
    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "dtype_note": "bf16 inputs, caches and outputs; attention products in fp16 (rows re-encoded exactly from "
                      "bf16, the normalised query split into two fp16 parts), fp32 accumulation and softmax; "
                      "indexer in bf16 with fp32 accumulation",
        "data": "synthetic: seeded N(0,1) caches, tokens, queries; N(0,0.02) biases (workloads.py)",
        "config": {"workload": cfg["name"], "name": args.workload, "batch": cfg.get("B", 1),
                   "l2": "caches larger than L2, and L2 flushed before every timed step (512 MiB written, "
                         "then 512 MiB read, outside the timed span)",
                   "timing": "device: CUDA-graph replays of the step, CUDA events; e2e: replays of the step "
                             "captured with its pinned-host input copies and its output copy (StepGraph), all "
                             "inside the timed span"},
        "roofline": res["roofline"],
        "step_roofline": res["step_roofline"],
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"],
        "clocks": res["clocks"],
        "device_error_word": res["device_error_word"],
    }
    if do_cpu:
        line["cpu_baseline"] = wk.cpu_sample(args.cpu_budget)
        if args.all_core_budget > 0:
            line["cpu_baseline"]["all_core"] = all_core_baseline(*oracle_units(args.workload, args.seed),
                                                                 args.all_core_budget)
    del wk
    if world == 1 and not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        extra = {}
        for name in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            wk_x, res_x = measure(name, args, flush, world, device, rank, args.seed)
            del wk_x
            extra[name] = res_x
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:    # pragma: no cover
        return os.cpu_count() or 1


def oracle_all_core(unit, budget_s: float, threads: int) -> float:
    """Units per second of the oracle on `threads` host threads at once, each running `unit()`
    (one token of the workload on shared read-only inputs) until `budget_s` of wall time has
    passed.  The oracle's C calls release the interpreter lock, so the threads run in parallel."""
    counts = [0] * threads
    start = threading.Barrier(threads + 1)
    stop_at = [0.0]

    def work(i):
        start.wait()
        while time.perf_counter() < stop_at[0]:
            unit()
            counts[i] += 1

    pool = [threading.Thread(target=work, args=(i,), daemon=True) for i in range(threads)]
    for t in pool:
        t.start()
    t0 = time.perf_counter()
    stop_at[0] = t0 + budget_s
    start.wait()
    for t in pool:
        t.join()
    return sum(counts) / (time.perf_counter() - t0)


def oracle_units(workload: str, seed: int):
    """One token of `workload` for the oracle on synthetic host inputs of the workload's shapes:
    (object with one_unit() and sample, tokens a unit stands for)."""
    cfg = wl.WORKLOADS[workload]
    if cfg["kind"] == "block_decode":
        # one token through one CSA and one HCA layer per step, scaled to the block's layer count
        parts = [_HostOnly("csa_decode_128k", dict(entries=cfg["csa_entries"], pos=cfg["pos"], shape=cfg["csa"]),
                           seed),
                 _HostOnly("hca_decode_1m", dict(entries=cfg["hca_entries"], pos=cfg["pos"], shape=cfg["hca"]),
                           seed)]
        scale = float(cfg["n_csa"])        # n_csa == n_hca: each step covers 1/n_csa of the block

        class _Pair:
            sample = ("one CSA layer (%d entries) and one HCA layer (%d entries), scaled to %d + %d layers"
                      % (cfg["csa_entries"], cfg["hca_entries"], cfg["n_csa"], cfg["n_hca"]))

            def one_unit(self):
                for p in parts:
                    p.one_unit()
        return _Pair(), scale
    return _HostOnly(workload, cfg, seed), 1.0


def all_core_baseline(wk, scale: float, budget_s: float) -> dict:
    """The oracle on every host core (threads over shared inputs), beside the single-thread figure."""
    wk.one_unit()                       # warm: first-call set-up outside the timed span
    n = host_cores()
    value = oracle_all_core(wk.one_unit, budget_s, n) / scale
    return {"value": round(value, 3), "unit": "tokens/s", "cores": n,
            "sample": "%d threads, each one token at a time (%s) for %.0f s of wall time" % (n, wk.sample, budget_s)}


def run_reference(args):
    """The oracle (CPU, fp64, single thread) as the reference arm: each step is a bounded sample."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    cfg = wl.WORKLOADS[args.workload]
    wk, scale = oracle_units(args.workload, args.seed)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        wk.one_unit()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_unit = float(np.mean(times)) * scale
    value = 1.0 / per_unit
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_unit * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded (workloads.py)",
        "config": {"workload": cfg["name"], "name": args.workload, "batch": cfg.get("B", 1)},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(value, 3), "unit": "tokens/s",
                         "sample": "one token of the workload per step: " + wk.sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if args.all_core_budget > 0:
        line["cpu_baseline"]["all_core"] = all_core_baseline(wk, scale, args.all_core_budget)
    print(json.dumps(line), flush=True)


class _HostOnly:
    """Host-side inputs of one token of a workload for the oracle arm (no GPU touched)."""

    def __init__(self, name, cfg, seed):
        import oracle
        from workloads import bf16_bits
        self.oracle = oracle
        s = cfg.get("shape")
        self.s = s
        rng = wl.Rng(seed)
        self.kind = name
        if name.startswith("mhc"):       # hyper-connections of one token: coefficients, pre, post
            n, d = cfg["n"], cfg["d"]
            K = 2 * n + n * n
            self.iters = cfg["iters"]
            self.x = bf16_bits(rng.normal_bf16((n, d)))
            self.y = bf16_bits(rng.normal_bf16((d,)))
            self.phi = bf16_bits(rng.normal_bf16((K, n * d), 1.0 / math.sqrt(n * d)))
            self.bias = rng.normal_f32((K,)).numpy()
            self.sample = "coefficients (Sinkhorn-Knopp, %d passes), layer input and new streams of one token" \
                % self.iters
            return
        if name.startswith("csa_"):      # a CSA layer: compression, indexer, top-k, attention
            entries = cfg["entries"]
            pos = cfg.get("pos", cfg.get("q_begin", 0) + cfg.get("Tq", 1) - 1)
            self.pos = pos
            self.kv = bf16_bits(rng.normal_bf16((entries, s.head_dim)))
            self.keys = bf16_bits(rng.normal_bf16((entries, s.idx_dim)))
            self.win = bf16_bits(rng.normal_bf16((s.window, s.head_dim)))
            self.tok_v = bf16_bits(rng.normal_bf16((2 * s.ratio, s.head_dim)))
            self.tok_vi = bf16_bits(rng.normal_bf16((2 * s.ratio, s.idx_dim)))
            self.tok_z = rng.normal_f32((2 * s.ratio,)).numpy()
            self.q = bf16_bits(rng.normal_bf16((s.heads, s.head_dim)))
            self.qi = bf16_bits(rng.normal_bf16((s.idx_heads, s.idx_dim)))
            self.wi = (rng.normal_f32((s.idx_heads,)) / math.sqrt(s.idx_heads)).numpy()
            self.sample = "compression, window row, indexer over %d entries, top-%d, attention" % (entries, s.topk)
            self.e4m3 = bool(cfg.get("idx_e4m3"))
            if self.e4m3:               # the key cache in e4m3 (state before the token, not timed)
                self.k8, self.ks = oracle.quantize_rows_e4m3(self.keys)
                self.sample = self.sample.replace("indexer", "e4m3 indexer (keys and queries quantised)")
            self.proj = None
            if "hidden" in cfg:         # the token's input projections come first
                self.proj = {k: bf16_bits(v) for k, v in wl.prefill_projection_weights(rng, s, cfg["hidden"]).items()}
                self.x_row = bf16_bits(rng.normal_bf16((1, cfg["hidden"])))
                self.sample = "input projections from hidden %d, " % cfg["hidden"] + self.sample
        else:
            entries = cfg["entries"]
            self.pos = cfg["pos"]
            self.kv = bf16_bits(rng.normal_bf16((entries, s.head_dim)))
            self.win = bf16_bits(rng.normal_bf16((s.window, s.head_dim)))
            self.tok_v = bf16_bits(rng.normal_bf16((s.ratio, s.head_dim)))
            self.tok_z = rng.normal_f32((s.ratio,)).numpy()
            self.q = bf16_bits(rng.normal_bf16((s.heads, s.head_dim)))
            self.sample = "compression of a %d-token block, window row, attention over %d entries" % (s.ratio, entries)
        self.ones = np.ones(s.head_dim, np.float32)
        self.sink = rng.normal_f32((s.heads,)).numpy()
        self.kv8 = None
        if cfg.get("kv_e4m3"):              # the KV cache in e4m3 (state before the token, not timed)
            self.kv8, self.kvs = oracle.quantize_rows_e4m3(self.kv)
            self.sample += " (e4m3 KV rows)"

    def _attend(self, **kw):
        o, s = self.oracle, self.s
        scale = 1.0 / math.sqrt(s.head_dim)
        if self.kv8 is not None:
            o.quantize_rows_e4m3(self.kv[-1:])                # the new entry's row
            return o.attend_e4m3(self.q, self.ones, self.pos, self.kv8, self.kvs, self.sink, self.win,
                                 self.win.shape[0], s.window, s.rope_dims, s.rope_base, s.rms_eps, scale, **kw)
        return o.attend(self.q, self.ones, self.pos, self.kv, self.sink, self.win, self.win.shape[0], s.window,
                        s.rope_dims, s.rope_base, s.rms_eps, scale, **kw)

    def one_unit(self):
        if getattr(self, "proj", None):
            for W in self.proj.values():
                self.oracle.gemm_bf16(self.x_row, W)
        if self.kind.startswith("mhc"):
            o = self.oracle
            a, c, B = o.mhc_coeffs(self.x, self.phi, self.bias, iters=self.iters)
            o.mhc_pre(self.x, a)
            o.mhc_post(self.x, B, c, self.y)
            return
        o, s = self.oracle, self.s
        span = s.ratio if self.kind.startswith("hca_") else 2 * s.ratio
        bias = np.zeros(span, np.float32)
        p0 = self.pos + 1 - span
        j = (self.pos + 1) // s.ratio - 1
        o.compress(self.tok_v, self.tok_z, p0, bias, self.ones, s.rms_eps, s.rope_dims, s.rope_base, span, s.ratio,
                   j, 1)
        o.window_row(self.tok_v[-1], self.ones, s.rms_eps, s.rope_dims, s.rope_base, self.pos)
        if not self.kind.startswith("hca_"):
            o.compress(self.tok_vi, self.tok_z, p0, bias, None, s.rms_eps, 0, s.rope_base, span, s.ratio, j, 1)
            n_vis = o.visible_entries(self.pos, s.ratio)
            if getattr(self, "e4m3", False):
                o.quantize_rows_e4m3(self.keys[-1:])             # the new key row
                q8, qs = o.quantize_rows_e4m3(self.qi)
                sc = o.indexer_scores_e4m3(q8, qs, self.wi, self.k8, self.ks, n_vis)
            else:
                sc = o.indexer_scores(self.qi, self.wi, self.keys, n_vis)
            idx = o.topk(sc, s.topk)
            self._attend(idx=idx)
        else:
            self._attend(n_dense=o.visible_entries(self.pos, s.ratio))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the chosen workload only (by default the headline run also times %s)"
                    % ", ".join(EXTRA_WORKLOADS))
    ap.add_argument("--all-core-budget", type=float, default=6.0,
                    help="seconds of wall time for the oracle on every host core (0: skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
