"""ctypes view of liblca.so (the C ABI declared in include/lca.h)."""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB_PATH, ROOT

HEADER = os.path.join(ROOT, "include", "lca.h")

c_int, c_float, c_size_t, c_int64, c_void_p = (ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                               ctypes.c_int64, ctypes.c_void_p)


class lca_attn_params(ctypes.Structure):
    _fields_ = [
        ("heads", c_int), ("head_dim", c_int), ("rope_dims", c_int),
        ("rope_base", c_float), ("rms_eps", c_float), ("softmax_scale", c_float),
        ("window", c_int), ("ratio", c_int), ("topk", c_int),
        ("idx_heads", c_int), ("idx_dim", c_int),
    ]


class lca_compress_variant(ctypes.Structure):
    _fields_ = [("per_channel", c_int), ("e4m3", c_int), ("cache_scale", c_void_p), ("scale_batch_stride", c_int64)]


P = ctypes.POINTER(lca_attn_params)
CV = ctypes.POINTER(lca_compress_variant)
V = c_void_p

# argument types of every entry point, in header order
SIGNATURES = {
    "csa_compress_kv": ([P, c_int, c_int, V, c_int64, c_int, V, c_int64, V, V, V, c_int, V, c_int, V, c_int64,
                         c_int64, V], c_int),
    "hca_compress_kv": ([P, c_int, c_int, V, c_int64, c_int, V, c_int64, V, V, V, c_int, V, c_int, V, c_int64,
                         c_int64, V], c_int),
    "lca_window_update": ([P, c_int, V, c_int64, c_int, V, V, V, c_int64, c_int, V], c_int),
    "csa_indexer_scores": ([P, c_int, c_int, V, V, V, c_int64, c_int64, V, V, c_int64, V], c_int),
    "lca_topk": ([P, c_int, c_int, V, c_int64, V, c_int64, V, V], c_int),
    "csa_indexer_workspace": ([P, c_int, c_int, c_int64], c_size_t),
    "csa_indexer_topk": ([P, c_int, c_int, V, V, V, c_int64, c_int64, V, V, V, c_size_t, V], c_int),
    "csa_attend_workspace": ([P, c_int, c_int], c_size_t),
    "hca_attend_workspace": ([P, c_int, c_int, c_int64], c_size_t),
    "csa_attend": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, V, c_int64, c_int, V, V, V, V, c_size_t, V],
                   c_int),
    "hca_attend": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, c_int64, c_int, V, V, V, V, c_size_t, V],
                   c_int),
    "csa_attend_prepare": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, V, c_int64, c_int, V, V, V, V, c_size_t,
                            V], c_int),
    "csa_attend_prepared": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, V, c_int64, c_int, V, V, V, V, c_size_t,
                             V], c_int),
    "hca_attend_prepare": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, c_int64, c_int, V, V, V, V, c_size_t, V],
                           c_int),
    "hca_attend_prepared": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, c_int64, c_int, V, V, V, V, c_size_t,
                             V], c_int),
    "hca_attend_noalloc": ([P, c_int, c_int, V, V, V, V, c_int64, c_int64, V, c_int64, c_int, V, V, V, V], c_int),
    "lca_grouped_oproj": ([c_int, c_int, c_int, c_int, c_int, c_int, V, V, V, V, V, V], c_int),
    "lca_gemm_bf16": ([c_int, c_int, c_int, V, c_int64, V, c_int64, V, c_int64, V], c_int),
    "lca_gemm_bf16_f32": ([c_int, c_int, c_int, V, c_int64, V, c_int64, V, c_int64, V], c_int),
    "lca_mhc_workspace": ([c_int, c_int], c_size_t),
    "lca_mhc_pre": ([c_int, c_int, c_int, c_int, V, V, V, V, V, V, V, V, c_size_t, V], c_int),
    "lca_mhc_post": ([c_int, c_int, c_int, V, V, V, V, V, V], c_int),
    "lca_quantize_rows_e4m3": ([V, c_int64, c_int, V, V, V], c_int),
    "csa_compress_kv_ex": ([P, CV, c_int, c_int, V, c_int64, c_int, V, c_int64, V, V, V, c_int, V, c_int, V, c_int64,
                            c_int64, V], c_int),
    "hca_compress_kv_ex": ([P, CV, c_int, c_int, V, c_int64, c_int, V, c_int64, V, V, V, c_int, V, c_int, V, c_int64,
                            c_int64, V], c_int),
    "csa_indexer_scores_e4m3": ([P, c_int, c_int, V, V, V, V, c_int64, V, c_int64, c_int64, V, V, c_int64, V], c_int),
    "csa_indexer_topk_e4m3": ([P, c_int, c_int, V, V, V, V, c_int64, V, c_int64, c_int64, V, V, V, c_size_t, V],
                              c_int),
    "csa_attend_e4m3": ([P, c_int, c_int, V, V, V, V, c_int64, V, c_int64, c_int64, V, V, c_int64, c_int, V, V, V, V,
                         c_size_t, V], c_int),
    "hca_attend_e4m3": ([P, c_int, c_int, V, V, V, V, c_int64, V, c_int64, c_int64, V, c_int64, c_int, V, V, V, V,
                         c_size_t, V], c_int),
    "lca_status_string": ([c_int], ctypes.c_char_p),
    "lca_last_error": ([], ctypes.c_char_p),
    "lca_device_error": ([V, ctypes.POINTER(ctypes.c_uint32)], c_int),
    "lca_test_hooks": ([ctypes.c_longlong, c_int], c_int),
    "lca_version": ([], ctypes.c_char_p),
}


def declared_functions() -> list[str]:
    """Names of the functions include/lca.h declares (parsed from the header text)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "return")]


_lib = None


def load() -> ctypes.CDLL:
    """Load liblca.so; raises if it has not been built (there is no other implementation)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("liblca.so is not built (%s); run long_context_attention_04_b300.build.build() "
                               "or __graft_entry__.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib
