"""Host-side checks of the C ABI: the library builds and loads, exports every function
include/lca.h declares, and rejects bad arguments before launching anything (these calls
return from host validation, so they need no GPU)."""
import ctypes
import subprocess

import pytest

from long_context_attention_04_b300 import _lib, build as lca_build


@pytest.fixture(scope="module")
def lib():
    lca_build.build()
    return _lib.load()


def test_every_declared_function_is_exported(lib):
    declared = _lib.declared_functions()
    assert len(declared) >= 17
    out = subprocess.run(["nm", "-D", "--defined-only", lca_build.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    for n in declared:
        assert hasattr(lib, n)
    # nothing but the ABI is exported from the library's own code
    ours = {n for n in exported if n.startswith(("lca", "csa", "hca"))}
    assert ours == set(declared)


def test_binding_signatures_cover_the_header():
    assert set(_lib.SIGNATURES) == set(_lib.declared_functions())


def _params(**kw):
    base = dict(heads=64, head_dim=512, rope_dims=64, rope_base=1e4, rms_eps=1e-6, softmax_scale=0.0,
                window=128, ratio=4, topk=512, idx_heads=64, idx_dim=128)
    base.update(kw)
    return _lib.lca_attn_params(*base.values())


FAKE = ctypes.c_void_p(0x10000)        # aligned, never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10002)


def _attend(lib, p, entry="csa_attend", **over):
    args = dict(p=ctypes.byref(p), batch=1, n_q=1, q=FAKE, gamma=FAKE, pos=FAKE, kv=FAKE, kv_bs=0,
                rows=1000, idx=FAKE, win=FAKE, win_bs=0, win_cap=128, sink=FAKE, out=FAKE, lse=None,
                ws=FAKE, ws_bytes=0, stream=None)
    args.update(over)
    return getattr(lib, entry)(*args.values())


def test_attend_rejects_bad_arguments(lib):
    assert _attend(lib, _params(), q=None) == 1                       # NULL
    assert _attend(lib, _params(), q=FAKE_ODD) == 1                   # misaligned
    assert _attend(lib, _params(head_dim=192)) == 2                   # unsupported c
    assert _attend(lib, _params(heads=65)) == 2                       # too many heads
    assert _attend(lib, _params(rope_dims=3)) == 2                    # odd R
    assert _attend(lib, _params(), win_cap=64) == 1                   # ring smaller than W
    assert _attend(lib, _params(), batch=0) == 1
    assert _attend(lib, _params(), ws_bytes=16) == 3                  # workspace too small
    assert b"workspace" in lib.lca_last_error()
    assert _attend(lib, _params(), idx=None) == 1


@pytest.mark.parametrize("entry", ["csa_attend_prepare", "csa_attend_prepared"])
def test_attention_halves_validate_like_the_whole_call(lib, entry):
    assert _attend(lib, _params(), entry, q=None) == 1
    assert _attend(lib, _params(head_dim=192), entry) == 2
    assert _attend(lib, _params(), entry, ws_bytes=16) == 3
    assert _attend(lib, _params(), entry, idx=None) == 1
    assert entry.encode() in lib.lca_last_error()


def test_workspace_sizes_are_positive_and_monotone(lib):
    p = _params()
    a = lib.csa_attend_workspace(ctypes.byref(p), 32, 1)
    b = lib.hca_attend_workspace(ctypes.byref(p), 16, 1, 8192)
    c = lib.csa_indexer_workspace(ctypes.byref(p), 32, 1, 32768)
    assert a > 0 and b > 0 and c >= 32 * 32768 * 4
    assert lib.csa_attend_workspace(ctypes.byref(p), 0, 1) == 0


def test_compress_and_indexer_reject_bad_arguments(lib):
    p = _params()
    # width not a multiple of 8
    assert lib.csa_compress_kv(ctypes.byref(p), 1, 100, FAKE, 0, 8, FAKE, 0, FAKE, FAKE, None, 0, FAKE, 1, FAKE,
                               0, 10, None) == 2
    # NULL cache
    assert lib.hca_compress_kv(ctypes.byref(p), 1, 512, FAKE, 0, 8, FAKE, 0, FAKE, FAKE, None, 0, FAKE, 1, None,
                               0, 10, None) == 1
    # window wider than the kernel's limit (m' = 512 -> span 512)
    assert lib.hca_compress_kv(ctypes.byref(_params(ratio=512)), 1, 512, FAKE, 0, 8, FAKE, 0, FAKE, FAKE, None,
                               0, FAKE, 1, FAKE, 0, 10, None) == 2
    # indexer: scores stride below cache rows
    assert lib.csa_indexer_scores(ctypes.byref(p), 1, 1, FAKE, FAKE, FAKE, 0, 1000, FAKE, FAKE, 996, None) == 1
    # indexer + top-k: workspace too small
    assert lib.csa_indexer_topk(ctypes.byref(p), 1, 1, FAKE, FAKE, FAKE, 0, 1000, FAKE, FAKE, FAKE, 100,
                                None) == 3
    # top-k: k = 0
    assert lib.lca_topk(ctypes.byref(_params(topk=0)), 1, 1, FAKE, 1000, FAKE, 1000, FAKE, None) == 1


def test_projection_rejects_bad_arguments(lib):
    assert lib.lca_gemm_bf16(0, 8, 64, FAKE, 64, FAKE, 64, FAKE, 8, None) == 2      # M = 0
    assert lib.lca_gemm_bf16(17, 8, 64, FAKE, 60, FAKE, 64, FAKE, 8, None) == 1     # lda % 8
    assert lib.lca_gemm_bf16_f32(17, 8, 64, FAKE, 64, FAKE, 64, None, 8, None) == 1  # NULL C
    assert lib.lca_gemm_bf16(4, 8, 60, FAKE, 64, FAKE, 64, FAKE, 8, None) == 2      # K % 8
    assert lib.lca_grouped_oproj(4, 64, 512, 7, 1024, 4096, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.lca_status_string(3) == b"workspace too small"


def test_null_and_zero_arguments_are_errors_not_crashes(lib):
    """Every entry point called with NULL pointers and zero sizes returns an error status (or a
    zero workspace size) from host validation, without touching memory."""
    for name, (argtypes, restype) in sorted(_lib.SIGNATURES.items()):
        if name in ("lca_version", "lca_status_string", "lca_last_error", "lca_device_error", "lca_test_hooks"):
            continue
        args = [None if t is ctypes.c_void_p or hasattr(t, "_type_") and not t.__name__.startswith("c_")
                else 0 for t in argtypes]
        r = getattr(lib, name)(*args)
        if name.endswith("_workspace"):
            assert r == 0, name
        else:
            assert r in (1, 2), (name, r)
