"""The C ABI library builds for sm_103a, loads, exports what include/tt_emb.h
declares, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import tensor_train_compressed_embeddingbag_gb300 as tt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tt_emb.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tt_emb_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    tt.build()
    return tt.load_library()


def test_header_declares_the_binding_names():
    assert header_functions() == sorted(tt.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", tt.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tt_emb_\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert getattr(lib, name)


def test_debug_library_exports_the_same_symbols():
    """libttemb_debug.so (the kernels' index checks compiled in) offers the same C ABI."""
    path = tt.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tt_emb_\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name


def test_build_targets_sm_103a_only():
    from tensor_train_compressed_embeddingbag_gb300 import _nvcc_build as b

    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(9):
        s = tt.tt_emb_status_string(code)
        assert isinstance(s, str) and s
    assert "index" in tt.tt_emb_status_string(tt.TT_ERR_INDEX)
    assert "debug" in tt.tt_emb_status_string(tt.TT_ERR_BOUNDS)


def _create(lib, E, p, q, r, cores=(256, 512, 768)):
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 3)(*cores)
    st = lib.tt_emb_create(E, (ctypes.c_int64 * 3)(*p), (ctypes.c_int32 * 3)(*q), (ctypes.c_int32 * 2)(*r),
                           ptrs, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize(
    "E,p,q,r",
    [
        (121, [4, 5, 6], [2, 2, 2], [4, 4]),     # p1 p2 p3 < E
        (0, [4, 5, 6], [2, 2, 2], [4, 4]),       # no rows
        (100, [4, 0, 6], [2, 2, 2], [4, 4]),     # zero factor
        (100, [4, 5, 6], [2, 2, 2], [0, 4]),     # rank 0
        (100, [4, 5, 6], [2, 2, 2], [4, 129]),   # rank above the limit
        (100, [4, 5, 6], [8, 8, 8], [4, 4]),     # D = 512 above the limit
    ],
)
def test_bad_shapes_rejected_before_any_cuda_call(lib, E, p, q, r):
    st, h = _create(lib, E, p, q, r)
    assert st == tt.TT_ERR_SHAPE
    assert not h.value


def test_null_arguments_rejected(lib):
    st, h = _create(lib, 120, [4, 5, 6], [2, 2, 2], [4, 4], cores=(256, 0, 256))
    assert st == tt.TT_ERR_ARG
    # cores must be 16-byte aligned (the kernels read them as float4)
    st, h = _create(lib, 120, [4, 5, 6], [2, 2, 2], [4, 4], cores=(256, 260, 256))
    assert st == tt.TT_ERR_ARG
    assert not h.value
    h = ctypes.c_void_p()
    assert lib.tt_emb_batch_create(0, None, ctypes.byref(h)) == tt.TT_ERR_ARG
    assert lib.tt_emb_forward(None, None, 0, None, 0, None, 0, None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_backward(None, None, ctypes.c_float(0.1), None) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(None, tt.TT_OPT_SGD, ctypes.c_float(0.0), None) == tt.TT_ERR_ARG
    assert lib.tt_emb_full_weight(None, 0, 0, 1, None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_lfu_enable(None, 64, 64) == tt.TT_ERR_ARG
    assert lib.tt_emb_lfu_populate(None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_lfu_disable(None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_set_trainable(None, 1, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_read(None, None, None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_write(None, None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_populate(None, None, 0, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_disable(None) == tt.TT_ERR_ARG
    assert lib.tt_emb_reserve(None, 1, 1) == tt.TT_ERR_ARG
    assert lib.tt_emb_get_last_error(None) == tt.TT_ERR_ARG
    assert lib.tt_emb_last_launch_count(None, 0) == -1
    lib.tt_emb_destroy(None)


def test_valid_shape_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _create(lib, 120, [4, 5, 6], [2, 2, 2], [4, 4])
    assert st == tt.TT_ERR_CUDA
    assert not h.value


def test_product_path_has_no_fallback(tmp_path, monkeypatch):
    """Without the built library the binding raises instead of computing anything."""
    import importlib

    mod = importlib.import_module("tensor_train_compressed_embeddingbag_gb300")
    monkeypatch.setattr(mod, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        mod.load_library()
