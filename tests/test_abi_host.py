"""The C ABI on the host: the library loads, exports every symbol that
include/are.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import all_reduce_epilogue_gb300 as are

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from all_reduce_epilogue_gb300 import build
    build.build()
    return are.load_library()


def test_header_declarations_are_exported(lib):
    text = open(os.path.join(ROOT, "include", "are.h")).read()
    declared = set(re.findall(r"\b(are_[a-z_]+)\s*\(", text))
    assert declared == set(are.EXPORTS), declared ^ set(are.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.are_version() >> 16 == 1


def test_status_strings(lib):
    for s in range(9):
        assert lib.are_status_string(s).decode().startswith("ARE_")


@pytest.mark.parametrize("args,ok", [
    ((are.OP_GEMM_RS, 2, 64, 256, 128), True),
    ((are.OP_GEMM_RS, 4, 8192, 4096, 2048), True),
    ((are.OP_GEMM_RS, 8, 8192, 8192, 4096), True),
    ((are.OP_GEMM_RS, 3, 264, 320, 136), True),
    ((are.OP_GEMM_RS, 0, 64, 256, 128), False),   # R < 1
    ((are.OP_GEMM_RS, 9, 72, 256, 128), False),   # R > 8
    ((are.OP_GEMM_RS, 3, 100, 256, 128), False),  # M % R
    ((are.OP_GEMM_RS, 4, 40, 256, 128), False),   # (M/R) % 8
    ((are.OP_GEMM_RS, 2, 64, 250, 128), False),   # N % 8
    ((are.OP_GEMM_RS, 2, 64, 256, 100), False),   # K % 8
    ((are.OP_GEMM_AR, 8, 64, 7168, 2048), True),
    ((are.OP_GEMM_AR, 8, 65, 7168, 2048), True),  # any M for AR
    ((are.OP_GEMM_AR, 8, 64, 7168, 2047), False),
    ((are.OP_ALLREDUCE_RMSNORM, 8, 4096, 7168, 0), True),
    ((are.OP_ALLREDUCE_RMSNORM, 8, 1, 7168, 0), True),
    ((are.OP_ALLREDUCE_RMSNORM, 8, 1, 7164, 0), False),   # N % 8
    ((are.OP_ALLREDUCE_RMSNORM, 8, 1, 32776, 0), False),  # N too large
    ((are.OP_ALLREDUCE_RMSNORM, 8, -1, 64, 0), False),
    ((99, 1, 8, 8, 8), False),
])
def test_supports(lib, args, ok):
    assert (lib.are_supports(*args) == are.OK) == ok


def test_calls_reject_bad_arguments_without_launching(lib):
    vp = ctypes.c_void_p
    A = (vp * 2)(16, 32)
    # NULL workspace
    assert lib.are_gemm_rs(A, A, A, 2, 64, 256, 128, None, None) == are.EINVAL
    assert lib.are_gemm_ar(A, A, A, 2, 64, 256, 128, None, None) == are.EINVAL
    assert lib.are_allreduce_rmsnorm(A, None, 16, ctypes.c_float(1e-6), 16, 2, 4, 64, None, None) == are.EINVAL
    assert lib.are_allreduce_add_rmsnorm(A, None, 16, ctypes.c_float(1e-6), 16, None, 2, 4, 64, None, None) == are.EINVAL
    assert lib.are_allreduce_rmsnorm_quant(A, None, 16, ctypes.c_float(1e-6), 16, 16, None, 2, 4, 64, None, None) == are.EINVAL
    # bad workspace-independent arguments fail the same way
    assert lib.are_workspace_create(None, None) == are.EINVAL
    assert lib.are_workspace_destroy(None) == are.OK
    assert lib.are_workspace_reset(None) == are.EINVAL
    assert lib.are_workspace_set_oneshot_max_bytes(None, 0) == are.EINVAL


def test_workspace_create_validates_caps(lib):
    h = ctypes.c_void_p()
    bad = are._Caps(0, 64, 64, 64, 0, 0, 0)
    assert lib.are_workspace_create(ctypes.byref(h), ctypes.byref(bad)) == are.EINVAL
    bad = are._Caps(2, 64, 60, 64, 0, 0, 0)  # N_max % 8
    assert lib.are_workspace_create(ctypes.byref(h), ctypes.byref(bad)) == are.EINVAL


def test_no_gpu_means_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    caps = are._Caps(2, 64, 256, 128, 0, 0, 0)
    assert lib.are_workspace_create(ctypes.byref(h), ctypes.byref(caps)) == are.ENODEV
    assert not h.value


def test_missing_library_fails_loudly(tmp_path):
    saved = are._lib
    try:
        are._lib = None
        with pytest.raises(are.AreLibraryMissing):
            are.load_library(str(tmp_path / "nope.so"))
    finally:
        are._lib = saved
