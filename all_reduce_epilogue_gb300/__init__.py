"""GB300-native tensor-parallel row-parallel linear epilogue.

Thin Python binding of ``libare.so`` (C ABI in ``include/are.h``): argument
marshalling only.  Every step of the computation runs in the library's CUDA
kernels; PyTorch supplies device memory and streams.  There is no CPU path:
calling any operation without the built library raises ``AreLibraryMissing``.

Operations (the same names as the C ABI, without the ``are_`` prefix):

* ``gemm_rs(A, B, out, ws)``      R partial GEMMs, ring-order fp32 sum,
  reduce-scattered into R owner row segments (bf16).
* ``gemm_ar(A, B, out, ws)``      R partial GEMMs rounded to bf16, all-reduced
  into every rank view.
* ``allreduce_rmsnorm(partials, residual, gamma, eps, out, ws)``
  all-reduce + residual + RMSNorm in one Lamport-synchronised kernel.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libare.so")

# status codes (are_status)
OK, EINVAL, ENOMEM, ECUDA, ETIMEOUT, EBUSY, ENODEV, ECAPACITY, ECAPTURE = range(9)
# ops
OP_GEMM_RS, OP_GEMM_AR, OP_ALLREDUCE_RMSNORM = 1, 2, 3
# debug flags
DEBUG_NO_REARM, DEBUG_LOG_PIECES, DEBUG_COUNT_CANON, DEBUG_SKIP_PUBLISH, DEBUG_SKIP_STAGE = 1, 2, 4, 8, 16
DEBUG_SINGLE_CTA, DEBUG_WAIT_PROFILE, DEBUG_AR_ONESHOT, DEBUG_AR_LAMPORT, DEBUG_PAIR_CTA = 32, 64, 128, 256, 512
DEBUG_RS_RING, DEBUG_RS_SPLIT = 1024, 2048
# device status codes
DEV_OK, DEV_MASK_TIMEOUT, DEV_STAGE_TIMEOUT, DEV_PIPE_TIMEOUT = 0, 1, 2, 3
# snapshot kinds
SNAP_MASKS, SNAP_STAGING, SNAP_PIECES, SNAP_COUNTERS, SNAP_CHUNKS = 1, 2, 3, 4, 5
CHUNK_CAP = 64          # chunk counters per owner segment in the workspace
CHUNK_Q = 1 << 32       # counter advance per completed chunk
# kernels (are_kernel), as reported by Workspace.last_launch()
KERNEL_NAMES = {0: "none", 1: "memset", 2: "gemm_reduce_kernel", 3: "gemm_pair_kernel", 4: "ar_rmsnorm_kernel",
                5: "ar_oneshot_kernel"}
PIECE_WORDS = 64
TILE_M, TILE_N = 128, 256

# Every C-ABI symbol declared in include/are.h.
EXPORTS = [
    "are_version", "are_status_string", "are_supports", "are_workspace_create", "are_workspace_destroy",
    "are_workspace_reset", "are_workspace_set_debug", "are_workspace_set_oneshot_max_bytes",
    "are_workspace_set_gemm_order", "are_workspace_set_chunks", "are_chunk_generation", "are_chunk_wait",
    "are_get_device_status", "are_debug_snapshot", "are_debug_last_launch",
    "are_gemm_rs", "are_gemm_ar", "are_allreduce_rmsnorm", "are_allreduce_add_rmsnorm", "are_allreduce_rmsnorm_quant",
    "are_allreduce_rmsnorm_noalloc", "are_noalloc_device_status",
]


class AreError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class AreLibraryMissing(RuntimeError):
    pass


class _Caps(ctypes.Structure):
    _fields_ = [("R_max", ctypes.c_int32), ("M_max", ctypes.c_int64), ("N_max", ctypes.c_int64),
                ("K_max", ctypes.c_int64), ("timeout_ns", ctypes.c_uint64), ("debug_flags", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class _DevStatus(ctypes.Structure):
    _fields_ = [("code", ctypes.c_uint32), ("where", ctypes.c_uint32), ("a", ctypes.c_int32), ("b", ctypes.c_int32)]


class _LaunchInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("cluster", ctypes.c_int32), ("rank_block", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("rank_group", ctypes.c_int32), ("group_m", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load ``libare.so`` (idempotent).  Raises AreLibraryMissing if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise AreLibraryMissing(
            f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
    lib.are_version.restype = i32
    lib.are_status_string.restype = ctypes.c_char_p
    lib.are_status_string.argtypes = [i32]
    lib.are_supports.restype = i32
    lib.are_supports.argtypes = [i32, i32, i64, i64, i64]
    lib.are_workspace_create.restype = i32
    lib.are_workspace_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(_Caps)]
    lib.are_workspace_destroy.restype = i32
    lib.are_workspace_destroy.argtypes = [vp]
    lib.are_workspace_reset.restype = i32
    lib.are_workspace_reset.argtypes = [vp]
    lib.are_workspace_set_debug.restype = i32
    lib.are_workspace_set_debug.argtypes = [vp, u32, i64]
    lib.are_workspace_set_oneshot_max_bytes.restype = i32
    lib.are_workspace_set_oneshot_max_bytes.argtypes = [vp, u64]
    lib.are_workspace_set_gemm_order.restype = i32
    lib.are_workspace_set_gemm_order.argtypes = [vp, i32, i32, i32]
    lib.are_workspace_set_chunks.restype = i32
    lib.are_workspace_set_chunks.argtypes = [vp, i32, i32]
    lib.are_chunk_generation.restype = i32
    lib.are_chunk_generation.argtypes = [vp, ctypes.POINTER(u64)]
    lib.are_chunk_wait.restype = i32
    lib.are_chunk_wait.argtypes = [vp, i32, i32, u64, u64]
    lib.are_get_device_status.restype = i32
    lib.are_get_device_status.argtypes = [vp, ctypes.POINTER(_DevStatus)]
    lib.are_debug_snapshot.restype = i32
    lib.are_debug_snapshot.argtypes = [vp, i32, vp, ctypes.c_size_t]
    lib.are_debug_last_launch.restype = i32
    lib.are_debug_last_launch.argtypes = [vp, ctypes.POINTER(_LaunchInfo)]
    lib.are_noalloc_device_status.restype = i32
    lib.are_noalloc_device_status.argtypes = [ctypes.POINTER(_DevStatus)]
    for name in ("are_gemm_rs", "are_gemm_ar"):
        f = getattr(lib, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp]
    lib.are_allreduce_rmsnorm.restype = i32
    lib.are_allreduce_rmsnorm.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i64, i64, vp, vp]
    lib.are_allreduce_add_rmsnorm.restype = i32
    lib.are_allreduce_add_rmsnorm.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, i32, i64, i64, vp, vp]
    lib.are_allreduce_rmsnorm_quant.restype = i32
    lib.are_allreduce_rmsnorm_quant.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i64, i64, vp, vp]
    lib.are_allreduce_rmsnorm_noalloc.restype = i32
    lib.are_allreduce_rmsnorm_noalloc.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i64, i64, vp]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().are_status_string(status).decode()
    except AreLibraryMissing:
        return f"status {status}"


def version() -> int:
    return load_library().are_version()


def supports(op: int, R: int, M: int, N: int, K: int = 0) -> bool:
    return load_library().are_supports(op, R, M, N, K) == OK


def _check(status: int, what: str):
    if status != OK:
        raise AreError(status, what)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptrs(tensors) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _check_bf16(t, what: str):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA bfloat16 tensor")


class Workspace:
    """Device workspace (tile masks, partial buffer, armed staging, status word).

    Sized once from the capacities; use one workspace per stream."""

    def __init__(self, R_max: int, M_max: int, N_max: int, K_max: int = 0, timeout_ns: int = 0,
                 debug_flags: int = 0):
        lib = load_library()
        caps = _Caps(R_max, M_max, N_max, K_max, timeout_ns, debug_flags, 0)
        h = ctypes.c_void_p()
        _check(lib.are_workspace_create(ctypes.byref(h), ctypes.byref(caps)), "are_workspace_create")
        self._h = h
        self.caps = dict(R_max=R_max, M_max=M_max, N_max=N_max, K_max=K_max)

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("workspace is closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            load_library().are_workspace_destroy(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        _check(load_library().are_workspace_reset(self.handle), "are_workspace_reset")

    def set_debug(self, flags: int, arg: int = -1):
        _check(load_library().are_workspace_set_debug(self.handle, flags, arg), "are_workspace_set_debug")

    def set_oneshot_max_bytes(self, nbytes: int):
        """Per-rank input size (M*N*2 bytes) up to which allreduce_rmsnorm uses
        its one-shot kernel (0: always the Lamport kernel)."""
        _check(load_library().are_workspace_set_oneshot_max_bytes(self.handle, nbytes),
               "are_workspace_set_oneshot_max_bytes")

    def device_status(self) -> dict:
        st = _DevStatus()
        rc = load_library().are_get_device_status(self.handle, ctypes.byref(st))
        if rc not in (OK, ETIMEOUT):
            raise AreError(rc, "are_get_device_status")
        return {"status": rc, "code": st.code, "where": st.where, "a": st.a, "b": st.b}

    def last_launch(self) -> dict:
        """Which kernel the last operation on this workspace launched, and its
        launch shape (host-side record; no device access)."""
        li = _LaunchInfo()
        _check(load_library().are_debug_last_launch(self.handle, ctypes.byref(li)), "are_debug_last_launch")
        return {"kernel": KERNEL_NAMES.get(li.kernel, str(li.kernel)), "grid": li.grid, "block": li.block,
                "cluster": li.cluster, "rank_block": li.rank_block, "variant": li.variant,
                "rank_group": li.rank_group, "group_m": li.group_m}

    def set_gemm_order(self, group_m: int = 0, block_pairs: int = 0, rank_group: int = 0):
        """Order of the CTA-pair GEMM kernel's work units (0 = the library's
        choice; block_pairs < 0 = a pair's R units consecutive).  Results do
        not depend on it."""
        _check(load_library().are_workspace_set_gemm_order(self.handle, group_m, block_pairs, rank_group),
               "are_workspace_set_gemm_order")

    def set_chunks(self, chunks: int, stripe: int = 0):
        """GEMM+RS chunked owner-segment completion: `chunks` per segment (0 =
        off); `stripe` 0 = destination-rotated chunk-major order, > 0 = striped,
        -1 = the usual order."""
        _check(load_library().are_workspace_set_chunks(self.handle, chunks, stripe), "are_workspace_set_chunks")

    def chunk_generation(self) -> int:
        g = ctypes.c_uint64()
        _check(load_library().are_chunk_generation(self.handle, ctypes.byref(g)), "are_chunk_generation")
        return g.value

    def chunk_wait(self, segment: int, chunk: int, generation: int, timeout_ns: int = 1_000_000_000) -> bool:
        """Host-side wait for a chunk to reach `generation`; False on timeout."""
        rc = load_library().are_chunk_wait(self.handle, segment, chunk, generation, timeout_ns)
        if rc not in (OK, ETIMEOUT):
            raise AreError(rc, "are_chunk_wait")
        return rc == OK

    def chunk_counters(self):
        """[R_max, CHUNK_CAP] uint64 completion counters (synchronises)."""
        import numpy as np
        n = self.caps["R_max"] * CHUNK_CAP * 8
        return self.snapshot(SNAP_CHUNKS, n).view(np.uint64).reshape(self.caps["R_max"], CHUNK_CAP)

    def snapshot(self, kind: int, nbytes: int):
        import numpy as np
        buf = np.empty(nbytes, dtype=np.uint8)
        _check(load_library().are_debug_snapshot(self.handle, kind, buf.ctypes.data, nbytes), "are_debug_snapshot")
        return buf


def gemm_rs(A: Sequence, B: Sequence, out, ws: Workspace, stream=None):
    """out[s] = rows [s*M/R, (s+1)*M/R) of bf16(sum_r A[r] @ B[r]).

    ``out`` is either a list of R segment tensors [M/R, N] or one [M, N]
    tensor (segments are then its consecutive row bands)."""
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    for t in list(A) + list(B):
        _check_bf16(t, "A/B")
    if isinstance(out, (list, tuple)):
        segs = list(out)
        for t in segs:
            _check_bf16(t, "out")
        seg_ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() for t in segs])
    else:
        _check_bf16(out, "out")
        S = M // R if R else 0
        seg_ptrs = (ctypes.c_void_p * R)(*[out.data_ptr() + s * S * N * 2 for s in range(R)])
    rc = load_library().are_gemm_rs(_ptrs(A), _ptrs(B), seg_ptrs, R, M, N, K, ws.handle, _stream_handle(stream))
    _check(rc, "are_gemm_rs")


def gemm_ar(A: Sequence, B: Sequence, out, ws: Workspace, stream=None):
    """Every view out[v] = bf16(sum_r f32(bf16(A[r] @ B[r]))).

    ``out`` is a list of R [M, N] views (they may alias) or one tensor used
    for every view."""
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    for t in list(A) + list(B):
        _check_bf16(t, "A/B")
    views = list(out) if isinstance(out, (list, tuple)) else [out] * R
    for t in views:
        _check_bf16(t, "out")
    rc = load_library().are_gemm_ar(_ptrs(A), _ptrs(B), _ptrs(views), R, M, N, K, ws.handle, _stream_handle(stream))
    _check(rc, "are_gemm_ar")


def allreduce_rmsnorm(partials: Sequence, residual, gamma, eps: float, out, ws: Workspace, stream=None):
    """out = bf16(rmsnorm(sum_r partials[r] + residual) * gamma)."""
    import torch
    R = len(partials)
    M, N = partials[0].shape
    for t in partials:
        _check_bf16(t, "partials")
    if residual is not None:
        _check_bf16(residual, "residual")
    _check_bf16(out, "out")
    if gamma.dtype != torch.float32 or not gamma.is_cuda or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous CUDA float32 tensor")
    rc = load_library().are_allreduce_rmsnorm(
        _ptrs(partials), residual.data_ptr() if residual is not None else None, gamma.data_ptr(), float(eps),
        out.data_ptr(), R, M, N, ws.handle, _stream_handle(stream))
    _check(rc, "are_allreduce_rmsnorm")


def allreduce_add_rmsnorm(partials: Sequence, residual, gamma, eps: float, out, residual_out, ws: Workspace,
                          stream=None):
    """As ``allreduce_rmsnorm``, and residual_out = bf16(sum_r partials[r] +
    residual), the residual the next layer takes (may be ``residual`` itself)."""
    import torch
    R = len(partials)
    M, N = partials[0].shape
    for t in partials:
        _check_bf16(t, "partials")
    if residual is not None:
        _check_bf16(residual, "residual")
    _check_bf16(out, "out")
    if residual_out is not None:
        _check_bf16(residual_out, "residual_out")
    if gamma.dtype != torch.float32 or not gamma.is_cuda or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous CUDA float32 tensor")
    rc = load_library().are_allreduce_add_rmsnorm(
        _ptrs(partials), residual.data_ptr() if residual is not None else None, gamma.data_ptr(), float(eps),
        out.data_ptr(), residual_out.data_ptr() if residual_out is not None else None, R, M, N, ws.handle,
        _stream_handle(stream))
    _check(rc, "are_allreduce_add_rmsnorm")


def allreduce_rmsnorm_quant(partials: Sequence, residual, gamma, eps: float, out_q, out_scale, ws: Workspace,
                            residual_out=None, stream=None):
    """Quantising variant: out_q (uint8 FP8 E4M3 codes [M, N]) and out_scale
    (fp32 [M]) with y ~= e4m3(out_q) * out_scale per row; residual_out optional."""
    import torch
    R = len(partials)
    M, N = partials[0].shape
    for t in partials:
        _check_bf16(t, "partials")
    if residual is not None:
        _check_bf16(residual, "residual")
    if residual_out is not None:
        _check_bf16(residual_out, "residual_out")
    if out_q.dtype != torch.uint8 or not out_q.is_cuda or not out_q.is_contiguous():
        raise ValueError("out_q must be a contiguous CUDA uint8 tensor")
    if out_scale.dtype != torch.float32 or not out_scale.is_cuda or not out_scale.is_contiguous():
        raise ValueError("out_scale must be a contiguous CUDA float32 tensor")
    if gamma.dtype != torch.float32 or not gamma.is_cuda or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous CUDA float32 tensor")
    rc = load_library().are_allreduce_rmsnorm_quant(
        _ptrs(partials), residual.data_ptr() if residual is not None else None, gamma.data_ptr(), float(eps),
        out_q.data_ptr(), out_scale.data_ptr(), residual_out.data_ptr() if residual_out is not None else None,
        R, M, N, ws.handle, _stream_handle(stream))
    _check(rc, "are_allreduce_rmsnorm_quant")


def allreduce_rmsnorm_noalloc(partials: Sequence, residual, gamma, eps: float, out, stream=None):
    """As ``allreduce_rmsnorm`` but without a workspace and without any device
    allocation, for callers that cannot let a library allocate: the scratch is
    a fixed array inside the library (M * N <= 2,097,152).  Calls that can
    overlap on the GPU race on that array."""
    import torch
    R = len(partials)
    M, N = partials[0].shape
    for t in partials:
        _check_bf16(t, "partials")
    if residual is not None:
        _check_bf16(residual, "residual")
    _check_bf16(out, "out")
    if gamma.dtype != torch.float32 or not gamma.is_cuda or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous CUDA float32 tensor")
    rc = load_library().are_allreduce_rmsnorm_noalloc(
        _ptrs(partials), residual.data_ptr() if residual is not None else None, gamma.data_ptr(), float(eps),
        out.data_ptr(), R, M, N, _stream_handle(stream))
    _check(rc, "are_allreduce_rmsnorm_noalloc")


def noalloc_device_status() -> dict:
    """Status word of the allocation-free entry point on the current device
    (synchronises the device; describes the last call only)."""
    st = _DevStatus()
    rc = load_library().are_noalloc_device_status(ctypes.byref(st))
    if rc not in (OK, ETIMEOUT):
        raise AreError(rc, "are_noalloc_device_status")
    return {"status": rc, "code": st.code, "where": st.where, "a": st.a, "b": st.b}
