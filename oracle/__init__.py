"""Python face of the CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py``.  The library package
never imports it, and it never imports the library.

All bf16 tensors are numpy ``uint16`` bit patterns; results are numpy
``float32`` (the unrounded fp32 reference) unless stated otherwise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_lock = threading.Lock()
_libs: dict = {}

# Tile shape of the per-tile ready bitmask named by the GEMM+RS workload
# ("per-tile ready bitmask over 128x256 output tiles").
MASK_TILE_M = 128
MASK_TILE_N = 256


def lib_path(plant: int = 0) -> str:
    return os.path.join(_LIBDIR, "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so")


def build(plant: int = 0, force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc.  ``plant > 0`` builds a copy with a known
    mistake planted (used only by the pin-strength tests)."""
    src = os.path.join(_HERE, "oracle.c")
    out = lib_path(plant)
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           f"-DORACLE_PLANT={plant}", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def _load(plant: int = 0):
    with _lock:
        if plant in _libs:
            return _libs[plant]
        path = build(plant)
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_rne_sat.restype = ctypes.c_uint8
        lib.oracle_e4m3_rne_sat.argtypes = [ctypes.c_float]
        lib.oracle_quant_rows.restype = None
        lib.oracle_quant_rows.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_bf16_rne_n.restype = None
        lib.oracle_bf16_rne_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_max_threads.restype = i32
        lib.oracle_partial_gemm.argtypes = [vp, vp, i64, i64, i64, vp, i32]
        lib.oracle_gemm_reduce_rows.argtypes = [vp, vp, i32, i64, i64, i64, vp, i64, i32, vp, i32]
        lib.oracle_owner_of_row.restype = i32
        lib.oracle_owner_of_row.argtypes = [i64, i64, i32]
        lib.oracle_tile_pieces.restype = i32
        lib.oracle_tile_pieces.argtypes = [i64, i64, i64, i32, vp, vp, vp]
        lib.oracle_expected_masks.restype = i64
        lib.oracle_expected_masks.argtypes = [i32, i64, i64, i64, i64, vp, i64]
        lib.oracle_chunk_pieces.restype = None
        lib.oracle_chunk_pieces.argtypes = [i32, i64, i64, i64, i64, i32, vp]
        lib.oracle_ar_stage.restype = i64
        lib.oracle_ar_stage.argtypes = [vp, i32, i64, i64, vp, i32]
        lib.oracle_rmsnorm_rows.argtypes = [vp, vp, vp, ctypes.c_float, i64, i64, vp, vp, i32]
        _libs[plant] = lib
        return lib


class Oracle:
    """The oracle's functions bound to one build (``plant=0`` is the real one)."""

    def __init__(self, plant: int = 0, nthreads: int = 0):
        self.lib = _load(plant)
        self.nthreads = nthreads

    # -- helpers ----------------------------------------------------------
    @staticmethod
    def _u16(a):
        a = np.ascontiguousarray(a)
        assert a.dtype == np.uint16
        return a

    @staticmethod
    def _ptr_array(arrs):
        return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    # -- bf16 ---------------------------------------------------------------
    def bf16_rne(self, x) -> np.ndarray:
        """fp32 -> bf16 bits, round to nearest even (scalar loop; small inputs)."""
        x = np.asarray(x, dtype=np.float32)
        flat = x.reshape(-1)
        out = np.empty(flat.shape, dtype=np.uint16)
        for i, v in enumerate(flat):
            out[i] = self.lib.oracle_bf16_rne(ctypes.c_float(float(v)))
        return out.reshape(x.shape)

    def bf16_rne_array(self, x) -> np.ndarray:
        """fp32 -> bf16 bits for a whole array (the same rounding function)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_bf16_rne_n(x.ctypes.data, out.ctypes.data, x.size)
        return out

    # -- GEMM ---------------------------------------------------------------
    def partial_gemm(self, A, B) -> np.ndarray:
        A, B = self._u16(A), self._u16(B)
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        P = np.empty((M, N), dtype=np.float32)
        self.lib.oracle_partial_gemm(A.ctypes.data, B.ctypes.data, M, N, K, P.ctypes.data, self.nthreads)
        return P

    def gemm_reduce_rows(self, A_list, B_list, rows=None, mode: str = "rs") -> np.ndarray:
        """Rows ``rows`` of the ring-order reduced result (``mode`` 'rs' or 'ar')."""
        A_list = [self._u16(a) for a in A_list]
        B_list = [self._u16(b) for b in B_list]
        R = len(A_list)
        M, K = A_list[0].shape
        N = B_list[0].shape[1]
        for a, b in zip(A_list, B_list):
            assert a.shape == (M, K) and b.shape == (K, N)
        if rows is None:
            rows = np.arange(M, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        Y = np.empty((rows.size, N), dtype=np.float32)
        self.lib.oracle_gemm_reduce_rows(self._ptr_array(A_list), self._ptr_array(B_list), R, M, N, K,
                                         rows.ctypes.data, rows.size, 1 if mode == "ar" else 0,
                                         Y.ctypes.data, self.nthreads)
        return Y

    def gemm_rs(self, A_list, B_list, rows=None) -> np.ndarray:
        return self.gemm_reduce_rows(A_list, B_list, rows, "rs")

    def gemm_ar(self, A_list, B_list, rows=None) -> np.ndarray:
        return self.gemm_reduce_rows(A_list, B_list, rows, "ar")

    # -- owner segments and masks --------------------------------------------
    def owner_of_row(self, row: int, M: int, R: int) -> int:
        return int(self.lib.oracle_owner_of_row(row, M, R))

    def tile_pieces(self, row0: int, BM: int, M: int, R: int):
        seg = np.zeros(BM + 1, dtype=np.int64)
        b = np.zeros(BM + 1, dtype=np.int64)
        e = np.zeros(BM + 1, dtype=np.int64)
        n = self.lib.oracle_tile_pieces(row0, BM, M, R, seg.ctypes.data, b.ctypes.data, e.ctypes.data)
        return [(int(seg[i]), int(b[i]), int(e[i])) for i in range(n)]

    def expected_masks(self, R: int, M: int, N: int, nwords: int,
                       BM: int = MASK_TILE_M, BN: int = MASK_TILE_N):
        words = np.zeros(nwords, dtype=np.uint32)
        T = self.lib.oracle_expected_masks(R, M, N, BM, BN, words.ctypes.data, nwords)
        return words, int(T)

    def chunk_pieces(self, R: int, M: int, N: int, C: int,
                     BM: int = MASK_TILE_M, BN: int = MASK_TILE_N) -> np.ndarray:
        """[R, C] int64: pieces (one tile's rows stored into one owner segment)
        that complete chunk c of segment s in one call; 0 for unused chunks."""
        out = np.zeros(R * C, dtype=np.int64)
        self.lib.oracle_chunk_pieces(R, M, N, BM, BN, C, out.ctypes.data)
        return out.reshape(R, C)

    def segments(self, Y: np.ndarray, R: int):
        """Split a full [M, N] result into the R owner segments."""
        M = Y.shape[0]
        S = M // R
        return [Y[s * S:(s + 1) * S] for s in range(R)]

    # -- all-reduce + RMSNorm --------------------------------------------------
    def ar_stage(self, x_list):
        """(s, count): canonicalised ring-order sum of R bf16 partials, and how
        many words were canonicalised from -0.0 to +0.0."""
        x_list = [self._u16(x) for x in x_list]
        M, N = x_list[0].shape
        s = np.empty((M, N), dtype=np.float32)
        n = self.lib.oracle_ar_stage(self._ptr_array(x_list), len(x_list), M, N, s.ctypes.data, self.nthreads)
        return s, int(n)

    def rmsnorm(self, s, residual, gamma, eps: float, return_h: bool = False):
        s = np.ascontiguousarray(s, dtype=np.float32)
        M, N = s.shape
        gamma = np.ascontiguousarray(gamma, dtype=np.float32)
        res_ptr = None
        if residual is not None:
            residual = self._u16(residual)
            res_ptr = residual.ctypes.data
        y = np.empty((M, N), dtype=np.float32)
        h = np.empty((M, N), dtype=np.float32) if return_h else None
        self.lib.oracle_rmsnorm_rows(s.ctypes.data, res_ptr, gamma.ctypes.data, ctypes.c_float(eps), M, N,
                                     y.ctypes.data, h.ctypes.data if return_h else None, self.nthreads)
        return (y, h) if return_h else y

    def allreduce_rmsnorm(self, x_list, residual, gamma, eps: float):
        s, _ = self.ar_stage(x_list)
        return self.rmsnorm(s, residual, gamma, eps)

    def e4m3(self, x) -> np.ndarray:
        """fp32 -> FP8 E4M3 codes (RNE, saturating), element by element."""
        x = np.asarray(x, dtype=np.float32)
        flat = x.reshape(-1)
        out = np.empty(flat.shape, dtype=np.uint8)
        for i, v in enumerate(flat):
            out[i] = self.lib.oracle_e4m3_rne_sat(ctypes.c_float(float(v)))
        return out.reshape(x.shape)

    def quant_rows(self, y):
        """(q, scale, x): per-row dynamic FP8 E4M3 quantisation of y [M, N]:
        scale = amax/448, x = y/scale, q = e4m3(x)."""
        y = np.ascontiguousarray(y, dtype=np.float32)
        M, N = y.shape
        q = np.empty((M, N), dtype=np.uint8)
        scale = np.empty(M, dtype=np.float32)
        x = np.empty((M, N), dtype=np.float32)
        self.lib.oracle_quant_rows(y.ctypes.data, M, N, q.ctypes.data, scale.ctypes.data, x.ctypes.data,
                                   self.nthreads)
        return q, scale, x

    def allreduce_rmsnorm_quant(self, x_list, residual, gamma, eps: float):
        """The quantising variant: (q, scale, x) of the RMSNorm output."""
        return self.quant_rows(self.allreduce_rmsnorm(x_list, residual, gamma, eps))

    def allreduce_residual_out(self, x_list, residual):
        """The updated residual stream a fused add-RMSNorm hands to the next
        layer: bf16 bits of h = canon(sum_r x_r) + residual (fp32 add; residual
        may be None), h as the RMSNorm step defines it."""
        s, _ = self.ar_stage(x_list)
        M, N = s.shape
        _, h = self.rmsnorm(s, residual, np.ones(N, np.float32), 1e-6, return_h=True)
        return self.bf16_rne_array(h)


_default = None


def get(nthreads: int = 0) -> Oracle:
    global _default
    if _default is None or nthreads:
        o = Oracle(0, nthreads)
        if not nthreads:
            _default = o
        return o
    return _default


# ----------------------------------------------------------------------------
# comparison helpers for the parity tests (the tolerance of the workloads)
# ----------------------------------------------------------------------------

REL_L2_MAX = 2e-3
ELEM_REL = 2.0 ** -7
ELEM_ABS = 1e-3


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.sum(ref * ref))
    num = np.sqrt(np.sum((got - ref) ** 2))
    return float(num / den) if den > 0 else float(num)


def elementwise_violations(got: np.ndarray, ref: np.ndarray) -> int:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = ELEM_REL * np.abs(ref) + ELEM_ABS
    return int(np.count_nonzero(~(np.abs(got - ref) <= bound)))


def check_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    """Raise AssertionError unless relL2 <= 2e-3 and |err| <= 2^-7|ref| + 1e-3."""
    r = rel_l2(got, ref)
    v = elementwise_violations(got, ref)
    info = {"rel_l2": r, "violations": v, "n": int(np.asarray(ref).size)}
    if not (r <= REL_L2_MAX and v == 0):
        raise AssertionError(f"{what}: parity failed {info}")
    return info
