"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

Only random draws live here (see ``synth.c`` for the generator's definition);
nothing in this package computes any part of the epilogue.  Every array comes
back as a host numpy array: bf16 tensors as ``uint16`` bit patterns, fp32 as
``float32``.

Workload recipes follow the shapes and value distributions of the five
benchmark configurations (tiny GEMM+RS+RMSNorm, GEMM+RS at R=4, GEMM+AR at
R=8, AR+residual+RMSNorm at R=8, large GEMM+RS at R=8); the seed of a
configuration is ``0xA11 + config_id`` and rank ``r`` of tensor ``t`` draws
from its own stream ``(seed, t, r)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIBPATH = os.path.join(_LIBDIR, "libsynth.so")
_lock = threading.Lock()
_lib = None

# tensor ids of the streams
T_A, T_B, T_RESIDUAL, T_GAMMA, T_PARTIAL, T_NEGZERO = 1, 2, 3, 4, 5, 6

BF16_NEG_ZERO = 0x8000


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_lib/libsynth.so`` with gcc (OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(src)):
        return _LIBPATH
    tmp = _LIBPATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIBPATH)
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_stream_key.restype = u64
            lib.synth_stream_key.argtypes = [u64, u64, u64]
            lib.synth_words.argtypes = [u64, u64, i64, vp]
            lib.synth_uniform_bf16.argtypes = [u64, i64, dbl, dbl, vp]
            lib.synth_normal_bf16.argtypes = [u64, i64, dbl, dbl, vp]
            lib.synth_normal_f32.argtypes = [u64, i64, dbl, dbl, vp]
            lib.synth_inject_bf16.restype = i64
            lib.synth_inject_bf16.argtypes = [u64, i64, dbl, ctypes.c_uint16, vp]
            _lib = lib
        return _lib


def stream_key(seed: int, tensor_id: int, rank: int = 0) -> int:
    return int(_get().synth_stream_key(seed, tensor_id, rank))


def words(seed: int, tensor_id: int, rank: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _get().synth_words(stream_key(seed, tensor_id, rank), start, n, out.ctypes.data)
    return out


def uniform_bf16(shape, seed, tensor_id, rank=0, lo=-1.0, hi=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _get().synth_uniform_bf16(stream_key(seed, tensor_id, rank), out.size, lo, hi, out.ctypes.data)
    return out


def normal_bf16(shape, seed, tensor_id, rank=0, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _get().synth_normal_bf16(stream_key(seed, tensor_id, rank), out.size, mean, std, out.ctypes.data)
    return out


def normal_f32(shape, seed, tensor_id, rank=0, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _get().synth_normal_f32(stream_key(seed, tensor_id, rank), out.size, mean, std, out.ctypes.data)
    return out


def inject_bf16(arr: np.ndarray, seed, tensor_id, rank, p: float, bits: int) -> int:
    """Overwrite about a fraction ``p`` of ``arr`` (uint16, C-contiguous) with ``bits``."""
    assert arr.dtype == np.uint16 and arr.flags.c_contiguous
    return int(_get().synth_inject_bf16(stream_key(seed, tensor_id, rank), arr.size, p, bits,
                                        arr.ctypes.data))


# ----------------------------------------------------------------------------
# workload recipes
# ----------------------------------------------------------------------------

def config_seed(config_id: int) -> int:
    return 0xA11 + config_id


def gemm_inputs(R: int, M: int, N: int, K: int, seed: int, dist: str = "normal"):
    """Per-rank A_r [M,K] and B_r [K,N] (bf16 bits).

    ``dist="normal"``: N(0,1)/sqrt(K) (the GEMM+RS / GEMM+AR workloads);
    ``dist="uniform"``: U[-1,1) (the tiny GEMM+RS+RMSNorm workload).
    """
    A, B = [], []
    for r in range(R):
        if dist == "uniform":
            A.append(uniform_bf16((M, K), seed, T_A, r))
            B.append(uniform_bf16((K, N), seed, T_B, r))
        else:
            s = 1.0 / np.sqrt(K)
            A.append(normal_bf16((M, K), seed, T_A, r, 0.0, s))
            B.append(normal_bf16((K, N), seed, T_B, r, 0.0, s))
    return A, B


def ar_inputs(R: int, M: int, N: int, seed: int, negzero_frac: float = 0.01):
    """R bf16 partials [M,N] ~ N(0,1) with a fraction of entries set to -0.0,
    bf16 residual [M,N] ~ N(0,1) and fp32 gamma [N] ~ N(1, 0.1)."""
    partials = []
    for r in range(R):
        x = normal_bf16((M, N), seed, T_PARTIAL, r)
        if negzero_frac > 0:
            inject_bf16(x, seed, T_NEGZERO, r, negzero_frac, BF16_NEG_ZERO)
        partials.append(x)
    residual = normal_bf16((M, N), seed, T_RESIDUAL, 0)
    gamma = normal_f32((N,), seed, T_GAMMA, 0, 1.0, 0.1)
    return partials, residual, gamma


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: a bf16 is the top half of an fp32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
