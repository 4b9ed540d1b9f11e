"""The quantising AR+RMSNorm variant (per-row dynamic FP8 E4M3) against the
oracle, through both kernels.

A code is an integer decided by floating point: the oracle and the kernel
both decide it in fp32 (the kernel's precision), from a y that differs only
in its last bits (rsqrt and the order of the sum of squares).  So a code may
differ from the oracle's only where the oracle's y/scale lies within a
relative 1e-5 of a rounding boundary, and then only to the neighbouring code
on the other side of it."""
import numpy as np
import pytest

import synth
from tests.gpu_util import dev_bf16, host_bits, need_gpu

pytestmark = pytest.mark.gpu

REL = 1e-5


def run_quant(ws, parts, res, gamma, flags, residual_out=False):
    import torch

    import all_reduce_epilogue_gb300 as are
    M, N = parts[0].shape
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    sc = torch.empty(M, dtype=torch.float32, device="cuda")
    ro = torch.empty((M, N), dtype=torch.bfloat16, device="cuda") if residual_out else None
    ws.set_debug(flags)
    try:
        are.allreduce_rmsnorm_quant([dev_bf16(x) for x in parts], dev_bf16(res) if res is not None else None,
                                    torch.from_numpy(gamma).cuda(), 1e-6, q, sc, ws, residual_out=ro)
        st = ws.device_status()
    finally:
        ws.set_debug(0)
    assert st["code"] == 0, st
    return q.cpu().numpy(), sc.cpu().numpy(), (host_bits(ro) if residual_out else None)


@pytest.mark.parametrize("R,M,N,resid", [(8, 16, 7168, True), (8, 300, 7168, True), (3, 37, 1024, False),
                                          (8, 1500, 7168, True)])
def test_quant_against_oracle_both_paths(oracle, R, M, N, resid):
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    parts, res, gamma = synth.ar_inputs(R, M, N, 7000 + R * M + N)
    r = res if resid else None
    y = oracle.allreduce_rmsnorm(parts, r, gamma, 1e-6)
    q_ref, s_ref, x_ref = oracle.quant_rows(y)
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=100_000_000) as ws:
        q1, s1, h1 = run_quant(ws, parts, r, gamma, are.DEBUG_AR_ONESHOT, residual_out=True)
        q2, s2, h2 = run_quant(ws, parts, r, gamma, are.DEBUG_AR_LAMPORT, residual_out=True)
    # the two kernels agree bit for bit
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    assert np.array_equal(h1, h2) and np.array_equal(h1, oracle.allreduce_residual_out(parts, r))
    # scales: fp32 noise only
    assert np.all(np.abs(s1.astype(np.float64) - s_ref) <= REL * s_ref), "scale"
    # codes: equal, or the neighbour across a boundary the oracle's value is within REL of
    diff = np.nonzero(q1 != q_ref)
    assert len(diff[0]) <= max(1, q1.size // 1000), f"{len(diff[0])} codes differ"
    if len(diff[0]):
        xs = x_ref[diff]
        lo = oracle.e4m3(xs * np.float32(1 - REL))
        hi = oracle.e4m3(xs * np.float32(1 + REL))
        ok = (q1[diff] == lo) | (q1[diff] == hi)
        assert np.all(ok), f"codes off by more than a boundary: {q1[diff][~ok][:5]} vs {q_ref[diff][~ok][:5]}"
    # the largest |y| of every row maps to +-448
    amax_code = np.take_along_axis(q1, np.argmax(np.abs(y), axis=1)[:, None], axis=1)[:, 0]
    assert np.all(amax_code & 0x7F == 0x7E)


def test_quant_zero_row_and_bad_arguments():
    """An all-zero row gets scale 1 and zero codes; the quantising call rejects
    missing outputs."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N = 2, 4, 256
    parts = [np.zeros((M, N), np.uint16) for _ in range(R)]
    gamma = np.ones(N, np.float32)
    with are.Workspace(R_max=8, M_max=M, N_max=N) as ws:
        q, sc, _ = run_quant(ws, parts, None, gamma, 0)
        assert np.all(q == 0) and np.all(sc == 1)
        lib = are.load_library()
        P = [torch.zeros((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        g = torch.ones(N, dtype=torch.float32, device="cuda")
        import ctypes
        ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() for t in P])
        rc = lib.are_allreduce_rmsnorm_quant(ptrs, None, g.data_ptr(), ctypes.c_float(1e-6), None, None, None, R, M,
                                             N, ws.handle, None)
        assert rc == are.EINVAL
