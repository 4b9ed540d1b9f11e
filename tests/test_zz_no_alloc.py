"""The allocation-free all-reduce + RMSNorm entry point.

Callers that cannot let a library allocate device memory (a framework whose
allocator must own every device byte, a fixed memory budget, code that cannot
afford the synchronisation of cudaMalloc/cudaFree) use
are_allreduce_rmsnorm_noalloc, whose scratch is a fixed array inside the
library.  Its output must match the workspace-based are_allreduce_rmsnorm
within the parity tolerance, on two calls in a row (the second call reuses
the array the first one left behind).  This file is collected last and must
also pass alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth
from oracle import check_close
from tests.gpu_util import dev_bf16, host_f32, need_gpu

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, parts, res, gamma, eps, out, stream):
    ptrs = (ctypes.c_void_p * len(parts))(*[t.data_ptr() for t in parts])
    return lib.are_allreduce_rmsnorm_noalloc(ptrs, res.data_ptr() if res is not None else None, gamma.data_ptr(),
                                            ctypes.c_float(eps), out.data_ptr(), len(parts), parts[0].shape[0],
                                            parts[0].shape[1], stream)


# 2048 x 1024 fills the array and laps the staging ring
@pytest.mark.parametrize("R,M,N,resid", [(8, 64, 7168, True), (3, 5, 1000, False), (4, 2048, 1024, True)])
def test_noalloc_matches_workspace_entry_point(R, M, N, resid):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    lib = are.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    calls = []
    for k in range(2):  # two calls in a row, different inputs
        parts_h, res_h, gamma_h = synth.ar_inputs(R, M, N, 1000 + 17 * k + R * M)
        parts = [dev_bf16(x) for x in parts_h]
        res = dev_bf16(res_h) if resid else None
        gamma = torch.from_numpy(gamma_h).cuda()
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, parts, res, gamma, 1e-6, out, stream) == are.OK
        calls.append((parts, res, gamma, out))
    torch.cuda.synchronize()
    with are.Workspace(R_max=8, M_max=M, N_max=N) as ws:
        for parts, res, gamma, out in calls:
            ref = torch.empty_like(out)
            are.allreduce_rmsnorm(parts, res, gamma, 1e-6, ref, ws)
            assert ws.device_status()["code"] == 0
            check_close(host_f32(out), host_f32(ref), "noalloc vs workspace entry point")


def test_noalloc_rejects_sizes_beyond_its_array():
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    lib = are.load_library()
    M, N = 293, 7168  # M * N > 2,097,152
    x = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(N, dtype=torch.float32, device="cuda")
    out = torch.empty_like(x)
    assert _call_noalloc(lib, [x], None, g, 1e-6, out, None) == are.ECAPACITY
