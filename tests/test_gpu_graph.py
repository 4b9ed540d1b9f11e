"""The operations inside a captured CUDA graph, replayed many times.

A call touches no host state that a replay would miss: the GEMM masks and the
Lamport staging words are re-armed inside the kernels (never by the host, and
never by a captured fill), so a graph captured once replays correctly while
its inputs change between replays."""
import numpy as np
import pytest

from oracle import check_close
import synth
from tests.gpu_util import dev_bf16, host_f32, need_gpu

pytestmark = pytest.mark.gpu

SENT = 0x80000000


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # outside the capture once: any lazy set-up happens here
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("path", ["oneshot", "lamport"])
@pytest.mark.parametrize("M", [16, 2000])
def test_allreduce_rmsnorm_graph_replays(oracle, path, M):
    """Capture one call, then for several input sets copy the inputs in and
    replay (20 replays per set): every result matches the oracle and every
    staging word is re-armed afterwards.  M=2000 laps the Lamport ring."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, N = 8, 7168
    P = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    res = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gamma = torch.empty(N, dtype=torch.float32, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=100_000_000) as ws:
        ws.set_debug(are.DEBUG_AR_ONESHOT if path == "oneshot" else are.DEBUG_AR_LAMPORT)
        for t in P + [res]:
            t.zero_()
        gamma.fill_(1.0)
        g = _capture(lambda: are.allreduce_rmsnorm(P, res, gamma, 1e-6, out, ws))
        for k in range(3):
            parts, r_h, g_h = synth.ar_inputs(R, M, N, 900 + k + M)
            for t, h in zip(P, parts):
                t.copy_(dev_bf16(h))
            res.copy_(dev_bf16(r_h))
            gamma.copy_(torch.from_numpy(g_h).cuda())
            for _ in range(20):
                g.replay()
            torch.cuda.synchronize()
            st = ws.device_status()
            assert st["code"] == 0, st
            check_close(host_f32(out), oracle.allreduce_rmsnorm(parts, r_h, g_h, 1e-6), f"replay set {k}")
        words = ws.snapshot(are.SNAP_STAGING, M * N * 4).view(np.uint32)
        assert np.all(words == SENT)


@pytest.mark.parametrize("reduction", ["default", "ring"])
def test_gemm_rs_and_ar_graph_replays(oracle, reduction):
    """GEMM+RS and GEMM+AR captured together and replayed: the tile masks are
    re-armed by the reducers (the ring's last rank, or the last of a tile's
    row-slice reducers, whose per-tile count also returns to 0), so every
    replay waits for that replay's own partials.  At this size GEMM+RS takes
    the row-slice split by default; the ring is forced in the second case."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 4, 512, 768, 256
    dA = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    dB = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    out_rs = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out_ar = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K, timeout_ns=100_000_000) as ws:
        if reduction == "ring":
            ws.set_debug(are.DEBUG_RS_RING)
        for t in dA + dB:
            t.zero_()

        def step():
            are.gemm_rs(dA, dB, out_rs, ws)
            are.gemm_ar(dA, dB, [out_ar] * R, ws)
        g = _capture(step)
        for k in range(3):
            A, B = synth.gemm_inputs(R, M, N, K, 50 + k)
            for t, h in zip(dA + dB, A + B):
                t.copy_(dev_bf16(h))
            for _ in range(10):
                g.replay()
            torch.cuda.synchronize()
            st = ws.device_status()
            assert st["code"] == 0, st
            check_close(host_f32(out_rs), oracle.gemm_rs(A, B), f"rs replay set {k}")
            check_close(host_f32(out_ar), oracle.gemm_ar(A, B), f"ar replay set {k}")
        masks = ws.snapshot(are.SNAP_MASKS, 4 * 4 * 3).view(np.uint32)
        assert np.all(masks == 0), "tile masks not re-armed"
