"""The one-shot AR+RMSNorm kernel (small messages) against the Lamport kernel
and the oracle, and the dispatch between the two.

The one-shot kernel sums, canonicalises and normalises with the same
arithmetic in the same order as the Lamport kernel's two phases, so the two
paths must agree bit for bit, not just within tolerance."""
import numpy as np
import pytest

from oracle import check_close
import synth
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu

pytestmark = pytest.mark.gpu

SENT = 0x80000000


def call(ws, parts_d, res_d, gamma_d, M, N, flags):
    import torch

    import all_reduce_epilogue_gb300 as are
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws.set_debug(flags)
    try:
        are.allreduce_rmsnorm(parts_d, res_d, gamma_d, 1e-6, out, ws)
        st = ws.device_status()
    finally:
        ws.set_debug(0)
    assert st["code"] == 0, st
    return out


@pytest.mark.parametrize("R,M,N,resid", [(8, 1, 7168, True), (8, 16, 7168, True), (8, 37, 7168, False),
                                          (3, 128, 1024, True), (1, 300, 4104, True), (8, 200, 7168, True),
                                          (5, 2, 8, True), (8, 160, 12288, False)])
def test_oneshot_equals_lamport_bitwise(oracle, R, M, N, resid):
    """Same inputs through both paths: identical output bits; both within the
    oracle's tolerance.  Rows of all -0.0 partials exercise the canonicalisation
    (with a -0.0 residual the sign of h depends on it)."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    parts, res, gamma = synth.ar_inputs(R, M, N, 4000 + R * M + N)
    rng = np.random.default_rng(M + N)
    forced = rng.choice(M * N, min(64, M * N), replace=False)
    for p in parts:
        p.reshape(-1)[forced] = 0x8000
    res.reshape(-1)[forced[: len(forced) // 2]] = 0x8000
    with are.Workspace(R_max=8, M_max=max(M, 8), N_max=N, timeout_ns=50_000_000) as ws:
        P = [dev_bf16(x) for x in parts]
        r = dev_bf16(res) if resid else None
        g = torch.from_numpy(gamma).cuda()
        a = call(ws, P, r, g, M, N, are.DEBUG_AR_ONESHOT)
        b = call(ws, P, r, g, M, N, are.DEBUG_AR_LAMPORT)
    assert np.array_equal(host_bits(a), host_bits(b)), "one-shot and Lamport outputs differ"
    check_close(host_f32(a), oracle.allreduce_rmsnorm(parts, res if resid else None, gamma, 1e-6), "one-shot")


def test_dispatch_by_message_size():
    """With re-arm off, a Lamport call leaves its staged sums in the staging
    words and a one-shot call leaves them untouched: small messages (per-rank
    input at or below the threshold) take the one-shot path, large ones the
    Lamport path, and each forcing flag overrides the size."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    N = 7168
    for M, expect_oneshot in [(16, True), (1024, False)]:  # 1024 rows: the Lamport path without ring laps
        parts, res, gamma = synth.ar_inputs(8, M, N, 77 + M)
        P = [dev_bf16(x) for x in parts]
        r = dev_bf16(res)
        g = torch.from_numpy(gamma).cuda()
        for flags, oneshot in [(0, expect_oneshot), (are.DEBUG_AR_ONESHOT, True), (are.DEBUG_AR_LAMPORT, False)]:
            with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=50_000_000) as ws:
                call(ws, P, r, g, M, N, flags | are.DEBUG_NO_REARM)
                words = ws.snapshot(are.SNAP_STAGING, min(M, 8) * N * 4).view(np.uint32)
                untouched = bool(np.all(words == SENT))
                assert untouched == oneshot, (M, flags)


def test_threshold_moves_the_dispatch():
    """are_workspace_set_oneshot_max_bytes: 0 sends a small message to the
    Lamport kernel, a large threshold sends a 1024-row message to the one-shot
    kernel."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    N = 7168
    for M, threshold, oneshot in [(16, 0, False), (1024, 1 << 40, True)]:
        parts, res, gamma = synth.ar_inputs(8, M, N, 55 + M)
        with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=50_000_000) as ws:
            ws.set_oneshot_max_bytes(threshold)
            call(ws, [dev_bf16(x) for x in parts], dev_bf16(res), torch.from_numpy(gamma).cuda(), M, N,
                 are.DEBUG_NO_REARM)
            words = ws.snapshot(are.SNAP_STAGING, min(M, 8) * N * 4).view(np.uint32)
            assert bool(np.all(words == SENT)) == oneshot, (M, threshold)


def test_oneshot_falls_back_when_a_row_does_not_fit(oracle):
    """R=8 rows of 16384 bf16 plus a residual do not fit one block's shared
    memory: even when forced, the call takes the Lamport path (staged words
    appear) and the result is right."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N = 8, 3, 16384
    parts, res, gamma = synth.ar_inputs(R, M, N, 91)
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=50_000_000) as ws:
        out = call(ws, [dev_bf16(x) for x in parts], dev_bf16(res), torch.from_numpy(gamma).cuda(), M, N,
                   are.DEBUG_AR_ONESHOT | are.DEBUG_NO_REARM)
        words = ws.snapshot(are.SNAP_STAGING, M * N * 4).view(np.uint32)
        assert not np.all(words == SENT)
    check_close(host_f32(out), oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6), "fallback")


def test_oneshot_many_rows_per_block(oracle):
    """Forced one-shot with more rows than blocks: each block walks several
    rows, reusing its shared memory while the next row's copies are in flight."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N = 8, 1000, 7168
    parts, res, gamma = synth.ar_inputs(R, M, N, 1234)
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=50_000_000) as ws:
        out = call(ws, [dev_bf16(x) for x in parts], dev_bf16(res), torch.from_numpy(gamma).cuda(), M, N,
                   are.DEBUG_AR_ONESHOT)
    check_close(host_f32(out), oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6), "one-shot M=1000")


@pytest.mark.parametrize("path", ["oneshot", "lamport"])
@pytest.mark.parametrize("R,M,N,resid,inplace", [(8, 16, 7168, True, False), (8, 300, 7168, True, True),
                                                  (3, 5, 1024, False, False), (8, 1500, 7168, True, True)])
def test_residual_out_bit_exact(oracle, path, R, M, N, resid, inplace):
    """residual_out = bf16(canon(sum) + residual) bit for bit against the
    oracle, through each kernel, also written in place over the residual; the
    normalised output is unchanged by asking for it."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    parts, res, gamma = synth.ar_inputs(R, M, N, 6000 + R * M + N)
    want_h = oracle.allreduce_residual_out(parts, res if resid else None)
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=100_000_000) as ws:
        ws.set_debug(are.DEBUG_AR_ONESHOT if path == "oneshot" else are.DEBUG_AR_LAMPORT)
        P = [dev_bf16(x) for x in parts]
        g = torch.from_numpy(gamma).cuda()
        r = dev_bf16(res) if resid else None
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ro = r if (inplace and resid) else torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.allreduce_add_rmsnorm(P, r, g, 1e-6, out, ro, ws)
        out2 = torch.empty_like(out)
        r2 = dev_bf16(res) if resid else None
        are.allreduce_rmsnorm(P, r2, g, 1e-6, out2, ws)
        st = ws.device_status()
    assert st["code"] == 0, st
    assert np.array_equal(host_bits(ro), want_h), "residual_out differs from the oracle"
    assert np.array_equal(host_bits(out), host_bits(out2)), "asking for residual_out changed out"
    check_close(host_f32(out), oracle.allreduce_rmsnorm(parts, res if resid else None, gamma, 1e-6), "add-rmsnorm")
