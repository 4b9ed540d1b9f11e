"""AR + residual + RMSNorm on the GPU against the CPU oracle: the Lamport
kernel, and for small messages the one-shot kernel the dispatch picks there."""
import numpy as np
import pytest

import oracle
from oracle import check_close
import synth
from tests.gpu_util import dev_bf16, host_f32, need_gpu

pytestmark = pytest.mark.gpu

SENT = 0x80000000


@pytest.fixture(scope="module")
def ws():
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    w = are.Workspace(R_max=8, M_max=4096, N_max=7168, K_max=0, timeout_ns=50_000_000)
    yield w
    w.close()


def run(ws, parts, res, gamma, eps=1e-6):
    import torch

    import all_reduce_epilogue_gb300 as are
    M, N = parts[0].shape
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    are.allreduce_rmsnorm([dev_bf16(x) for x in parts], dev_bf16(res) if res is not None else None,
                          torch.from_numpy(gamma).cuda(), eps, out, ws)
    st = ws.device_status()
    assert st["code"] == 0, st
    return host_f32(out)


def staging_words(ws, M, N):
    import all_reduce_epilogue_gb300 as are
    return ws.snapshot(are.SNAP_STAGING, M * N * 4).view(np.uint32).reshape(M, N)


@pytest.mark.parametrize("path", ["default", "lamport", "oneshot"])
@pytest.mark.parametrize("M", [1, 16, 128, 1024, 4096])
def test_workload_shapes(ws, oracle, M, path):
    """R=8 bf16 partials [M, 7168], 1% -0.0 entries, residual, gamma ~ N(1, 0.1),
    through the default dispatch and through each path forced."""
    import all_reduce_epilogue_gb300 as are
    flags = {"default": 0, "lamport": are.DEBUG_AR_LAMPORT, "oneshot": are.DEBUG_AR_ONESHOT}[path]
    parts, res, gamma = synth.ar_inputs(8, M, 7168, synth.config_seed(3))
    ws.set_debug(flags)
    try:
        got = run(ws, parts, res, gamma)
    finally:
        ws.set_debug(0)
    ref = oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6)
    oracle_mod_check(got, ref, f"M={M} {path}")
    # every staged word consumed and re-armed with -0.0 (the ring's odd-lap
    # sentinel never survives a call)
    assert np.all(staging_words(ws, M, 7168) == SENT)


def oracle_mod_check(got, ref, what):
    info = check_close(got, ref, what)
    assert info["rel_l2"] < 2e-3


@pytest.mark.parametrize("R,M,N,resid", [(1, 3, 200, False), (2, 5, 8, True), (3, 7, 2048, True),
                                          (5, 300, 4104, True), (8, 613, 7168, False), (8, 2, 16384, True),
                                          (4, 9, 32768, True)])
def test_ragged_shapes(oracle, R, M, N, resid):
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    with are.Workspace(R_max=8, M_max=1024, N_max=32768, timeout_ns=50_000_000) as w:
        parts, res, gamma = synth.ar_inputs(R, M, N, 100 + R * M + N)
        got = run(w, parts, res if resid else None, gamma)
        ref = oracle.allreduce_rmsnorm(parts, res if resid else None, gamma, 1e-6)
        check_close(got, ref, f"R={R} M={M} N={N}")


def test_staging_snapshot_bit_exact(oracle):
    """With re-arm off, the staged words equal the oracle's canonicalised
    ring-order sums bit for bit (integer-valued partials: every sum is exact),
    including positions forced to all -0.0 (staged +0.0), and the count of
    canonicalised words matches."""
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    R, M, N = 8, 37, 1024
    rng = np.random.default_rng(3)
    parts = [(np.rint(rng.standard_normal((M, N)) * 4)).astype(np.float32) for _ in range(R)]
    parts = [synth_bits(p) for p in parts]
    forced = rng.choice(M * N, 500, replace=False)
    for p in parts:
        p.reshape(-1)[forced] = 0x8000
        p.reshape(-1)[rng.choice(M * N, 50, replace=False)] = 0x8000  # single -0.0: not a sentinel sum
    res = synth.normal_bf16((M, N), 4, synth.T_RESIDUAL)
    gamma = synth.normal_f32((N,), 4, synth.T_GAMMA, 0, 1.0, 0.1)
    with are.Workspace(R_max=8, M_max=64, N_max=N, timeout_ns=50_000_000,
                       debug_flags=are.DEBUG_NO_REARM | are.DEBUG_COUNT_CANON | are.DEBUG_AR_LAMPORT) as w:
        got = run(w, parts, res, gamma)
        s_ref, count = oracle.ar_stage(parts)
        snap = staging_words(w, M, N)
        assert np.array_equal(snap, s_ref.view(np.uint32)), "staged words differ from the oracle"
        assert not np.any(snap == SENT)
        counters = w.snapshot(are.SNAP_COUNTERS, 32).view(np.uint64)
        assert int(counters[0]) == count and count >= 500
        check_close(got, oracle.rmsnorm(s_ref, res, gamma, 1e-6), "snapshot case")


def synth_bits(x_f32):
    from tests.pins import to_bf16_bits
    return to_bf16_bits(x_f32)


def test_repeat_rearm(ws, oracle):
    """Back-to-back calls with changing M and inputs: a pack re-armed late would
    leak an old value into a later call."""
    import torch

    import all_reduce_epilogue_gb300 as are
    N = 7168
    cases = []
    for i, M in enumerate([64, 1, 2000, 513, 8, 300, 4096]):
        parts, res, gamma = synth.ar_inputs(8, M, N, 500 + i)
        cases.append(([dev_bf16(x) for x in parts], dev_bf16(res), torch.from_numpy(gamma).cuda(),
                      torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                      oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6)))
    for it in range(1000):
        p, r, g, out, _ = cases[it % len(cases)]
        are.allreduce_rmsnorm(p, r, g, 1e-6, out, ws)
    st = ws.device_status()
    assert st["code"] == 0, st
    for p, r, g, out, ref in cases:
        check_close(host_f32(out), ref, "repeat")
    assert np.all(staging_words(ws, 4096, N) == SENT)


def test_missing_pack_times_out_and_reset_recovers(oracle):
    """A pack that is never staged makes its consumer's bounded spin expire:
    the status names the row and pack, the kernel returns, and after a reset
    the workspace works again."""
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    M, N = 20, 1024
    parts, res, gamma = synth.ar_inputs(4, M, N, 9)
    with are.Workspace(R_max=8, M_max=64, N_max=N, timeout_ns=20_000_000) as w:
        pack = 5 * (N // 8) + 17  # row 5, pack 17
        w.set_debug(are.DEBUG_SKIP_STAGE | are.DEBUG_AR_LAMPORT, pack)
        import torch
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.allreduce_rmsnorm([dev_bf16(x) for x in parts], dev_bf16(res), torch.from_numpy(gamma).cuda(), 1e-6,
                              out, w)
        st = w.device_status()
        assert st["status"] == are.ETIMEOUT and st["code"] == are.DEV_STAGE_TIMEOUT
        assert st["a"] == 5 and st["b"] == 17
        w.set_debug(0)
        w.reset()
        got = run(w, parts, res, gamma)
        check_close(got, oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6), "after reset")


def test_bad_arguments(ws):
    import torch

    import all_reduce_epilogue_gb300 as are
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.float32, device="cuda")
    out = torch.empty_like(x)
    with pytest.raises(are.AreError) as e:
        are.allreduce_rmsnorm([x], None, g, 0.0, out, ws)  # eps <= 0
    assert e.value.status == are.EINVAL
    with pytest.raises(are.AreError) as e:
        are.allreduce_rmsnorm([x] * 9, None, g, 1e-6, out, ws)  # R > 8
    assert e.value.status == are.EINVAL
    big = torch.zeros((4097, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(are.AreError) as e:
        are.allreduce_rmsnorm([big], None, g, 1e-6, torch.empty_like(big), ws)  # M > M_max
    assert e.value.status == are.ECAPACITY
    empty = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    are.allreduce_rmsnorm([empty], None, g, 1e-6, torch.empty_like(empty), ws)  # M = 0: no-op


@pytest.mark.parametrize("M", [8192, 7000])
def test_ring_many_laps_repeat(oracle, M):
    """Many laps of the staging ring with a partial last chunk, called
    repeatedly: every staging position must be overwritten only after its
    consumer re-armed it (a producer running laps ahead would corrupt or
    stall a later lap)."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    N = 7168
    parts, res, gamma = synth.ar_inputs(8, M, N, 77 + M)
    ref = oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6)
    P = [dev_bf16(x) for x in parts]
    r = dev_bf16(res)
    g = torch.from_numpy(gamma).cuda()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=100_000_000) as w:
        for _ in range(30):
            are.allreduce_rmsnorm(P, r, g, 1e-6, out, w)
        st = w.device_status()
        assert st["code"] == 0, st
        check_close(host_f32(out), ref, f"ring M={M}")
        assert np.all(staging_words(w, M, N) == SENT)


def test_ring_reuse_waits_for_rearm(oracle):
    """Without re-arming, no staged word of lap 0 turns back into the lap-1
    sentinel, so every producer's bounded check before it overwrites its row of
    the first slot in lap 1 (chunk 8) expires: the status names that check and
    chunk, the kernel returns, and after a reset the workspace works again."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    M, N = 4096, 1024  # more than 8 chunks of at most 2 x 152 rows: the ring laps
    parts, res, gamma = synth.ar_inputs(2, M, N, 31)
    P = [dev_bf16(x) for x in parts]
    r = dev_bf16(res)
    g = torch.from_numpy(gamma).cuda()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, timeout_ns=20_000_000) as w:
        w.set_debug(are.DEBUG_NO_REARM | are.DEBUG_AR_LAMPORT)
        are.allreduce_rmsnorm(P, r, g, 1e-6, out, w)
        st = w.device_status()
        assert st["status"] == are.ETIMEOUT and st["code"] == are.DEV_PIPE_TIMEOUT, st
        assert st["a"] == -3 and st["b"] == 8, st
        w.set_debug(0)
        w.reset()
        are.allreduce_rmsnorm(P, r, g, 1e-6, out, w)
        assert w.device_status()["code"] == 0
        check_close(host_f32(out), oracle.allreduce_rmsnorm(parts, res, gamma, 1e-6), "after reset")
        assert np.all(staging_words(w, M, N) == SENT)
