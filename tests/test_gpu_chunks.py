"""Chunked owner-segment completion for GEMM+RS (ROCm/mori PR #662, the fused
GEMM -> scatter follow-ups: per-(destination, chunk) completion counters,
monotonic, with a modulo election; the destination-rotated tile order).

The counters are bookkeeping with one exact answer, stated by the oracle
(``chunk_pieces``): after one call with re-arming off, every counter equals
its chunk's piece count; with re-arming on, every completed chunk advances
its counter by exactly 2^32 per call, whatever the shapes of the calls.  The
tile order must not change a single output byte.  A host-side waiter sees a
chunk complete while the kernel is still running, and in the rotated order
every segment's first chunk completes before any segment's last."""
import time

import numpy as np
import pytest

import synth
from oracle import check_close
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu

pytestmark = pytest.mark.gpu

Q = 1 << 32


def _inputs(R, M, N, K, seed):
    A, B = synth.gemm_inputs(R, M, N, K, seed)
    return A, B, [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]


@pytest.mark.parametrize("R,M,N,K,C,flags", [
    (2, 64, 256, 128, 4, 0),              # tiny: one tile row shared by two segments (one-CTA kernel)
    (4, 256, 4096, 128, 2, 0),            # segments inside one tile row (one-CTA kernel)
    (4, 1024, 4096, 128, 8, "pair"),      # two tile rows per segment, C halves to 2 (CTA pairs)
    (3, 264, 320, 136, 2, "pair"),        # straddling tiles, unequal tile rows per segment, ragged N
    (8, 4096, 1024, 64, 8, "pair"),       # C halves to 4
    (8, 4096, 1024, 64, 6, "single"),     # C = 6 halves to 1, one-CTA kernel
])
def test_chunk_counters_match_oracle_bit_exact(oracle, R, M, N, K, C, flags):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    A, B, Ad, Bd = _inputs(R, M, N, K, 77 + M + C)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        extra = {"pair": are.DEBUG_PAIR_CTA, "single": are.DEBUG_SINGLE_CTA, 0: 0}[flags]
        ws.set_chunks(C, 0)
        ws.set_debug(are.DEBUG_NO_REARM | extra)
        are.gemm_rs(Ad, Bd, out, ws)
        assert ws.device_status()["code"] == 0
        got = ws.chunk_counters()
        want = oracle.chunk_pieces(R, M, N, C)
        assert np.array_equal(got[:R, :C].astype(np.int64), want), (got[:R, :C], want)
        assert np.all(got[:, C:] == 0) and np.all(got[R:] == 0)
        check_close(host_f32(out), oracle.gemm_rs(A, B), "gemm_rs with chunk counting")
        # a normal call after a reset: every used chunk advances by exactly 2^32, generation 1
        ws.set_debug(extra)
        ws.reset()
        are.gemm_rs(Ad, Bd, out, ws)
        assert ws.device_status()["code"] == 0
        got = ws.chunk_counters()
        assert np.array_equal(got[:R, :C], np.where(want > 0, Q, 0).astype(np.uint64))
        assert ws.chunk_generation() == 1
        for s in range(R):
            for c in range(C):
                assert ws.chunk_wait(s, c, 1, timeout_ns=0) == (want[s, c] > 0), (s, c)


def test_counters_stay_exact_across_calls_of_different_shapes(oracle):
    """Monotonic counters never reset: a call starts at a multiple of 2^32, so
    calls of different shapes (different piece counts per chunk) each elect
    exactly one completion per used chunk."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, N, K, C = 4, 1024, 128, 8
    shapes = [1024, 512, 2048, 1024, 256]
    with are.Workspace(R_max=8, M_max=2048, N_max=N, K_max=K) as ws:
        ws.set_chunks(C, 0)
        want = np.zeros((R, C), np.uint64)
        for i, M in enumerate(shapes):
            ws.set_debug(are.DEBUG_PAIR_CTA if i % 2 else 0)
            A, B, Ad, Bd = _inputs(R, M, N, K, 300 + i)
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            are.gemm_rs(Ad, Bd, out, ws)
            want += np.where(oracle.chunk_pieces(R, M, N, C) > 0, Q, 0).astype(np.uint64)
            assert ws.device_status()["code"] == 0
            check_close(host_f32(out), oracle.gemm_rs(A, B), f"gemm_rs M={M}")
        assert np.array_equal(ws.chunk_counters()[:R, :C], want)
        assert ws.chunk_generation() == len(shapes)
        gens = (want >> np.uint64(32)).astype(np.int64)
        for s in range(R):
            for c in range(C):
                if gens[s, c]:
                    assert ws.chunk_wait(s, c, int(gens[s, c]), timeout_ns=0)
                    assert not ws.chunk_wait(s, c, int(gens[s, c]) + 1, timeout_ns=1000)


@pytest.mark.parametrize("stripe", [-1, 0, 1, 3])
def test_rotated_order_changes_no_output_byte(oracle, stripe):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 4, 2048, 1000, 256   # segments of 512 rows: two tile pairs each; ragged N
    A, B, Ad, Bd = _inputs(R, M, N, K, 41)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(ref)
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_PAIR_CTA)
        are.gemm_rs(Ad, Bd, ref, ws)
        ws.set_chunks(4, stripe)
        are.gemm_rs(Ad, Bd, out, ws)
        assert ws.device_status()["code"] == 0
        assert ws.last_launch()["kernel"] == "gemm_pair_kernel"
        assert np.array_equal(host_bits(out), host_bits(ref))
        check_close(host_f32(out), oracle.gemm_rs(A, B), "rotated order")


@pytest.mark.slow
@pytest.mark.parametrize("stripe", [0, -1])
def test_host_sees_chunks_while_the_kernel_runs(stripe):
    """The large GEMM+RS (R=8, M=N=8192, K=4096, 8 chunks per segment).  The
    host polls every chunk from the moment the call is enqueued; as soon as a
    segment's first chunk is published it copies that chunk on another stream,
    while the kernel still runs, and the copies equal the final output.  In the
    rotated order every segment's first chunk completes before segment 0's
    last; in the usual order segment 0 completes entirely first."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K, C = 8, 8192, 8192, 4096, 8
    torch.manual_seed(5)
    Ad = [(torch.randn(M, K, device="cuda") * K ** -0.5).to(torch.bfloat16) for _ in range(R)]
    Bd = [(torch.randn(K, N, device="cuda") * K ** -0.5).to(torch.bfloat16) for _ in range(R)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    S = M // R
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_chunks(C, stripe)
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        with torch.cuda.stream(sa):
            are.gemm_rs(Ad, Bd, out, ws)   # warm-up
        torch.cuda.synchronize()
        copies = [torch.empty((S // C, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        with torch.cuda.stream(sa):
            are.gemm_rs(Ad, Bd, out, ws)
        gen = ws.chunk_generation()
        assert gen == 2
        t = np.full((R, C), np.nan)
        busy = {}
        t0 = time.perf_counter()
        while np.isnan(t).any():
            for s in range(R):
                for c in range(C):
                    if np.isnan(t[s, c]) and ws.chunk_wait(s, c, gen, timeout_ns=0):
                        t[s, c] = time.perf_counter() - t0
                        if c == 0:
                            busy[s] = not sa.query()
                            with torch.cuda.stream(sb):
                                copies[s].copy_(out[s * S:s * S + S // C])
            assert time.perf_counter() - t0 < 10.0, "chunks did not complete"
        torch.cuda.synchronize()
        assert ws.device_status()["code"] == 0
        assert any(busy.values()), "no first chunk was seen before the kernel ended"
        for s in range(R):
            assert torch.equal(copies[s].view(torch.int16), out[s * S:s * S + S // C].view(torch.int16)), s
        if stripe == 0:
            assert t[R - 1, 0] < t[0, C - 1], t
        else:
            assert t[0, C - 1] < t[R - 1, 0], t


def test_chunk_counters_across_graph_replays(oracle):
    """Counters advance by 2^32 per replay of a captured call (never reset, so
    the capture needs no host step between replays)."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K, C = 4, 1024, 512, 128, 4
    A, B, Ad, Bd = _inputs(R, M, N, K, 9)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_chunks(C, 0)
        ws.set_debug(are.DEBUG_PAIR_CTA)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            are.gemm_rs(Ad, Bd, out, ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            are.gemm_rs(Ad, Bd, out, ws)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert ws.device_status()["code"] == 0
        used = oracle.chunk_pieces(R, M, N, C) > 0
        assert np.array_equal(ws.chunk_counters()[:R, :C], np.where(used, 4 * Q, 0).astype(np.uint64))
        for sg in range(R):
            for c in range(C):
                assert ws.chunk_wait(sg, c, 4, timeout_ns=0) == bool(used[sg, c])
        check_close(host_f32(out), oracle.gemm_rs(A, B), "gemm_rs after replays")


def test_chunk_wait_arguments_and_timeout():
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    with are.Workspace(R_max=4, M_max=256, N_max=256, K_max=64) as ws:
        with pytest.raises(are.AreError):
            ws.set_chunks(65)
        with pytest.raises(are.AreError):
            ws.chunk_wait(4, 0, 1)
        t0 = time.perf_counter()
        assert not ws.chunk_wait(0, 0, 1, timeout_ns=2_000_000)
        assert time.perf_counter() - t0 < 1.0
    with are.Workspace(R_max=2, M_max=64, N_max=64) as ws:   # no GEMM buffers
        with pytest.raises(are.AreError):
            ws.set_chunks(2)
