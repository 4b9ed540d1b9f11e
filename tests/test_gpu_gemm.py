"""GEMM + reduce-scatter / all-reduce on the GPU against the CPU oracle."""
import numpy as np
import pytest

import oracle
import oracle as oracle_mod
from oracle import check_close
import synth
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu, sample_rows

pytestmark = pytest.mark.gpu


def make_ws(R_max=8, M_max=1024, N_max=1024, K_max=1024, **kw):
    import all_reduce_epilogue_gb300 as are
    return are.Workspace(R_max=R_max, M_max=M_max, N_max=N_max, K_max=K_max, timeout_ns=kw.pop("timeout_ns", 50_000_000),
                         **kw)


def run_rs(ws, A, B, segmented=False):
    import torch

    import all_reduce_epilogue_gb300 as are
    R = len(A)
    M, K = A[0].shape
    N = B[0].shape[1]
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    if segmented:
        out = [torch.empty((M // R, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        are.gemm_rs(dA, dB, out, ws)
        full = torch.cat(out, 0)
    else:
        full = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(dA, dB, full, ws)
    st = ws.device_status()
    assert st["code"] == 0, st
    return full


def run_ar(ws, A, B, nviews=None):
    import torch

    import all_reduce_epilogue_gb300 as are
    R = len(A)
    M = A[0].shape[0]
    N = B[0].shape[1]
    nviews = R if nviews is None else nviews
    views = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(nviews)]
    out = [views[v % nviews] for v in range(R)]
    are.gemm_ar([dev_bf16(a) for a in A], [dev_bf16(b) for b in B], out, ws)
    st = ws.device_status()
    assert st["code"] == 0, st
    return views


# ----------------------------------------------------------------------------- GEMM+RS

def test_tiny_gemm_rs(oracle):
    """R=2, M=64, N=256, K=128, U[-1,1]: one 128x256 tile holding two 32-row
    owner segments."""
    need_gpu()
    A, B = synth.gemm_inputs(2, 64, 256, 128, synth.config_seed(0), dist="uniform")
    with make_ws() as ws:
        got = host_f32(run_rs(ws, A, B))
    check_close(got, oracle.gemm_rs(A, B), "tiny gemm_rs")


@pytest.mark.parametrize("R,M,N,K", [(3, 264, 320, 136), (1, 8, 8, 8), (2, 16, 264, 72), (4, 512, 768, 64),
                                     (8, 192, 512, 200), (5, 40, 1024, 1024), (7, 56, 8, 24)])
def test_ragged_gemm_rs(oracle, R, M, N, K):
    need_gpu()
    A, B = synth.gemm_inputs(R, M, N, K, 7 * R + M + N + K)
    with make_ws() as ws:
        got = host_f32(run_rs(ws, A, B))
    check_close(got, oracle.gemm_rs(A, B), f"gemm_rs R={R} M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [256, 1024])
def test_gemm_rs_r4_full(oracle, M):
    """GEMM+RS at R=4, N=4096, K=2048 (the full result)."""
    need_gpu()
    A, B = synth.gemm_inputs(4, M, 4096, 2048, synth.config_seed(1))
    with make_ws(R_max=4, M_max=M, N_max=4096, K_max=2048) as ws:
        got = host_f32(run_rs(ws, A, B))
    check_close(got, oracle.gemm_rs(A, B), f"gemm_rs R=4 M={M}")


@pytest.mark.slow
@pytest.mark.parametrize("M", [4096, 8192])
def test_gemm_rs_r4_sampled(oracle, M):
    need_gpu()
    A, B = synth.gemm_inputs(4, M, 4096, 2048, synth.config_seed(1))
    rows = sample_rows(M, 4)
    with make_ws(R_max=4, M_max=M, N_max=4096, K_max=2048) as ws:
        got = host_f32(run_rs(ws, A, B))[rows]
    check_close(got, oracle.gemm_rs(A, B, rows), f"gemm_rs R=4 M={M} sampled")


@pytest.mark.parametrize("R,N", [(4, 4096), (8, 7168)])
def test_gemm_rs_single_tile_row_split(oracle, R, N):
    """GEMM+RS with a single 128-row tile at R >= 4 takes the CTA-pair kernel's
    row-slice split by default (the pair's second tile is absent): the launch
    record says so, the bytes equal the one-CTA kernel's, and the full result
    matches the oracle.  M=128, K=2048, owner segments of 128/R rows."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    M, K = 128, 2048
    A, B = synth.gemm_inputs(R, M, N, K, 4100 + R)
    dA, dB = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    with make_ws(M_max=M, N_max=N, K_max=K) as ws:
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(dA, dB, out, ws)
        assert ws.device_status()["code"] == 0
        li = ws.last_launch()
        assert li["kernel"] == "gemm_pair_kernel" and li["variant"] == 1, li
        ref = torch.empty_like(out)
        ws.set_debug(are.DEBUG_SINGLE_CTA)
        are.gemm_rs(dA, dB, ref, ws)
        assert ws.device_status()["code"] == 0
    assert np.array_equal(host_bits(out), host_bits(ref))
    check_close(host_f32(out), oracle.gemm_rs(A, B), f"gemm_rs R={R} M={M} N={N} single tile row")


def test_integer_inputs_bit_exact(oracle):
    """Small integer operands: every partial and sum is exact in fp32, so the
    bf16 output must equal the oracle's rounding bit for bit."""
    need_gpu()
    from tests.pins import small_ints_bf16
    rng = np.random.default_rng(11)
    R, M, N, K = 4, 256, 512, 192
    A = [small_ints_bf16((M, K), rng) for _ in range(R)]
    B = [small_ints_bf16((K, N), rng) for _ in range(R)]
    with make_ws() as ws:
        got = host_bits(run_rs(ws, A, B))
        views = run_ar(ws, A, B)
    want = oracle.bf16_rne(oracle.gemm_rs(A, B))
    assert np.array_equal(got, want)
    for v in views:
        assert np.array_equal(host_bits(v), oracle.bf16_rne(oracle.gemm_ar(A, B)))


def test_segments_equal_contiguous(oracle):
    """Passing R separate segment buffers gives the same bytes as one
    contiguous [M, N] output (each segment holds its owner's rows)."""
    need_gpu()
    A, B = synth.gemm_inputs(4, 256, 512, 256, 33)
    with make_ws() as ws:
        a = host_bits(run_rs(ws, A, B, segmented=False))
        b = host_bits(run_rs(ws, A, B, segmented=True))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kernel", ["default", "pair", "pair_split"])
def test_masks_and_owner_pieces_bit_exact(oracle, kernel):
    """With re-arm off, every tile's ready word is (1 << R) - 1 (and words past
    the last tile are 0); each reducer's stored owner pieces equal the
    oracle's cut of the tile at owner boundaries.  After a normal call every
    word is 0 again.  Through the default kernel choice and with the CTA-pair
    kernel forced wherever it applies, with either of its GEMM+RS reductions
    (the ring's last rank, or the last of a tile's R row-slice reducers, logs
    the tile's pieces and re-arms its word)."""
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    extra = {"default": 0, "pair": are.DEBUG_PAIR_CTA | are.DEBUG_RS_RING,
             "pair_split": are.DEBUG_PAIR_CTA | are.DEBUG_RS_SPLIT}[kernel]
    for (R, M, N, K) in [(2, 64, 256, 128), (4, 256, 1024, 128), (3, 264, 320, 64), (8, 1024, 512, 64)]:
        A, B = synth.gemm_inputs(R, M, N, K, 5)
        with make_ws(debug_flags=are.DEBUG_NO_REARM | are.DEBUG_LOG_PIECES | extra) as ws:
            run_rs(ws, A, B)
            T = ((M + 127) // 128) * ((N + 255) // 256)
            words = ws.snapshot(are.SNAP_MASKS, (T + 8) * 4).view(np.uint32)
            want, t = oracle.expected_masks(R, M, N, T + 8)
            assert t == T and np.array_equal(words, want), (R, M, N)
            log = ws.snapshot(are.SNAP_PIECES, T * are.PIECE_WORDS * 4).view(np.int32).reshape(T, -1)
            seen = set()
            for t in range(T):
                tm, tn, n = log[t, :3]
                seen.add((int(tm), int(tn)))
                got = [tuple(int(v) for v in log[t, 3 + 3 * i: 6 + 3 * i]) for i in range(n)]
                assert got == oracle.tile_pieces(int(tm) * 128, 128, M, R), (R, M, N, t)
            assert len(seen) == T
            ws.set_debug(extra)
            ws.reset()
            run_rs(ws, A, B)
            assert np.all(ws.snapshot(are.SNAP_MASKS, T * 4).view(np.uint32) == 0)


@pytest.mark.parametrize("kernel", ["single", "pair", "pair_split"])
def test_unpublished_tile_times_out_and_reset_recovers(oracle, kernel):
    """A producer that never sets its ready bit makes the tile's reducer time
    out: the status names the tile, every CTA returns, and a reset recovers.
    Unit 0 is the first producer of tile 0 for the one-CTA kernel, and of the
    first tile pair (tiles 0 and N/256) for the CTA-pair kernel, where with the
    row-slice split every unit of that pair waits for it."""
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 4, 256, 512, 128
    A, B = synth.gemm_inputs(R, M, N, K, 8)
    single_cta = kernel == "single"
    base = {"single": are.DEBUG_SINGLE_CTA, "pair": are.DEBUG_PAIR_CTA | are.DEBUG_RS_RING,
            "pair_split": are.DEBUG_PAIR_CTA | are.DEBUG_RS_SPLIT}[kernel]
    with make_ws(timeout_ns=20_000_000) as ws:
        ws.set_debug(base | are.DEBUG_SKIP_PUBLISH, 0)
        import torch
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs([dev_bf16(a) for a in A], [dev_bf16(b) for b in B], out, ws)
        st = ws.device_status()
        assert st["status"] == are.ETIMEOUT and st["code"] == are.DEV_MASK_TIMEOUT, st
        assert st["a"] in ((0,) if single_cta else (0, N // 256)), st
        ws.set_debug(base)
        ws.reset()
        got = host_f32(run_rs(ws, A, B))
    check_close(got, oracle.gemm_rs(A, B), "after reset")


def test_ring_rank_unpublished_mid_chain_times_out(oracle):
    """GEMM+RS on the CTA-pair kernel's push ring, broken in the middle of a
    tile's chain: rank 2 of the first tile pair adds S_1 and stores S_2 but never
    sets its ready bit, so rank 3's loader times out waiting for it; every CTA
    returns with a timeout status naming one of the pair's tiles, and a reset
    recovers.  The ranks run one after the other over a single block of all
    tile pairs, so the unit of rank r and tile pair p is r * pairs + p
    (here 2 pairs: unit 4)."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 4, 256, 512, 128
    A, B = synth.gemm_inputs(R, M, N, K, 23)
    dA, dB = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with make_ws(timeout_ns=20_000_000) as ws:
        ws.set_debug(are.DEBUG_PAIR_CTA | are.DEBUG_RS_RING | are.DEBUG_SKIP_PUBLISH, 4)
        are.gemm_rs(dA, dB, out, ws)
        st = ws.device_status()
        assert ws.last_launch()["kernel"] == "gemm_pair_kernel" and ws.last_launch()["variant"] == 0
        assert st["status"] == are.ETIMEOUT and st["code"] in (are.DEV_MASK_TIMEOUT, are.DEV_PIPE_TIMEOUT), st
        if st["code"] == are.DEV_MASK_TIMEOUT:
            assert st["a"] in (0, N // 256), st
        ws.set_debug(are.DEBUG_PAIR_CTA | are.DEBUG_RS_RING)
        ws.reset()
        got = host_f32(run_rs(ws, A, B))
    check_close(got, oracle.gemm_rs(A, B), "after reset")


def test_gemm_ar_unpublished_unit_times_out_with_own_slice(oracle):
    """GEMM+AR at R = 8 through the CTA-pair kernel, where each unit keeps its
    own row slice on chip and a drain waits for the reduction two units back:
    when unit 0 never publishes, every slice reducer of that tile pair times out
    on the mask, the drains waiting on those reductions give up with the abort,
    every CTA returns with a timeout status, and a reset recovers the workspace
    (the next call matches the oracle)."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 8, 512, 512, 128
    A, B = synth.gemm_inputs(R, M, N, K, 18)
    dA, dB = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    views = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    with make_ws(timeout_ns=20_000_000) as ws:
        ws.set_debug(are.DEBUG_PAIR_CTA | are.DEBUG_SKIP_PUBLISH, 0)
        are.gemm_ar(dA, dB, views, ws)
        st = ws.device_status()
        assert st["status"] == are.ETIMEOUT and st["code"] in (are.DEV_MASK_TIMEOUT, are.DEV_PIPE_TIMEOUT), st
        assert ws.last_launch()["kernel"] == "gemm_pair_kernel"
        ws.set_debug(are.DEBUG_PAIR_CTA)
        ws.reset()
        are.gemm_ar(dA, dB, views, ws)
        assert ws.device_status()["code"] == 0
        ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws.set_debug(are.DEBUG_SINGLE_CTA)
        are.gemm_ar(dA, dB, ref, ws)
        assert ws.device_status()["code"] == 0
    for v in views:  # after the reset: the one-CTA kernel's bytes, and the oracle's values
        assert np.array_equal(host_bits(v), host_bits(ref))
    assert oracle_mod.rel_l2(host_f32(ref), oracle.gemm_ar(A, B)) <= 2e-3


def test_k_zero_and_empty(oracle):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    with make_ws() as ws:
        A = [torch.zeros((64, 0), dtype=torch.bfloat16, device="cuda")] * 2
        B = [torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")] * 2
        out = torch.full((64, 256), 1.0, dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(A, B, out, ws)
        assert torch.all(out == 0)
        E = [torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")] * 2
        are.gemm_rs(E, [torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")] * 2,
                    torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), ws)
        with pytest.raises(are.AreError) as e:
            are.gemm_rs([torch.zeros((60, 64), dtype=torch.bfloat16, device="cuda")] * 2,
                        [torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")] * 2,
                        torch.empty((60, 256), dtype=torch.bfloat16, device="cuda"), ws)  # S = 30
        assert e.value.status == are.EINVAL
        torch.cuda.synchronize()


# ----------------------------------------------------------------------------- GEMM+AR

@pytest.mark.parametrize("R,M,N,K,nviews", [(8, 64, 7168, 2048, 8), (8, 512, 7168, 2048, 1), (3, 200, 328, 72, 2),
                                            (1, 5, 16, 8, 1), (2, 130, 520, 136, 2)])
def test_gemm_ar(oracle, R, M, N, K, nviews):
    need_gpu()
    A, B = synth.gemm_inputs(R, M, N, K, synth.config_seed(2) + M)
    with make_ws(M_max=1024, N_max=7168, K_max=2048) as ws:
        views = run_ar(ws, A, B, nviews)
    ref = oracle.gemm_ar(A, B)
    first = host_bits(views[0])
    check_close(synth.bf16_bits_to_f32(first), ref, f"gemm_ar R={R} M={M}")
    for v in views[1:]:
        assert np.array_equal(host_bits(v), first)


@pytest.mark.slow
def test_gemm_ar_m4096_sampled(oracle):
    need_gpu()
    A, B = synth.gemm_inputs(8, 4096, 7168, 2048, synth.config_seed(2))
    rows = sample_rows(4096, 8)
    with make_ws(M_max=4096, N_max=7168, K_max=2048) as ws:
        views = run_ar(ws, A, B, 1)
    check_close(host_f32(views[0])[rows], oracle.gemm_ar(A, B, rows), "gemm_ar M=4096 sampled")


# ----------------------------------------------------------------------------- large GEMM+RS

@pytest.mark.slow
def test_large_gemm_rs_sampled_and_deterministic(oracle):
    """R=8, M=N=8192, K=4096: sampled rows against the oracle, and two runs with
    the same inputs give identical bytes."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 8, 8192, 8192, 4096
    A, B = synth.gemm_inputs(R, M, N, K, synth.config_seed(4))
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    rows = sample_rows(M, R, n_random=8)
    with make_ws(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        o1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        o2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(dA, dB, o1, ws)
        are.gemm_rs(dA, dB, o2, ws)
        st = ws.device_status()
        assert st["code"] == 0, st
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), "not deterministic"
        got = host_f32(o1)[rows]
    check_close(got, oracle.gemm_rs(A, B, rows), "large gemm_rs sampled")


@pytest.mark.parametrize("mode,R,M,N,K", [("rs", 8, 1024, 1024, 512), ("rs", 3, 384, 520, 136), ("ar", 8, 640, 7168, 256),
                                          ("ar", 2, 512, 1024, 1024)])
def test_pair_kernel_matches_single_cta_kernel(mode, R, M, N, K):
    """The CTA-pair kernel (256-row tiles, cta_group::2) and the one-CTA kernel
    compute each output element with the same operations in the same order,
    so their outputs are bitwise identical (several waves, an odd number of
    tile rows where one CTA of the last pair has no tile); for GEMM+RS so are
    the pair kernel's two reductions, the ring and the row-slice split."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    A, B = synth.gemm_inputs(R, M, N, K, 321 + M + R)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    outs = []
    kinds = (are.DEBUG_PAIR_CTA, are.DEBUG_SINGLE_CTA)
    if mode == "rs":
        kinds += (are.DEBUG_PAIR_CTA | are.DEBUG_RS_RING, are.DEBUG_PAIR_CTA | are.DEBUG_RS_SPLIT)
    for flags in kinds:
        with make_ws(M_max=M, N_max=N, K_max=K, debug_flags=flags) as ws:
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            if mode == "rs":
                are.gemm_rs(dA, dB, out, ws)
            else:
                are.gemm_ar(dA, dB, [out] * R, ws)
            assert ws.device_status()["code"] == 0
            outs.append(host_bits(out))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


@pytest.mark.gpu
def test_wait_profile_counts_and_leaves_results_unchanged():
    """With the wait profile on, the pair kernel's output is bitwise the same
    and every role has reported: one producer per CTA, the MMA span covers the
    MMA waits, and no wait fraction exceeds its span."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 4, 1024, 1024, 512
    A, B = synth.gemm_inputs(R, M, N, K, 777)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in B]
    with make_ws(M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_PAIR_CTA)
        out0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(dA, dB, out0, ws)
        ws.reset()
        ws.set_debug(are.DEBUG_WAIT_PROFILE | are.DEBUG_PAIR_CTA)
        out1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        are.gemm_rs(dA, dB, out1, ws)
        assert ws.device_status()["code"] == 0
        c = ws.snapshot(are.SNAP_COUNTERS, 128).view(np.uint64)
    assert np.array_equal(host_bits(out0), host_bits(out1))
    ctas = int(c[8])
    assert ctas >= 2 and ctas % 2 == 0
    assert c[4] > 0 and c[2] + c[3] <= c[4]
