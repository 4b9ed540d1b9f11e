"""The CTA-pair kernel's unit order (raster groups, rank blocks, rank groups)
and the destination-rotated order of chunked GEMM+RS change the order in which
work units run, never the arithmetic: every order must give the same output
bytes, in both modes, with odd numbers of tile rows (a pair whose second tile
does not exist) and ragged N; every tile mask is re-armed to 0 after each
call.  GEMM+AR splits each tile's reduction into R row slices, one per unit of
the pair (two-shot), which also must not change a byte; GEMM+RS runs every
order with each of its two reductions, the ring and the row-slice split."""
import numpy as np
import pytest

import synth
from oracle import check_close
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu

pytestmark = pytest.mark.gpu

# (group_m, block_pairs, rank_group)
ORDERS = [
    (0, -1, 0),      # a pair's R units consecutive
    (1, -1, 0),
    (2, 2, 1),       # rank by rank in blocks of 2 pairs
    (2, 3, 2),       # ranks in groups of 2, blocks of 3
    (1, 4, 3),       # groups of 3 ranks (the last group smaller when 3 does not divide R)
    (0, 0, 0),       # the library's choice
]


@pytest.mark.parametrize("mode", ["rs", "rs_split", "ar"])
@pytest.mark.parametrize("R,M,N,K", [(4, 1152, 1000, 192), (3, 768, 520, 64), (8, 2048, 768, 128),
                                     (5, 1280, 256, 128)])
def test_order_changes_no_output_byte(oracle, mode, R, M, N, K):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    A, B = synth.gemm_inputs(R, M, N, K, 500 + M + R)
    Ad, Bd = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    call = are.gemm_ar if mode == "ar" else are.gemm_rs
    reduction = {"rs": are.DEBUG_RS_RING, "rs_split": are.DEBUG_RS_SPLIT, "ar": 0}[mode]
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_SINGLE_CTA)       # the one-CTA kernel: whole-tile reduction
        call(Ad, Bd, ref, ws)
        assert ws.device_status()["code"] == 0
        Y = oracle.gemm_ar(A, B) if mode == "ar" else oracle.gemm_rs(A, B)
        check_close(host_f32(ref), Y, f"gemm_{mode} one-CTA kernel")
        ws.set_debug(are.DEBUG_PAIR_CTA | reduction)
        T = -(-M // 128) * -(-N // 256)
        for order in ORDERS:
            ws.set_gemm_order(*order)
            for _ in range(2):
                out = torch.zeros_like(ref)
                call(Ad, Bd, out, ws)
                st = ws.device_status()
                assert st["code"] == 0, (order, st)
                assert ws.last_launch()["kernel"] == "gemm_pair_kernel"
                assert np.array_equal(host_bits(out), host_bits(ref)), order
                masks = ws.snapshot(are.SNAP_MASKS, T * 4).view(np.uint32)
                assert np.all(masks == 0), order


def test_orders_with_chunks_and_rotation(oracle):
    """The rank blocks compose with chunk counting and the destination-rotated
    order: same bytes, exact counters."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K, C = 4, 2048, 768, 128, 4
    A, B = synth.gemm_inputs(R, M, N, K, 808)
    Ad, Bd = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(ref)
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_PAIR_CTA)
        are.gemm_rs(Ad, Bd, ref, ws)
        ws.set_chunks(C, 1)
        for order in [(0, -1, 0), (0, 3, 1), (0, 0, 0)]:
            ws.set_gemm_order(*order)
            are.gemm_rs(Ad, Bd, out, ws)
            assert ws.device_status()["code"] == 0
            assert np.array_equal(host_bits(out), host_bits(ref)), order
        used = oracle.chunk_pieces(R, M, N, C) > 0
        assert np.array_equal(ws.chunk_counters()[:R, :C], np.where(used, 3 << 32, 0).astype(np.uint64))
        check_close(host_f32(out), oracle.gemm_rs(A, B), "orders + chunks + rotation")


@pytest.mark.parametrize("order", [(0, 76, 1), (0, 76, 2), (2, 38, 8), (0, -1, 0), (0, 19, 1), (4, 19, 4), (0, 9, 2)])
def test_ar_rank_blocks_spanning_many_steps(order):
    """GEMM+AR at R = 8 keeps a unit's own row slice on chip only while a
    pair's units lie within two steps of the persistent loop; a rank-blocked
    order that spreads a pair over up to R steps (blocks of 76 pairs, ranks in
    groups of 1 or 2) must run through memory instead, with no expired wait
    and the same bytes as the one-CTA kernel (whole-tile reduction in the same
    rank order) and the library's own order.  Blocks of 19 pairs (two waves of
    76 clusters) or of 9 (under one wave) keep the own slice on chip."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, M, N, K = 8, 4096, 2560, 128  # 160 tile pairs, 1280 units: many steps of 76 clusters
    A, B = synth.gemm_inputs(R, M, N, K, 4242)
    Ad, Bd = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(ref)
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_SINGLE_CTA)
        are.gemm_ar(Ad, Bd, ref, ws)
        assert ws.device_status()["code"] == 0
        ws.set_debug(are.DEBUG_PAIR_CTA)
        are.gemm_ar(Ad, Bd, out, ws)
        assert ws.device_status()["code"] == 0
        assert np.array_equal(host_bits(out), host_bits(ref))
        ws.set_gemm_order(*order)
        for _ in range(2):
            out.zero_()
            are.gemm_ar(Ad, Bd, out, ws)
            st = ws.device_status()
            assert st["code"] == 0, (order, st)
            assert ws.last_launch()["kernel"] == "gemm_pair_kernel"
            assert np.array_equal(host_bits(out), host_bits(ref)), order


@pytest.mark.parametrize("R,M,N,K", [(8, 600, 1000, 192), (8, 1300, 264, 128)])
def test_ar_own_slice_odd_tile_rows_ragged(oracle, R, M, N, K):
    """GEMM+AR at R = 8 with an odd number of tile rows (the last pair's second
    CTA has no tile, so the two CTAs of a cluster count their units differently),
    M not a multiple of 16 (slices past the last row) and ragged N: the pair
    kernel, which keeps each unit's own row slice on chip and writes the views
    with TMA tensor stores, gives the one-CTA kernel's bytes and the oracle's
    values, with no expired wait."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    A, B = synth.gemm_inputs(R, M, N, K, 9000 + M)
    Ad, Bd = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    views = [torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_SINGLE_CTA)
        are.gemm_ar(Ad, Bd, ref, ws)
        assert ws.device_status()["code"] == 0
        ws.set_debug(are.DEBUG_PAIR_CTA)
        for _ in range(2):
            are.gemm_ar(Ad, Bd, views, ws)
            st = ws.device_status()
            assert st["code"] == 0, st
            assert ws.last_launch()["kernel"] == "gemm_pair_kernel"
            for v in views:
                assert np.array_equal(host_bits(v), host_bits(ref))
    check_close(host_f32(views[0]), oracle.gemm_ar(A, B), f"gemm_ar R={R} M={M} N={N} K={K}")
