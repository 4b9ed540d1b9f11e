"""Which kernel each call launches (the host-side launch record), for the
workload shapes and the dispatch boundaries: for GEMM+RS CTA pairs wherever
there are at least two 128-row tiles, with the row-slice split for R = 4 and 8
with K <= 2048 up to three quarters of a wave of tile pairs and otherwise up to
half a wave (then also with a single tile row), and the ring beyond; for GEMM+AR CTA pairs
from one wave of pair units on (also with a single tile row), one CTA per tile
otherwise; the one-shot AR+RMSNorm kernel up to the per-rank
byte threshold, the Lamport kernel above it; memsets for an empty
contraction.  The results themselves are covered by the parity tests."""
import pytest

from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _gemm(op, R, M, N, K, flags=0):
    import torch

    import all_reduce_epilogue_gb300 as are
    A = [torch.zeros((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    B = [torch.zeros((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=R, M_max=M, N_max=N, K_max=max(K, 64)) as ws:
        ws.set_debug(flags)
        assert ws.last_launch()["kernel"] == "none"
        (are.gemm_rs if op == "rs" else are.gemm_ar)(A, B, out, ws)
        assert ws.device_status()["code"] == 0
        return ws.last_launch()


@pytest.mark.parametrize("op,R,M,N,K,kernel,split", [
    ("rs", 2, 64, 256, 128, "gemm_reduce_kernel", 0),      # tiny: one tile row, R < 4
    ("rs", 4, 128, 4096, 2048, "gemm_pair_kernel", 1),     # one tile row, the split (the pair's second tile absent)
    ("rs", 8, 128, 7168, 2048, "gemm_pair_kernel", 1),
    ("rs", 4, 256, 4096, 2048, "gemm_pair_kernel", 1),     # below one wave of pairs
    ("rs", 4, 512, 4096, 2048, "gemm_pair_kernel", 1),     # 32 tile pairs
    ("rs", 8, 384, 4096, 2048, "gemm_pair_kernel", 1),     # 32 tile pairs, 3.4 waves of units
    ("rs", 6, 384, 4096, 2048, "gemm_pair_kernel", 1),     # R = 6: 32 tile pairs, up to half a wave
    ("rs", 6, 768, 4096, 2048, "gemm_pair_kernel", 0),     # R = 6: 48 tile pairs, the ring
    ("rs", 8, 384, 7168, 2048, "gemm_pair_kernel", 1),     # 56 tile pairs, K = 2048: the split
    ("rs", 8, 384, 7168, 4096, "gemm_pair_kernel", 0),     # 56 tile pairs, K = 4096: the ring
    ("rs", 2, 256, 4096, 2048, "gemm_pair_kernel", 0),     # a ring of two
    ("rs", 4, 1024, 4096, 2048, "gemm_pair_kernel", 0),    # 64 tile pairs: the ring (a padded block)
    ("rs", 4, 8192, 4096, 2048, "gemm_pair_kernel", 0),
    ("rs", 8, 8192, 8192, 4096, "gemm_pair_kernel", 0),
    ("ar", 8, 64, 7168, 2048, "gemm_pair_kernel", 1),     # one tile row: the pair's second tile is empty
    ("ar", 8, 1, 1000, 128, "gemm_reduce_kernel", 0),     # below one wave of pairs
    ("ar", 8, 4096, 7168, 2048, "gemm_pair_kernel", 1),
    ("rs", 2, 64, 256, 0, "memset", 0),
])
def test_gemm_dispatch(op, R, M, N, K, kernel, split):
    """The thresholds are stated for the GB300s (76 co-resident clusters
    of two)."""
    need_gpu()
    li = _gemm(op, R, M, N, K)
    assert li["kernel"] == kernel, li
    if kernel == "gemm_pair_kernel":
        assert li["variant"] == split, li
    if kernel == "gemm_pair_kernel":
        assert li["cluster"] == 2 and li["grid"] % 2 == 0 and li["block"] == 384, li
    if kernel == "gemm_reduce_kernel":
        assert li["cluster"] == 1 and li["block"] == 256, li


def test_ring_block_is_padded_to_a_wave_for_short_units():
    """GEMM+RS on the ring with most of a wave of tile pairs but not a whole one
    runs each rank in a wave of its own (a block padded to the co-resident
    clusters) when its units are short (K <= 2048); otherwise one block of the
    actual pairs."""
    need_gpu()
    li = _gemm("rs", 4, 1024, 4096, 2048)        # 64 tile pairs
    clusters = li["grid"] // 2
    assert li["variant"] == 0 and li["rank_block"] == clusters > 64, li
    li = _gemm("rs", 8, 512, 8192, 4096)         # 64 tile pairs, K = 4096
    assert li["variant"] == 0 and li["rank_block"] == 64, li
    li = _gemm("rs", 2, 256, 4096, 2048)         # 16 tile pairs: a sparse wave
    assert li["variant"] == 0 and li["rank_block"] == 16, li


def test_gemm_debug_flags_force_kernels():
    need_gpu()
    import all_reduce_epilogue_gb300 as are
    assert _gemm("rs", 4, 256, 4096, 2048, are.DEBUG_SINGLE_CTA)["kernel"] == "gemm_reduce_kernel"
    assert _gemm("rs", 4, 8192, 4096, 2048, are.DEBUG_SINGLE_CTA)["kernel"] == "gemm_reduce_kernel"
    assert _gemm("ar", 2, 256, 512, 128, are.DEBUG_PAIR_CTA)["kernel"] == "gemm_pair_kernel"
    li = _gemm("rs", 4, 256, 4096, 2048, are.DEBUG_RS_RING)
    assert li["kernel"] == "gemm_pair_kernel" and li["variant"] == 0, li
    li = _gemm("rs", 4, 8192, 4096, 2048, are.DEBUG_RS_SPLIT)
    assert li["kernel"] == "gemm_pair_kernel" and li["variant"] == 1, li


@pytest.mark.parametrize("M,kernel", [(1, "ar_oneshot_kernel"), (16, "ar_oneshot_kernel"),
                                      (128, "ar_rmsnorm_kernel"), (4096, "ar_rmsnorm_kernel")])
def test_allreduce_rmsnorm_dispatch(M, kernel):
    """Default threshold 448 KiB per rank: at N=7168 one row is 14 KiB, so
    M <= 32 takes the one-shot kernel."""
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    R, N = 8, 7168
    P = [torch.zeros((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    g = torch.ones(N, dtype=torch.float32, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with are.Workspace(R_max=8, M_max=M, N_max=N) as ws:
        are.allreduce_rmsnorm(P, None, g, 1e-6, out, ws)
        assert ws.device_status()["code"] == 0
        li = ws.last_launch()
        assert li["kernel"] == kernel, li
        assert li["variant"] == 4, li  # 896 packs of 8 over 256 threads
        for flag, forced in ((are.DEBUG_AR_ONESHOT, "ar_oneshot_kernel"), (are.DEBUG_AR_LAMPORT, "ar_rmsnorm_kernel")):
            ws.set_debug(flag)
            are.allreduce_rmsnorm(P, None, g, 1e-6, out, ws)
            assert ws.last_launch()["kernel"] == forced
        ws.set_debug(0)
        assert ws.device_status()["code"] == 0
