"""Seeded random shapes for GEMM+RS and GEMM+AR: every rank count of the
workloads, ragged M and N, several K.  For each shape the CTA-pair kernel (or
the one-CTA kernel when there is a single tile row; for GEMM+RS both of its reductions,
the ring and the row-slice split) must return the one-CTA kernel's bytes, no wait may expire, and the result must match the oracle
within the parity tolerance."""
import numpy as np
import pytest

import synth
from oracle import check_close
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu

pytestmark = pytest.mark.gpu


def _shapes(seed: int, n: int):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        mode = str(rng.choice(["ar", "rs"]))
        R = int(rng.choice([1, 2, 3, 4, 5, 8, 8, 8]))
        if mode == "rs":
            M = int(rng.choice([8, 16, 24, 40, 64, 128, 136])) * R  # owner segments of M/R rows, 8 | M/R
        else:
            M = int(rng.integers(129, 1500))
        N = int(rng.integers(1, 160)) * 8
        K = int(rng.integers(1, 5)) * 64
        out.append((mode, R, M, N, K))
    return out


@pytest.mark.parametrize("case", range(16))
def test_random_shapes_pair_equals_one_cta_and_oracle(oracle, case):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    mode, R, M, N, K = _shapes(2026, 16)[case]
    A, B = synth.gemm_inputs(R, M, N, K, 3000 + case)
    Ad, Bd = [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(ref)
    call = are.gemm_ar if mode == "ar" else are.gemm_rs
    with are.Workspace(R_max=8, M_max=M, N_max=N, K_max=K) as ws:
        ws.set_debug(are.DEBUG_SINGLE_CTA)
        call(Ad, Bd, ref, ws)
        assert ws.device_status()["code"] == 0
        ws.set_debug(are.DEBUG_PAIR_CTA if M > 128 else 0)
        call(Ad, Bd, out, ws)
        st = ws.device_status()
        assert st["code"] == 0, st
        assert np.array_equal(host_bits(out), host_bits(ref)), (mode, R, M, N, K)
        if mode == "rs" and M > 128:
            # both GEMM+RS reductions of the pair kernel: the ring and the row-slice split
            for flag in (are.DEBUG_RS_RING, are.DEBUG_RS_SPLIT):
                out.zero_()
                ws.set_debug(are.DEBUG_PAIR_CTA | flag)
                call(Ad, Bd, out, ws)
                st = ws.device_status()
                assert st["code"] == 0, (flag, st)
                assert ws.last_launch()["variant"] == (1 if flag == are.DEBUG_RS_SPLIT else 0)
                assert np.array_equal(host_bits(out), host_bits(ref)), (flag, mode, R, M, N, K)
    Y = oracle.gemm_ar(A, B) if mode == "ar" else oracle.gemm_rs(A, B)
    check_close(host_f32(out), Y, f"{mode} R={R} M={M} N={N} K={K}")
