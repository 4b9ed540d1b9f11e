"""Mixed GEMM calls on one workspace: the GEMM+RS row-slice split, the ring,
the single-tile-row split, the one-CTA kernel and GEMM+AR (whose two-shot
reduction shares the per-tile slice count with the split) in a seeded random
order.  Every call must finish without a device error and return the same
bytes as the first call of its shape, the first call of each shape must match
the oracle, and every tile's mask word must be 0 again at the end (each
call's last reader re-armed it)."""
import numpy as np
import pytest

import synth
from oracle import check_close
from tests.gpu_util import dev_bf16, host_bits, host_f32, need_gpu

pytestmark = pytest.mark.gpu

# (mode, R, M, N, K, the pair kernel's reduction: 1 = row slices, 0 = ring, None = one-CTA kernel);
# the dispatch thresholds are the GB300s' (76 co-resident clusters of two)
CASES = [
    ("rs", 4, 256, 4096, 512, 1),     # the row-slice split below one wave
    ("rs", 2, 1024, 1024, 256, 0),    # the ring (R < 4)
    ("rs", 8, 128, 2048, 256, 1),     # the split with a single tile row
    ("rs", 2, 64, 256, 128, None),    # the one-CTA kernel
    ("ar", 8, 512, 4096, 256, 1),     # GEMM+AR (two-shot), 3.4 waves of pair units
]


def test_mixed_gemm_calls_share_a_workspace(oracle):
    need_gpu()
    import torch

    import all_reduce_epilogue_gb300 as are
    inputs, firsts = [], []
    for i, (mode, R, M, N, K, _) in enumerate(CASES):
        A, B = synth.gemm_inputs(R, M, N, K, 7700 + i)
        inputs.append((A, B, [dev_bf16(a) for a in A], [dev_bf16(b) for b in B]))
    rng = np.random.default_rng(77)
    order = list(range(len(CASES))) + [int(v) for v in rng.integers(0, len(CASES), 35)]
    with are.Workspace(R_max=8, M_max=1024, N_max=4096, K_max=512) as ws:
        seen = {}
        for i in order:
            mode, R, M, N, K, split = CASES[i]
            A, B, dA, dB = inputs[i]
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            if mode == "rs":
                are.gemm_rs(dA, dB, out, ws)
            else:
                are.gemm_ar(dA, dB, [out] * R, ws)
            st = ws.device_status()
            assert st["code"] == 0, (CASES[i], st)
            li = ws.last_launch()
            if split is None:
                assert li["kernel"] == "gemm_reduce_kernel", li
            else:
                assert li["kernel"] == "gemm_pair_kernel" and li["variant"] == split, (CASES[i], li)
            bits = host_bits(out)
            if i not in seen:
                seen[i] = bits
                Y = oracle.gemm_rs(A, B) if mode == "rs" else oracle.gemm_ar(A, B)
                check_close(host_f32(out), Y, f"{CASES[i]}")
            else:
                assert np.array_equal(bits, seen[i]), CASES[i]
        T = max(-(-M // 128) * -(-N // 256) for (_, _, M, N, _, _) in CASES)
        masks = ws.snapshot(are.SNAP_MASKS, T * 4).view(np.uint32)
        assert np.all(masks == 0)
