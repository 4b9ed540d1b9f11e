"""bench.py's host-side arithmetic on the CPU: the work model every roofline
fraction divides by, the choice of the burst or the sustained bf16 peak from
the clock samples of the timed region, the roofline as the larger of the
compute and the memory bound, and the ncu traffic figures being dropped once
the kernel source they were taken on has changed."""
import numpy as np

import bench


def _bytes(shapes, itemsize):
    return float(sum(int(np.prod(s)) * itemsize for s in shapes))


def test_gemm_work_counts_every_multiply_add_and_each_tensor_once():
    # FLOPs: one multiply and one add per (rank, row, column, k) term of the R products
    R, M, N, K = 2, 3, 4, 5
    terms = sum(1 for r in range(R) for i in range(M) for j in range(N) for k in range(K))
    assert bench.work_of("gemm_rs", R, M, N, K)[0] == 2 * terms
    assert bench.work_of("gemm_ar", R, M, N, K)[0] == 2 * terms
    # bytes: the R bf16 operand pairs read once, the bf16 output written once (GEMM+RS: the
    # M x N result split over the owner segments; GEMM+AR: one full view per rank)
    R, M, N, K = 8, 8192, 8192, 4096
    rs = [(M, K)] * R + [(K, N)] * R + [(M // R, N)] * R
    assert bench.work_of("gemm_rs", R, M, N, K)[1] == _bytes(rs, 2)
    R, M, N, K = 8, 4096, 7168, 2048
    ar = [(M, K)] * R + [(K, N)] * R + [(M, N)] * R
    assert bench.work_of("gemm_ar", R, M, N, K)[1] == _bytes(ar, 2)


def test_allreduce_rmsnorm_work_is_its_tensors():
    R, M, N = 8, 4096, 7168
    with_res = _bytes([(M, N)] * R + [(M, N), (M, N)], 2) + _bytes([(N,)], 4)  # partials, residual, out; gamma
    no_res = _bytes([(M, N)] * R + [(M, N)], 2) + _bytes([(N,)], 4)
    assert bench.work_of("allreduce_rmsnorm", R, M, N) == (0.0, with_res)
    assert bench.work_of("allreduce_rmsnorm", R, M, N, residual=False) == (0.0, no_res)
    assert abs(with_res - 587.3e6) < 0.1e6  # the figure the roofline fractions quote


def test_roofline_is_the_larger_of_the_compute_and_memory_bounds():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1000.0}
    assert bench.roofline_seconds_of(2e12, 1e9, peaks, "burst") == 1e-3      # compute: 2e12 / 2e15
    assert bench.roofline_seconds_of(2e12, 1e9, peaks, "sustained") == 2e-3  # compute: 2e12 / 1e15
    assert bench.roofline_seconds_of(1e9, 4e9, peaks, "burst") == 4e-3       # memory: 4e9 / 1e12


def test_peak_regime_follows_the_clock_samples():
    def clocks(sm, reasons=(), window="timed region"):
        return {"sm_mhz": sm, "sm_max_mhz": 2070.0, "reasons": list(reasons), "window": window}
    assert bench.peak_regime(clocks(2070.0))[0] == "burst"
    assert bench.peak_regime(clocks(2010.0))[0] == "burst"                    # within 3 % of the maximum
    assert bench.peak_regime(clocks(1900.0))[0] == "sustained"                # clock held low
    assert bench.peak_regime(clocks(2070.0, ["sw_power_cap"]))[0] == "sustained"
    assert bench.peak_regime(clocks(None))[0] == "burst"                      # no sample: the larger peak
    assert bench.peak_regime(clocks(1400.0, window="whole run"))[0] == "burst"
    peaks = {"hbm_gbs": 1.0, "bf16_tflops": 1896.2, "bf16_tflops_sustained": 1698.0}
    assert bench.bf16_peak(peaks, "burst") == 1896.2 and bench.bf16_peak(peaks, "sustained") == 1698.0


def test_ncu_traffic_is_dropped_once_the_kernel_source_changes(monkeypatch):
    part = "gemm_rs"
    val, sha = bench.NCU_TRAFFIC[part]
    monkeypatch.setattr(bench, "source_sha16", lambda name: sha)
    assert bench.ncu_traffic(part) == val
    monkeypatch.setattr(bench, "source_sha16", lambda name: "0" * 16)
    assert bench.ncu_traffic(part) is None
