"""Pins of the CPU oracle to facts outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with something the pages or the mathematics fix: fp64 brute
force, exact integer products, identity / one-hot operands, sums whose fp32
result depends on the order, torch's own ``rms_norm`` and bf16 rounding, the
closed forms of RMSNorm, and hand-derived fixtures under ``tests/golden/``.
They are plain functions so that the pin-strength test can run every one of
them against oracle builds with a planted mistake.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16))


def to_bf16_bits(x_f32):
    """Round fp32 -> bf16 with torch (a library routine, round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def small_ints_bf16(shape, rng, lo=-3, hi=3):
    return to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def pin_bf16_rne(o):
    # hand-derived: ties go to even, NaN stays NaN, overflow rounds to inf
    cases = {0x3F800000: 0x3F80, 0x3F808000: 0x3F80, 0x3F818000: 0x3F82, 0x3F808001: 0x3F81,
             0x80000000: 0x8000, 0x7F800000: 0x7F80, 0x7F7FFFFF: 0x7F80, 0xBF7FFFFF: 0xBF80}
    for xb, want in cases.items():
        x = np.array([xb], dtype=np.uint32).view(np.float32)
        got = int(o.bf16_rne(x)[0])
        assert got == want, f"bf16_rne({xb:#x}) = {got:#x}, want {want:#x}"
    nan = np.array([0x7FC00001], dtype=np.uint32).view(np.float32)
    g = int(o.bf16_rne(nan)[0])
    assert (g & 0x7F80) == 0x7F80 and (g & 0x7F) != 0, "NaN must stay NaN"
    # against torch on random fp32 values
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(2000) * np.exp2(rng.integers(-20, 20, 2000))).astype(np.float32)
    assert np.array_equal(o.bf16_rne(x), to_bf16_bits(x)), "bf16_rne disagrees with torch"


# ---------------------------------------------------------------------------
# partial GEMM
# ---------------------------------------------------------------------------

def pin_partial_vs_fp64(o):
    """fp32 oracle vs an fp64 matmul of the same bf16 values (K <= 128)."""
    for (M, N, K, seed) in [(7, 33, 128, 3), (16, 64, 96, 4), (5, 9, 1, 5)]:
        A = synth.uniform_bf16((M, K), seed, synth.T_A)
        B = synth.uniform_bf16((K, N), seed, synth.T_B)
        P = o.partial_gemm(A, B).astype(np.float64)
        ref = f32(A).astype(np.float64) @ f32(B).astype(np.float64)
        # fp32 accumulation bound: |err_ij| <= K * 2^-24 * sum_k |a_ik||b_kj|
        bound = K * 2.0 ** -24 * (np.abs(f32(A)).astype(np.float64) @ np.abs(f32(B)).astype(np.float64))
        assert np.all(np.abs(P - ref) <= bound + 1e-30), "partial GEMM outside the fp32 error bound"
        den = np.linalg.norm(ref)
        assert np.linalg.norm(P - ref) / den <= 1e-6, "partial GEMM relL2 vs fp64 > 1e-6"


def pin_partial_exact_integers(o):
    """Small integer operands: every product and partial sum is exact in fp32."""
    rng = np.random.default_rng(7)
    A = small_ints_bf16((9, 40), rng)
    B = small_ints_bf16((40, 17), rng)
    P = o.partial_gemm(A, B)
    ref = f32(A).astype(np.int64) @ f32(B).astype(np.int64)
    assert np.array_equal(P.astype(np.int64), ref) and np.all(P == ref), "integer GEMM not exact"


def pin_partial_rectangular(o):
    """A [M,K] times B [K,N] with M, N, K distinct: a transposed operand cannot
    even produce the right values (checked by brute force on a 3x4x5 case)."""
    A = to_bf16_bits(np.arange(1, 16, dtype=np.float32).reshape(3, 5))
    B = to_bf16_bits(np.arange(-10, 10, dtype=np.float32).reshape(5, 4))
    P = o.partial_gemm(A, B)
    a, b = f32(A), f32(B)
    for i in range(3):
        for j in range(4):
            want = sum(float(a[i, k]) * float(b[k, j]) for k in range(5))
            assert float(P[i, j]) == want, f"P[{i},{j}] = {P[i, j]}, brute force {want}"


# ---------------------------------------------------------------------------
# ring-order reduce
# ---------------------------------------------------------------------------

def pin_rs_vs_fp64(o):
    """Y = sum_r A_r B_r against fp64 brute force (R <= 3, tiny shapes)."""
    for (R, M, N, K, seed) in [(3, 12, 40, 64, 11), (2, 5, 7, 128, 12), (1, 8, 16, 32, 13)]:
        A, B = synth.gemm_inputs(R, M, N, K, seed, dist="uniform")
        Y = o.gemm_rs(A, B).astype(np.float64)
        ref = sum(f32(A[r]).astype(np.float64) @ f32(B[r]).astype(np.float64) for r in range(R))
        assert np.linalg.norm(Y - ref) / np.linalg.norm(ref) <= 1e-6, "GEMM+RS relL2 vs fp64 > 1e-6"
        if R == 1:
            assert np.array_equal(Y.astype(np.float32), o.partial_gemm(A[0], B[0])), "R=1 is not the plain GEMM"


def pin_rs_identity_ring_order(o):
    """B_r = I (K = N): P_r = A_r exactly, so Y is the fp32 sum of the A_r in
    ring order.  The values 2^24, 1, -2^24 make the order visible:
    (2^24 + 1) rounds to 2^24 in fp32, so ((2^24 + 1) - 2^24) = 0 while any
    order that adds 1 last gives 1."""
    N = 8
    eye = to_bf16_bits(np.eye(N, dtype=np.float32))
    a0 = np.zeros((2, N), np.float32); a1 = np.zeros((2, N), np.float32); a2 = np.zeros((2, N), np.float32)
    a0[0, 0], a1[0, 0], a2[0, 0] = 2.0 ** 24, 1.0, -(2.0 ** 24)   # ring order -> 0
    a0[0, 1], a1[0, 1], a2[0, 1] = 1.0, 2.0 ** 24, -(2.0 ** 24)   # ring order -> 0
    a0[1, 2], a1[1, 2], a2[1, 2] = 2.0 ** 24, -(2.0 ** 24), 1.0   # ring order -> 1
    a0[1, 3], a1[1, 3], a2[1, 3] = 3.0, -5.0, 0.5                  # -1.5
    A = [to_bf16_bits(a) for a in (a0, a1, a2)]
    Y = o.gemm_rs(A, [eye, eye, eye])
    want = np.zeros((2, N), np.float32)
    want[1, 2] = 1.0
    want[1, 3] = -1.5
    assert np.array_equal(Y, want), f"ring-order sum wrong: {Y}"


def pin_rs_one_hot(o):
    """A_r rows one-hot at column pi_r(i): row i of Y is the ring-order sum of
    row pi_r(i) of each B_r (exact here: B values are small integers)."""
    R, M, N, K = 3, 6, 10, 12
    rng = np.random.default_rng(5)
    A, B, picks = [], [], []
    for r in range(R):
        p = rng.permutation(K)[:M]
        a = np.zeros((M, K), np.float32)
        a[np.arange(M), p] = 1.0
        A.append(to_bf16_bits(a))
        B.append(small_ints_bf16((K, N), rng, -50, 50))
        picks.append(p)
    Y = o.gemm_rs(A, B)
    want = np.zeros((M, N), np.float64)
    for r in range(R):
        want += f32(B[r])[picks[r]]
    assert np.array_equal(Y, want.astype(np.float32)), "one-hot GEMM+RS wrong"


def pin_rs_rows_subset(o):
    """Selected rows equal the same rows of the full result."""
    A, B = synth.gemm_inputs(2, 20, 24, 40, 21, dist="normal")
    full = o.gemm_rs(A, B)
    rows = np.array([19, 0, 7, 7, 13])
    assert np.array_equal(o.gemm_rs(A, B, rows), full[rows]), "row subset differs from full result"


def pin_ar_rounds_partials(o):
    """GEMM+AR rounds each partial to bf16 before the sum.  With K = 2,
    a = [1, 2^-9], b = [1, 1]: P = 1 + 2^-9 (exact in fp32), a tie in bf16 that
    rounds to even (1.0), so for R = 2 the AR result is 2.0 and the RS result
    is 2 + 2^-8.  Integer inputs (bf16-exact partials) make AR equal RS."""
    a = to_bf16_bits(np.array([[1.0, 2.0 ** -9]], np.float32))
    b = to_bf16_bits(np.array([[1.0], [1.0]], np.float32))
    y_ar = o.gemm_ar([a, a], [b, b])
    y_rs = o.gemm_rs([a, a], [b, b])
    assert float(y_ar[0, 0]) == 2.0, f"AR partial rounding: {y_ar[0, 0]}"
    assert float(y_rs[0, 0]) == 2.0 + 2.0 ** -8, f"RS must not round partials: {y_rs[0, 0]}"
    rng = np.random.default_rng(9)
    A = [small_ints_bf16((4, 8), rng) for _ in range(3)]
    B = [small_ints_bf16((8, 5), rng) for _ in range(3)]
    assert np.array_equal(o.gemm_ar(A, B), o.gemm_rs(A, B)), "AR != RS on bf16-exact partials"


# ---------------------------------------------------------------------------
# owner segments and masks
# ---------------------------------------------------------------------------

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                lhs, rhs = line.split(":")
                rows.append((lhs.split(), rhs.split()))
    return rows


def pin_owner_pieces_golden(o):
    for lhs, rhs in _read_golden("owner_pieces.txt"):
        M, R, row0 = map(int, lhs)
        want = [tuple(int(v) for v in p.split(",")) for p in rhs]
        got = o.tile_pieces(row0, 128, M, R)
        assert got == want, f"pieces(M={M},R={R},row0={row0}) = {got}, want {want}"


def pin_owner_pieces_partition(o):
    """Over all tiles the pieces partition [0, M); each lies in one segment
    [sS, (s+1)S) and owner(row) is constant on it; a new piece starts exactly
    where a tile or a segment starts."""
    for (M, R, BM) in [(264, 3, 128), (64, 2, 128), (4096, 8, 128), (48, 6, 16), (1000, 8, 128)]:
        S = M // R
        cover = np.zeros(M, np.int32)
        starts = set()
        for row0 in range(0, M, BM):
            for (s, b, e) in o.tile_pieces(row0, BM, M, R):
                assert s * S <= b < e <= (s + 1) * S and e <= M, (M, R, s, b, e)
                assert o.owner_of_row(b, M, R) == s and o.owner_of_row(e - 1, M, R) == s
                cover[b:e] += 1
                starts.add(b)
        assert np.all(cover == 1), "pieces do not partition the rows"
        want_starts = set(range(0, M, BM)) | {s * S for s in range(R) if s * S < M}
        assert starts == want_starts, "pieces start elsewhere than tile or segment starts"


def pin_masks_golden(o):
    for lhs, rhs in _read_golden("masks.txt"):
        R, M, N = map(int, lhs)
        T, full = int(rhs[0]), int(rhs[1], 16)
        words, t = o.expected_masks(R, M, N, T + 5)
        assert t == T, f"T({R},{M},{N}) = {t}, want {T}"
        assert np.all(words[:T] == full) and np.all(words[T:] == 0), "mask words wrong"


def pin_chunk_pieces_golden(o):
    for lhs, rhs in _read_golden("chunks.txt"):
        R, M, N, C = map(int, lhs)
        want = np.array([[int(v) for v in seg.split(",")] for seg in rhs], dtype=np.int64)
        got = o.chunk_pieces(R, M, N, C)
        assert got.shape == want.shape and np.array_equal(got, want), \
            f"chunk_pieces(R={R},M={M},N={N},C={C}) =\n{got}\nwant\n{want}"


def pin_chunk_pieces_cover_owner_pieces(o):
    """Over the chunks of a segment the counts add up to the number of owner
    pieces stored into that segment in one call (from the owner-piece cut,
    pinned on its own), every used chunk has the same count, and the used
    chunks are a prefix whose length divides the segment's tile rows."""
    for (R, M, N, C) in [(3, 264, 320, 2), (8, 4096, 7168, 8), (4, 1024, 4096, 3), (6, 4800, 512, 4),
                         (8, 8192, 8192, 16), (2, 64, 256, 4), (5, 1000, 1000, 8)]:
        tiles_n = -(-N // 256)
        per_seg = np.zeros(R, np.int64)
        rows_of_seg = [set() for _ in range(R)]
        for row0 in range(0, M, 128):
            for (s, b, e) in o.tile_pieces(row0, 128, M, R):
                per_seg[s] += tiles_n
                rows_of_seg[s].add(row0 // 128)
        got = o.chunk_pieces(R, M, N, C)
        for s in range(R):
            assert got[s].sum() == per_seg[s], (R, M, N, C, s, got[s], per_seg[s])
            used = got[s][got[s] > 0]
            k = len(used)
            assert k >= 1 and np.all(got[s][:k] > 0) and np.all(got[s][k:] == 0), (R, M, C, got[s])
            assert np.all(used == used[0]), (R, M, C, got[s])
            assert len(rows_of_seg[s]) % k == 0 and k <= C, (R, M, C, got[s])


# ---------------------------------------------------------------------------
# Lamport stage: ring-order sum + canonicalisation
# ---------------------------------------------------------------------------

def pin_sentinels_golden(o):
    vals = {}
    with open(os.path.join(GOLDEN, "sentinels.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v, 16)
    neg = np.full((1, 8), vals["bf16_sentinel"], np.uint16)
    s, n = o.ar_stage([neg, neg])
    assert s.view(np.uint32)[0, 0] == vals["fp32_canonical_zero"] and n == 8, "all -0.0 must stage +0.0"
    # -0.0 (fp32 sentinel) never staged
    x = synth.normal_bf16((16, 64), 3, synth.T_PARTIAL)
    synth.inject_bf16(x, 3, synth.T_NEGZERO, 0, 0.3, vals["bf16_sentinel"])
    s, _ = o.ar_stage([x, x.copy()])
    assert not np.any(s.view(np.uint32) == vals["fp32_sentinel"]), "a sentinel was staged"


def pin_stage_r1_and_order(o):
    """R = 1 stages x exactly (bar -0.0 -> +0.0); R = 3 with 2^24, 1, -2^24
    shows the fixed order r = 0..R-1; mixed-sign zeros are not sentinels."""
    rng = np.random.default_rng(2)
    x = to_bf16_bits(rng.standard_normal((5, 16)).astype(np.float32))
    x[0, :3] = 0x8000
    s, n = o.ar_stage([x])
    want = f32(x).copy()
    want[0, :3] = 0.0
    assert n == 3 and np.array_equal(s.view(np.uint32), want.view(np.uint32)), "R=1 stage wrong"
    a = np.zeros((1, 8), np.float32); b = np.zeros((1, 8), np.float32); c = np.zeros((1, 8), np.float32)
    a[0, 0], b[0, 0], c[0, 0] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    a[0, 1], b[0, 1], c[0, 1] = 2.0 ** 24, -(2.0 ** 24), 1.0
    bits = [to_bf16_bits(v) for v in (a, b, c)]
    bits[0][0, 2] = 0x8000   # -0 + +0 + +0 = +0 : not canonicalised
    for t in bits:
        t[0, 3] = 0x8000     # all -0 : canonicalised
    s, n = o.ar_stage(bits)
    assert float(s[0, 0]) == 0.0 and float(s[0, 1]) == 1.0, f"stage order wrong: {s[0, :2]}"
    assert n == 1 and s.view(np.uint32)[0, 3] == 0, "canonicalisation count wrong"


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def pin_rmsnorm_vs_torch(o):
    """Against torch.nn.functional.rms_norm in fp64 (eps inside the sqrt)."""
    M, N = 6, 7168
    partials, residual, gamma = synth.ar_inputs(3, M, N, 17)
    s, _ = o.ar_stage(partials)
    y, h = o.rmsnorm(s, residual, gamma, 1e-6, return_h=True)
    # h = s + residual in fp32 (an exact check: both are sums of a few bf16 values)
    assert np.array_equal(h, (s + f32(residual)).astype(np.float32)), "h != s + residual"
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h.astype(np.float64)), (N,),
                                       weight=torch.from_numpy(gamma.astype(np.float64)),
                                       eps=float(np.float32(1e-6))).numpy()
    assert np.max(np.abs(y - ref) / (np.abs(ref) + 1e-30)) <= 2.0 ** -23, "rms_norm disagrees with torch"


def pin_rmsnorm_closed_forms(o):
    N, eps = 64, 1e-6
    eps32 = float(np.float32(eps))
    # constant row c with gamma = 1: y = c / sqrt(c^2 + eps)
    for c in (3.0, -0.25, 1e-3):
        s = np.full((1, N), c, np.float32)
        y = o.rmsnorm(s, None, np.ones(N, np.float32), eps)
        want = np.float32(c / np.sqrt(c * c + eps32))
        assert np.all(y == want), f"constant row {c}: {y[0, 0]} vs {want}"
    # zero row -> 0 (eps prevents 0/0)
    y = o.rmsnorm(np.zeros((1, N), np.float32), None, np.ones(N, np.float32), eps)
    assert np.all(y == 0), "zero row"
    # mean((y/gamma)^2) = ms / (ms + eps)
    rng = np.random.default_rng(4)
    s = (rng.standard_normal((4, N)) * 3).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(N)).astype(np.float32)
    y = o.rmsnorm(s, None, g, eps).astype(np.float64)
    ms = np.mean(s.astype(np.float64) ** 2, axis=1)
    got = np.mean((y / g.astype(np.float64)) ** 2, axis=1)
    assert np.allclose(got, ms / (ms + eps32), rtol=1e-6, atol=0), "unit-RMS closed form"
    # scale invariance y(a*h) ~ y(h) for a >> sqrt(eps)
    y2 = o.rmsnorm((s * 8).astype(np.float32), None, g, eps).astype(np.float64)
    assert np.allclose(y, y2, rtol=1e-6, atol=1e-7), "scale invariance"


def pin_bf16_rne_array(o):
    """The array rounding is the scalar function element by element, and both
    agree with torch's bf16 conversion (finite values, ties included)."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(4096) * 100).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** 100 * (1 + 2.0 ** -8)], np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])
    got = o.bf16_rne_array(x)
    assert np.array_equal(got, o.bf16_rne(x)), "array rounding differs from the scalar function"
    assert np.array_equal(got, to_bf16_bits(x)), "array rounding differs from torch"


def pin_residual_out(o):
    """bf16(h), h = canon(sum_r x_r) + residual:
    R = 1 and no residual is the identity except -0.0 -> +0.0;
    a residual equal to -x_0 gives +0.0 everywhere;
    small-integer inputs give the exact integer sum."""
    rng = np.random.default_rng(22)
    x0 = synth.normal_bf16((5, 64), 23, synth.T_PARTIAL, 0)
    x0.reshape(-1)[rng.choice(320, 20, replace=False)] = 0x8000
    want = x0.copy()
    want[want == 0x8000] = 0
    assert np.array_equal(o.allreduce_residual_out([x0], None), want), "R=1 identity"
    neg = x0 ^ np.uint16(0x8000)
    assert np.all(o.allreduce_residual_out([x0], neg) == 0), "x - x must be +0.0"
    ints = [rng.integers(-8, 9, size=(3, 40)) for _ in range(4)]
    res = rng.integers(-8, 9, size=(3, 40))
    got = f32(o.allreduce_residual_out([to_bf16_bits(a.astype(np.float32)) for a in ints],
                                       to_bf16_bits(res.astype(np.float32))))
    assert np.array_equal(got, (sum(ints) + res).astype(np.float32)), "integer sums"


def pin_e4m3_vs_torch(o):
    """FP8 E4M3 rounding agrees with torch's float8_e4m3fn conversion on
    finite values within range (normals, subnormals, exact ties), and
    saturates what torch turns into NaN."""
    rng = np.random.default_rng(31)
    mags = 2.0 ** rng.uniform(-12, 8.8, 6000)
    x = (mags * rng.choice([-1.0, 1.0], 6000)).astype(np.float32)
    ties = []
    for e in range(-6, 9):  # halfway between neighbouring codes, both parities of the lower one
        for m in range(8):
            lo = (1 + m / 8) * 2.0 ** e
            ties.append(lo + 2.0 ** e / 16)
    ties += [(k + 0.5) * 2.0 ** -9 for k in range(8)]  # subnormal ties
    x = np.concatenate([x, np.array(ties, np.float32), -np.array(ties, np.float32)])
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3(x), want), "e4m3 rounding differs from torch"
    sat = o.e4m3(np.array([464.0, 1e6, np.inf, -1e30, -np.inf], np.float32))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE], "saturation"
    assert o.e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F, "NaN"


def pin_quant_rows(o):
    """Per-row dynamic quantisation: the largest |y| maps to +-448 (code 0x7E);
    dequantised codes are within half an E4M3 step (2^-4 relative) of y where
    y/scale is a normal E4M3 value; a zero row gets scale 1 and zero codes."""
    rng = np.random.default_rng(32)
    y = (rng.standard_normal((5, 700)) * rng.uniform(0.01, 50, (5, 1))).astype(np.float32)
    y[4] = 0
    q, scale, x = o.quant_rows(y)
    assert scale[4] == 1 and np.all(q[4] == 0), "zero row"
    for i in range(4):
        j = int(np.argmax(np.abs(y[i])))
        assert q[i, j] & 0x7F == 0x7E, "amax element is not +-448"
        vals = torch.from_numpy(q[i].copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
        deq = vals.astype(np.float64) * float(scale[i])
        normal = np.abs(x[i]) >= 2.0 ** -6
        err = np.abs(deq - y[i]) / np.abs(y[i].astype(np.float64))
        assert np.all(err[normal] <= 2.0 ** -4 * (1 + 1e-6)), "dequantised value off by more than half a step"


ALL_PINS = [
    pin_bf16_rne, pin_partial_vs_fp64, pin_partial_exact_integers, pin_partial_rectangular,
    pin_rs_vs_fp64, pin_rs_identity_ring_order, pin_rs_one_hot, pin_rs_rows_subset, pin_ar_rounds_partials,
    pin_owner_pieces_golden, pin_owner_pieces_partition, pin_masks_golden,
    pin_chunk_pieces_golden, pin_chunk_pieces_cover_owner_pieces,
    pin_sentinels_golden, pin_stage_r1_and_order,
    pin_rmsnorm_vs_torch, pin_rmsnorm_closed_forms, pin_bf16_rne_array, pin_residual_out,
    pin_e4m3_vs_torch, pin_quant_rows,
]
