"""Helpers shared by the GPU parity tests: moving bf16 bit patterns between
numpy (the generator's and the oracle's side) and torch CUDA tensors."""
import numpy as np
import pytest

import synth


def need_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t):
    return synth.bf16_bits_to_f32(host_bits(t))


def sample_rows(M, R, n_random=16, seed=0):
    """Rows that touch every owner segment's edges, every 128-row tile edge
    near them, and a few random rows."""
    S = M // R
    rows = {0, M - 1}
    for s in range(R):
        for r in (s * S, s * S + 1, (s + 1) * S - 1):
            if 0 <= r < M:
                rows.add(r)
    for t in range(0, M, 128):
        rows.update(r for r in (t, t + 127) if r < M)
        if len(rows) > 64:
            break
    rng = np.random.default_rng(seed)
    rows.update(int(v) for v in rng.integers(0, M, n_random))
    return np.array(sorted(rows), dtype=np.int64)
