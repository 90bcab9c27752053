"""Shared helpers for the parity tests: tolerances and comparison against the oracle.

Tolerances: output max-abs <= 2e-2 and mean-abs <= 2e-3, LSE max-abs <= 1e-3,
measured against the fp64 oracle on the same rounded inputs.  These bound the
error of a 16-bit output after fp32 accumulation with P rounded to 16 bits
before the second GEMM ("Skill: Write a Triton Attention Kernel", step 5h).
"""
from __future__ import annotations

import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def np64(t):
    """A torch tensor (any device, 16-bit or fp32) as an fp64 numpy array."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what=""):
    o = np64(o_gpu) if not isinstance(o_gpu, np.ndarray) else o_gpu
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        l = np64(lse_gpu) if not isinstance(lse_gpu, np.ndarray) else lse_gpu
        assert l.shape == lse_ref.shape, (l.shape, lse_ref.shape)
        le = np.abs(l - lse_ref)
        assert le.max() <= LSE_MAX_ABS, f"{what}: LSE max-abs {le.max():.3e} at {np.unravel_index(le.argmax(), le.shape)}"
    return float(err.max())


def sample_rows(B, H, N, n_random=48, seed=0, tile=128):
    """(b, h, i) triples: first/last rows, tile boundaries and diagonal rows, plus random ones."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, N - 1, N // 2}
    for t in range(0, N, tile):
        fixed.update({t, min(t + tile - 1, N - 1)})
    fixed = sorted(i for i in fixed if 0 <= i < N)
    rows = []
    for j, i in enumerate(fixed):
        rows.append((j % B, (7 * j) % H, i))
    for _ in range(n_random):
        rows.append((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))))
    return np.array(rows, dtype=np.int64)
