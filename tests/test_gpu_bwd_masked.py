"""GPU parity of attn_bwd_ex with the forward's windows, ALiBi and key ranges
against the pinned fp64 backward oracle (oracle.masked.attention_bwd_masked),
through the C ABI.

Each case runs the masked forward (attn_fwd_prefill_ex with the same options)
for O and LSE, then the backward, and compares dQ, dK, dV with the oracle
under the bounds of the plain backward tests (max error 2 % of the largest
reference magnitude, mean error 1 % of the mean magnitude).  Covered: left and
two-sided windows, causal and not, ALiBi alone and with windows, key ranges
with empty, full and past-the-end rows, rows that a window leaves without
keys (dQ = 0), GQA, fp16/bf16, D 64/128, ragged and unequal lengths, and no
options gives the plain kernels' result.  (Rotary embeddings: test_gpu_bwd_rope.)
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from attention_fa2_fwd_gb300 import inputs as I
from oracle import masked as M
from tests.helpers import np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def grad_close(g, ref, what):
    x = np64(g)
    assert np.isfinite(x).all(), f"{what}: non-finite"
    err = np.abs(x - ref)
    top, mean = np.abs(ref).max(), np.abs(ref).mean()
    assert err.max() <= 2e-2 * top, f"{what}: max err {err.max():.3e} vs max |ref| {top:.3e}"
    assert err.mean() <= 1e-2 * mean, f"{what}: mean err {err.mean():.3e} vs mean |ref| {mean:.3e}"


def _ranges(B, Nq, Nkv, seed):
    """Random [lo, hi) rows, with an empty, a full and a past-the-end row in each batch."""
    r = np.random.default_rng(seed)
    lo = r.integers(0, Nkv, size=(B, Nq))
    hi = lo + r.integers(0, Nkv, size=(B, Nq))
    kr = np.stack([lo, hi], axis=-1).astype(np.int32)
    kr[:, 0] = (5, 5)               # empty
    kr[:, 1] = (0, Nkv)             # full
    kr[:, 2] = (Nkv - 3, Nkv + 50)  # past the end
    return kr


def _slopes(Hq):
    return np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=np.float32)


CASES = [
    # id, B, Hq, Hkv, Nq, Nkv, D, dtype, causal, window, alibi, ranges
    ("causal_wl64", 1, 4, 2, 300, 300, 128, "bf16", True, (64, -1), False, False),
    ("full_w50_30_f16_d64", 1, 4, 2, 300, 300, 64, "f16", False, (50, 30), False, False),
    ("causal_alibi", 2, 4, 1, 257, 257, 128, "bf16", True, (-1, -1), True, False),
    ("full_w100_alibi_cross", 1, 2, 2, 200, 350, 128, "bf16", False, (100, 100), True, False),
    ("causal_ranges", 1, 4, 2, 300, 300, 128, "bf16", True, (-1, -1), False, True),
    ("full_ranges_alibi_d64", 2, 4, 2, 180, 260, 64, "bf16", False, (-1, -1), True, True),
    ("rows_without_keys", 1, 2, 1, 400, 200, 128, "bf16", False, (10, 0), False, False),
    ("causal_w_alibi_ranges_f16", 1, 8, 2, 520, 520, 128, "f16", True, (200, -1), True, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_masked_backward_against_oracle(case):
    import attention_fa2_fwd_gb300 as A
    name, B, Hq, Hkv, Nq, Nkv, D, dtype, causal, window, alibi, ranges = case
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + 3 * Nkv)
    g = torch.Generator().manual_seed(Nq + Nkv + D)
    dout = torch.randn((B, Hq, Nq, D), generator=g).to(q.dtype)
    slopes = _slopes(Hq) if alibi else None
    kr = _ranges(B, Nq, Nkv, Nq * 7 + Nkv) if ranges else None
    kw = dict(window=window,
              alibi_slopes=torch.from_numpy(slopes).cuda() if alibi else None,
              kv_ranges=torch.from_numpy(kr).cuda() if ranges else None)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    scale = 1 / math.sqrt(D)
    o, lse = A.prefill(qd, kd, vd, causal=causal, **kw)
    dq, dk, dv = A.backward(qd, kd, vd, o, lse, gd, causal=causal, **kw)
    torch.cuda.synchronize()
    A.check_device_error()
    ref = M.attention_bwd_masked(np64(q), np64(k), np64(v), np64(dout), causal, scale, window_left=window[0],
                                 window_right=window[1], alibi_slopes=slopes, kv_ranges=kr)
    for what, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        grad_close(got, want, f"{name} {what}")
    if name == "rows_without_keys":
        # rows i > N_kv - 1 + window_left see no key: their dQ is exactly zero
        assert torch.count_nonzero(dq[:, :, Nkv + window[0]:]) == 0


def test_masked_backward_without_options_matches_plain():
    """attn_bwd_ex with unbounded windows runs the plain kernels: bit-identical to attn_bwd."""
    import attention_fa2_fwd_gb300 as A
    q, k, v = (t.cuda() for t in I.prefill_inputs(1, 4, 2, 300, 300, 128, "bf16", seed=8))
    dout = torch.randn_like(q)
    o, lse = A.prefill(q, k, v, causal=True)
    a = A.backward(q, k, v, o, lse, dout, causal=True)
    b = A.backward(q, k, v, o, lse, dout, causal=True, window=(-1, -1))
    for x, y in zip(a, b):
        assert torch.equal(x, y)
