"""GPU parity of attn_bwd_ex with rotary position embeddings against the pinned fp64 backward oracle
(oracle.rope.attention_bwd), through the C ABI.

Each case runs the rotary forward (attn_fwd_prefill_ex with the same options) for O and LSE, then the
backward, and compares dQ, dK, dV with the oracle under the bounds of the other backward tests (max error
2 % of the largest reference magnitude, mean error 1 % of the mean magnitude).  Covered: both pair layouts,
keys rotated by the call or given rotated, causal and not, GQA, fp16/bf16, D 64/128, ragged and unequal
lengths, and RoPE together with windows, ALiBi and key ranges.  The workspace size and the caller's inputs
(which the call must not modify) are checked too.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from attention_fa2_fwd_gb300 import inputs as I
from oracle import rope as R
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
    r = np.random.default_rng(seed)
    lo = r.integers(0, Nkv, size=(B, Nq))
    hi = lo + r.integers(0, Nkv, size=(B, Nq))
    kr = np.stack([lo, hi], axis=-1).astype(np.int32)
    kr[:, 0] = (5, 5)    # empty
    kr[:, 1] = (0, Nkv)  # full
    return kr


CASES = [
    # id, B, Hq, Hkv, Nq, Nkv, D, dtype, causal, interleaved, rotated_keys, theta, window, alibi, ranges
    ("causal_half_d128", 1, 4, 2, 300, 300, 128, "bf16", True, False, False, 10000.0, (-1, -1), False, False),
    ("full_interleaved_f16_d64", 2, 4, 4, 200, 333, 64, "f16", False, True, False, 10000.0, (-1, -1), False, False),
    ("causal_rotated_keys", 1, 8, 2, 257, 257, 128, "bf16", True, False, True, 500000.0, (-1, -1), False, False),
    ("full_interleaved_rotated_keys_d64", 1, 2, 1, 130, 400, 64, "bf16", False, True, True, 10000.0, (-1, -1),
     False, False),
    ("causal_window_alibi", 1, 4, 2, 520, 520, 128, "bf16", True, False, False, 10000.0, (128, -1), True, False),
    ("full_ranges_f16", 2, 4, 2, 180, 260, 128, "f16", False, True, False, 10000.0, (-1, -1), False, True),
    ("long_positions", 1, 2, 1, 2100, 2100, 128, "bf16", True, False, False, 100.0, (-1, -1), False, False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rope_backward_against_oracle(case):
    import attention_fa2_fwd_gb300 as A
    name, B, Hq, Hkv, Nq, Nkv, D, dtype, causal, inter, rk, theta, window, alibi, ranges = case
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + 5 * Nkv + D)
    g = torch.Generator().manual_seed(Nq + Nkv + 3 * D)
    dout = torch.randn((B, Hq, Nq, D), generator=g).to(q.dtype)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=np.float32) if alibi else None
    kr = _ranges(B, Nq, Nkv, Nq + Nkv) if ranges else None
    kw = dict(window=window, alibi_slopes=torch.from_numpy(slopes).cuda() if alibi else None,
              kv_ranges=torch.from_numpy(kr).cuda() if ranges else None, rope_theta=theta,
              rope_interleaved=inter, rope_rotated_keys=rk)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    q0, k0 = qd.clone(), kd.clone()
    scale = 1 / math.sqrt(D)
    o, lse = A.prefill(qd, kd, vd, causal=causal, **kw)
    dq, dk, dv = A.backward(qd, kd, vd, o, lse, gd, causal=causal, **kw)
    torch.cuda.synchronize()
    A.check_device_error()
    assert torch.equal(qd, q0) and torch.equal(kd, k0), "the caller's Q and K must not be modified"
    ref = R.attention_bwd(np64(q), np64(k), np64(v), np64(dout), causal, scale, theta, inter, rotated_keys=rk,
                          window_left=window[0], window_right=window[1], alibi_slopes=slopes, kv_ranges=kr)
    for what, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        grad_close(got, want, f"{name} {what}")


def test_rope_backward_strided_outputs():
    """dQ and dK turned back in place in strided (non-contiguous) output views."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D = 1, 4, 2, 200, 128
    q, k, v = (t.cuda() for t in I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=17))
    dout = torch.randn_like(q)
    o, lse = A.prefill(q, k, v, causal=True, rope_theta=10000.0)
    opts = A.make_options(rope_theta=10000.0)
    n = A.attn_bwd_ex_workspace_size(B, Hq, Hkv, N, N, D, opts)
    ws = torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device="cuda")
    dq_big = torch.zeros((B, N, Hq, D), dtype=q.dtype, device="cuda")      # (B, N, H, D) memory, viewed (B, H, N, D)
    dk_big = torch.zeros((B, Hkv, N, 2 * D), dtype=q.dtype, device="cuda")  # every row padded to 2 D
    dq = dq_big.transpose(1, 2)
    dk = dk_big[..., :D]
    dv = torch.empty_like(k)
    st = A.attn_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), A.ATTN_BF16, B, Hq, Hkv, N, N, D, q.stride(),
                       k.stride(), v.stride(), o.stride(), dout.stride(), dq.stride(), dk.stride(), dv.stride(), 1,
                       1 / math.sqrt(D), opts, ws.data_ptr(), n, None)
    assert st == A.ATTN_OK
    ref = A.backward(q, k, v, o, lse, dout, causal=True, rope_theta=10000.0)
    torch.cuda.synchronize()
    assert torch.equal(dq, ref[0]) and torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert torch.count_nonzero(dk_big[..., D:]) == 0, "padding beyond D must stay untouched"


def test_rope_backward_workspace_too_small():
    import attention_fa2_fwd_gb300 as A
    q, k, v = (t.cuda() for t in I.prefill_inputs(1, 4, 2, 128, 128, 128, "bf16", seed=1))
    o, lse = A.prefill(q, k, v, causal=True, rope_theta=10000.0)
    opts = A.make_options(rope_theta=10000.0)
    n_plain = A.attn_bwd_workspace_size(1, 4, 128)
    n = A.attn_bwd_ex_workspace_size(1, 4, 2, 128, 128, 128, opts)
    assert n == n_plain + 2 * 4 * 128 * 128 + 2 * 2 * 128 * 128
    ws = torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device="cuda")
    out = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = A.attn_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), q.data_ptr(), lse.data_ptr(),
                       out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), A.ATTN_BF16, 1, 4, 2, 128, 128, 128,
                       q.stride(), k.stride(), v.stride(), o.stride(), q.stride(), out[0].stride(), out[1].stride(),
                       out[2].stride(), 1, 0.088, opts, ws.data_ptr(), n - 16, None)
    assert st == A.ATTN_ERR_WORKSPACE
