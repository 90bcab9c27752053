"""GPU parity of attn_bwd (gradients from the saved LSE) through the C ABI, against the
fp64 oracle's gradients on the same inputs.

The forward is the library's own (O and LSE as a training step would keep them).
Tolerance: max |err| <= 2e-2 * max |ref| and mean |err| <= 1e-2 * mean |ref| per
gradient tensor.  The GPU rounds P and dS to 16 bits before their products (about
2^-9 relative each), builds D from the 16-bit O, and rounds the result to 16 bits
(2^-9 for bf16); sums over up to N_q or N_kv terms with random signs keep the
relative error well under 1 %.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
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


CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal, dtype
    (1, 2, 2, 128, 128, 64, False, "f16"),
    (2, 8, 2, 257, 257, 128, True, "bf16"),
    (2, 8, 2, 257, 257, 128, False, "bf16"),
    (1, 4, 1, 100, 300, 64, True, "bf16"),
    (1, 4, 4, 300, 100, 128, True, "f16"),
    (1, 16, 4, 1024, 1024, 128, True, "bf16"),
    (1, 32, 1, 385, 385, 64, True, "f16"),       # MQA: every q head's dK, dV summed into one kv head
    (2, 8, 8, 129, 640, 128, False, "bf16"),     # more keys than queries, one row past a tile
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}_h{c[1]}-{c[2]}_n{c[3]}x{c[4]}_d{c[5]}_{'c' if c[6] else 'nc'}_{c[7]}"
                                             for c in CASES])
def test_bwd_matches_oracle(case):
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, Nq, Nkv, D, causal, dtype = case
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + Nkv + D)
    dout = I.prefill_inputs(B, Hq, Hq, Nq, Nq, D, dtype, seed=7)[0]
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, lse = A.prefill(qd, kd, vd, causal=causal)
    dq, dk, dv = A.backward(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_bwd(np64(q), np64(k), np64(v), np64(dout), causal, 1 / math.sqrt(D))
    grad_close(dq, rq, "dQ")
    grad_close(dk, rk, "dK")
    grad_close(dv, rv, "dV")


def test_bwd_is_deterministic():
    import attention_fa2_fwd_gb300 as A
    q, k, v = (t.cuda() for t in I.prefill_inputs(2, 8, 2, 512, 512, 128, "bf16", seed=3))
    dout = I.prefill_inputs(2, 8, 8, 512, 512, 128, "bf16", seed=4)[0].cuda()
    o, lse = A.prefill(q, k, v, causal=True)
    g1 = A.backward(q, k, v, o, lse, dout, causal=True)
    g2 = A.backward(q, k, v, o, lse, dout, causal=True)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_bwd_keys_past_the_last_query_get_zero_gradients():
    """Causal with N_kv > N_q: keys no query attends to have dK = dV = 0."""
    import attention_fa2_fwd_gb300 as A
    q, k, v = (t.cuda() for t in I.prefill_inputs(1, 2, 2, 64, 400, 64, "f16", seed=5))
    dout = I.prefill_inputs(1, 2, 2, 64, 64, 64, "f16", seed=6)[0].cuda()
    o, lse = A.prefill(q, k, v, causal=True)
    dq, dk, dv = A.backward(q, k, v, o, lse, dout, causal=True)
    torch.cuda.synchronize()
    assert (dk[:, :, 64:] == 0).all() and (dv[:, :, 64:] == 0).all()
