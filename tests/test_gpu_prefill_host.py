"""GPU parity of attn_fwd_prefill_host (host-resident tensors, copies pipelined
against the compute in chunks): equal, bit for bit, to attn_fwd_prefill_ex on
the same inputs in device memory, and within tolerance of the fp64 oracle."""
from __future__ import annotations

import math

import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
from tests.helpers import assert_close, np64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


CASES = [
    # (B, H_q, H_kv, N_q, N_kv, D, causal, dtype): several chunks per batch element, ragged lengths, MHA and GQA
    (2, 32, 8, 1000, 1000, 128, True, "bf16"),
    (3, 16, 4, 300, 777, 64, False, "f16"),
    (1, 8, 8, 2048, 2048, 128, True, "bf16"),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,causal,dtype", CASES)
def test_prefill_host_equals_device_prefill(B, Hq, Hkv, Nq, Nkv, D, causal, dtype):
    import attention_fa2_fwd_gb300 as A
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + Nkv)
    hq, hk, hv = (t.contiguous().pin_memory() for t in (q, k, v))
    o_h, l_h = A.prefill_host(hq, hk, hv, causal=causal)
    o_d, l_d = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    rows = sample_rows(B, Hq, Nq, n_random=32, seed=Nq)
    o_ref, l_ref = oracle.attention_rows(np64(q), np64(k), np64(v), causal, 1 / math.sqrt(D), rows)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    assert_close(np64(o_h)[b, h, i], o_ref, np64(l_h)[b, h, i], l_ref, "host prefill vs oracle")


def test_prefill_host_window_alibi_equals_device():
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D = 2, 16, 4, 900, 128
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=5)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32, device="cuda")
    hq, hk, hv = (t.contiguous().pin_memory() for t in (q, k, v))
    o_h, l_h = A.prefill_host(hq, hk, hv, causal=True, window=(200, -1), alibi_slopes=slopes)
    o_d, l_d = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, window=(200, -1), alibi_slopes=slopes)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
