"""GPU parity of attn_fwd_prefill_varlen (packed sequences of different lengths)
through the C ABI, against the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def _packed(lens_q, lens_k, Hq, Hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    tq, tk = sum(lens_q), sum(lens_k)
    q = torch.randn((tq, Hq, D), generator=g).to(dt)
    k = torch.randn((tk, Hkv, D), generator=g).to(dt)
    v = torch.randn((tk, Hkv, D), generator=g).to(dt)
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return q, k, v, cq, ck


CASES = [
    ("self", [1, 33, 300, 127, 1000, 256], None),
    ("cross", [5, 130, 257, 64], [700, 1, 256, 129]),
]


@pytest.mark.parametrize("name,lens_q,lens_k", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype,Hq,Hkv", [(128, "bf16", 16, 4), (64, "f16", 8, 8)])
def test_varlen_matches_oracle(name, lens_q, lens_k, causal, D, dtype, Hq, Hkv):
    import attention_fa2_fwd_gb300 as A
    lens_k = lens_k or lens_q
    q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, dtype, seed=len(lens_q) + D)
    o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), max(lens_q), max(lens_k),
                              causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.prefill_varlen(np64(q), np64(k), np64(v), cq.numpy(), ck.numpy(), causal,
                                           1 / math.sqrt(D))
    assert_close(o, o_ref, lse, lse_ref, f"{name} causal={causal} D={D}")


def test_varlen_equal_lengths_match_dense_prefill():
    import attention_fa2_fwd_gb300 as A
    B, N, Hq, Hkv, D = 3, 512, 32, 8, 128
    q, k, v, cq, ck = _packed([N] * B, [N] * B, Hq, Hkv, D, "bf16", seed=3)
    o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), N, N, causal=True)
    to_bhnd = lambda x: x.view(B, N, x.shape[1], D).permute(0, 2, 1, 3)
    od, ld = A.prefill(to_bhnd(q.cuda()), to_bhnd(k.cuda()), to_bhnd(v.cuda()), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(to_bhnd(o), od)
    assert torch.equal(lse.view(Hq, B, N).permute(1, 0, 2), ld)


def test_varlen_neighbouring_rows_never_leak():
    """Non-finite values in another sequence's rows (read by the TMA tile that runs past a
    sequence's end) do not reach the sequence's result."""
    import attention_fa2_fwd_gb300 as A
    lens = [100, 200]
    Hq, Hkv, D = 4, 2, 128
    q, k, v, cq, ck = _packed(lens, lens, Hq, Hkv, D, "bf16", seed=9)
    v[100:] = float("inf")
    k[100:] = float("nan")
    o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), 200, 200, causal=False)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.prefill_varlen(np64(q[:100]), np64(k[:100]), np64(v[:100]), [0, 100], [0, 100], False,
                                           1 / math.sqrt(D))
    assert_close(o[:100], o_ref, lse[:, :100], lse_ref, "first sequence")


def test_varlen_empty_sequences():
    """A sequence with no keys gets O = 0, LSE = -inf; one with no queries writes nothing."""
    import attention_fa2_fwd_gb300 as A
    lens_q, lens_k = [3, 0, 50], [0, 10, 77]
    Hq, Hkv, D = 2, 2, 64
    q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, "f16", seed=4)
    o = torch.full((sum(lens_q), Hq, D), 5.0, dtype=torch.float16, device="cuda")
    lse = torch.full((Hq, sum(lens_q)), 7.0, dtype=torch.float32, device="cuda")
    A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), 50, 77, causal=True, out=o, lse_out=lse)
    torch.cuda.synchronize()
    assert (o[:3] == 0).all() and torch.isneginf(lse[:, :3]).all()
    o_ref, lse_ref = oracle.prefill_varlen(np64(q), np64(k), np64(v), cq.numpy(), ck.numpy(), True, 1 / 8)
    assert_close(o[3:], o_ref[3:], lse[:, 3:], lse_ref[:, 3:], "third sequence")


def test_varlen_bad_offsets_are_reported():
    import attention_fa2_fwd_gb300 as A
    lens = [64, 64]
    q, k, v, cq, ck = _packed(lens, lens, 2, 2, 64, "f16", seed=5)
    bad = torch.tensor([0, 100, 64], dtype=torch.int32)  # out of order
    A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), bad.cuda(), ck.cuda(), 64, 64)
    assert A.attn_get_device_error(torch.cuda.current_stream().cuda_stream) == A.ATTN_ERR_DEVICE_INDEX
    A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), 32, 64)  # length above max_seqlen_q
    assert A.attn_get_device_error(torch.cuda.current_stream().cuda_stream) == A.ATTN_ERR_DEVICE_INDEX


@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (False, (-1, -1)), (True, (32, -1)), (False, (16, 16))])
def test_varlen_many_short_sequences(causal, window):
    """1500 packed sequences with independent query and key lengths in 0..400
    (zeros included): every CTA runs dozens of units that mix full, ragged,
    key-less (windows, more queries than keys) and empty sequences."""
    import attention_fa2_fwd_gb300 as A
    from oracle import masked as M
    rng = np.random.default_rng(5)
    n = 1500
    lens_q = rng.integers(0, 401, n)
    lens_k = rng.integers(0, 401, n)
    lens_q[::97] = 0
    lens_k[::89] = 0
    q, k, v, cq, ck = _packed(lens_q.tolist(), lens_k.tolist(), 4, 2, 64, "bf16", seed=17)
    o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), int(lens_q.max()),
                              int(lens_k.max()), causal=causal, window=window)
    torch.cuda.synchronize()
    o_ref, lse_ref = M.prefill_varlen_masked(np64(q), np64(k), np64(v), cq.numpy(), ck.numpy(), causal, 1 / 8,
                                             window[0], window[1])
    o, lse = np64(o), np64(lse)
    empty = np.isneginf(lse_ref)  # (H_q, total_q): rows that see no key
    assert (np.isneginf(lse) == empty).all(), "rows without keys differ"
    assert (o.transpose(1, 0, 2)[empty] == 0).all(), "rows without keys are not zero"
    full = ~empty
    assert_close(o.transpose(1, 0, 2)[full], o_ref.transpose(1, 0, 2)[full], lse[full], lse_ref[full],
                 f"many sequences causal={causal} window={window}")
