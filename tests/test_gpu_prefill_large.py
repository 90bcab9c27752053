"""Prefill and decode at the large end of their size range, through the C ABI.

* a 131035-token causal sequence (1024 query-tile pairs per head, a ragged
  last tile, row offsets past 2^24 elements), sampled rows against the fp64
  oracle plus the one-key first row;
* 4096 units of one short tile each (B = 2048): the persistent schedule's
  many rounds, every batch element checked at its first and last row;
* a short query block over a 100003-key cache (non-causal, D = 64);
* decode over a 262141-token cache at two lengths.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
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


def _rows(B, H, N, fixed, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = [(j % B, (3 * j) % H, i) for j, i in enumerate(sorted(set(i for i in fixed if 0 <= i < N)))]
    rows += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(n_random)]
    return np.array(rows, dtype=np.int64)


def _check_rows(q, k, v, o, lse, causal, rows, name):
    D = q.shape[-1]
    o_ref, lse_ref = oracle.attention_rows(np64(q), np64(k), np64(v), causal, 1.0 / np.sqrt(D), rows)
    og = np64(o)[rows[:, 0], rows[:, 1], rows[:, 2]]
    lg = np64(lse)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(og, o_ref, lg, lse_ref, name)


def test_long_causal_sequence():
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D = 1, 2, 1, 131035, 128
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=11)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    fixed = [0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1] + [t * 128 + 127 for t in (511, 512, 1022)]
    _check_rows(q, k, v, o, lse, True, _rows(B, Hq, N, fixed, 24, seed=1), "long causal")
    # row 0 sees one key: O equals that key's value exactly, LSE the scaled score
    assert torch.equal(o[:, :, 0, :].cpu(), v[:, :, 0, :].repeat_interleave(Hq // Hkv, dim=1))
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_many_short_units():
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D = 2048, 2, 2, 200, 64
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "f16", seed=12)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    # every batch element at its first and last row (alternating heads), plus random rows
    rows = [(b, b % Hq, 0) for b in range(B)] + [(b, (b + 1) % Hq, N - 1) for b in range(B)]
    rng = np.random.default_rng(2)
    rows += [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(N))) for _ in range(64)]
    _check_rows(q, k, v, o, lse, False, np.array(rows, dtype=np.int64), "many units")


def test_short_queries_long_cache():
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, Nq, Nkv, D = 2, 8, 2, 300, 100003, 64
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, "bf16", seed=13)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    rows = _rows(B, Hq, Nq, [0, 127, 128, 255, 256, Nq - 1], 32, seed=3)
    _check_rows(q, k, v, o, lse, False, rows, "long cache")


def test_decode_long_cache():
    """One query token over a 262141-token cache (every split holds thousands of keys)."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, D, L = 1, 8, 2, 128, 262141
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=14)
    q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=14)[:, :, 0]
    kc, vc = k.cuda(), v.cuda()
    for cl in (L, L - 130000):
        o, lse = A.decode(q.cuda(), kc, vc, cl)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), cl, 1 / np.sqrt(D))
        assert_close(o, o_ref, lse, lse_ref, f"decode L={cl}")
