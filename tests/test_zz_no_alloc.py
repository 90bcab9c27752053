"""attn_fwd_decode_noalloc: decode for callers that may not allocate device memory.

Some callers cannot call cudaMalloc or pass the library a workspace -- a
plugin whose host framework owns all device memory, or a serving loop that
must not risk an allocation's device synchronisation or failure mid-request.
For them the library keeps a 4 MiB scratch array of its own.  These tests call
that entry point through the C ABI and check its output against the fp64
oracle and against the workspace-taking attn_fwd_decode on the same inputs,
for two calls in a row (the second call finds the first call's partials still
in the shared scratch array and must not be affected by them): bf16 with
D = 128 and many splits, fp16 with D = 64, and short caches that need one
split and no scratch at all.

The file is named so that pytest collects it last.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
from tests.helpers import assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    return A


def _call_noalloc(A, q, kc, vc, cache_len):
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    q4, o4 = q.unsqueeze(2), o.unsqueeze(2)
    code = A.ATTN_BF16 if q.dtype == torch.bfloat16 else A.ATTN_F16
    st = A.attn_fwd_decode_noalloc(q4.data_ptr(), kc.data_ptr(), vc.data_ptr(), o4.data_ptr(), lse.data_ptr(),
                                   code, B, Hq, Hkv, cache_len, D, q4.stride(), kc.stride(), vc.stride(),
                                   o4.stride(), 1.0 / math.sqrt(D), torch.cuda.current_stream().cuda_stream)
    assert st == A.ATTN_OK, A.attn_status_string(st)
    return o, lse


# (dtype, D, B, H_q, H_kv, cache lengths of the two calls, whether the split scratch is used)
CASES = [
    ("bf16", 128, 2, 32, 8, (4097, 2001), True),   # many splits: the scratch array holds the partials
    ("f16", 64, 3, 16, 4, (3000, 777), True),      # fp16, D = 64
    ("bf16", 128, 4, 32, 8, (200, 130), False),    # short caches: one split, the scratch is not touched
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_d{c[1]}_b{c[2]}_{'split' if c[6] else 'onepass'}"
                                             for c in CASES])
def test_noalloc_decode_matches_workspace_decode_twice(A, case):
    """Two calls in a row, each checked against the fp64 oracle and against the
    workspace-taking attn_fwd_decode on the same inputs."""
    dt, D, B, Hq, Hkv, lens, split = case
    L = max(lens)
    for cl in lens:
        assert (A.attn_decode_splits(B, Hq, Hkv, cl, D) > 1) == split
    k, v = I.decode_stream(B, Hkv, L, D, dt, seed=21 + D)
    kc, vc = k.cuda(), v.cuda()
    queries = I.decode_queries(B, Hq, D, [cl - 1 for cl in lens], dt, seed=21 + D)
    for j, cache_len in enumerate(lens):
        q = queries[:, :, j].contiguous().cuda()
        o_ws, lse_ws = A.decode(q, kc, vc, cache_len)
        o, lse = _call_noalloc(A, q, kc, vc, cache_len)
        torch.cuda.synchronize()
        A.check_device_error()
        o_ref, lse_ref = oracle.decode(np64(queries[:, :, j]), np64(k), np64(v), cache_len, 1 / math.sqrt(D))
        assert_close(o, o_ref, lse, lse_ref, f"call {j + 1} vs oracle")
        assert_close(o, np64(o_ws), lse, np64(lse_ws), f"call {j + 1} vs attn_fwd_decode")


def test_noalloc_decode_rejects_scratch_beyond_limit(A):
    # B=64, H_q=32, H_kv=8 at cache_len 8192 splits each kv head in four on a
    # 152-SM GB300, which needs 4 * 64 * 32 * 4 * 129 bytes (4.2 MB) of
    # partials: more than the 4 MiB array.
    B, Hq, Hkv, D, L = 64, 32, 8, 128, 8192
    splits = A.attn_decode_splits(B, Hq, Hkv, L, D)
    need = 4 * B * Hq * splits * (D + 1) if splits > 1 else 0
    if need <= (4 << 20):
        pytest.skip("on this device the case fits the scratch array")
    P = 0x7F0000000000  # never dereferenced: the size check returns before any launch
    st = A.attn_fwd_decode_noalloc(P, P, P, P, None, A.ATTN_BF16, B, Hq, Hkv, L, D, (Hq * D, D, D, 1),
                                   (Hkv * L * D, L * D, D, 1), (Hkv * L * D, L * D, D, 1), (Hq * D, D, D, 1),
                                   0.088, None)
    assert st == A.ATTN_ERR_WORKSPACE
