"""Failure detection on the GPU without a fault: a bounded wait that runs out.

attn_selftest_wait_timeout launches one kernel whose thread waits on an
mbarrier that nothing arrives on, through the library's bounded wait.  The
wait must give up after its wall-clock limit and record the time-out; the
host reads ATTN_ERR_DEVICE_TIMEOUT once (the read clears it), kernels that run
while the word is set compute nothing, and after the read the library computes
correct results again on the same context.
"""
from __future__ import annotations

import math
import time

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


def test_bounded_wait_times_out_and_the_context_stays_usable():
    import attention_fa2_fwd_gb300 as A
    q, k, v = I.prefill_inputs(1, 4, 2, 200, 300, 64, "bf16", seed=3)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert A.attn_get_device_error() == A.ATTN_OK

    t0 = time.perf_counter()
    assert A.attn_selftest_wait_timeout() == A.ATTN_OK
    # a prefill enqueued behind the timed-out kernel sees the error word and computes nothing
    sentinel = torch.full((1, 4, 200, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    A.prefill(qd, kd, vd, causal=True, out=sentinel, return_lse=False)
    # so does a split decode (split and merge kernels)
    Bd, Hq, Hkv, Dd, L = 2, 32, 8, 128, 8192
    kc, vc = (t.cuda() for t in I.decode_stream(Bd, Hkv, L, Dd, "bf16", seed=9))
    qdec = I.decode_queries(Bd, Hq, Dd, [L - 1], "bf16", seed=9)[:, :, 0].cuda()
    ws = A.decode_workspace(Bd, Hq, Hkv, Dd)
    assert A.attn_decode_splits(Bd, Hq, Hkv, L, Dd) > 1
    dec_sentinel = torch.full((Bd, Hq, Dd), 7.0, dtype=torch.bfloat16, device="cuda")
    A.decode(qdec, kc, vc, L, out=dec_sentinel, return_lse=False, workspace=ws)
    assert A.attn_get_device_error() == A.ATTN_ERR_DEVICE_TIMEOUT
    waited = time.perf_counter() - t0
    assert 1.0 < waited < 60.0, f"the wait gave up after {waited:.1f} s"
    assert bool((sentinel == 7.0).all()), "a kernel ran while the error word was set"
    assert bool((dec_sentinel == 7.0).all()), "a decode ran while the error word was set"

    # the read cleared the word: the next read is clean and the library computes again
    assert A.attn_get_device_error() == A.ATTN_OK
    o, lse = A.prefill(qd, kd, vd, causal=True)
    assert A.attn_get_device_error() == A.ATTN_OK
    o_ref, lse_ref = oracle.attention(np64(q), np64(k), np64(v), True, 1 / math.sqrt(64))
    assert_close(o, o_ref, lse, lse_ref, "after a time-out")
    # and so does the decode, on the same workspace
    od, ld = A.decode(qdec, kc, vc, L, workspace=ws)
    assert A.attn_get_device_error() == A.ATTN_OK
    od_ref, ld_ref = oracle.decode(np64(qdec.cpu()), np64(kc.cpu()), np64(vc.cpu()), L, 1 / math.sqrt(Dd))
    assert_close(od, od_ref, ld, ld_ref, "decode after a time-out")
