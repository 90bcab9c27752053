"""GPU parity of kv_cache_write and attn_fwd_decode, through the C ABI.

Decode workload: bf16, H_q=32, H_kv=8, D=128, B in {2, 64}; the cache is
filled token by token with kv_cache_write and decoded at cache_len in
{1, 33, 257, 1024, 4097, 8192}.  Checks: against the fp64 oracle (all heads,
batches sampled at B=64), autoregressive equivalence with the causal prefill
("Triton-FlashAttention", Phase 2: per-token decode outputs concatenated equal
the prefill output), bit-exact cache writes with untouched neighbours.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.masked
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


def test_kv_cache_write_bit_exact():
    import attention_fa2_fwd_gb300 as A
    for D, dt in ((128, "bf16"), (64, "f16")):
        B, Hkv, L = 3, 4, 50
        kc0, vc0, _ = I.prefill_inputs(B, Hkv, Hkv, L, L, D, dt, seed=1)
        kn, vn, _ = I.prefill_inputs(B, Hkv, Hkv, 7, 7, D, dt, seed=2)
        kc, vc = kc0.cuda(), vc0.cuda()
        A.write_kv_cache(kc, vc, kn.cuda(), vn.cuda(), 20)
        torch.cuda.synchronize()
        kr, vr = oracle.kv_cache_write(kc0.float().numpy(), vc0.float().numpy(), kn.float().numpy(),
                                       vn.float().numpy(), 20)
        assert np.array_equal(kc.cpu().float().numpy(), kr)
        assert np.array_equal(vc.cpu().float().numpy(), vr)


def test_kv_cache_write_strided_new_tokens():
    """New tokens given as a (B,N,H,D)-memory view are written to a (B,H,N,D) cache."""
    import attention_fa2_fwd_gb300 as A
    B, Hkv, L, D = 2, 8, 16, 128
    kc = torch.zeros((B, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn, vn, _ = I.prefill_inputs(B, Hkv, Hkv, 3, 3, D, "bf16", layout="bnhd", seed=4)
    kn_d = kn.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    vn_d = vn.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    A.write_kv_cache(kc, vc, kn_d, vn_d, L - 3)
    torch.cuda.synchronize()
    assert torch.equal(kc[:, :, L - 3:].cpu(), kn) and torch.equal(vc[:, :, L - 3:].cpu(), vn)
    assert (kc[:, :, :L - 3] == 0).all() and (vc[:, :, :L - 3] == 0).all()


def _fill_and_decode(B, L_max, lens, check_ar_upto=0, b_sample=None):
    """Fill a cache token by token; decode; compare at `lens` with the oracle and
    the first `check_ar_upto` decode steps with the causal prefill."""
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D = 32, 8, 128
    scale = 1 / np.sqrt(D)
    k, v = I.decode_stream(B, Hkv, L_max, D, "bf16", seed=B)
    steps = sorted(set(range(check_ar_upto)) | {L - 1 for L in lens})
    col = {t: j for j, t in enumerate(steps)}
    q = I.decode_queries(B, Hq, D, steps, "bf16", seed=B)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    kc = torch.zeros((B, Hkv, L_max, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ws = A.decode_workspace(B, Hq, Hkv, D)
    outs, lses = {}, {}
    n_ar = max(check_ar_upto, 1)
    o_steps = torch.empty((B, Hq, n_ar, D), dtype=torch.bfloat16, device="cuda")
    l_steps = torch.empty((B, Hq, n_ar), dtype=torch.float32, device="cuda")
    for t in range(L_max):
        A.write_kv_cache(kc, vc, kd[:, :, t:t + 1], vd[:, :, t:t + 1], t)
        if t in col:
            o, lse = A.decode(qd[:, :, col[t]], kc, vc, t + 1, workspace=ws)
            if t < check_ar_upto:
                o_steps[:, :, t] = o
                l_steps[:, :, t] = lse
            if (t + 1) in lens:
                outs[t + 1], lses[t + 1] = o.clone(), lse.clone()
    torch.cuda.synchronize()
    A.check_device_error()
    bs = np.arange(B) if b_sample is None else np.array(b_sample)
    for L in sorted(lens):
        o_ref, lse_ref = oracle.decode(np64(q[bs][:, :, col[L - 1]]), np64(k[bs]), np64(v[bs]), L, scale)
        assert_close(np64(outs[L])[bs], o_ref, np64(lses[L])[bs], lse_ref, f"B={B} L={L}")
    if check_ar_upto:
        n = check_ar_upto
        o_pre, l_pre = A.prefill(qd[:, :, :n], kd[:, :, :n], vd[:, :, :n], causal=True)
        torch.cuda.synchronize()
        assert_close(o_steps, np64(o_pre), l_steps, np64(l_pre), "autoregressive")


def test_decode_b2_all_lengths_and_autoregressive():
    _fill_and_decode(2, 8192, set(I.DECODE_LENS), check_ar_upto=8192)


def test_decode_b64_lengths():
    _fill_and_decode(64, 8192, set(I.DECODE_LENS), check_ar_upto=1024, b_sample=[0, 17, 42, 63])


def test_decode_against_oracle_gqa_ratios():
    """Group sizes 1..32 (MHA to MQA) and D = 64 / 128, non-aligned cache lengths."""
    import attention_fa2_fwd_gb300 as A
    for Hkv in (32, 16, 8, 4, 2, 1):
        for D in (64, 128):
            B, Hq, L = 2, 32, 300
            k, v = I.decode_stream(B, Hkv, L, D, "f16", seed=Hkv * D)
            lens = (1, 31, 33, 257, 300)
            q = I.decode_queries(B, Hq, D, [c - 1 for c in lens], "f16", seed=Hkv * D)
            kc, vc = k.cuda(), v.cuda()
            for j, cl in enumerate(lens):
                o, lse = A.decode(q[:, :, j].cuda(), kc, vc, cl)
                torch.cuda.synchronize()
                o_ref, lse_ref = oracle.decode(np64(q[:, :, j]), np64(k), np64(v), cl, 1 / np.sqrt(D))
                assert_close(o, o_ref, lse, lse_ref, f"Hkv={Hkv} D={D} L={cl}")


def test_decode_workspace_errors():
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, D, L = 2, 32, 8, 128, 8192
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    need = A.attn_decode_workspace_size(B, Hq, Hkv, D)
    assert need > 0  # B=2 splits the cache over many CTAs
    assert A.attn_decode_splits(B, Hq, Hkv, L, D) > 1
    small = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.decode(q, kc, kc, L, workspace=small)
    assert e.value.status == A.ATTN_ERR_WORKSPACE
    # A workspace of attn_decode_workspace_size bytes serves every cache length.
    ws = A.decode_workspace(B, Hq, Hkv, D)
    for cl in (1, 255, 256, 257, 4097, 8192):
        A.decode(q, kc, kc, cl, workspace=ws)
    torch.cuda.synchronize()


def test_decode_split_count_does_not_change_result():
    """B=2 uses many splits, B=64 few; the same (b, h) rows must agree within tolerance."""
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D, L = 32, 8, 128, 4097
    k, v = I.decode_stream(2, Hkv, L, D, "bf16", seed=77)
    q = I.decode_queries(2, Hq, D, [L - 1], "bf16", seed=77)[:, :, 0]
    o2, l2 = A.decode(q.cuda(), k.cuda(), v.cuda(), L)
    kk = k.repeat(32, 1, 1, 1).cuda()
    vv = v.repeat(32, 1, 1, 1).cuda()
    o64, l64 = A.decode(q.repeat(32, 1, 1).cuda(), kk, vv, L)
    torch.cuda.synchronize()
    assert A.attn_decode_splits(2, Hq, Hkv, L, D) != A.attn_decode_splits(64, Hq, Hkv, L, D)
    assert_close(o64[:2], np64(o2), l64[:2], np64(l2), "splits")


@pytest.mark.parametrize("B", [2, 64])
def test_decode_one_split_equals_automatic_split(B):
    """The same problem with the cache read in one pass (num_splits = 1), in the
    automatic number of splits, and in a forced 3: all match the oracle and each other."""
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D, L = 32, 8, 128, 8192
    assert A.attn_decode_splits(B, Hq, Hkv, L, D) > 1
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=90 + B)
    q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=90 + B)[:, :, 0]
    qd, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o_auto, l_auto = A.decode(qd, kc, vc, L)
    o_one, l_one = A.decode(qd, kc, vc, L, num_splits=1)
    ws3 = A.decode_workspace(B, Hq, Hkv, D, num_splits=3)
    o_three, l_three = A.decode(qd, kc, vc, L, num_splits=3, workspace=ws3)
    torch.cuda.synchronize()
    A.check_device_error()
    bs = np.arange(B) if B <= 4 else np.array([0, 21, 63])
    o_ref, lse_ref = oracle.decode(np64(q[bs]), np64(k[bs]), np64(v[bs]), L, 1 / np.sqrt(D))
    for name, o, l in (("auto", o_auto, l_auto), ("one", o_one, l_one), ("three", o_three, l_three)):
        assert_close(np64(o)[bs], o_ref, np64(l)[bs], lse_ref, f"B={B} {name}")
    assert_close(o_one, np64(o_auto), l_one, np64(l_auto), f"B={B} one vs auto")


def test_decode_forced_splits_need_their_workspace():
    """A forced split count above the automatic one needs a larger workspace."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, D, L = 64, 32, 8, 128, 8192
    auto = A.attn_decode_splits(B, Hq, Hkv, L, D)
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    ws = A.decode_workspace(B, Hq, Hkv, D)
    with pytest.raises(A.AttnError) as e:
        A.decode(q, kc, kc, L, workspace=ws, num_splits=auto + 4)
    assert e.value.status == A.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,L", [(2, 8192), (64, 4097), (3, 200)])
def test_decode_guard_bands(B, L):
    """Nothing is written outside O, LSE and the first attn_decode_workspace_size
    bytes of the workspace: canary values around each of them stay untouched."""
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D = 32, 8, 128
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=5 + B)
    q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=5 + B)[:, :, 0].cuda()
    kc, vc = k.cuda(), v.cuda()
    pad = 1024
    n_o = B * Hq * D
    o_buf = torch.full((n_o + 2 * pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    o = o_buf[pad:pad + n_o].view(B, Hq, D)
    # Interleaved guard: O as every other row of a (B, H_q, 2, D) buffer.
    o2_buf = torch.full((B, Hq, 2, D), 5.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * Hq + 2 * pad,), 9.0, dtype=torch.float32, device="cuda")
    lse = l_buf[pad:pad + B * Hq].view(B, Hq)
    need = A.attn_decode_workspace_size(B, Hq, Hkv, D)
    ws_buf = torch.full((need // 4 + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    ws = ws_buf[pad:pad + need // 4]
    A.decode(q, kc, vc, L, out=o, lse_out=lse, workspace=ws if need else None)
    A.decode(q, kc, vc, L, out=o2_buf[:, :, 0, :], return_lse=False, workspace=ws if need else None)
    torch.cuda.synchronize()
    A.check_device_error()
    assert (o_buf[:pad] == 3.0).all() and (o_buf[pad + n_o:] == 3.0).all()
    assert (o2_buf[:, :, 1, :] == 5.0).all()
    assert (l_buf[:pad] == 9.0).all() and (l_buf[pad + B * Hq:] == 9.0).all()
    assert (ws_buf[:pad] == -7.0).all() and (ws_buf[pad + need // 4:] == -7.0).all()
    o_ref, lse_ref = oracle.decode(np64(q[:2]), np64(k[:2]), np64(v[:2]), L, 1 / np.sqrt(D))
    assert_close(np64(o)[:2], o_ref, np64(lse)[:2], lse_ref, "guarded")
    assert torch.equal(o2_buf[:, :, 0, :], o)


def test_decode_workspace_reused_across_sizes_and_split_counts():
    """One workspace serves a series of calls with different batch sizes, cache lengths, windows and
    forced split counts: each result matches the oracle, whatever garbage the workspace holds between calls
    (its contents need not be initialised)."""
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D = 32, 8, 128
    ws = A.decode_workspace(8, Hq, Hkv, D, num_splits=40)
    cases = [(2, 8192, 0, -1), (8, 3000, 0, -1), (1, 9000, 17, -1), (2, 5000, 40, 700), (8, 300, 3, -1),
             (2, 8192, 0, -1)]
    for i, (B, L, splits, wl) in enumerate(cases):
        k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=300 + i)
        q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=300 + i)[:, :, 0]
        ws.view(torch.int32).fill_(0x7fc00000 + i)  # NaN garbage
        o, lse = A.decode(q.cuda(), k.cuda(), v.cuda(), L, workspace=ws, num_splits=splits, window_left=wl)
        torch.cuda.synchronize()
        A.check_device_error()
        bs = np.arange(min(B, 2))
        if wl >= 0:
            o_ref, lse_ref = oracle.masked.decode_masked(np64(q[bs]), np64(k[bs]), np64(v[bs]), L, 1 / np.sqrt(D),
                                                         window_left=wl)
        else:
            o_ref, lse_ref = oracle.decode(np64(q[bs]), np64(k[bs]), np64(v[bs]), L, 1 / np.sqrt(D))
        assert_close(np64(o)[bs], o_ref, np64(lse)[bs], lse_ref, f"case {i}")
