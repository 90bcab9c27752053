"""GPU parity of the CTA-pair prefill kernel (attn_options_t.prefill_kernel = 2)
against the fp64 oracle, through the C ABI.

The pair kernel computes the same function as the one-CTA kernel: every case
compares the whole O and LSE tensors with the oracle under the standard
bounds -- ragged and unequal lengths, GQA/MQA ratios, fp16 and bf16, the GQA
causal prefill at N = 2048, the (B,N,H,D)-strided cross-attention -- plus the
exact causal row 0, rows past N_q untouched, determinism, agreement with the
one-CTA kernel, the host-buffer call, and the cases the pair kernel refuses.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
from tests.helpers import assert_close, np64

pytestmark = pytest.mark.gpu

PAIR = 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def run(q, k, v, causal, kernel=PAIR, **kw):
    import attention_fa2_fwd_gb300 as A
    o, lse = A.prefill(q if q.is_cuda else q.cuda(), k if k.is_cuda else k.cuda(), v if v.is_cuda else v.cuda(),
                       causal=causal, prefill_kernel=kernel, **kw)
    torch.cuda.synchronize()
    return o, lse


CASES = [
    # B, Hq, Hkv, Nq, Nkv, causal, dtype
    (1, 2, 1, 1, 1, True, "bf16"),
    (1, 2, 2, 7, 7, False, "f16"),
    (2, 4, 1, 130, 130, True, "bf16"),
    (1, 8, 2, 300, 300, True, "f16"),
    (1, 4, 4, 511, 511, False, "bf16"),
    (1, 4, 2, 512, 512, True, "bf16"),
    (2, 2, 2, 513, 513, True, "f16"),
    (1, 8, 1, 1000, 1000, True, "bf16"),
    (1, 4, 2, 700, 1000, True, "bf16"),
    (1, 4, 2, 1000, 300, True, "f16"),
    (1, 2, 1, 257, 2000, False, "bf16"),
    (2, 16, 2, 1100, 1100, False, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%dh%dk%d_q%d_k%d_%s_%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", c[6]))
def test_pair_against_oracle(case):
    B, Hq, Hkv, Nq, Nkv, causal, dtype = case
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, 128, dtype, seed=Nq * 7 + Nkv)
    o, lse = run(q, k, v, causal)
    o_ref, lse_ref = oracle.attention(np64(q), np64(k), np64(v), causal, 1 / np.sqrt(128))
    assert_close(o, o_ref, lse, lse_ref, "pair %s" % (case,))


def test_pair_gqa_causal_2048():
    """The GQA causal prefill at N = 2048, every element."""
    cfg = I.GQA_CAUSAL[2048]
    q, k, v = cfg.make()
    o, lse = run(q, k, v, cfg.causal)
    o_ref, lse_ref = oracle.attention(np64(q), np64(k), np64(v), cfg.causal, cfg.scale)
    assert_close(o, o_ref, lse, lse_ref, cfg.name + " (pair)")
    # Causal row 0 equals V[kv_head, 0] exactly (one key, weight 1).
    g = cfg.Hq // cfg.Hkv
    assert torch.equal(o[:, :, 0, :], v[:, :, 0, :].repeat_interleave(g, dim=1).cuda())


@pytest.mark.parametrize("cfg", [I.CROSS[128], I.CROSS_STD2[128]], ids=lambda c: c.name)
def test_pair_cross_attention_bnhd(cfg):
    """The (B,N,H,D)-strided cross-attention (D = 128) on the pair kernel, every element."""
    q, k, v = cfg.make()
    qd = q.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    kd = k.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    vd = v.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    out = torch.empty((cfg.B, cfg.Nq, cfg.Hq, cfg.D), dtype=q.dtype, device="cuda").permute(0, 2, 1, 3)
    o, lse = run(qd, kd, vd, False, out=out)
    o_ref, lse_ref = oracle.attention(np64(q), np64(k), np64(v), False, cfg.scale)
    assert_close(o, o_ref, lse, lse_ref, cfg.name + " (pair)")


def test_pair_rows_past_nq_untouched():
    """Rows >= N_q of a larger output buffer and LSE past its end keep their contents."""
    B, H, N, D = 1, 2, 37, 128
    q, k, v = I.prefill_inputs(B, H, H, N, N, D, "bf16", seed=11)
    big = torch.full((B, H, N + 600, D), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, :, :N, :]
    lse_big = torch.full((B * H * N + 64,), 9.0, dtype=torch.float32, device="cuda")
    lse = lse_big[:B * H * N].view(B, H, N)
    run(q, k, v, True, out=out, lse_out=lse)
    assert (big[:, :, N:, :] == 7.0).all()
    assert (lse_big[B * H * N:] == 9.0).all()
    o_ref, lse_ref = oracle.attention(np64(q), np64(k), np64(v), True, 1 / np.sqrt(D))
    assert_close(out, o_ref, lse, lse_ref, "pair guard")


def test_pair_deterministic_and_close_to_one_cta():
    """Two pair runs are bit-identical; the pair and one-CTA kernels agree within twice the oracle bound."""
    q, k, v = I.prefill_inputs(2, 8, 2, 1500, 1500, 128, "bf16", seed=21)
    o1, l1 = run(q, k, v, True)
    o2, l2 = run(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = run(q, k, v, True, kernel=1)
    assert (o1.float() - o3.float()).abs().max().item() <= 4e-2
    assert (l1 - l3).abs().max().item() <= 2e-3


def test_pair_host_buffer_call_matches_device_call():
    """The host-buffer call with the pair kernel gives the device call's results bit for bit."""
    import attention_fa2_fwd_gb300 as A
    q, k, v = I.prefill_inputs(2, 8, 2, 600, 600, 128, "bf16", seed=23)
    o_d, l_d = run(q, k, v, True)
    o_h, l_h = A.prefill_host(q.contiguous(), k.contiguous(), v.contiguous(), causal=True, prefill_kernel=PAIR)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("kw", [
    dict(D=64),
    dict(window=(64, -1)),
    dict(alibi=True),
    dict(rope_theta=10000.0),
], ids=["d64", "window", "alibi", "rope"])
def test_pair_refuses_unsupported_cases(kw):
    """Head dimension 64, windows, ALiBi and RoPE are not on the pair kernel: ATTN_ERR_UNSUPPORTED,
    nothing enqueued, and the library stays usable."""
    import attention_fa2_fwd_gb300 as A
    D = kw.pop("D", 128)
    q, k, v = (t.cuda() for t in I.prefill_inputs(1, 4, 2, 256, 256, D, "bf16", seed=5))
    if kw.pop("alibi", False):
        kw["alibi_slopes"] = torch.full((4,), 0.1, dtype=torch.float32, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.prefill(q, k, v, causal=True, prefill_kernel=PAIR, **kw)
    assert e.value.status == A.ATTN_ERR_UNSUPPORTED
    o, lse = run(q, k, v, True, kernel=0, **kw)
    assert torch.isfinite(o.float()).all()
