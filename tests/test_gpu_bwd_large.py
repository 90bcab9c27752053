"""GPU parity of the backward at the benchmark's own size -- causal GQA, B=2, H_q=32, H_kv=8,
N=8192, D=128, bf16, the launch configuration ``bench.py`` times -- on sampled rows the oracle computes
one by one (oracle.attention_bwd_dq_rows / attention_bwd_dkv_rows, pinned to the full backward).

Sampled: dQ rows of three (b, h) including tile edges and the last row; dK and dV rows of two (b, kv head)
groups including the first and last keys and tile edges; plus the RoPE backward on one group.  Bounds as in
the other backward tests, over the sampled rows: max error 2 % of the largest reference magnitude, mean
error 1 % of the mean magnitude.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
from oracle import rope as R
from tests.helpers import np64

pytestmark = pytest.mark.gpu

B, HQ, HKV, N, D = 2, 32, 8, 8192, 128
SCALE = 1 / math.sqrt(D)


@pytest.fixture(scope="module")
def full_size():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    q, k, v = I.prefill_inputs(B, HQ, HKV, N, N, D, "bf16", seed=2024)
    g = torch.Generator().manual_seed(2025)
    dout = torch.randn((B, HQ, N, D), generator=g).to(torch.bfloat16)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    yield A, (q, k, v, dout), (qd, kd, vd, gd)
    A.check_device_error()


def close(got, ref, what):
    err = np.abs(got - ref)
    top, mean = np.abs(ref).max(), np.abs(ref).mean()
    assert np.isfinite(got).all(), f"{what}: non-finite"
    assert err.max() <= 2e-2 * top, f"{what}: max err {err.max():.3e} vs max |ref| {top:.3e}"
    assert err.mean() <= 1e-2 * mean, f"{what}: mean err {err.mean():.3e} vs mean |ref| {mean:.3e}"


def _rows(seed, n_random=16):
    r = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 255, 256, 4095, 4096, 8063, 8064, 8190, 8191]
    return sorted(set(edges) | set(r.integers(0, N, size=n_random).tolist()))


def test_bwd_full_size_sampled_rows(full_size):
    A, host, dev = full_size
    q, k, v, dout = (np64(t) for t in host)
    qd, kd, vd, gd = dev
    o, lse = A.prefill(qd, kd, vd, causal=True)
    dq, dk, dv = A.backward(qd, kd, vd, o, lse, gd, causal=True)
    torch.cuda.synchronize()
    A.check_device_error()
    for b, h in ((0, 0), (0, 31), (1, 17)):
        rows = _rows(100 * b + h)
        ref = oracle.attention_bwd_dq_rows(q, k, v, dout, True, SCALE, b, h, rows)
        close(np64(dq[b, h, rows]), ref, f"dQ b{b} h{h}")
    for b, hk in ((0, 0), (1, 7)):
        keys = _rows(1000 + 10 * b + hk)
        rk, rv = oracle.attention_bwd_dkv_rows(q, k, v, dout, True, SCALE, b, hk, keys)
        close(np64(dk[b, hk, keys]), rk, f"dK b{b} hk{hk}")
        close(np64(dv[b, hk, keys]), rv, f"dV b{b} hk{hk}")


def test_bwd_rope_full_size_sampled_rows(full_size):
    """The RoPE backward at the same size: the oracle's samples on the rotated rows, dQ and dK turned back."""
    A, host, dev = full_size
    q, k, v, dout = (np64(t) for t in host)
    qd, kd, vd, gd = dev
    theta = 10000.0
    o, lse = A.prefill(qd, kd, vd, causal=True, rope_theta=theta)
    dq, dk, dv = A.backward(qd, kd, vd, o, lse, gd, causal=True, rope_theta=theta)
    torch.cuda.synchronize()
    A.check_device_error()
    pos = np.arange(N)
    qr, kr = R.rotate(q, pos, theta), R.rotate(k, pos, theta)
    b, h, hk = 1, 5, 1
    rows = _rows(7)
    ref = oracle.attention_bwd_dq_rows(qr, kr, v, dout, True, SCALE, b, h, rows)
    close(np64(dq[b, h, rows]), R.rotate(ref[None, None], -np.asarray(rows), theta)[0, 0], "RoPE dQ")
    keys = _rows(8)
    rk, rv = oracle.attention_bwd_dkv_rows(qr, kr, v, dout, True, SCALE, b, hk, keys)
    close(np64(dk[b, hk, keys]), R.rotate(rk[None, None], -np.asarray(keys), theta)[0, 0], "RoPE dK")
    close(np64(dv[b, hk, keys]), rv, "RoPE dV")
