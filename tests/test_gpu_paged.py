"""GPU parity of attn_fwd_decode_paged and kv_cache_write_paged (paged KV caches
with per-request lengths), through the C ABI, against the fp64 oracle.

The page pool is (num_pages, H_kv, page_size, D); request b's cache rows are
the rows of pages block_table[b][0], [1], ...  Page ids are shuffled so that
no request's pages are contiguous in the pool.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def _pool(B, Hkv, max_len, D, page_size, dtype, seed, spare=3):
    """A shuffled page pool holding B requests of max_len rows each (plus spare pages)."""
    max_pages = (max_len + page_size - 1) // page_size
    num_pages = B * max_pages + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)
    kp = (torch.randn((num_pages, Hkv, page_size, D), generator=g)).to(I.DTYPES[dtype])
    vp = (torch.randn((num_pages, Hkv, page_size, D), generator=g)).to(I.DTYPES[dtype])
    return kp, vp, table


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f16")])
def test_paged_decode_matches_oracle(page_size, D, dtype):
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv = 32, 8
    lens = [1, 33, 257, 1000, 0, 64, 129]
    B, max_len = len(lens), max(lens)
    kp, vp, table = _pool(B, Hkv, max_len, D, page_size, dtype, seed=page_size + D)
    q = I.decode_queries(B, Hq, D, [0], dtype, seed=page_size)[:, :, 0]
    cl = torch.tensor(lens, dtype=torch.int32)
    o, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cl.cuda(), max_len)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_paged(np64(q), np64(kp), np64(vp), table.numpy(), cl.numpy(), 1 / math.sqrt(D))
    nz = [b for b in range(B) if lens[b] > 0]
    assert_close(np64(o)[nz], o_ref[nz], np64(lse)[nz], lse_ref[nz], f"ps={page_size} D={D}")
    z = [b for b in range(B) if lens[b] == 0]
    assert (o[z] == 0).all() and torch.isneginf(lse[z]).all()


def test_paged_identity_layout_matches_contiguous_decode():
    """Pages laid out in order with an identity table reproduce the contiguous decode (B=2: many splits)."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, L, D, ps = 2, 32, 8, 4097, 128, 64
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=5)
    q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=5)[:, :, 0].cuda()
    npb = (L + ps - 1) // ps
    kpad = torch.zeros((B, Hkv, npb * ps, D), dtype=torch.bfloat16)
    vpad = torch.zeros_like(kpad)
    kpad[:, :, :L], vpad[:, :, :L] = k, v
    kp = kpad.view(B, Hkv, npb, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npb, Hkv, ps, D).contiguous()
    vp = vpad.view(B, Hkv, npb, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npb, Hkv, ps, D).contiguous()
    table = torch.arange(B * npb, dtype=torch.int32).view(B, npb)
    lens = torch.full((B,), L, dtype=torch.int32)
    o_p, l_p = A.decode_paged(q, kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), L)
    o_c, l_c = A.decode(q, k.cuda(), v.cuda(), L)
    torch.cuda.synchronize()
    assert_close(o_p, np64(o_c), l_p, np64(l_c), "paged vs contiguous")
    o_ref, l_ref = oracle.decode(np64(q), np64(k), np64(v), L, 1 / math.sqrt(D))
    assert_close(o_p, o_ref, l_p, l_ref, "paged vs oracle")


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_cache_write_bit_exact(page_size):
    import attention_fa2_fwd_gb300 as A
    B, Hkv, D, n = 3, 4, 128, 5
    kp, vp, table = _pool(B, Hkv, 4 * page_size, D, page_size, "bf16", seed=11)
    g = torch.Generator().manual_seed(12)
    kn = torch.randn((B, Hkv, n, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((B, Hkv, n, D), generator=g).to(torch.bfloat16)
    pos = torch.tensor([0, page_size - 2, 2 * page_size + 3], dtype=torch.int32)
    kd, vd = kp.cuda(), vp.cuda()
    A.write_kv_cache_paged(kd, vd, kn.cuda(), vn.cuda(), table.cuda(), pos.cuda())
    torch.cuda.synchronize()
    kr, vr = oracle.kv_cache_write_paged(kp.float().numpy(), vp.float().numpy(), kn.float().numpy(),
                                         vn.float().numpy(), table.numpy(), pos.numpy())
    assert np.array_equal(kd.cpu().float().numpy(), kr)
    assert np.array_equal(vd.cpu().float().numpy(), vr)


def test_paged_write_then_decode_token_by_token():
    """Requests of different lengths filled token by token: each step matches the oracle."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, D, ps, L = 3, 16, 4, 128, 32, 70
    kp, vp, table = _pool(B, Hkv, L, D, ps, "bf16", seed=21)
    kd, vd, td = kp.cuda(), vp.cuda(), table.cuda()
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=22)
    start = torch.tensor([0, 5, 20], dtype=torch.int32)  # request b has start[b] tokens before step 0
    for b in range(B):  # pre-fill the first start[b] tokens in one call per request
        if start[b] > 0:
            sel = torch.tensor([b])
            A.write_kv_cache_paged(kd, vd, k[sel, :, :start[b]].cuda(), v[sel, :, :start[b]].cuda(), td[sel],
                                   torch.zeros(1, dtype=torch.int32, device="cuda"))
    steps = 40
    q = I.decode_queries(B, Hq, D, list(range(steps)), "bf16", seed=23)
    for s in range(steps):
        pos = start + s
        kn = torch.stack([k[b, :, pos[b]] for b in range(B)])[:, :, None].cuda()
        vn = torch.stack([v[b, :, pos[b]] for b in range(B)])[:, :, None].cuda()
        A.write_kv_cache_paged(kd, vd, kn, vn, td, pos.cuda())
        lens = (pos + 1).to(torch.int32)
        o, lse = A.decode_paged(q[:, :, s].cuda(), kd, vd, td, lens.cuda(), L)
        if s in (0, 1, 13, steps - 1):
            torch.cuda.synchronize()
            for b in range(B):
                n = int(lens[b])
                o_ref, l_ref = oracle.decode(np64(q[b:b + 1, :, s]), np64(k[b:b + 1]), np64(v[b:b + 1]), n,
                                             1 / math.sqrt(D))
                assert_close(np64(o[b:b + 1]), o_ref, np64(lse[b:b + 1]), l_ref, f"step {s} req {b}")
    A.check_device_error()


def test_paged_out_of_range_indices_are_reported():
    """A page id past the pool, a length past max_cache_len and a write past the table are
    caught on the device: ATTN_ERR_DEVICE_INDEX, no out-of-range access."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, D, ps = 2, 8, 2, 128, 16
    kp, vp, table = _pool(B, Hkv, 64, D, ps, "bf16", seed=31)
    kd, vd = kp.cuda(), vp.cuda()
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    bad = table.clone()
    bad[1, 2] = kp.shape[0] + 1000
    A.decode_paged(q, kd, vd, bad.cuda(), torch.tensor([64, 64], dtype=torch.int32, device="cuda"), 64)
    assert A.attn_get_device_error(stream) == A.ATTN_ERR_DEVICE_INDEX
    A.decode_paged(q, kd, vd, table.cuda(), torch.tensor([64, 65], dtype=torch.int32, device="cuda"), 64)
    assert A.attn_get_device_error(stream) == A.ATTN_ERR_DEVICE_INDEX
    kn = torch.zeros((B, Hkv, 1, D), dtype=torch.bfloat16, device="cuda")
    before = kd.clone()
    A.write_kv_cache_paged(kd, vd, kn, kn, table.cuda(), torch.tensor([3, 64], dtype=torch.int32, device="cuda"))
    assert A.attn_get_device_error(stream) == A.ATTN_ERR_DEVICE_INDEX
    # request 0's valid write landed; request 1's was skipped
    changed = (kd != before).any(dim=(1, 2, 3)).nonzero().flatten().tolist()
    assert set(changed) <= {int(table[0, 0])}
    assert A.attn_get_device_error(stream) == A.ATTN_OK
