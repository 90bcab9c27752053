"""GPU parity of the sliding-window and ALiBi options (the *_ex entry points)
through the C ABI, against the fp64 windowed / ALiBi oracle.

Readings (the pages name these variants without defining them): row i and key
j sit at positions i and j; key j is visible iff
i - window_left <= j <= i + window_right (-1: unbounded side, causal adds
j <= i); ALiBi adds -slope_h |i - j| to the scaled score; decode's query sits at
position cache_len - 1.  Rows whose band holds no key give O = 0, LSE = -inf.
ALiBi slopes are the usual geometric ones, 2^(-8 (h + 1) / H_q).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from attention_fa2_fwd_gb300 import inputs as I
from oracle import masked as M
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


def _slopes(H):
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=np.float32)


def _dev_slopes(s):
    return None if s is None else torch.tensor(s, dtype=torch.float32, device="cuda")


def _assert_masked(o, lse, o_ref, lse_ref, what):
    """Rows with keys compare within tolerance; rows without keys must be exactly O = 0, LSE = -inf."""
    o, lse = np64(o), np64(lse)
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all(), f"{what}: empty-row pattern differs"
    assert (o[empty] == 0).all(), f"{what}: empty rows not zero"
    full = ~empty
    assert_close(o[full], o_ref[full], lse[full], lse_ref[full], what)


PREFILL_CASES = [
    # (name, Nq, Nkv, causal, window_left, window_right, alibi)
    ("causal-w100", 700, 700, True, 100, -1, False),
    ("causal-w0", 700, 700, True, 0, -1, False),
    ("causal-w300-alibi", 700, 700, True, 300, -1, True),
    ("causal-alibi", 700, 700, True, -1, -1, True),
    ("band-37-300", 700, 700, False, 37, 300, False),
    ("right0-is-causal", 700, 700, False, -1, 0, False),
    ("full-alibi", 700, 700, False, -1, -1, True),
    ("band-200-5-alibi", 700, 700, False, 200, 5, True),
    ("band-128-127", 700, 700, False, 128, 127, False),
    ("wide-window", 700, 700, True, 5000, -1, False),
    ("cross-short-q", 300, 900, False, 50, 600, True),
    ("cross-tall-q-empty-rows", 900, 300, False, 10, 10, False),
    ("cross-tall-q-causal", 900, 300, True, 20, -1, True),
]


@pytest.mark.parametrize("name,Nq,Nkv,causal,wl,wr,alibi", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f16")])
def test_prefill_window_alibi(name, Nq, Nkv, causal, wl, wr, alibi, D, dtype):
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv = 2, 8, 2
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, seed=Nq + 3 * Nkv + D)
    sl = _slopes(Hq) if alibi else None
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=(wl, wr), alibi_slopes=_dev_slopes(sl))
    torch.cuda.synchronize()
    o_ref, lse_ref = M.attention_masked(np64(q), np64(k), np64(v), causal, 1 / math.sqrt(D), wl, wr, sl)
    _assert_masked(o, lse, o_ref, lse_ref, name)


def test_prefill_many_keyless_units_after_one_with_keys():
    """Window (0, 0) over 128 keys and 8192 queries: each CTA runs one unit with
    keys and then ~31 units whose bands hold none (no Q load, no products) --
    the MMA thread's Q waits must stay in step with the producer's loads."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, Nq, Nkv, D = 1, 152, 8, 8192, 128, 64
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, "bf16", seed=21)
    for _ in range(3):
        o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=False, window=(0, 0))
    torch.cuda.synchronize()
    o, lse = np64(o), np64(lse)
    # row i < Nkv sees key i alone: O = V[i] exactly, LSE = the scaled score
    g = Hq // Hkv
    v_rows = np64(v)[:, np.arange(Hq) // g]  # (B, Hq, Nkv, D)
    assert (o[:, :, :Nkv] == v_rows).all()
    s = (np64(q)[:, :, :Nkv] * np64(k)[:, np.arange(Hq) // g]).sum(-1) / math.sqrt(D)
    assert np.abs(lse[:, :, :Nkv] - s).max() <= 1e-3
    # rows past the keys: O = 0, LSE = -inf
    assert (o[:, :, Nkv:] == 0).all() and np.isneginf(lse[:, :, Nkv:]).all()


def test_prefill_window_bhnd_and_bnhd_layouts_agree():
    """The options do not depend on the memory layout of Q, K, V, O."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D = 2, 8, 4, 513, 128
    sl = _dev_slopes(_slopes(Hq))
    outs = []
    for layout in ("bhnd", "bnhd"):
        q, k, v = (t.cuda() for t in I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", layout, seed=9))
        assert layout == "bhnd" or q.stride(1) == D  # the (B,N,H,D) memory order survived the copy
        outs.append(A.prefill(q, k, v, causal=True, window=(70, -1), alibi_slopes=sl))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("causal,wl,wr", [(True, 64, -1), (False, 100, 50), (False, 0, 0)])
def test_varlen_window_alibi(causal, wl, wr):
    import attention_fa2_fwd_gb300 as A
    lens = [1, 33, 300, 127, 1000, 256]
    Hq, Hkv, D = 16, 4, 128
    g = torch.Generator().manual_seed(sum(lens) + wl)
    tq = sum(lens)
    q = torch.randn((tq, Hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((tq, Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((tq, Hkv, D), generator=g).to(torch.bfloat16)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sl = _slopes(Hq)
    o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), cu.cuda(), max(lens), max(lens),
                              causal=causal, window=(wl, wr), alibi_slopes=_dev_slopes(sl))
    torch.cuda.synchronize()
    o_ref, lse_ref = M.prefill_varlen_masked(np64(q), np64(k), np64(v), cu.numpy(), cu.numpy(), causal,
                                             1 / math.sqrt(D), wl, wr, sl)
    # LSE is (H_q, total_q): compare it row-major with O's (total_q, H_q) rows
    _assert_masked(o, lse.t(), o_ref, lse_ref.T, f"varlen causal={causal} window=({wl},{wr})")


@pytest.mark.parametrize("B,L", [(4, 4097), (2, 8192), (64, 1000)])
@pytest.mark.parametrize("wl", [0, 63, 64, 1000, 9000])
@pytest.mark.parametrize("alibi", [False, True])
def test_decode_window_alibi(B, L, wl, alibi):
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D = 32, 8, 128
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=L + wl)
    q = I.decode_queries(B, Hq, D, [L - 1], "bf16", seed=L)[:, :, 0]
    sl = _slopes(Hq) if alibi else None
    o, lse = A.decode(q.cuda(), k.cuda(), v.cuda(), L, window_left=wl, alibi_slopes=_dev_slopes(sl))
    torch.cuda.synchronize()
    rows = slice(None) if B <= 4 else [0, 17, 63]
    o_ref, lse_ref = M.decode_masked(np64(q)[rows], np64(k)[rows], np64(v)[rows], L, 1 / math.sqrt(D), wl, sl)
    assert_close(np64(o)[rows], o_ref, np64(lse)[rows], lse_ref, f"decode B={B} L={L} wl={wl} alibi={alibi}")


def test_decode_window_is_last_row_of_windowed_prefill():
    """Decode at cache_len n with window w equals row n - 1 of the causal prefill with window (w, -1)."""
    import attention_fa2_fwd_gb300 as A
    B, Hq, Hkv, N, D, w = 2, 8, 2, 777, 128, 200
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=77)
    sl = _dev_slopes(_slopes(Hq))
    o_p, l_p = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, window=(w, -1), alibi_slopes=sl)
    o_d, l_d = A.decode(q[:, :, -1].contiguous().cuda(), k.cuda(), v.cuda(), N, window_left=w, alibi_slopes=sl)
    torch.cuda.synchronize()
    assert_close(o_d, np64(o_p[:, :, -1]), l_d, np64(l_p[:, :, -1]), "decode vs prefill last row")


def _pool(B, Hkv, max_len, D, page_size, seed):
    max_pages = (max_len + page_size - 1) // page_size
    num_pages = B * max_pages + 2
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)
    kp = torch.randn((num_pages, Hkv, page_size, D), generator=g).to(torch.bfloat16)
    vp = torch.randn((num_pages, Hkv, page_size, D), generator=g).to(torch.bfloat16)
    return kp, vp, table


@pytest.mark.parametrize("page_size", [16, 64, 128])
@pytest.mark.parametrize("wl,alibi", [(0, False), (100, True), (-1, True), (700, False)])
def test_paged_decode_window_alibi(page_size, wl, alibi):
    import attention_fa2_fwd_gb300 as A
    Hq, Hkv, D = 32, 8, 128
    lens = [1, 33, 257, 1000, 0, 64, 129]
    B, max_len = len(lens), max(lens)
    kp, vp, table = _pool(B, Hkv, max_len, D, page_size, seed=page_size + wl)
    q = I.decode_queries(B, Hq, D, [0], "bf16", seed=page_size)[:, :, 0]
    cl = torch.tensor(lens, dtype=torch.int32)
    sl = _slopes(Hq) if alibi else None
    o, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), cl.cuda(), max_len, window_left=wl,
                            alibi_slopes=_dev_slopes(sl))
    torch.cuda.synchronize()
    o_ref, lse_ref = M.decode_paged_masked(np64(q), np64(kp), np64(vp), table.numpy(), cl.numpy(),
                                           1 / math.sqrt(D), wl, sl)
    _assert_masked(o, lse, o_ref, lse_ref, f"paged ps={page_size} wl={wl} alibi={alibi}")


# ---------------------------------------------------------------- custom masks: per-row key ranges

def _ranges(rng, B, Nq, Nkv):
    """Random [lo, hi) per row, with a full row, an empty row and ranges reaching past N_kv."""
    lo = rng.integers(-5, Nkv, size=(B, Nq))
    hi = lo + rng.integers(0, Nkv // 2 + 2, size=(B, Nq))
    r = np.stack([lo, hi], axis=-1).astype(np.int32)
    r[:, 0] = (0, Nkv)
    r[:, 1] = (7, 7)
    r[:, 2] = (Nkv - 3, Nkv + 40)
    return r


RANGE_CASES = [(dt, D, causal) for dt in ("bf16", "f16") for D in (64, 128) for causal in (False, True)]


@pytest.mark.parametrize("case", RANGE_CASES, ids=[f"{c[0]}_d{c[1]}_{'c' if c[2] else 'nc'}" for c in RANGE_CASES])
def test_key_ranges_prefill(case):
    import attention_fa2_fwd_gb300 as A
    dt, D, causal = case
    B, Hq, Hkv, Nq, Nkv = 2, 8, 2, 300, 333
    q, k, v = I.prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dt, seed=D + causal)
    kr = _ranges(np.random.default_rng(D + 3 * causal), B, Nq, Nkv)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_ranges=torch.from_numpy(kr).cuda())
    torch.cuda.synchronize()
    o_ref, l_ref = M.attention_masked(np64(q), np64(k), np64(v), causal, 1 / math.sqrt(D), kv_ranges=kr)
    _assert_masked(o, lse, o_ref, l_ref, f"ranges {case}")


def test_document_mask_equals_separate_documents():
    """Block-diagonal ranges over one long row: each query sees only its own document (causal within
    it); documents of 1000, 1, 3000 and 4191 tokens."""
    import attention_fa2_fwd_gb300 as A
    lens = [1000, 1, 3000, 4191]
    cu = np.concatenate([[0], np.cumsum(lens)])
    N, Hq, Hkv, D = int(cu[-1]), 8, 2, 128
    q, k, v = I.prefill_inputs(1, Hq, Hkv, N, N, D, "bf16", seed=80)
    kr = np.zeros((1, N, 2), dtype=np.int32)
    for d in range(len(lens)):
        kr[0, cu[d]:cu[d + 1]] = (cu[d], cu[d + 1])
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, kv_ranges=torch.from_numpy(kr).cuda())
    torch.cuda.synchronize()
    import oracle
    o_ref, l_ref = oracle.prefill_varlen(np64(q)[0].transpose(1, 0, 2), np64(k)[0].transpose(1, 0, 2),
                                         np64(v)[0].transpose(1, 0, 2), cu, cu, True, 1 / math.sqrt(D))
    assert_close(np64(o)[0], o_ref.transpose(1, 0, 2), np64(lse)[0], l_ref, "document mask")


def test_key_ranges_with_window_alibi_and_rope():
    import attention_fa2_fwd_gb300 as A
    from oracle import rope as R
    B, Hq, Hkv, N, D = 1, 4, 1, 500, 128
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=81)
    kr = _ranges(np.random.default_rng(81), B, N, N)
    s = _slopes(Hq)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=False, window=(120, 30), alibi_slopes=_dev_slopes(s),
                       kv_ranges=torch.from_numpy(kr).cuda())
    torch.cuda.synchronize()
    o_ref, l_ref = M.attention_masked(np64(q), np64(k), np64(v), False, 1 / math.sqrt(D), 120, 30, s.astype(np.float64),
                                      kv_ranges=kr)
    _assert_masked(o, lse, o_ref, l_ref, "ranges + window + ALiBi")
    # with rotary embeddings: the oracle's rotation rounded to 16 bits, then the masked oracle
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope_theta=10000.0,
                       kv_ranges=torch.from_numpy(kr).cuda())
    torch.cuda.synchronize()
    qr = torch.from_numpy(R.rotate(np64(q), np.arange(N), 10000.0)).to(torch.bfloat16).double().numpy()
    kr_ = torch.from_numpy(R.rotate(np64(k), np.arange(N), 10000.0)).to(torch.bfloat16).double().numpy()
    o_ref, l_ref = M.attention_masked(qr, kr_, np64(v), True, 1 / math.sqrt(D), kv_ranges=kr)
    _assert_masked(o, lse, o_ref, l_ref, "ranges + RoPE")


def test_key_ranges_varlen_and_host_path():
    import attention_fa2_fwd_gb300 as A
    lq, lk = [300, 1, 129, 700], [300, 50, 129, 900]
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    Hq, Hkv, D = 8, 2, 64
    g = torch.Generator().manual_seed(82)
    q = torch.randn((int(cq[-1]), Hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((int(ck[-1]), Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((int(ck[-1]), Hkv, D), generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(82)
    kr = np.zeros((int(cq[-1]), 2), dtype=np.int32)
    for b in range(len(lq)):
        kr[cq[b]:cq[b + 1]] = _ranges(rng, 1, lq[b] + 3, lk[b])[0][:lq[b]]
    for causal in (False, True):
        o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cq, dtype=torch.int32).cuda(),
                                  torch.tensor(ck, dtype=torch.int32).cuda(), max(lq), max(lk), causal=causal,
                                  kv_ranges=torch.from_numpy(kr).cuda())
        torch.cuda.synchronize()
        o_ref, l_ref = M.prefill_varlen_masked(np64(q), np64(k), np64(v), cq, ck, causal, 1 / math.sqrt(D),
                                               kv_ranges=kr)
        # varlen LSE is (H_q, total_q): compare it row-aligned with O (total_q, H_q, D)
        _assert_masked(o, lse.t(), o_ref, l_ref.T, f"varlen ranges causal={causal}")
    # the host-buffer call cuts the problem per batch element: its result equals the device call's
    qd, kd, vd = I.prefill_inputs(2, 16, 4, 700, 700, 128, "bf16", seed=83)
    krd = torch.from_numpy(_ranges(np.random.default_rng(83), 2, 700, 700)).cuda()
    o_d, l_d = A.prefill(qd.cuda(), kd.cuda(), vd.cuda(), causal=True, kv_ranges=krd)
    o_h, l_h = A.prefill_host(qd.pin_memory(), kd.pin_memory(), vd.pin_memory(), causal=True, kv_ranges=krd)
    torch.cuda.synchronize()
    assert torch.equal(o_d.cpu(), o_h) and torch.equal(l_d.cpu(), l_h)
