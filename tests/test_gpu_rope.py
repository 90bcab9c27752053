"""GPU parity of the rotary-embedding (RoPE) paths against the fp64 oracle, through the C ABI.

The kernels rotate Q and K on chip in fp32 and -- because the tensor core
multiplies 16-bit operands -- round the rotated rows to the input type before
Q K^T (prefill); decode keeps the rotated query in fp32 and reads keys that
the cache write rotated and rounded once.  So every case is checked twice:

* tight: against the plain oracle (``oracle.attention`` / ``oracle.decode`` /
  ``oracle.masked``) fed with the oracle's exact rotation (``oracle.rope``)
  rounded to the 16-bit type by this test -- the standard tolerances (O max
  2e-2, mean 2e-3; LSE max 1e-3);
* exact: against ``oracle.rope`` itself, within a bound derived from that one
  rounding: each rotated operand carries a relative error of at most u
  (2^-8 bf16, 2^-11 fp16: half an ulp), so a score moves by at most
  E_ij = 2 u scale sum_d |q'_d| |k'_d| and, to first order,
  |dLSE_i| <= max_j E_ij and |dO_i| <= 2 max_j E_ij max_j |v_j| beyond the
  standard tolerances.

Cases: prefill in both pair layouts, bf16 and fp16, D = 64 and 128, causal
and not, GQA, ragged and unequal lengths, large angles (small and large
theta), with windows and ALiBi, the GQA causal workload at N = 2048, packed
variable-length batches, the host-buffer path; the RoPE cache write (dense
and paged), decode and paged decode over rotated caches, and autoregressive
decode = causal prefill rows.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa2_fwd_gb300 import inputs as I
from oracle import masked
from oracle import rope as R
from tests.helpers import LSE_MAX_ABS, O_MAX_ABS, assert_close, np64

pytestmark = pytest.mark.gpu

# unit roundoff (half an ulp, relative) of the 16-bit types: 8 and 11 significant bits
U16 = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
THETA = 10000.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def A_():
    import attention_fa2_fwd_gb300 as A
    return A


def round16(x, dt):
    """fp64 array rounded to the 16-bit type (round to nearest even), back in fp64."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(dt).double().numpy()


def rot(x, theta, inter, offset=0):
    """Oracle rotation of a (B, H, N, D) tensor, row n at position offset + n."""
    x = np64(x)
    return R.rotate(x, offset + np.arange(x.shape[2]), theta, inter)


def exact_bounds(qr, kr, v, scale, u, causal):
    """Per-row (E_i, max|v|) of the derived bound: E_i = max over allowed keys of 2u scale sum_d |q'||k'|."""
    B, Hq, Nq, D = qr.shape
    Hkv, Nkv = kr.shape[1], kr.shape[2]
    g = Hq // Hkv
    E = np.zeros((B, Hq, Nq))
    vmax = np.zeros((B, Hq, 1))
    for b in range(B):
        for h in range(Hq):
            M = (np.abs(qr[b, h]) @ np.abs(kr[b, h // g]).T) * (2 * u * scale)
            if causal:
                M = np.where(np.arange(Nkv)[None, :] <= np.arange(Nq)[:, None], M, 0.0)
            E[b, h] = M.max(axis=1)
            vmax[b, h] = np.abs(v[b, h // g]).max()
    return E, vmax


def assert_within_derived(o, lse, o_ref, lse_ref, E, vmax, what):
    o, lse = np64(o), np64(lse)
    dl = np.abs(lse - lse_ref)
    assert (dl <= LSE_MAX_ABS + E).all(), f"{what}: LSE beyond the derived bound by {(dl - LSE_MAX_ABS - E).max():.3e}"
    do = np.abs(o - o_ref)
    lim = O_MAX_ABS + 2 * E[..., None] * vmax[..., None]
    assert (do <= lim).all(), f"{what}: O beyond the derived bound by {(do - lim).max():.3e}"


def check_prefill(q, k, v, causal, theta, inter, what, window=(-1, -1), slopes=None):
    A = A_()
    dt = q.dtype
    D = q.shape[-1]
    scale = 1 / math.sqrt(D)
    o, lse = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window,
                       alibi_slopes=None if slopes is None else torch.tensor(slopes, dtype=torch.float32).cuda(),
                       rope_theta=theta, rope_interleaved=inter)
    torch.cuda.synchronize()
    th = float(np.float32(theta))
    qr, kr = rot(q, th, inter), rot(k, th, inter)
    qh, kh = round16(qr, dt), round16(kr, dt)
    plain = window == (-1, -1) and slopes is None
    if plain:
        o_t, l_t = oracle.attention(qh, kh, np64(v), causal, scale)
    else:
        o_t, l_t = masked.attention_masked(qh, kh, np64(v), causal, scale, window[0], window[1], slopes)
    assert_close(o, o_t, lse, l_t, what + " (rounded rotation)")
    o_x, l_x = R.attention(np64(q), np64(k), np64(v), causal, scale, th, inter, window[0], window[1], slopes)
    E, vmax = exact_bounds(qr, kr, np64(v), scale, U16[dt], causal)
    assert_within_derived(o, lse, o_x, l_x, E, vmax, what + " (exact oracle)")
    return o, lse


PREFILL_CASES = [(dt, D, causal, inter) for dt in ("bf16", "f16") for D in (64, 128) for causal in (False, True)
                 for inter in (False, True)]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[f"{c[0]}_d{c[1]}_{'c' if c[2] else 'nc'}_{'il' if c[3] else 'half'}"
                                                    for c in PREFILL_CASES])
def test_rope_prefill_small(case):
    dt, D, causal, inter = case
    q, k, v = I.prefill_inputs(2, 8, 2, 300, 300, D, dt, seed=D + 7 * causal + 3 * inter)
    check_prefill(q, k, v, causal, THETA, inter, f"{case}")


def test_rope_prefill_unequal_lengths_and_angles():
    """Cross lengths, and bases whose angles wrap many times (theta 1.5) or barely move (500000)."""
    q, k, v = I.prefill_inputs(1, 4, 4, 200, 700, 128, "bf16", seed=71)
    check_prefill(q, k, v, False, THETA, False, "200x700")
    q, k, v = I.prefill_inputs(1, 4, 2, 1024, 1024, 64, "f16", seed=72)
    for theta in (1.5, 500000.0):
        check_prefill(q, k, v, True, theta, True, f"theta={theta}")


def test_rope_prefill_with_window_and_alibi():
    q, k, v = I.prefill_inputs(1, 4, 1, 500, 500, 128, "bf16", seed=73)
    check_prefill(q, k, v, False, THETA, False, "window+alibi", window=(100, 20), slopes=[0.5, 0.25, 0.125, 0.0625])
    check_prefill(q, k, v, True, THETA, True, "causal window", window=(64, -1))


def test_rope_gqa_causal_prefill_n2048():
    cfg = I.GQA_CAUSAL[2048]
    q, k, v = cfg.make(seed=5)
    o, _ = check_prefill(q, k, v, True, THETA, False, cfg.name + " rope")
    g = cfg.Hq // cfg.Hkv
    assert torch.equal(o[:, :, 0, :].cpu(), v[:, :, 0, :].repeat_interleave(g, dim=1))  # row 0: one key, weight 1


def test_rope_prefill_host_path_equals_device():
    A = A_()
    q, k, v = I.prefill_inputs(2, 16, 4, 700, 700, 128, "bf16", seed=74)
    o_d, l_d = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope_theta=THETA)
    o_h, l_h = A.prefill_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True, rope_theta=THETA)
    torch.cuda.synchronize()
    assert torch.equal(o_d.cpu(), o_h) and torch.equal(l_d.cpu(), l_h)


def _positions(cu):
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for b in range(len(cu) - 1):
        pos[cu[b]:cu[b + 1]] = np.arange(cu[b + 1] - cu[b])
    return pos


@pytest.mark.parametrize("inter", [False, True])
def test_rope_varlen(inter):
    A = A_()
    lq = [300, 1, 0, 129, 513]
    lk = [300, 40, 17, 129, 513]
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    Hq, Hkv, D = 8, 2, 128
    g = torch.Generator().manual_seed(75)
    q = torch.randn((int(cq[-1]), Hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((int(ck[-1]), Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((int(ck[-1]), Hkv, D), generator=g).to(torch.bfloat16)
    cu_q = torch.tensor(cq, dtype=torch.int32).cuda()
    cu_k = torch.tensor(ck, dtype=torch.int32).cuda()
    for causal in (False, True):
        o, lse = A.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q, cu_k, max(lq), max(lk), causal=causal,
                                  rope_theta=THETA, rope_interleaved=inter)
        torch.cuda.synchronize()
        qr = R.rotate(np64(q).transpose(1, 0, 2), _positions(cq), THETA, inter).transpose(1, 0, 2)
        kr = R.rotate(np64(k).transpose(1, 0, 2), _positions(ck), THETA, inter).transpose(1, 0, 2)
        o_t, l_t = oracle.prefill_varlen(round16(qr, torch.bfloat16), round16(kr, torch.bfloat16), np64(v), cq, ck,
                                         causal, 1 / math.sqrt(D))
        assert_close(o, o_t, lse, l_t, f"varlen causal={causal}")
        o_x, l_x = R.prefill_varlen(np64(q), np64(k), np64(v), cq, ck, causal, 1 / math.sqrt(D), THETA, inter)
        assert np.abs(np64(o) - o_x).max() < 5e-2 and np.nanmax(np.abs(np.where(np.isinf(l_x), 0, np64(lse) - l_x))) < 3e-2


def pair_norm(x, inter):
    """|(x_a, x_b)| of the pair each coordinate belongs to (rotations keep it)."""
    D = x.shape[-1]
    if inter:
        n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
        return np.repeat(n, 2, axis=-1)
    n = np.sqrt(x[..., :D // 2] ** 2 + x[..., D // 2:] ** 2)
    return np.concatenate([n, n], axis=-1)


def assert_rotated_keys(got, k_exact, u, inter, what):
    """Keys rotated in fp32 and rounded once: within half an ulp of the exact rotation plus the fp32
    rotation's own error (a few 1e-7 of the pair's norm, which matters where the rotation cancels);
    and equal to the rounded exact rotation for all but a few elements."""
    lim = u * np.abs(k_exact) + 2e-6 * pair_norm(k_exact, inter) + 1e-30
    err = np.abs(got - k_exact)
    assert (err <= lim).all(), f"{what}: rotated key off by {(err - lim).max():.3e} beyond the bound"


def _fill_rope_cache(k, v, chunks, theta, inter, max_len=None):
    """Cache written by the GPU RoPE cache write in the given (pos, n) chunks."""
    A = A_()
    B, Hkv, L, D = k.shape
    kc = torch.zeros((B, Hkv, max_len or L, D), dtype=k.dtype, device="cuda")
    vc = torch.zeros_like(kc)
    kd, vd = k.cuda(), v.cuda()
    for pos, n in chunks:
        A.write_kv_cache(kc, vc, kd[:, :, pos:pos + n], vd[:, :, pos:pos + n], pos, rope_theta=theta,
                         rope_interleaved=inter)
    torch.cuda.synchronize()
    return kc, vc


@pytest.mark.parametrize("dt,D,inter", [("bf16", 128, False), ("f16", 64, True), ("bf16", 64, True)])
def test_rope_cache_write_and_decode(dt, D, inter):
    A = A_()
    B, Hq, Hkv, L = 2, 32, 8, 1200
    k, v = I.decode_stream(B, Hkv, L, D, dt, seed=D + inter)
    chunks = [(0, 1), (1, 7), (8, 500), (508, 1), (509, L - 509)]
    kc, vc = _fill_rope_cache(k, v, chunks, THETA, inter, max_len=L + 64)
    tdt = I.DTYPES[dt]
    # the cache: keys rotated at their positions (one rounding), values copied bit for bit
    k_exact = R.rotate(np64(k), np.arange(L), THETA, inter)
    k_round = round16(k_exact, tdt)
    got = np64(kc[:, :, :L])
    assert_rotated_keys(got, k_exact, U16[tdt], inter, "cache")
    assert np.mean(got != k_round) < 1e-3, "too many rotated keys differ from the rounded exact rotation"
    assert torch.equal(vc[:, :, :L].cpu(), v) and (kc[:, :, L:] == 0).all() and (vc[:, :, L:] == 0).all()
    lens = (1, 33, 257, 700, 1200)
    qs = I.decode_queries(B, Hq, D, [n - 1 for n in lens], dt, seed=D)
    for j, n in enumerate(lens):
        o, lse = A.decode(qs[:, :, j].cuda(), kc, vc, n, rope_theta=THETA, rope_interleaved=inter)
        torch.cuda.synchronize()
        qr = R.rotate(np64(qs[:, :, j])[:, :, None, :], [n - 1], THETA, inter)[:, :, 0, :]
        o_t, l_t = oracle.decode(qr, k_round, np64(v), n, 1 / math.sqrt(D))
        assert_close(o, o_t, lse, l_t, f"decode L={n} (rounded cache)")
        o_x, l_x = R.decode(np64(qs[:, :, j]), k_exact, np64(v), n, 1 / math.sqrt(D), THETA, inter)
        E, vmax = exact_bounds(qr[:, :, None, :], k_exact[:, :, :n], np64(v)[:, :, :n], 1 / math.sqrt(D),
                               U16[tdt] / 2, False)
        assert_within_derived(o, lse, o_x, l_x, E[:, :, 0], vmax[:, :, 0], f"decode L={n} (exact oracle)")


def test_rope_autoregressive_decode_equals_prefill_rows():
    A = A_()
    B, Hq, Hkv, D, L = 2, 8, 2, 128, 300
    q, k, v = I.prefill_inputs(B, Hq, Hkv, L, L, D, "bf16", seed=76)
    o_pre, l_pre = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope_theta=THETA)
    kc, vc = _fill_rope_cache(k, v, [(t, 1) for t in range(L)], THETA, False)
    o_steps = torch.empty_like(o_pre)
    l_steps = torch.empty_like(l_pre)
    qd = q.cuda()
    for t in range(L):
        o, lse = A.decode(qd[:, :, t], kc, vc, t + 1, rope_theta=THETA)
        o_steps[:, :, t], l_steps[:, :, t] = o, lse
    torch.cuda.synchronize()
    # Both sides round the rotated keys once; the prefill also rounds the rotated query
    # (decode keeps it in fp32), so the two differ by that one rounding.
    qr, kr = rot(q, THETA, False), rot(k, THETA, False)
    E, vmax = exact_bounds(qr, kr, np64(v), 1 / math.sqrt(D), U16[torch.bfloat16] / 2, True)
    assert_within_derived(o_steps, l_steps, np64(o_pre), np64(l_pre), E, vmax, "autoregressive")


@pytest.mark.parametrize("page_size,inter", [(16, False), (64, True)])
def test_rope_paged_write_and_decode(page_size, inter):
    A = A_()
    B, Hq, Hkv, D = 3, 16, 4, 128
    lens = [700, 0, 129]
    L = max(lens)
    max_pages = (L + page_size - 1) // page_size
    num_pages = B * max_pages + 5
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(9))[:B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)
    k, v = I.decode_stream(B, Hkv, L, D, "bf16", seed=page_size)
    kp = torch.zeros((num_pages, Hkv, page_size, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    bt = table.cuda()
    for pos0, n in ((0, 100), (100, 1), (101, L - 101)):
        A.write_kv_cache_paged(kp, vp, k[:, :, pos0:pos0 + n].cuda(), v[:, :, pos0:pos0 + n].cuda(), bt,
                               torch.full((B,), pos0, dtype=torch.int32).cuda(), rope_theta=THETA,
                               rope_interleaved=inter)
    q = I.decode_queries(B, Hq, D, [max(n - 1, 0) for n in lens], "bf16", seed=3)[:, :, 0]
    cl = torch.tensor(lens, dtype=torch.int32).cuda()
    o, lse = A.decode_paged(q.cuda(), kp, vp, bt, cl, L, rope_theta=THETA, rope_interleaved=inter)
    torch.cuda.synchronize()
    # expected pages: the oracle's RoPE paged write, rounded to bf16
    kp_x, vp_x = R.kv_cache_write_paged(np.zeros(kp.shape), np.zeros(vp.shape), np64(k), np64(v), table.numpy(),
                                        np.zeros(B, dtype=np.int64), THETA, inter)
    kp_r = round16(kp_x, torch.bfloat16)
    assert torch.equal(vp.cpu().double(), torch.from_numpy(vp_x))
    assert_rotated_keys(np64(kp), kp_x, U16[torch.bfloat16], inter, "pages")
    assert np.mean(np64(kp) != kp_r) < 1e-3
    qr = np.stack([R.rotate(np64(q[b])[:, None, :], [max(lens[b] - 1, 0)], THETA, inter)[:, 0, :] for b in range(B)])
    o_t, l_t = masked.decode_paged_masked(qr, kp_r, np64(vp), table.numpy(), lens, 1 / math.sqrt(D))
    nz = [b for b in range(B) if lens[b] > 0]
    assert_close(np64(o)[nz], o_t[nz], np64(lse)[nz], l_t[nz], f"paged page_size={page_size}")
    assert (o[1] == 0).all() and torch.isneginf(lse[1]).all()  # the empty request


@pytest.mark.parametrize("dt,D,causal,inter", [("bf16", 128, True, False), ("f16", 64, False, True)])
def test_rope_prefill_with_rotated_keys(dt, D, causal, inter):
    """rope_rotated_keys: the keys come in rotated (here: the oracle's rotation, rounded to 16 bits);
    the kernel rotates only the queries."""
    A = A_()
    tdt = I.DTYPES[dt]
    q, k, v = I.prefill_inputs(2, 8, 2, 400, 400, D, dt, seed=77 + D)
    kr = rot(k, THETA, inter)
    k_in = torch.from_numpy(kr).to(tdt)
    o, lse = A.prefill(q.cuda(), k_in.cuda(), v.cuda(), causal=causal, rope_theta=THETA, rope_interleaved=inter,
                       rope_rotated_keys=True)
    torch.cuda.synchronize()
    qh = round16(rot(q, THETA, inter), tdt)
    o_t, l_t = oracle.attention(qh, np64(k_in), np64(v), causal, 1 / math.sqrt(D))
    assert_close(o, o_t, lse, l_t, "rotated keys")


def test_rope_prefill_over_rope_cache_equals_fused():
    """The serving flow: keys written to a cache by the RoPE cache write, then a prefill over the
    cache with rope_rotated_keys, equals the prefill that rotates the raw keys itself."""
    A = A_()
    B, Hq, Hkv, N, D = 2, 16, 4, 777, 128
    q, k, v = I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=78)
    kc, vc = _fill_rope_cache(k, v, [(0, 500), (500, N - 500)], THETA, False)
    o_c, l_c = A.prefill(q.cuda(), kc, vc, causal=True, rope_theta=THETA, rope_rotated_keys=True)
    o_f, l_f = A.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope_theta=THETA)
    torch.cuda.synchronize()
    assert_close(o_c, np64(o_f), l_c, np64(l_f), "cache flow vs fused")
