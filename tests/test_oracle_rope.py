"""Pins of the rotary-embedding oracle (``oracle.rope``) to facts that do not come from it.

* Hand-derived rotations of one D = 4 row in both pair layouts
  (``tests/golden/rope_d4.json``), and the identity at position 0.
* A second formulation: pair c as the complex number x_a + i x_b multiplied
  by e^{i p theta_c} (numpy complex arithmetic, pairs and frequencies written
  independently).
* Closed forms for D = 2: unit vectors rotated at i and j have dot products
  cos(i - j) and sin(i - j).
* Rotations preserve each row's norm; scores depend only on i - j (a Toeplitz
  score matrix for constant rows, unchanged when every position is shifted).
* Attention with RoPE is the C oracle's plain attention (or the windowed /
  ALiBi oracle) on the independently rotated rows; GQA equals MHA with the
  K/V heads repeated.
* A cache filled by the RoPE cache write, then decoded, gives the last row of
  the causal RoPE prefill (dense and paged); packed variable-length batches
  count positions per sequence.
Every planted mistake in ``oracle/rope.py`` (MUTANTS) fails at least one pin.
"""
from __future__ import annotations

import json
import os
import types
import zlib

import numpy as np
import pytest

import oracle
from oracle import masked
from oracle import rope as ROPE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_d4.json")
TOL = 1e-10


def _rng(*key):
    return np.random.default_rng(zlib.crc32(repr(key).encode()))


def complex_rotate(x, positions, theta, interleaved):
    """Second formulation: pair c as a complex number, multiplied by exp(i * p * theta^(-2c/D))."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    if interleaved:
        z = x[..., 0::2] + 1j * x[..., 1::2]
    else:
        z = x[..., :D // 2] + 1j * x[..., D // 2:]
    freq = np.power(float(theta), -np.arange(0, D, 2, dtype=np.float64) / D)
    z = z * np.exp(1j * np.outer(np.asarray(positions, dtype=np.float64), freq))
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = z.real, z.imag
    else:
        out[..., :D // 2], out[..., D // 2:] = z.real, z.imag
    return out


def check_golden_d4(R):
    g = json.load(open(GOLDEN))
    x = np.array(g["x"])[None, :]
    for layout, inter in (("half", False), ("interleaved", True)):
        got = R.rotate(x, [g["position"]], g["theta"], inter)[0]
        assert np.allclose(got, g["expected"][layout], rtol=0, atol=1e-13), (layout, got)
        assert np.array_equal(R.rotate(x, [0], g["theta"], inter), x)


def check_complex_formulation(R):
    for D in (2, 4, 64, 128):
        for inter in (False, True):
            r = _rng("cx", D, inter)
            x = r.normal(size=(3, 17, D))
            pos = r.integers(0, 100000, size=17)
            for theta in (10000.0, 500000.0, 7.5):
                assert np.allclose(R.rotate(x, pos, theta, inter), complex_rotate(x, pos, theta, inter),
                                   rtol=0, atol=1e-9), (D, inter, theta)


def check_d2_closed_forms(R):
    n = 9
    i = np.arange(n)
    e0 = np.tile([1.0, 0.0], (n, 1))
    e1 = np.tile([0.0, 1.0], (n, 1))
    for inter in (False, True):  # D = 2: both layouts pair (0, 1)
        qr = R.rotate(e0, i, 1234.0, inter)
        s_cos = qr @ R.rotate(e0, i, 1234.0, inter).T
        s_sin = qr @ R.rotate(e1, i, 1234.0, inter).T
        d = (i[:, None] - i[None, :]).astype(np.float64)
        assert np.allclose(s_cos, np.cos(d), atol=1e-12) and np.allclose(s_sin, np.sin(d), atol=1e-12)


def check_norm_and_relative_position(R):
    r = _rng("rel")
    for inter in (False, True):
        x = r.normal(size=(40, 64))
        pos = r.integers(0, 50000, size=40)
        xr = R.rotate(x, pos, 10000.0, inter)
        assert np.allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
        q, k = r.normal(size=64), r.normal(size=64)
        n = 24
        p = np.arange(n)
        s = R.rotate(np.tile(q, (n, 1)), p, 10000.0, inter) @ R.rotate(np.tile(k, (n, 1)), p, 10000.0, inter).T
        assert np.allclose(s[1:, 1:], s[:-1, :-1], atol=1e-10)  # depends on i - j only
        s_shift = (R.rotate(np.tile(q, (n, 1)), p + 777, 10000.0, inter)
                   @ R.rotate(np.tile(k, (n, 1)), p + 777, 10000.0, inter).T)
        assert np.allclose(s, s_shift, atol=1e-9)
        assert not np.allclose(s[0, 0], s[0, 5])  # positions matter at all


def check_attention_is_plain_on_rotated_rows(R):
    for inter in (False, True):
        for causal in (False, True):
            r = _rng("att", inter, causal)
            q, k, v = r.normal(size=(2, 4, 37, 64)), r.normal(size=(2, 2, 41, 64)), r.normal(size=(2, 2, 41, 64))
            o, lse = R.attention(q, k, v, causal, 0.125, 10000.0, inter)
            qr = complex_rotate(q, np.arange(37), 10000.0, inter)
            kr = complex_rotate(k, np.arange(41), 10000.0, inter)
            o_ref, lse_ref = oracle.attention(qr, kr, v, causal, 0.125)
            assert np.allclose(o, o_ref, atol=TOL) and np.allclose(lse, lse_ref, atol=TOL)
    # with a window and ALiBi slopes
    r = _rng("att-masked")
    q, k, v = r.normal(size=(1, 4, 50, 32)), r.normal(size=(1, 1, 50, 32)), r.normal(size=(1, 1, 50, 32))
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    o, lse = R.attention(q, k, v, False, 0.2, 500000.0, False, 7, 3, slopes)
    o_ref, lse_ref = masked.attention_masked(complex_rotate(q, np.arange(50), 500000.0, False),
                                             complex_rotate(k, np.arange(50), 500000.0, False), v, False, 0.2, 7,
                                             3, slopes)
    assert np.allclose(o, o_ref, atol=TOL) and np.allclose(lse, lse_ref, atol=TOL)


def check_gqa_is_mha_expanded(R):
    r = _rng("gqa")
    q, k, v = r.normal(size=(1, 8, 20, 64)), r.normal(size=(1, 2, 20, 64)), r.normal(size=(1, 2, 20, 64))
    o, lse = R.attention(q, k, v, True, 0.125, 10000.0, False)
    o2, lse2 = R.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), True, 0.125, 10000.0, False)
    assert np.allclose(o, o2, atol=TOL) and np.allclose(lse, lse2, atol=TOL)


def check_cache_write_rotates_keys_only(R):
    r = _rng("write")
    for inter in (False, True):
        kc, vc = r.normal(size=(2, 2, 30, 64)), r.normal(size=(2, 2, 30, 64))
        kn, vn = r.normal(size=(2, 2, 5, 64)), r.normal(size=(2, 2, 5, 64))
        k2, v2 = R.kv_cache_write(kc, vc, kn, vn, 11, 10000.0, inter)
        assert np.allclose(k2[:, :, 11:16], complex_rotate(kn, np.arange(11, 16), 10000.0, inter), atol=1e-12)
        assert np.array_equal(v2[:, :, 11:16], vn)
        for sl in (slice(0, 11), slice(16, 30)):
            assert np.array_equal(k2[:, :, sl], kc[:, :, sl]) and np.array_equal(v2[:, :, sl], vc[:, :, sl])


def _fill_cache(R, k, v, theta, inter, chunks):
    """Cache written in the given chunks (pos, n) by the RoPE cache write."""
    kc, vc = np.zeros_like(k), np.zeros_like(v)
    for pos, n in chunks:
        kc, vc = R.kv_cache_write(kc, vc, k[:, :, pos:pos + n], v[:, :, pos:pos + n], pos, theta, inter)
    return kc, vc


def check_decode_is_last_prefill_row(R):
    for inter in (False, True):
        r = _rng("dec", inter)
        B, Hq, Hkv, L, D = 2, 4, 2, 45, 64
        q, k, v = r.normal(size=(B, Hq, L, D)), r.normal(size=(B, Hkv, L, D)), r.normal(size=(B, Hkv, L, D))
        kc, vc = _fill_cache(R, k, v, 10000.0, inter, [(0, 20), (20, 1), (21, 24)])
        o_pre, lse_pre = R.attention(q, k, v, True, 0.125, 10000.0, inter)
        for n in (1, 21, 45):
            o, lse = R.decode(q[:, :, n - 1], kc, vc, n, 0.125, 10000.0, inter)
            assert np.allclose(o, o_pre[:, :, n - 1], atol=TOL) and np.allclose(lse, lse_pre[:, :, n - 1], atol=TOL)
        slopes = np.array([0.3, 0.2, 0.1, 0.05])
        o_w, lse_w = R.attention(q, k, v, True, 0.125, 10000.0, inter, 9, -1, slopes)
        o, lse = R.decode(q[:, :, L - 1], kc, vc, L, 0.125, 10000.0, inter, 9, slopes)
        assert np.allclose(o, o_w[:, :, L - 1], atol=TOL) and np.allclose(lse, lse_w[:, :, L - 1], atol=TOL)


def check_paged_equals_dense(R):
    r = _rng("paged")
    B, Hq, Hkv, D, page, L = 3, 4, 2, 64, 16, 40
    lens = np.array([40, 17, 1])
    k, v = r.normal(size=(B, Hkv, L, D)), r.normal(size=(B, Hkv, L, D))
    q = r.normal(size=(B, Hq, D))
    n_pages = 3 * ((L + page - 1) // page)
    table = r.permutation(n_pages).reshape(B, -1)
    kp, vp = np.zeros((n_pages, Hkv, page, D)), np.zeros((n_pages, Hkv, page, D))
    kp, vp = R.kv_cache_write_paged(kp, vp, k[:, :, :10], v[:, :, :10], table, np.zeros(B, dtype=int), 10000.0)
    kp, vp = R.kv_cache_write_paged(kp, vp, k[:, :, 10:], v[:, :, 10:], table, np.full(B, 10), 10000.0)
    o, lse = R.decode_paged(q, kp, vp, table, lens, 0.125, 10000.0)
    kc, vc = _fill_cache(R, k, v, 10000.0, False, [(0, L)])
    for b in range(B):
        ob, lb = R.decode(q[b:b + 1], kc[b:b + 1], vc[b:b + 1], int(lens[b]), 0.125, 10000.0)
        assert np.allclose(o[b], ob[0], atol=TOL) and np.allclose(lse[b], lb[0], atol=TOL)


def check_varlen_positions_per_sequence(R):
    r = _rng("varlen")
    lq, lk = [13, 30, 1], [20, 30, 7]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, k, v = r.normal(size=(sum(lq), 4, 64)), r.normal(size=(sum(lk), 2, 64)), r.normal(size=(sum(lk), 2, 64))
    for causal in (False, True):
        o, lse = R.prefill_varlen(q, k, v, cu_q, cu_k, causal, 0.125, 10000.0, True)
        for b in range(3):
            qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            ob, lb = R.attention(q[qs:qe].transpose(1, 0, 2)[None], k[ks:ke].transpose(1, 0, 2)[None],
                                 v[ks:ke].transpose(1, 0, 2)[None], causal, 0.125, 10000.0, True)
            assert np.allclose(o[qs:qe], ob[0].transpose(1, 0, 2), atol=TOL)
            assert np.allclose(lse[:, qs:qe], lb[0], atol=TOL)


def _fd_check(R, grads, loss, base, what):
    """Every entry of grads (dict name -> array) against central differences of loss(**inputs)."""
    eps = 1e-5
    for name, grad in grads.items():
        for idx in np.ndindex(base[name].shape):
            xp, xm = base[name].copy(), base[name].copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = dict(base), dict(base)
            ap[name], am[name] = xp, xm
            fd = (loss(**ap) - loss(**am)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (what, name, idx, fd, grad[idx])


def check_bwd_matches_finite_differences(R):
    """Gradients of the rotary attention against central finite differences through ``attention`` (both
    pair layouts, causal and windowed + ALiBi, key ranges) and, with keys given rotated, through attention of
    the rotated queries over those keys."""
    r = _rng("bwd-fd")
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 4, 6, 4
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    g = r.normal(size=q.shape)
    base = {"q": q, "k": k, "v": v}
    for inter, causal, kw in ((False, True, {}), (True, False, dict(window_left=2, window_right=1,
                                                                   alibi_slopes=[0.4, 0.15]))):
        dq, dk, dv = R.attention_bwd(q, k, v, g, causal, 0.7, 100.0, inter, **kw)

        def loss(q, k, v):
            o, _ = R.attention(q, k, v, causal, 0.7, 100.0, inter, **kw)
            return float(np.sum(o * g))
        _fd_check(R, {"q": dq, "k": dk, "v": dv}, loss, base, f"inter={inter}")
    kr = np.array([[[0, 3], [2, 6], [1, 1], [0, 6]]], dtype=np.int32)  # one row without keys
    dq, dk, dv = R.attention_bwd(q, k, v, g, False, 0.7, 100.0, True, kv_ranges=kr)

    def loss_ranges(q, k, v):
        o, _ = masked.attention_masked(R.rotate(q, np.arange(Nq), 100.0, True), R.rotate(k, np.arange(Nkv), 100.0,
                                                                                          True), v, False, 0.7,
                                       kv_ranges=kr)
        return float(np.sum(o * g))
    _fd_check(R, {"q": dq, "k": dk, "v": dv}, loss_ranges, base, "key ranges")
    dq, dk, dv = R.attention_bwd(q, k, v, g, True, 0.7, 100.0, False, rotated_keys=True)

    def loss_rk(q, k, v):
        o, _ = oracle.attention(R.rotate(q, np.arange(Nq), 100.0), k, v, True, 0.7)
        return float(np.sum(o * g))
    _fd_check(R, {"q": dq, "k": dk, "v": dv}, loss_rk, base, "rotated keys")


def check_bwd_at_position_zero_is_plain(R):
    """One query and one key at position 0: no rotation, so the plain backward."""
    r = _rng("bwd-p0")
    q, k, v, g = (r.normal(size=(2, 4, 1, 8)), r.normal(size=(2, 2, 1, 8)), r.normal(size=(2, 2, 1, 8)),
                  r.normal(size=(2, 4, 1, 8)))
    got = R.attention_bwd(q, k, v, g, True, 0.3, 10000.0)
    ref = oracle.attention_bwd(q, k, v, g, True, 0.3)
    for a, b in zip(got, ref):
        assert np.allclose(a, b, atol=TOL)


CHECKS = [check_golden_d4, check_complex_formulation, check_d2_closed_forms, check_norm_and_relative_position,
          check_attention_is_plain_on_rotated_rows, check_gqa_is_mha_expanded, check_cache_write_rotates_keys_only,
          check_decode_is_last_prefill_row, check_paged_equals_dense, check_varlen_positions_per_sequence,
          check_bwd_matches_finite_differences, check_bwd_at_position_zero_is_plain]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_rope_oracle_pin(check):
    check(ROPE)


# Planted mistakes in oracle/rope.py: (anchor, replacement), every occurrence replaced.
MUTANTS = {
    "frequency exponent halved": ("-2.0 * c / D", "-1.0 * c / D"),
    "first coordinate sign": ("out[..., a] = xa * cs - xb * sn", "out[..., a] = xa * cs + xb * sn"),
    "second coordinate sign": ("out[..., b] = xb * cs + xa * sn", "out[..., b] = xb * cs - xa * sn"),
    "rotate-half pairs shifted": ("a, b = c, c + D // 2", "a, b = c, (c + D // 2 + 1) % D"),
    "interleaved pair order swapped": ("a, b = 2 * c, 2 * c + 1", "a, b = 2 * c + 1, 2 * c"),
    "query positions from 1": ("qr = rotate(q, np.arange(q.shape[2])", "qr = rotate(q, 1 + np.arange(q.shape[2])"),
    "keys not rotated": ("kr = rotate(k, np.arange(k.shape[2]), theta, interleaved)", "kr = k"),
    "decode query at cache_len": ("[cache_len - 1]", "[cache_len]"),
    "cache write one position late": ("kr = rotate(k_new, pos + np.arange(k_new.shape[2])",
                                      "kr = rotate(k_new, pos + 1 + np.arange(k_new.shape[2])"),
    "values rotated on write": ("kr, _f64(v_new), pos)",
                                "kr, rotate(_f64(v_new), pos + np.arange(k_new.shape[2]), theta, interleaved), pos)"),
    "varlen positions not reset": ("pos[s:e] = np.arange(e - s)", "pos[s:e] = np.arange(s, e)"),
    "paged write one position late": ("int(positions[b]) + np.arange(k_new.shape[2])",
                                      "int(positions[b]) + 1 + np.arange(k_new.shape[2])"),
    "paged decode query at the length": ("[int(cache_lens[b]) - 1]", "[int(cache_lens[b])]"),
    "bwd dQ not rotated back": ("dq = rotate(dqr, -qpos, theta, interleaved)", "dq = dqr"),
    "bwd dQ rotated forward again": ("dq = rotate(dqr, -qpos, theta, interleaved)",
                                     "dq = rotate(dqr, qpos, theta, interleaved)"),
    "bwd dK not rotated back": ("dk = dkr if rotated_keys else rotate(dkr, -kpos, theta, interleaved)", "dk = dkr"),
    "bwd rotated keys rotated again": ("kr = k if rotated_keys else rotate(k, kpos, theta, interleaved)",
                                       "kr = rotate(k, kpos, theta, interleaved)"),
    "bwd keys rotated at query positions": ("kr = k if rotated_keys else rotate(k, kpos, theta, interleaved)",
                                            "kr = k if rotated_keys else rotate(k, np.arange(k.shape[2]) + 1, "
                                            "theta, interleaved)"),
}


def _mutant(old, new):
    with open(ROPE.__file__) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("rope_mutant")
    exec(compile(src.replace(old, new), "rope_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_rope_planted_mistakes_are_caught(name):
    mk = _mutant(*MUTANTS[name])
    caught = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mk)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"mutant '{name}' passed every pin"
