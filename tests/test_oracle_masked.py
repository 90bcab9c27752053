"""Pins of the windowed / ALiBi oracle (``oracle.masked``) to facts that do not come from it.

* A window wider than the sequences changes nothing: the C oracle's plain
  attention (an independent implementation).
* Each row of a windowed prefill is the C oracle's decode over the slice of
  keys in the row's band; a row whose band is empty gives O = 0, LSE = -inf.
* window_left = 0 with the causal mask leaves row i only key i: O_i = V_i and
  LSE_i = scale q_i . k_i.
* ALiBi with slope 0 is plain attention; with all keys equal the weights are
  geometric in |i - j|, so O and LSE have closed forms.
* ALiBi as an extra dimension: -slope (i - j) = slope j - slope i, and the
  per-row constant -slope i leaves the softmax unchanged, so appending slope_h
  to q and j / scale to k_j turns the causal ALiBi problem into a plain one for
  the C oracle (LSE shifted by -slope i).  Without the causal mask the keys
  left and right of i are two such problems merged by their LSEs.
* Decode is the last row of a causal prefill of cache_len rows, and paged
  decode is decode over the gathered rows for any page order.
* Per-row key ranges: each row equals the C oracle's decode over the keys of
  its range (intersected with the causal bound; empty ranges give 0 / -inf);
  full ranges are plain attention; block-diagonal ranges over one packed
  batch equal the C oracle's variable-length attention of the blocks.
Every planted mistake in ``oracle/masked.py`` (MUTANTS) fails at least one pin.
"""
from __future__ import annotations

import math
import types
import zlib

import numpy as np
import pytest

import oracle
from oracle import masked as M

TOL = 1e-12


def _rng(*key):
    return np.random.default_rng(zlib.crc32(repr(key).encode()))


def _qkv(B, Hq, Hkv, Nq, Nkv, D, *key):
    r = _rng(*key)
    return r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))


def _band(i, Nkv, causal, wl, wr):
    lo = 0 if wl < 0 else max(0, i - wl)
    hi = Nkv - 1
    if wr >= 0:
        hi = min(hi, i + wr)
    if causal:
        hi = min(hi, i)
    return lo, hi


def _close(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    same_inf = np.isneginf(a) == np.isneginf(b)
    assert same_inf.all(), f"{what}: -inf pattern differs"
    fin = np.isfinite(b)
    assert np.allclose(a[fin], b[fin], rtol=0, atol=1e-10), f"{what}: max err {np.abs(a[fin] - b[fin]).max():.3e}"


WINDOWS = [(2, 1), (0, 3), (4, -1), (-1, 2), (0, 0), (1, 1)]
SHAPES = [(7, 7), (9, 6), (5, 11)]


def check_unbounded_window_is_plain(mk):
    for causal in (False, True):
        for Nq, Nkv in SHAPES:
            q, k, v = _qkv(2, 4, 2, Nq, Nkv, 3, "plain", causal, Nq, Nkv)
            o_ref, l_ref = oracle.attention(q, k, v, causal, 0.7)
            for wl, wr in ((-1, -1), (Nq + Nkv, Nq + Nkv)):
                o, l = mk.attention_masked(q, k, v, causal, 0.7, wl, wr)
                _close(o, o_ref, "O unbounded window")
                _close(l, l_ref, "LSE unbounded window")


def check_band_rows_are_decode_over_slice(mk):
    scale = 0.6
    for causal in (False, True):
        for Nq, Nkv in SHAPES:
            q, k, v = _qkv(2, 4, 2, Nq, Nkv, 3, "band", causal, Nq, Nkv)
            for wl, wr in WINDOWS:
                o, l = mk.attention_masked(q, k, v, causal, scale, wl, wr)
                for i in range(Nq):
                    lo, hi = _band(i, Nkv, causal, wl, wr)
                    if lo > hi:
                        assert (o[:, :, i] == 0).all() and np.isneginf(l[:, :, i]).all(), f"empty band row {i}"
                        continue
                    ks, vs = k[:, :, lo:hi + 1], v[:, :, lo:hi + 1]
                    o_ref, l_ref = oracle.decode(q[:, :, i], ks, vs, hi - lo + 1, scale)
                    _close(o[:, :, i], o_ref, f"O row {i} window ({wl},{wr}) causal={causal}")
                    _close(l[:, :, i], l_ref, f"LSE row {i} window ({wl},{wr}) causal={causal}")


def check_identity_window(mk):
    q, k, v = _qkv(1, 4, 2, 8, 8, 3, "identity")
    scale = 0.9
    for causal, wr in ((True, -1), (False, 0)):
        o, l = mk.attention_masked(q, k, v, causal, scale, 0, wr)
        for h in range(4):
            np.testing.assert_allclose(o[0, h], v[0, h // 2], rtol=0, atol=TOL)
            np.testing.assert_allclose(l[0, h], scale * np.einsum("nd,nd->n", q[0, h], k[0, h // 2]), rtol=0,
                                       atol=TOL)
    # more queries than keys: rows past the last key see nothing
    q, k, v = _qkv(1, 2, 2, 9, 5, 3, "identity-tall")
    o, l = mk.attention_masked(q, k, v, False, scale, 0, 0)
    assert (o[0, :, 5:] == 0).all() and np.isneginf(l[0, :, 5:]).all()
    np.testing.assert_allclose(o[0, :, :5], v[0], rtol=0, atol=TOL)


def check_alibi_zero_slope_is_plain(mk):
    for causal in (False, True):
        q, k, v = _qkv(2, 4, 2, 6, 8, 3, "slope0", causal)
        o, l = mk.attention_masked(q, k, v, causal, 0.5, alibi_slopes=np.zeros(4))
        o_ref, l_ref = oracle.attention(q, k, v, causal, 0.5)
        _close(o, o_ref, "O slope 0")
        _close(l, l_ref, "LSE slope 0")


def check_alibi_identical_keys_closed_form(mk):
    N, D, scale = 9, 3, 0.8
    r = _rng("alibi-identical")
    q = r.normal(size=(1, 3, N, D))
    kap = r.normal(size=D)
    k = np.broadcast_to(kap, (1, 1, N, D)).copy()
    v = r.normal(size=(1, 1, N, D))
    slopes = np.array([0.25, 0.5, 1.5])
    for causal in (True, False):
        o, l = mk.attention_masked(q, k, v, causal, scale, alibi_slopes=slopes)
        for h, sl in enumerate(slopes):
            rho = math.exp(-sl)
            for i in range(N):
                # weights rho^|i-j| over the visible keys; sums of geometric series
                left = (1 - rho ** (i + 1)) / (1 - rho)
                right = 0.0 if causal else rho * (1 - rho ** (N - 1 - i)) / (1 - rho)
                lse = scale * float(q[0, h, i] @ kap) + math.log(left + right)
                assert abs(l[0, h, i] - lse) < 1e-10, (causal, h, i)
                js = np.arange(i + 1) if causal else np.arange(N)
                w = rho ** np.abs(i - js) / (left + right)
                np.testing.assert_allclose(o[0, h, i], w @ v[0, 0, js], rtol=0, atol=1e-10)


def _augment(x, col):
    """Append one column (broadcast over the leading axes) to the last axis."""
    return np.concatenate([x, np.broadcast_to(col, x.shape[:-1] + (1,))], axis=-1)


def check_alibi_causal_is_plain_with_extra_dimension(mk):
    B, Hq, Hkv, N, D, scale = 2, 4, 2, 10, 3, 0.7
    q, k, v = _qkv(B, Hq, Hkv, N, N, D, "alibi-aug")
    slopes = np.array([0.1, 0.3, 0.9, 2.0])
    o, l = mk.attention_masked(q, k, v, True, scale, alibi_slopes=slopes)
    qa = _augment(q, slopes[None, :, None, None])
    ka = _augment(k, (np.arange(N) / scale)[None, None, :, None])
    o_ref, l_ref = oracle.attention(qa, ka, _augment(v, 0.0), True, scale)
    _close(o, o_ref[..., :D], "O ALiBi causal")
    _close(l, l_ref - slopes[None, :, None] * np.arange(N)[None, None, :], "LSE ALiBi causal")


def check_alibi_window_two_sided_by_merge(mk):
    """Non-causal windowed ALiBi: keys left and right of row i are two plain problems, merged by LSE."""
    B, Hq, Hkv, Nq, Nkv, D, scale = 1, 2, 1, 7, 9, 3, 0.6
    q, k, v = _qkv(B, Hq, Hkv, Nq, Nkv, D, "alibi-merge")
    slopes = np.array([0.4, 1.1])
    for wl, wr in ((-1, -1), (2, 3), (0, 1), (3, 0)):
        o, l = mk.attention_masked(q, k, v, False, scale, wl, wr, alibi_slopes=slopes)
        for i in range(Nq):
            lo, hi = _band(i, Nkv, False, wl, wr)
            parts = []
            for side, a, z in ((+1, lo, min(hi, i)), (-1, max(lo, i + 1), hi)):
                if a > z:
                    continue
                # side +1: bias slope*j - slope*i ; side -1: -slope*j + slope*i
                qa = _augment(q[:, :, i], (side * slopes)[None, :, None])
                ka = _augment(k[:, :, a:z + 1], (np.arange(a, z + 1) / scale)[None, None, :, None])
                op, lp = oracle.decode(qa, ka, _augment(v[:, :, a:z + 1], 0.0), z - a + 1, scale)
                parts.append((op[..., :D], lp - side * slopes[None, :] * i))
            if not parts:
                assert (o[:, :, i] == 0).all() and np.isneginf(l[:, :, i]).all()
                continue
            lse = np.logaddexp.reduce([p[1] for p in parts], axis=0)
            om = sum(np.exp(p[1] - lse)[..., None] * p[0] for p in parts)
            _close(o[:, :, i], om, f"O row {i} window ({wl},{wr})")
            _close(l[:, :, i], lse, f"LSE row {i} window ({wl},{wr})")


def check_decode_is_last_prefill_row(mk):
    B, Hq, Hkv, D, scale = 2, 4, 2, 3, 0.5
    slopes = np.array([0.2, 0.7, 1.3, 0.05])
    for n in (1, 2, 9):
        q, k, v = _qkv(B, Hq, Hkv, n, n + 3, D, "dec-last", n)  # caches longer than n: tail ignored
        for wl in (-1, 0, 3, 50):
            for sl in (None, slopes):
                o, l = mk.decode_masked(q[:, :, -1], k, v, n, scale, wl, sl)
                o_ref, l_ref = mk.attention_masked(q, k[:, :, :n], v[:, :, :n], True, scale, wl, -1, sl)
                _close(o, o_ref[:, :, -1], f"decode O n={n} wl={wl}")
                _close(l, l_ref[:, :, -1], f"decode LSE n={n} wl={wl}")
    o, l = mk.decode_masked(q[:, :, -1], k, v, 0, scale, 3, slopes)
    assert (o == 0).all() and np.isneginf(l).all()


def check_decode_alibi_extra_dimension(mk):
    B, Hq, Hkv, L, D, scale = 2, 4, 2, 12, 3, 0.9
    r = _rng("dec-aug")
    q = r.normal(size=(B, Hq, D))
    k, v = r.normal(size=(B, Hkv, L, D)), r.normal(size=(B, Hkv, L, D))
    slopes = np.array([0.3, 0.6, 1.2, 2.4])
    for n, wl in ((12, -1), (12, 4), (7, 0), (5, 10)):
        o, l = mk.decode_masked(q, k, v, n, scale, wl, slopes)
        lo = 0 if wl < 0 else max(0, n - 1 - wl)
        qa = _augment(q, slopes[None, :, None])
        ka = _augment(k[:, :, lo:n], (np.arange(lo, n) / scale)[None, None, :, None])
        o_ref, l_ref = oracle.decode(qa, ka, _augment(v[:, :, lo:n], 0.0), n - lo, scale)
        _close(o, o_ref[..., :D], f"decode ALiBi O n={n} wl={wl}")
        _close(l, l_ref - slopes[None, :] * (n - 1), f"decode ALiBi LSE n={n} wl={wl}")


def check_paged_is_decode_over_gathered_rows(mk):
    B, Hq, Hkv, D, ps, scale = 3, 4, 2, 3, 4, 0.7
    lens = [0, 7, 13]
    max_pages = 4
    r = _rng("paged-masked")
    num_pages = B * max_pages + 2
    kp, vp = r.normal(size=(num_pages, Hkv, ps, D)), r.normal(size=(num_pages, Hkv, ps, D))
    table = r.permutation(num_pages)[:B * max_pages].reshape(B, max_pages)
    q = r.normal(size=(B, Hq, D))
    slopes = np.array([0.5, 0.25, 0.125, 1.0])
    for wl in (-1, 0, 5):
        o, l = mk.decode_paged_masked(q, kp, vp, table, lens, scale, wl, slopes)
        for b in range(B):
            n = lens[b]
            if n == 0:
                assert (o[b] == 0).all() and np.isneginf(l[b]).all()
                continue
            kc = np.stack([kp[table[b][t // ps], :, t % ps] for t in range(n)], axis=1)[None]
            vc = np.stack([vp[table[b][t // ps], :, t % ps] for t in range(n)], axis=1)[None]
            o_ref, l_ref = mk.decode_masked(q[b:b + 1], kc, vc, n, scale, wl, slopes)
            _close(o[b], o_ref[0], f"paged O b={b} wl={wl}")
            _close(l[b], l_ref[0], f"paged LSE b={b} wl={wl}")


def check_varlen_equal_lengths_is_dense_batch(mk):
    B, Hq, Hkv, N, D, scale = 3, 4, 2, 6, 3, 0.8
    q, k, v = _qkv(B, Hq, Hkv, N, N, D, "varlen-masked")
    slopes = np.array([0.3, 0.1, 0.7, 0.2])
    cu = np.arange(B + 1) * N
    for causal, wl, wr in ((True, 2, -1), (False, 1, 2)):
        o, l = mk.prefill_varlen_masked(q.transpose(0, 2, 1, 3).reshape(B * N, Hq, D),
                                        k.transpose(0, 2, 1, 3).reshape(B * N, Hkv, D),
                                        v.transpose(0, 2, 1, 3).reshape(B * N, Hkv, D), cu, cu, causal, scale,
                                        wl, wr, slopes)
        o_ref, l_ref = mk.attention_masked(q, k, v, causal, scale, wl, wr, slopes)
        _close(o, o_ref.transpose(0, 2, 1, 3).reshape(B * N, Hq, D), "varlen O")
        _close(l, l_ref.transpose(1, 0, 2).reshape(Hq, B * N), "varlen LSE")


def _random_ranges(rng, B, Nq, Nkv):
    lo = rng.integers(0, Nkv + 1, size=(B, Nq))
    hi = rng.integers(0, Nkv + 1, size=(B, Nq))
    lo, hi = np.minimum(lo, hi), np.maximum(lo, hi)
    r = np.stack([lo, hi], axis=-1)
    r[:, 0] = (0, Nkv)                    # a full row
    r[:, min(1, Nq - 1)] = (Nkv // 2, Nkv // 2)  # an empty row
    return r


def check_range_rows_are_decode_over_slice(mk):
    scale = 0.7
    for causal in (False, True):
        for Nq, Nkv in ((9, 9), (5, 13), (16, 7)):
            q, k, v = _qkv(2, 4, 2, Nq, Nkv, 3, "ranges", causal, Nq, Nkv)
            kr = _random_ranges(_rng("kr", causal, Nq, Nkv), 2, Nq, Nkv)
            o, l = mk.attention_masked(q, k, v, causal, scale, kv_ranges=kr)
            for b in range(2):
                for i in range(Nq):
                    lo, hi = int(kr[b, i, 0]), int(kr[b, i, 1])
                    if causal:
                        hi = min(hi, i + 1)
                    if lo >= hi:
                        assert (o[b, :, i] == 0).all() and np.isneginf(l[b, :, i]).all(), f"empty range row {i}"
                        continue
                    o_ref, l_ref = oracle.decode(q[b:b + 1, :, i], k[b:b + 1, :, lo:hi], v[b:b + 1, :, lo:hi],
                                                 hi - lo, scale)
                    _close(o[b, :, i], o_ref[0], f"O b={b} row {i} range [{lo},{hi}) causal={causal}")
                    _close(l[b, :, i], l_ref[0], f"LSE b={b} row {i} range [{lo},{hi}) causal={causal}")


def check_full_ranges_are_plain(mk):
    q, k, v = _qkv(2, 4, 2, 11, 17, 3, "fullranges")
    kr = np.zeros((2, 11, 2), dtype=np.int64)
    kr[..., 1] = 17
    for causal in (False, True):
        o, l = mk.attention_masked(q, k, v, causal, 0.5, kv_ranges=kr)
        o_ref, l_ref = oracle.attention(q, k, v, causal, 0.5)
        _close(o, o_ref, "full ranges O")
        _close(l, l_ref, "full ranges LSE")


def check_block_diagonal_ranges_are_varlen(mk):
    """Documents of lengths 4, 1, 6 packed in one row of 11: each query sees only its own document."""
    lens = [4, 1, 6]
    cu = np.concatenate([[0], np.cumsum(lens)])
    N = int(cu[-1])
    q, k, v = _qkv(1, 4, 2, N, N, 3, "blockdiag")
    kr = np.zeros((1, N, 2), dtype=np.int64)
    for d in range(len(lens)):
        kr[0, cu[d]:cu[d + 1]] = (cu[d], cu[d + 1])
    for causal in (False, True):
        o, l = mk.attention_masked(q, k, v, False, 0.8, kv_ranges=kr) if not causal else \
            mk.attention_masked(q, k, v, True, 0.8, kv_ranges=kr)
        o_ref, l_ref = oracle.prefill_varlen(q[0].transpose(1, 0, 2), k[0].transpose(1, 0, 2),
                                             v[0].transpose(1, 0, 2), cu, cu, causal, 0.8)
        _close(o[0], o_ref.transpose(1, 0, 2), f"block-diagonal O causal={causal}")
        _close(l[0], l_ref, f"block-diagonal LSE causal={causal}")


def check_varlen_ranges_count_from_sequence_start(mk):
    lq, lk = [5, 3], [7, 4]
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    r = _rng("varlen-ranges")
    q, k, v = r.normal(size=(8, 4, 3)), r.normal(size=(11, 2, 3)), r.normal(size=(11, 2, 3))
    kr = np.stack([r.integers(0, 3, size=8), r.integers(3, 8, size=8)], axis=1)
    kr[5:, 1] = np.minimum(kr[5:, 1], 4)
    o, l = mk.prefill_varlen_masked(q, k, v, cq, ck, False, 0.6, kv_ranges=kr)
    for b in range(2):
        ob, lb = mk.attention_masked(q[cq[b]:cq[b + 1]].transpose(1, 0, 2)[None], k[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None],
                                     v[ck[b]:ck[b + 1]].transpose(1, 0, 2)[None], False, 0.6,
                                     kv_ranges=kr[cq[b]:cq[b + 1]][None])
        _close(o[cq[b]:cq[b + 1]], ob[0].transpose(1, 0, 2), f"varlen ranges O seq {b}")
        _close(l[:, cq[b]:cq[b + 1]], lb[0], f"varlen ranges LSE seq {b}")
    # and against the slice definition for one row of the second sequence
    i = 6
    lo, hi = int(kr[i, 0]), int(kr[i, 1])
    o_ref, l_ref = oracle.decode(q[i][None], k[ck[1] + lo:ck[1] + hi].transpose(1, 0, 2)[None],
                                 v[ck[1] + lo:ck[1] + hi].transpose(1, 0, 2)[None], hi - lo, 0.6)
    _close(o[i], o_ref[0], "varlen range row O")


def check_bwd_without_options_is_plain_bwd(mk):
    """No window, bias or ranges: the masked backward is the plain backward oracle."""
    q, k, v = _qkv(2, 4, 2, 6, 9, 3, "bwd-plain")
    g = _rng("bwd-plain-g").normal(size=q.shape)
    for causal in (False, True):
        got = mk.attention_bwd_masked(q, k, v, g, causal, 0.7)
        ref = oracle.attention_bwd(q, k, v, g, causal, 0.7)
        for name, a, b in zip("qkv", got, ref):
            _close(a, b, f"plain bwd d{name} causal={causal}")


def _fd_loss(mk, q, k, v, g, causal, scale, **kw):
    o, _ = mk.attention_masked(q, k, v, causal, scale, **kw)
    return float(np.sum(o * g))


def check_bwd_matches_finite_differences(mk):
    """Every gradient entry of a small GQA case with a window, ALiBi and key ranges (one row empty) against
    central finite differences of L = sum(O * G) through the masked forward."""
    q, k, v = _qkv(1, 4, 2, 5, 7, 3, "bwd-fd")
    r = _rng("bwd-fd-g")
    g = r.normal(size=q.shape)
    kr = np.array([[[0, 7], [1, 5], [2, 2], [0, 4], [3, 7]]])
    for causal, kw in ((False, dict(window_left=2, window_right=1, alibi_slopes=[0.5, 0.25, 0.8, 0.1])),
                       (True, dict(window_left=3, alibi_slopes=[0.3, 0.0, 1.1, 0.7], kv_ranges=kr))):
        dq, dk, dv = mk.attention_bwd_masked(q, k, v, g, causal, 0.6, **kw)
        eps = 1e-5
        for name, grad in (("q", dq), ("k", dk), ("v", dv)):
            base = {"q": q, "k": k, "v": v}
            for idx in np.ndindex(base[name].shape):
                xp, xm = base[name].copy(), base[name].copy()
                xp[idx] += eps
                xm[idx] -= eps
                ap, am = dict(base), dict(base)
                ap[name], am[name] = xp, xm
                fd = (_fd_loss(mk, ap["q"], ap["k"], ap["v"], g, causal, 0.6, **kw)
                      - _fd_loss(mk, am["q"], am["k"], am["v"], g, causal, 0.6, **kw)) / (2 * eps)
                assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx], causal)


def check_bwd_empty_row_has_zero_dq(mk):
    """A query row whose key range is empty gets dQ = 0 and leaves dK, dV as if it were absent."""
    q, k, v = _qkv(1, 2, 1, 4, 6, 3, "bwd-empty")
    g = _rng("bwd-empty-g").normal(size=q.shape)
    kr = np.array([[[0, 6], [2, 2], [1, 4], [0, 6]]])
    dq, dk, dv = mk.attention_bwd_masked(q, k, v, g, False, 0.9, kv_ranges=kr)
    if not np.all(dq[:, :, 1] == 0.0):
        raise AssertionError("empty row has a non-zero dQ")
    g0 = g.copy()
    g0[:, :, 1] = 0.0
    _, dk0, dv0 = mk.attention_bwd_masked(q, k, v, g0, False, 0.9, kv_ranges=kr)
    _close(dk, dk0, "empty row dK")
    _close(dv, dv0, "empty row dV")


CHECKS = [check_unbounded_window_is_plain, check_band_rows_are_decode_over_slice, check_identity_window,
          check_alibi_zero_slope_is_plain, check_alibi_identical_keys_closed_form,
          check_alibi_causal_is_plain_with_extra_dimension, check_alibi_window_two_sided_by_merge,
          check_decode_is_last_prefill_row, check_decode_alibi_extra_dimension,
          check_paged_is_decode_over_gathered_rows, check_varlen_equal_lengths_is_dense_batch,
          check_range_rows_are_decode_over_slice, check_full_ranges_are_plain, check_block_diagonal_ranges_are_varlen,
          check_varlen_ranges_count_from_sequence_start, check_bwd_without_options_is_plain_bwd,
          check_bwd_matches_finite_differences, check_bwd_empty_row_has_zero_dq]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_masked_oracle_pin(check):
    check(M)


# Planted mistakes in oracle/masked.py: (anchor, replacement), every occurrence replaced.
MUTANTS = {
    "left window off by one": ("keep &= j >= i - window_left", "keep &= j > i - window_left"),
    "right window off by one": ("keep &= j <= i + window_right", "keep &= j < i + window_right"),
    "window sides swapped": ("keep &= j >= i - window_left", "keep &= j >= i - window_right"),
    "causal ignored": ("    if causal:\n        keep &= j <= i", "    if causal:\n        keep &= j <= i + Nkv"),
    "ALiBi sign flipped": ("s = s - slopes[h] * dist", "s = s + slopes[h] * dist"),
    "ALiBi inside the scale": ("s = s - slopes[h] * dist", "s = s - scale * slopes[h] * dist"),
    "ALiBi signed distance": ("dist = np.abs(np.arange(Nq)[:, None] - np.arange(Nkv)[None, :])",
                              "dist = (np.arange(Nq)[:, None] - np.arange(Nkv)[None, :])"),
    "ALiBi slope of the kv head": ("slopes[h] * dist", "slopes[hk] * dist"),
    "decode query position n": ("pos = n - 1", "pos = n"),
    "decode window off by one": ("t >= pos - window_left", "t > pos - window_left"),
    "empty rows uniform": ("rows = np.isfinite(s).any(axis=1)", "rows = np.ones(n, dtype=bool)"),
    "paged row index": ("rows = [(int(block_table[b][t // page_size]), t % page_size)",
                        "rows = [(int(block_table[b][t // page_size]), (t + 1) % page_size)"),
    "range lower bound off by one": ("keep &= (j >= kr[:, 0:1]) & (j < kr[:, 1:2])",
                                     "keep &= (j > kr[:, 0:1]) & (j < kr[:, 1:2])"),
    "range upper bound inclusive": ("keep &= (j >= kr[:, 0:1]) & (j < kr[:, 1:2])",
                                    "keep &= (j >= kr[:, 0:1]) & (j <= kr[:, 1:2])"),
    "ranges of batch 0 for every batch": ("None if kv_ranges is None else np.asarray(kv_ranges)[b]",
                                          "None if kv_ranges is None else np.asarray(kv_ranges)[0]"),
    "varlen ranges of the wrong rows": ("np.asarray(kv_ranges)[qs:qe][None]", "np.asarray(kv_ranges)[:qe - qs][None]"),
    "bwd rowsum term dropped": ("dscore = prob * (dprob - (gb * out).sum(axis=1, keepdims=True))",
                                "dscore = prob * dprob"),
    "bwd dK without the scale": ("dk[b, hk] += scale * (dscore.T @ qb)", "dk[b, hk] += dscore.T @ qb"),
    "bwd dV of the unnormalised P": ("prob[live] = ex / ex.sum(axis=1, keepdims=True)", "prob[live] = ex"),
    "bwd bias ignored": ("                scores = scores - slopes[h] * dist", "                scores = scores"),
    "bwd mask ignored": ("scores = np.where(keeps[b], scores, -np.inf)", "scores = scores"),
    "bwd dK of the first head only": ("dk[b, hk] += scale", "dk[b, hk] = scale"),
    "varlen keys of the next sequence": ("kb = k[ks:ke]", "kb = k[ke:ke + (ke - ks)] if ke + (ke - ks) <= len(k) "
                                                          "else k[ks:ke][::-1]"),
}


def _mutant(old, new):
    with open(M.__file__) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("masked_mutant")
    exec(compile(src.replace(old, new), "masked_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_masked_planted_mistakes_are_caught(name):
    mk = _mutant(*MUTANTS[name])
    caught = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mk)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"mutant '{name}' passed every pin"
