"""Pins for the CPU fp64 oracle, checked against facts that do not come from it.

Each check below is a function of an oracle object so the same checks can be
run against deliberately broken copies of the oracle (``test_planted_mistakes``)
to show that a plausible slip in the oracle would be caught.

Sources of the pinned facts:
* hand-derived worked examples in ``tests/golden`` (each cites the passage);
* closed forms of softmax attention (zero query, identical keys, all-ones V,
  causal row 0, a dominant key);
* invariances of the definition (GQA head mapping equals MHA with K/V
  expanded by repeat_interleave -- "Triton-FlashAttention", GQA phase;
  permutation of KV positions; shift of all scores of a row; scale folding;
  split-KV log-sum-exp merge);
* autoregressive equivalence of decode and causal prefill
  ("Triton-FlashAttention", Phase 2);
* an independent second formulation (scipy's logsumexp) on small inputs.
"""
from __future__ import annotations

import glob
import json
import math
import os
import shutil
import subprocess
import tempfile
import zlib

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NON_ALIGNED = (1, 31, 33, 63, 65, 127, 257)


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle(oracle.build())


def _rng(*key):
    return np.random.default_rng(zlib.crc32(repr(key).encode()))


def _counts(Nq, Nkv, causal):
    """|A_i|: keys row i may attend to (top-left causal: j <= i)."""
    i = np.arange(Nq)
    return np.minimum(i + 1, Nkv) if causal else np.full(Nq, Nkv)


def _prefix_mean(v, Nq, causal):
    """Mean of V over each row's allowed keys. v: (B,H,Nkv,D) -> (B,H,Nq,D)."""
    Nkv = v.shape[2]
    if not causal:
        return np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape[:2] + (Nq, v.shape[3]))
    cs = np.cumsum(v, axis=2)
    n = _counts(Nq, Nkv, True)
    return cs[:, :, n - 1, :] / n[None, None, :, None]


def _expand(x, group):
    """torch.repeat_interleave(x, group, dim=1) in numpy."""
    return np.repeat(x, group, axis=1)


# ----------------------------------------------------------------------------- checks

def check_golden(orc):
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    assert files, "no golden fixtures found"
    for path in files:
        with open(path) as f:
            g = json.load(f)
        if "shape" not in g:  # paged-layout fixtures are checked by test_paged_golden
            continue
        s = g["shape"]
        q = np.array(g["q"], dtype=np.float64).reshape(s["B"], s["Hq"], s["Nq"], s["D"])
        k = np.array(g["k"], dtype=np.float64).reshape(s["B"], s["Hkv"], s["Nkv"], s["D"])
        v = np.array(g["v"], dtype=np.float64).reshape(s["B"], s["Hkv"], s["Nkv"], s["D"])
        for mode, exp in g["expected"].items():
            o, lse = orc.attention(q, k, v, causal=(mode == "causal"), scale=g["scale"])
            np.testing.assert_allclose(o.ravel(), exp["o"], rtol=0, atol=1e-12, err_msg=path)
            np.testing.assert_allclose(lse.ravel(), exp["lse"], rtol=0, atol=1e-12, err_msg=path)
    # causal_prefix_mean: N_q=2 < N_kv=3, top-left alignment keeps the first two causal rows
    with open(os.path.join(GOLDEN, "causal_prefix_mean_d1.json")) as f:
        g = json.load(f)
    q = np.array(g["q"][:2]).reshape(1, 1, 2, 1)
    k = np.array(g["k"]).reshape(1, 1, 3, 1)
    v = np.array(g["v"]).reshape(1, 1, 3, 1)
    o, lse = orc.attention(q, k, v, causal=True, scale=g["scale"])
    np.testing.assert_allclose(o.ravel(), g["expected"]["causal"]["o"][:2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.ravel(), g["expected"]["causal"]["lse"][:2], rtol=0, atol=1e-12)


def check_zero_query(orc):
    """Q = 0: every allowed score is 0, so O = mean of allowed V and LSE = ln|A_i|."""
    shapes = [(n, n) for n in NON_ALIGNED] + [(5, 9), (9, 5)]
    for Nq, Nkv in shapes:
        for causal in (False, True):
            B, Hq, Hkv, D = 2, 4, 2, 8
            r = _rng("zq", Nq, Nkv, causal)
            q = np.zeros((B, Hq, Nq, D))
            k = r.normal(size=(B, Hkv, Nkv, D))
            v = r.normal(size=(B, Hkv, Nkv, D))
            o, lse = orc.attention(q, k, v, causal, scale=0.37)
            ve = _expand(v, Hq // Hkv)
            np.testing.assert_allclose(o, _prefix_mean(ve, Nq, causal), rtol=0, atol=1e-12)
            want = np.log(_counts(Nq, Nkv, causal)).astype(np.float64)
            np.testing.assert_allclose(lse, np.broadcast_to(want, lse.shape), rtol=0, atol=1e-12)


def check_identical_keys(orc):
    """All keys of a head equal: O = mean of allowed V, LSE = scale*q.k + ln|A_i|."""
    for n in (1, 33, 65):
        for causal in (False, True):
            B, Hq, Hkv, D = 1, 6, 3, 16
            r = _rng("ik", n, causal)
            q = r.normal(size=(B, Hq, n, D))
            kvec = r.normal(size=(B, Hkv, 1, D))
            k = np.repeat(kvec, n, axis=2)
            v = r.normal(size=(B, Hkv, n, D))
            scale = 0.25
            o, lse = orc.attention(q, k, v, causal, scale)
            g = Hq // Hkv
            np.testing.assert_allclose(o, _prefix_mean(_expand(v, g), n, causal), rtol=0, atol=1e-12)
            s = scale * np.einsum("bhnd,bhd->bhn", q, _expand(kvec, g)[:, :, 0, :])
            want = s + np.log(_counts(n, n, causal))[None, None, :]
            np.testing.assert_allclose(lse, want, rtol=0, atol=1e-12)


def check_rows_sum_to_one(orc):
    """V = 1 everywhere: the softmax weights of every row sum to one, so O = 1."""
    for causal in (False, True):
        r = _rng("ones", causal)
        B, Hq, Hkv, Nq, Nkv, D = 2, 4, 4, 33, 31, 8
        q = r.normal(size=(B, Hq, Nq, D)) * 3
        k = r.normal(size=(B, Hkv, Nkv, D))
        v = np.ones((B, Hkv, Nkv, D))
        o, _ = orc.attention(q, k, v, causal, scale=0.5)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


def check_causal_row0(orc):
    """Causal row 0 sees key 0 only: O = V[0] exactly, LSE = scale * q0.k0."""
    r = _rng("row0")
    B, Hq, Hkv, N, D = 2, 8, 2, 17, 32
    q, k, v = (r.normal(size=s) for s in ((B, Hq, N, D), (B, Hkv, N, D), (B, Hkv, N, D)))
    o, lse = orc.attention(q, k, v, True, scale=0.125)
    ke, ve = _expand(k, 4), _expand(v, 4)
    np.testing.assert_array_equal(o[:, :, 0, :], ve[:, :, 0, :])
    np.testing.assert_allclose(lse[:, :, 0], 0.125 * np.einsum("bhd,bhd->bh", q[:, :, 0], ke[:, :, 0]),
                               rtol=0, atol=1e-12)


def check_gqa_equals_mha(orc):
    """GQA/MQA equals MHA with K/V expanded by repeat_interleave over the head axis."""
    B, Hq, N, D = 2, 16, 33, 8
    for Hkv in (16, 8, 4, 2, 1):
        for causal in (False, True):
            r = _rng("gqa", Hkv, causal)
            q = r.normal(size=(B, Hq, N, D))
            k = r.normal(size=(B, Hkv, N, D))
            v = r.normal(size=(B, Hkv, N, D))
            o1, l1 = orc.attention(q, k, v, causal, 0.35)
            o2, l2 = orc.attention(q, _expand(k, Hq // Hkv), _expand(v, Hq // Hkv), causal, 0.35)
            np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
            np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def check_permutation(orc):
    """Non-causal attention does not depend on the order of the KV positions."""
    r = _rng("perm")
    B, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 7, 29, 16
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    p = r.permutation(Nkv)
    o1, l1 = orc.attention(q, k, v, False, 0.3)
    o2, l2 = orc.attention(q, k[:, :, p], v[:, :, p], False, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def check_shift_large(orc):
    """K + u shifts every score of a row by scale*q.u: O unchanged, LSE shifted.

    With |scale*q.u| near 700 an implementation without the max subtraction
    overflows or underflows exp and returns inf/nan.
    """
    r = _rng("shift")
    B, Hq, Hkv, N, D = 1, 2, 2, 33, 8
    q = r.normal(size=(B, Hq, N, D)) * 0.1 + 1.0
    k = r.normal(size=(B, Hkv, N, D))
    v = r.normal(size=(B, Hkv, N, D))
    for sign in (1.0, -1.0):
        for causal in (False, True):
            u = np.full((B, Hkv, 1, D), sign * 700.0 / D / 0.5)
            o1, l1 = orc.attention(q, k, v, causal, 0.5)
            o2, l2 = orc.attention(q, k + u, v, causal, 0.5)
            assert np.isfinite(o2).all() and np.isfinite(l2).all()
            shift = 0.5 * np.einsum("bhnd,bhd->bhn", q, u[:, :, 0, :])
            np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-9)
            np.testing.assert_allclose(l2, l1 + shift, rtol=1e-12, atol=1e-9)


def check_split_merge(orc):
    """Attention over KV[:c] and KV[c:] merged by their LSE equals attention over all of KV.

    lse = ln(e^lse1 + e^lse2); O = e^(lse1-lse) O1 + e^(lse2-lse) O2.  This pins
    the LSE definition (m + ln l, natural log) as well as the normalisation.
    """
    r = _rng("split")
    B, Hq, Hkv, Nq, Nkv, D = 2, 4, 1, 3, 65, 16
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    o, lse = orc.attention(q, k, v, False, 0.4)
    for c in (1, 31, 64):
        o1, l1 = orc.attention(q, k[:, :, :c], v[:, :, :c], False, 0.4)
        o2, l2 = orc.attention(q, k[:, :, c:], v[:, :, c:], False, 0.4)
        lm = np.logaddexp(l1, l2)
        om = np.exp(l1 - lm)[..., None] * o1 + np.exp(l2 - lm)[..., None] * o2
        np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)
        np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)


def check_autoregressive(orc):
    """Decode of token t over a cache of t+1 positions equals causal prefill row t."""
    r = _rng("ar")
    B, Hq, Hkv, N, D = 2, 8, 2, 33, 16
    q, k, v = r.normal(size=(B, Hq, N, D)), r.normal(size=(B, Hkv, N, D)), r.normal(size=(B, Hkv, N, D))
    o, lse = orc.attention(q, k, v, True, 0.25)
    kc = np.zeros((B, Hkv, N + 7, D))
    vc = np.zeros((B, Hkv, N + 7, D))
    for t in range(N):
        kc, vc = oracle.kv_cache_write(kc, vc, k[:, :, t:t + 1], v[:, :, t:t + 1], t)
        od, ld = orc.decode(q[:, :, t], kc, vc, t + 1, 0.25)
        np.testing.assert_allclose(od, o[:, :, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(ld, lse[:, :, t], rtol=0, atol=1e-12)


def check_causal_prefix(orc):
    """Causal row i equals non-causal attention over keys 0..i and ignores later keys."""
    r = _rng("prefix")
    B, Hq, Hkv, N, D = 1, 2, 1, 20, 8
    q, k, v = r.normal(size=(B, Hq, N, D)), r.normal(size=(B, Hkv, N, D)), r.normal(size=(B, Hkv, N, D))
    o, lse = orc.attention(q, k, v, True, 0.6)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 11:] += 5.0
    v2[:, :, 11:] -= 3.0
    o2, lse2 = orc.attention(q, k2, v2, True, 0.6)
    np.testing.assert_array_equal(o2[:, :, :11], o[:, :, :11])
    for i in (0, 5, 10, 19):
        oi, li = orc.attention(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], False, 0.6)
        np.testing.assert_allclose(oi[:, :, 0], o[:, :, i], rtol=0, atol=1e-12)
        np.testing.assert_allclose(li[:, :, 0], lse[:, :, i], rtol=0, atol=1e-12)


def check_scale_folding(orc):
    """Scaling Q by c and the softmax scale by 1/c leaves the result unchanged."""
    r = _rng("scale")
    B, Hq, Hkv, N, D = 1, 2, 2, 9, 8
    q, k, v = r.normal(size=(B, Hq, N, D)), r.normal(size=(B, Hkv, N, D)), r.normal(size=(B, Hkv, N, D))
    for causal in (False, True):
        o1, l1 = orc.attention(q, k, v, causal, 0.125)
        o2, l2 = orc.attention(q * 4.0, k, v, causal, 0.125 / 4.0)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def check_dominant_key(orc):
    """A key whose score exceeds every other by 60 takes all the weight: O = its V row."""
    B, Hq, Hkv, N, D = 1, 1, 1, 12, 4
    r = _rng("dom")
    k = r.normal(size=(B, Hkv, N, D)) * 0.1
    v = r.normal(size=(B, Hkv, N, D))
    k[0, 0, 7] = np.array([10.0, 0, 0, 0])
    q = np.zeros((B, Hq, 1, D))
    q[0, 0, 0, 0] = 6.0
    o, lse = orc.attention(q, k, v, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 7], rtol=0, atol=1e-20 + 12 * math.exp(-55) * 10)
    np.testing.assert_allclose(lse[0, 0, 0], 60.0, rtol=0, atol=1e-20 + 12 * math.exp(-55))


def check_second_formulation(orc):
    """Agreement with an independent formulation built on scipy's logsumexp."""
    from scipy.special import logsumexp
    for (B, Hq, Hkv, Nq, Nkv, D, causal) in [(1, 2, 2, 3, 3, 4, False), (1, 2, 1, 3, 3, 4, True),
                                             (2, 4, 2, 5, 7, 3, True), (1, 3, 1, 6, 2, 5, False)]:
        r = _rng("2nd", B, Hq, Hkv, Nq, Nkv, D, causal)
        q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
        o, lse = orc.attention(q, k, v, causal, 0.7)
        g = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                for i in range(Nq):
                    sc = np.array([0.7 * sum(q[b, h, i, d] * k[b, h // g, j, d] for d in range(D))
                                   if (not causal or j <= i) else -np.inf for j in range(Nkv)])
                    L = logsumexp(sc)
                    w = np.exp(sc - L)
                    assert abs(lse[b, h, i] - L) < 1e-12
                    np.testing.assert_allclose(o[b, h, i], w @ v[b, h // g], rtol=0, atol=1e-12)


def check_rows_api(orc):
    """attention_rows returns exactly the selected rows of the full result."""
    r = _rng("rows")
    B, Hq, Hkv, Nq, Nkv, D = 2, 4, 2, 19, 23, 8
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.3)
        rows = np.array([[0, 0, 0], [1, 3, 18], [0, 2, 7], [1, 1, 1]])
        orow, lrow = orc.attention_rows(q, k, v, causal, 0.3, rows)
        np.testing.assert_array_equal(orow, o[rows[:, 0], rows[:, 1], rows[:, 2]])
        np.testing.assert_array_equal(lrow, lse[rows[:, 0], rows[:, 1], rows[:, 2]])


CHECKS = [check_golden, check_zero_query, check_identical_keys, check_rows_sum_to_one, check_causal_row0,
          check_gqa_equals_mha, check_permutation, check_shift_large, check_split_merge, check_autoregressive,
          check_causal_prefix, check_scale_folding, check_dominant_key, check_second_formulation, check_rows_api]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    check(orc)


def test_invalid_shapes_rejected(orc):
    q = np.zeros((1, 3, 2, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        orc.attention(q, k, k, False, 1.0)  # H_q not a multiple of H_kv


def test_kv_cache_write_places_tokens():
    r = _rng("kvw")
    kc, vc = r.normal(size=(2, 3, 10, 4)), r.normal(size=(2, 3, 10, 4))
    kn, vn = r.normal(size=(2, 3, 2, 4)), r.normal(size=(2, 3, 2, 4))
    k2, v2 = oracle.kv_cache_write(kc, vc, kn, vn, 5)
    np.testing.assert_array_equal(k2[:, :, 5:7], kn)
    np.testing.assert_array_equal(v2[:, :, 5:7], vn)
    np.testing.assert_array_equal(np.delete(k2, [5, 6], axis=2), np.delete(kc, [5, 6], axis=2))
    np.testing.assert_array_equal(np.delete(v2, [5, 6], axis=2), np.delete(vc, [5, 6], axis=2))
    with pytest.raises(ValueError):
        oracle.kv_cache_write(kc, vc, kn, vn, 9)


# Plausible slips in the oracle; each must make at least one check above fail.
MUTANTS = {
    "kv head h % H_kv": ("const int64_t hk = h / group;", "const int64_t hk = h % J->Hkv;"),
    "causal mask j >= i": ("if (J->causal && j > i)", "if (J->causal && j >= i)"),
    "causal mask reversed": ("if (J->causal && j > i)", "if (J->causal && j < i)"),
    "mask to 0 not -inf": ("if (J->causal && j > i) sj = -INFINITY;", "if (J->causal && j > i) sj = 0.0;"),
    "lse = m only": ("*lse_out = m + log(l);", "*lse_out = m;"),
    "lse in log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "no max subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "exp sign flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "no normalisation": ("const double w = s[j] / l;", "const double w = s[j];"),
    "no scale": ("double sj = J->scale * dot;", "double sj = dot;"),
    "K used for V": ("o_row[d] += w * vh[j * D + d];", "o_row[d] += w * kh[j * D + d];"),
    "reversed d of K": ("dot += qrow[d] * kh[j * D + d];", "dot += qrow[d] * kh[j * D + (D - 1 - d)];"),
    "off-by-one key": ("dot += qrow[d] * kh[j * D + d];", "dot += qrow[d] * kh[((j + 1) % Nkv) * D + d];"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.compile_source(path, os.path.join(td, "libmutant.so"))
        mutant = oracle.Oracle(lib)
        caught = []
        for check in CHECKS:
            try:
                with np.errstate(all="ignore"):
                    check(mutant)
            except AssertionError:
                caught.append(check.__name__)
        assert caught, f"mutant '{name}' passed every pin"


# ----------------------------------------------------------------------------- paged layout

def test_paged_golden():
    with open(os.path.join(GOLDEN, "paged_gather_d1.json")) as f:
        g = json.load(f)
    o, lse = oracle.decode_paged(np.array(g["q"]), np.array(g["k_pages"]), np.array(g["v_pages"]),
                                 np.array(g["block_table"]), np.array(g["cache_lens"]), g["scale"])
    np.testing.assert_allclose(o, np.array(g["expected"]["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["expected"]["lse"]), rtol=0, atol=1e-12)


def _paged_from_contiguous(kc, page_size, perm):
    """Split a contiguous cache (B, H, L, D) into a page pool whose page ids are shuffled by perm."""
    B, H, L, D = kc.shape
    npb = L // page_size
    pool = np.empty((B * npb, H, page_size, D))
    table = np.empty((B, npb), dtype=np.int64)
    for b in range(B):
        for i in range(npb):
            pid = perm[b * npb + i]
            pool[pid] = kc[b, :, i * page_size:(i + 1) * page_size, :]
            table[b, i] = pid
    return pool, table


def test_paged_equals_contiguous_under_any_page_order():
    r = _rng("paged")
    B, Hq, Hkv, L, D, ps = 3, 8, 2, 48, 16, 16
    q = r.normal(size=(B, Hq, D))
    kc, vc = r.normal(size=(B, Hkv, L, D)), r.normal(size=(B, Hkv, L, D))
    lens = np.array([48, 17, 1])
    for perm in (np.arange(B * (L // ps)), r.permutation(B * (L // ps))):
        kp, table = _paged_from_contiguous(kc, ps, perm)
        vp, _ = _paged_from_contiguous(vc, ps, perm)
        o, lse = oracle.decode_paged(q, kp, vp, table, lens, 0.25)
        for b in range(B):
            ob, lb = oracle.decode(q[b:b + 1], kc[b:b + 1], vc[b:b + 1], int(lens[b]), 0.25)
            np.testing.assert_array_equal(o[b], ob[0])
            np.testing.assert_array_equal(lse[b], lb[0])


def test_paged_length_zero_convention():
    q = np.ones((1, 2, 4))
    pool = np.ones((1, 1, 16, 4))
    o, lse = oracle.decode_paged(q, pool, pool, np.zeros((1, 1), dtype=np.int64), np.array([0]), 1.0)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_paged_write_then_gather_roundtrip():
    r = _rng("pwrite")
    B, H, D, ps, npages = 2, 2, 8, 16, 6
    kp, vp = np.zeros((npages, H, ps, D)), np.zeros((npages, H, ps, D))
    table = np.array([[4, 1, 5], [0, 3, 2]])
    pos = np.array([14, 0])
    kn, vn = r.normal(size=(B, H, 5, D)), r.normal(size=(B, H, 5, D))
    kp2, vp2 = oracle.kv_cache_write_paged(kp, vp, kn, vn, table, pos)
    for b in range(B):
        got = oracle.gather_pages(kp2, table[b], pos[b] + 5)[:, pos[b]:, :]
        np.testing.assert_array_equal(got, kn[b])
        got = oracle.gather_pages(vp2, table[b], pos[b] + 5)[:, pos[b]:, :]
        np.testing.assert_array_equal(got, vn[b])
    # request 0 wrote rows 14, 15 of page 4 and rows 0..2 of page 1; nothing else changed
    touched = np.zeros((npages, ps), dtype=bool)
    touched[4, 14:] = True
    touched[1, :3] = True
    touched[0, :5] = True
    assert (kp2[~touched[:, None, :, None].repeat(H, 1).repeat(D, 3)] == 0).all()


# ----------------------------------------------------------------------------- variable length

def test_varlen_golden_is_the_concatenation_of_fixtures():
    """Two hand-derived fixtures packed back to back give their own expected values."""
    with open(os.path.join(GOLDEN, "two_keys_d1.json")) as f:
        g1 = json.load(f)
    with open(os.path.join(GOLDEN, "causal_prefix_mean_d1.json")) as f:
        g2 = json.load(f)
    assert g1["scale"] == 1.0
    # rescale fixture 2's queries so both use scale 1 (scores are the same: its keys are all 0)
    q = np.array(g1["q"] + g2["q"]).reshape(-1, 1, 1)
    k = np.array(g1["k"] + g2["k"]).reshape(-1, 1, 1)
    v = np.array(g1["v"] + g2["v"]).reshape(-1, 1, 1)
    cu = np.array([0, 2, 5])
    for mode in ("noncausal", "causal"):
        o, lse = oracle.prefill_varlen(q, k, v, cu, cu, mode == "causal", 1.0)
        want_o = g1["expected"][mode]["o"] + g2["expected"][mode]["o"]
        want_l = g1["expected"][mode]["lse"] + g2["expected"][mode]["lse"]
        np.testing.assert_allclose(o.ravel(), want_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.ravel(), want_l, rtol=0, atol=1e-12)


def test_varlen_equal_lengths_equal_dense_batch():
    r = _rng("varlen")
    B, Hq, Hkv, N, D = 3, 4, 2, 21, 8
    q, k, v = r.normal(size=(B, Hq, N, D)), r.normal(size=(B, Hkv, N, D)), r.normal(size=(B, Hkv, N, D))
    cu = np.arange(B + 1) * N
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * N, x.shape[1], D)
    for causal in (False, True):
        o, lse = oracle.prefill_varlen(pack(q), pack(k), pack(v), cu, cu, causal, 0.3)
        od, ld = oracle.attention(q, k, v, causal, 0.3)
        np.testing.assert_array_equal(o, pack(od))
        np.testing.assert_array_equal(lse, ld.transpose(1, 0, 2).reshape(Hq, B * N))


def test_varlen_sequences_do_not_interact():
    """Changing one sequence's keys and values leaves the other sequences' results unchanged."""
    r = _rng("varlen2")
    H, D = 2, 8
    cu_q, cu_k = np.array([0, 5, 12, 13]), np.array([0, 9, 10, 30])
    q, k, v = r.normal(size=(13, H, D)), r.normal(size=(30, H, D)), r.normal(size=(30, H, D))
    o1, l1 = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[9:10] += 3.0
    v2[9:10] -= 7.0
    o2, l2 = oracle.prefill_varlen(q, k2, v2, cu_q, cu_k, True, 0.5)
    np.testing.assert_array_equal(o1[:5], o2[:5])
    np.testing.assert_array_equal(o1[12:], o2[12:])
    assert not np.allclose(o1[5:12], o2[5:12])


# ----------------------------------------------------------------------------- backward

def _loss(q, k, v, g, causal, scale):
    """L = sum(O * G), O from the forward oracle."""
    o, _ = oracle.attention(q, k, v, causal, scale)
    return float(np.sum(o * g))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_central_finite_differences(causal):
    """Every gradient entry of a small GQA case against (L(x+e) - L(x-e)) / 2e through the forward oracle."""
    r = _rng("fd", causal)
    B, Hq, Hkv, Nq, Nkv, D, scale = 1, 4, 2, 5, 7, 3, 0.7
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    g = r.normal(size=(B, Hq, Nq, D))
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, causal, scale)
    eps = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (_loss(args_p["q"], args_p["k"], args_p["v"], g, causal, scale)
                  - _loss(args_m["q"], args_m["k"], args_m["v"], g, causal, scale)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_bwd_gqa_equals_group_sum_of_mha():
    """GQA dK, dV equal the MHA gradients of repeat_interleave-expanded K, V summed over each group."""
    r = _rng("bwdgqa")
    B, Hq, Hkv, N, D = 2, 8, 2, 9, 4
    q, k, v = r.normal(size=(B, Hq, N, D)), r.normal(size=(B, Hkv, N, D)), r.normal(size=(B, Hkv, N, D))
    g = r.normal(size=(B, Hq, N, D))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, g, causal, 0.5)
        dq2, dk2, dv2 = oracle.attention_bwd(q, _expand(k, 4), _expand(v, 4), g, causal, 0.5)
        np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, 4, N, D).sum(axis=2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, 4, N, D).sum(axis=2), rtol=0, atol=1e-12)


def test_bwd_rows_of_ds_sum_to_zero():
    """Adding the same vector to every key leaves the weights unchanged, so dL/du = sum_j dK_j = 0."""
    r = _rng("dssum")
    q, k, v = r.normal(size=(1, 2, 6, 4)), r.normal(size=(1, 2, 6, 4)), r.normal(size=(1, 2, 6, 4))
    g = r.normal(size=(1, 2, 6, 4))
    for causal in (False, True):
        _, dk, _ = oracle.attention_bwd(q, k, v, g, causal, 0.9)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_sampled_rows_equal_full_backward(causal):
    """The sampled-row gradients equal the pinned full backward on every row and key (GQA, unequal lengths,
    blocks of query rows smaller than N_q)."""
    r = _rng("bwdrows", causal)
    B, Hq, Hkv, Nq, Nkv, D, scale = 2, 6, 2, 11, 13, 5, 0.6
    q, k, v = r.normal(size=(B, Hq, Nq, D)), r.normal(size=(B, Hkv, Nkv, D)), r.normal(size=(B, Hkv, Nkv, D))
    g = r.normal(size=(B, Hq, Nq, D))
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, causal, scale)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(oracle.attention_bwd_dq_rows(q, k, v, g, causal, scale, b, h, range(Nq)),
                                       dq[b, h], rtol=0, atol=1e-12)
        for hk in range(Hkv):
            keys = [12, 0, 5, 6]
            rk, rv = oracle.attention_bwd_dkv_rows(q, k, v, g, causal, scale, b, hk, keys, block=4)
            np.testing.assert_allclose(rk, dk[b, hk, keys], rtol=0, atol=1e-12)
            np.testing.assert_allclose(rv, dv[b, hk, keys], rtol=0, atol=1e-12)
