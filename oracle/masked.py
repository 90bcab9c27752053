"""Attention with sliding windows and ALiBi biases, numpy fp64 -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the CPU-baseline leg of the
benchmark may import this module; the CUDA library never calls it.  It shares
no code with the CUDA path.

What is computed.  "Skill: Write a Triton Attention Kernel" (When to use, and
Required reasoning process, question 3 on masking) names sliding-window
attention, custom masks and ALiBi biases as the variants a hand-written kernel
is for, and "Triton-FlashAttention" (Deferred / explicitly out of scope) lists
sliding windows and attention biases such as ALiBi without defining them.  The
pages fix no formula, so this module takes the plainest readings, which are
the ones in common use:

* Query row i of a prefill sits at position i and key j at position j (the same
  top-left alignment as the causal mask j <= i of the plain oracle).
* Sliding window (window_left, window_right), -1 meaning unbounded on that
  side: key j is visible to row i iff i - window_left <= j <= i + window_right.
  With ``causal`` the right bound is j <= i as well.
* ALiBi: one slope per query head h; the score becomes
  scale * q_i . k_j - slope_h * |i - j|, in natural-log units (the bias is added
  after the scale).
* Decode: the single query sits at position cache_len - 1, so key t is visible
  iff t >= cache_len - 1 - window_left, and its bias is
  -slope_h * (cache_len - 1 - t).
* Custom masks as per-query-row key ranges (a reading of the pages' "custom
  masks", in the general form that covers block-diagonal, document and
  prefix masks): row i of batch b sees only keys j with
  kv_ranges[b][i][0] <= j < kv_ranges[b][i][1], in addition to the other
  bounds; for packed variable-length batches the ranges are per packed row and
  count keys from the start of the row's own sequence.
* A row with no visible key gets O = 0 and LSE = -inf (the convention of the
  plain oracle for empty sequences).

Every function forms the full score matrix of one (batch, head) explicitly,
masks it with -inf, and applies softmax in the order of the plain oracle:
m = row max, p = exp(s - m), l = sum p, O = p V / l, LSE = m + ln l.

Parity status: pinned by ``tests/test_oracle_masked.py`` against the C oracle
on band slices, the identity window, closed forms for identical keys, an
ALiBi-as-extra-dimension construction, and planted-mistake checks; the
backward (``attention_bwd_masked``) against the plain backward oracle without
options and against central finite differences through ``attention_masked``
with windows, ALiBi and key ranges.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def visible(Nq: int, Nkv: int, causal: bool, window_left: int = -1, window_right: int = -1,
            kv_range=None) -> np.ndarray:
    """Boolean (Nq, Nkv): key j visible to query row i (kv_range: optional (Nq, 2) [lo, hi) per row)."""
    i = np.arange(Nq)[:, None]
    j = np.arange(Nkv)[None, :]
    keep = np.ones((Nq, Nkv), dtype=bool)
    if kv_range is not None:
        kr = np.asarray(kv_range, dtype=np.int64).reshape(Nq, 2)
        keep &= (j >= kr[:, 0:1]) & (j < kr[:, 1:2])
    if causal:
        keep &= j <= i
    if window_left >= 0:
        keep &= j >= i - window_left
    if window_right >= 0:
        keep &= j <= i + window_right
    return keep


def _softmax_rows(s: np.ndarray, v: np.ndarray):
    """(O, LSE) of score rows s (-inf where masked) against values v; empty rows give 0, -inf."""
    n = s.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    rows = np.isfinite(s).any(axis=1)
    if rows.any():
        sr = s[rows]
        m = sr.max(axis=1, keepdims=True)
        p = np.exp(sr - m)
        l = p.sum(axis=1, keepdims=True)
        o[rows] = (p @ v) / l
        lse[rows] = (m + np.log(l))[:, 0]
    return o, lse


def attention_bwd_masked(q, k, v, dout, causal: bool, scale: float, window_left: int = -1, window_right: int = -1,
                         alibi_slopes=None, kv_ranges=None):
    """(dQ, dK, dV) of attention_masked for the incoming gradient dout, in fp64.

    With P the masked softmax of S = scale Q K^T - slope_h |i - j| (-inf where
    masked) and O = P V:  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
    dQ = scale dS K,  dK = scale dS^T Q.  The bias and the mask do not depend on
    Q or K, so they enter the gradients only through P; a row with no visible
    key has P = 0 and contributes nothing.  GQA heads of a group add into their
    kv head's dK, dV.  q, dout (B,H_q,N_q,D); k, v (B,H_kv,N_kv,D).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    group = Hq // Hkv
    keeps = [visible(Nq, Nkv, causal, window_left, window_right,
                     None if kv_ranges is None else np.asarray(kv_ranges)[b]) for b in range(B)]
    dist = np.abs(np.arange(Nq)[:, None] - np.arange(Nkv)[None, :]).astype(np.float64)
    slopes = None if alibi_slopes is None else np.asarray(alibi_slopes, dtype=np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            qb, kb, vb, gb = q[b, h], k[b, hk], v[b, hk], dout[b, h]
            scores = scale * (qb @ kb.T)
            if slopes is not None:
                scores = scores - slopes[h] * dist
            scores = np.where(keeps[b], scores, -np.inf)
            prob = np.zeros((Nq, Nkv))
            live = np.isfinite(scores).any(axis=1)
            if live.any():
                sl = scores[live]
                ex = np.exp(sl - sl.max(axis=1, keepdims=True))
                prob[live] = ex / ex.sum(axis=1, keepdims=True)
            out = prob @ vb
            dv[b, hk] += prob.T @ gb
            dprob = gb @ vb.T
            dscore = prob * (dprob - (gb * out).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (dscore @ kb)
            dk[b, hk] += scale * (dscore.T @ qb)
    return dq, dk, dv


def attention_masked(q, k, v, causal: bool, scale: float, window_left: int = -1, window_right: int = -1,
                     alibi_slopes=None, kv_ranges=None):
    """O (B,H_q,N_q,D) and LSE (B,H_q,N_q) of windowed / ALiBi / key-range attention; K, V are (B,H_kv,N_kv,D).

    kv_ranges: optional (B, N_q, 2) int array, [lo, hi) of the keys each query row may see.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    group = Hq // Hkv
    keeps = [visible(Nq, Nkv, causal, window_left, window_right,
                     None if kv_ranges is None else np.asarray(kv_ranges)[b]) for b in range(B)]
    dist = np.abs(np.arange(Nq)[:, None] - np.arange(Nkv)[None, :]).astype(np.float64)
    slopes = None if alibi_slopes is None else np.asarray(alibi_slopes, dtype=np.float64)
    o = np.zeros((B, Hq, Nq, D))
    lse = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            s = scale * (q[b, h] @ k[b, hk].T)
            if slopes is not None:
                s = s - slopes[h] * dist
            s = np.where(keeps[b], s, -np.inf)
            o[b, h], lse[b, h] = _softmax_rows(s, v[b, hk])
    return o, lse


def decode_masked(q, k_cache, v_cache, cache_len: int, scale: float, window_left: int = -1, alibi_slopes=None):
    """One query per (b, h) at position cache_len - 1 over cache rows [0, cache_len).

    q: (B,H_q,D); caches (B,H_kv,L,D).  Returns O (B,H_q,D), LSE (B,H_q).
    """
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    group = Hq // Hkv
    n = int(cache_len)
    t = np.arange(n)
    pos = n - 1
    keep = np.ones(n, dtype=bool) if window_left < 0 else t >= pos - window_left
    dist = (pos - t).astype(np.float64)
    slopes = None if alibi_slopes is None else np.asarray(alibi_slopes, dtype=np.float64)
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    if n == 0:
        return o, lse
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            s = scale * (kc[b, hk, :n] @ q[b, h])
            if slopes is not None:
                s = s - slopes[h] * dist
            s = np.where(keep, s, -np.inf)
            ob, lb = _softmax_rows(s[None, :], vc[b, hk, :n])
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def decode_paged_masked(q, k_pages, v_pages, block_table, cache_lens, scale: float, window_left: int = -1,
                        alibi_slopes=None):
    """``decode_masked`` of each request over its rows gathered from the page pool.

    Row t of request b is row t % page_size of page block_table[b][t // page_size].
    """
    kp, vp = _f64(k_pages), _f64(v_pages)
    q = _f64(q)
    B = q.shape[0]
    page_size = kp.shape[2]
    o = np.zeros(q.shape)
    lse = np.full(q.shape[:2], -np.inf)
    for b in range(B):
        n = int(cache_lens[b])
        rows = [(int(block_table[b][t // page_size]), t % page_size) for t in range(n)]
        kb = np.stack([kp[pg, :, r, :] for pg, r in rows], axis=1) if n else np.zeros((kp.shape[1], 0, kp.shape[3]))
        vb = np.stack([vp[pg, :, r, :] for pg, r in rows], axis=1) if n else np.zeros((vp.shape[1], 0, vp.shape[3]))
        ob, lb = decode_masked(q[b:b + 1], kb[None], vb[None], n, scale, window_left, alibi_slopes)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def prefill_varlen_masked(q, k, v, cu_q, cu_k, causal: bool, scale: float, window_left: int = -1,
                          window_right: int = -1, alibi_slopes=None, kv_ranges=None):
    """``attention_masked`` of each packed sequence with positions counted from its own start.

    q: (total_q,H_q,D); k, v: (total_k,H_kv,D); kv_ranges: optional (total_q, 2), per packed row,
    keys counted from the row's sequence start.  Returns O (total_q,H_q,D), LSE (H_q,total_q).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    total_q, Hq, D = q.shape
    o = np.zeros((total_q, Hq, D))
    lse = np.full((Hq, total_q), -np.inf)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if qe == qs:
            continue
        qb = q[qs:qe].transpose(1, 0, 2)[None]
        kb = k[ks:ke].transpose(1, 0, 2)[None]
        vb = v[ks:ke].transpose(1, 0, 2)[None]
        kr = None if kv_ranges is None else np.asarray(kv_ranges)[qs:qe][None]
        ob, lb = attention_masked(qb, kb, vb, causal, scale, window_left, window_right, alibi_slopes, kr)
        o[qs:qe] = ob[0].transpose(1, 0, 2)
        lse[:, qs:qe] = lb[0]
    return o, lse
