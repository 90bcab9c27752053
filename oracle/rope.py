"""Attention with rotary position embeddings (RoPE), numpy fp64 -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the CPU-baseline leg of the
benchmark may import this module; the CUDA library never calls it.  It shares
no code with the CUDA path.

What is computed.  "Skill: Write a Triton Attention Kernel" (Use this when)
names RoPE-fused attention among the variants a hand-written kernel is for, and
"Triton-FlashAttention" (Deferred / explicitly out of scope) lists fused rotary
embeddings; neither page defines them.  This module takes the standard reading
of rotary position embeddings (rotary embeddings as introduced for the
RoFormer transformer):

* the D coordinates of a query or key row form D/2 pairs; pair c is rotated in
  its plane by the angle p * theta^(-2c/D), p the row's position and theta the
  base (10000 in common use):
      x_a' = x_a cos(angle) - x_b sin(angle),   x_b' = x_b cos(angle) + x_a sin(angle);
* pair c is (c, c + D/2) in the "rotate half" layout, or (2c, 2c + 1) in the
  interleaved layout;
* positions are those of the causal mask: query row i at i and key j at j
  (per sequence for packed variable-length batches); the decode query sits at
  cache_len - 1 (per request for the paged cache);
* queries and keys are rotated, values never; attention then proceeds on the
  rotated rows exactly as without RoPE (including windows and ALiBi);
* a KV cache holds rotated keys: a key written at cache position p is rotated
  at p when it is written, and decode rotates only the query.

Every function rotates explicitly in fp64 and then calls the plain C oracle
(``oracle.attention`` / ``oracle.decode``) or the windowed / ALiBi oracle
(``oracle.masked``), both pinned on their own.

Parity status: pinned by ``tests/test_oracle_rope.py`` against hand-derived
rotations (``tests/golden/rope_d4.json``), closed forms for D = 2, a matrix
formulation of the rotation, the relative-position property, norm
preservation, decode = last causal prefill row, and planted-mistake checks;
the backward (``attention_bwd``) against central finite differences through
``attention`` (both layouts, windows and ALiBi, keys given rotated) and the
plain backward at position 0.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import masked


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def inv_freq(D: int, theta: float) -> np.ndarray:
    """Angle per unit position of each of the D/2 pairs: theta^(-2c/D), c = 0 .. D/2 - 1."""
    c = np.arange(D // 2, dtype=np.float64)
    return float(theta) ** (-2.0 * c / D)


def pair_index(D: int, interleaved: bool):
    """(a, b): the two coordinates of each pair c."""
    c = np.arange(D // 2)
    if interleaved:
        a, b = 2 * c, 2 * c + 1
    else:
        a, b = c, c + D // 2
    return a, b


def rotate(x, positions, theta: float, interleaved: bool = False) -> np.ndarray:
    """x (..., N, D) with row n at position positions[n], each pair rotated by its angle."""
    x = _f64(x)
    D = x.shape[-1]
    pos = np.asarray(positions, dtype=np.float64).reshape(-1)
    if pos.shape[0] != x.shape[-2]:
        raise ValueError("one position per row")
    ang = pos[:, None] * inv_freq(D, theta)[None, :]          # (N, D/2)
    cs, sn = np.cos(ang), np.sin(ang)
    a, b = pair_index(D, interleaved)
    xa, xb = x[..., a], x[..., b]
    out = np.empty_like(x)
    out[..., a] = xa * cs - xb * sn
    out[..., b] = xb * cs + xa * sn
    return out


def _plain(window_left, window_right, alibi_slopes):
    return window_left < 0 and window_right < 0 and alibi_slopes is None


def attention(q, k, v, causal: bool, scale: float, theta: float, interleaved: bool = False,
              window_left: int = -1, window_right: int = -1, alibi_slopes=None):
    """O (B,H_q,N_q,D) and LSE (B,H_q,N_q): q row i rotated at i, k row j at j, then attention."""
    q, k = _f64(q), _f64(k)
    qr = rotate(q, np.arange(q.shape[2]), theta, interleaved)
    kr = rotate(k, np.arange(k.shape[2]), theta, interleaved)
    if _plain(window_left, window_right, alibi_slopes):
        return oracle.attention(qr, kr, v, causal, scale)
    return masked.attention_masked(qr, kr, v, causal, scale, window_left, window_right, alibi_slopes)


def attention_bwd(q, k, v, dout, causal: bool, scale: float, theta: float, interleaved: bool = False,
                  rotated_keys: bool = False, window_left: int = -1, window_right: int = -1, alibi_slopes=None,
                  kv_ranges=None):
    """(dQ, dK, dV) of ``attention`` (queries and keys rotated at their positions) for the incoming
    gradient dout, in fp64; kv_ranges: per-row key ranges as in ``masked.attention_masked``, applied to the
    rotated rows.

    With R the per-row rotation, the forward is attention(R q, R k, v); the gradients of attention with
    respect to its rotated inputs (dQ', dK', dV) come from the backward oracles, and by the chain rule
    dQ = R^T dQ', dK = R^T dK' -- R is orthogonal, so R^T is the rotation by the opposite angle -- while
    dV is unchanged.  rotated_keys: the keys were given already rotated (not rotated here), so dK is the
    gradient with respect to those rotated keys, dK'.
    """
    q, k = _f64(q), _f64(k)
    qpos, kpos = np.arange(q.shape[2]), np.arange(k.shape[2])
    qr = rotate(q, qpos, theta, interleaved)
    kr = k if rotated_keys else rotate(k, kpos, theta, interleaved)
    if _plain(window_left, window_right, alibi_slopes) and kv_ranges is None:
        dqr, dkr, dv = oracle.attention_bwd(qr, kr, v, dout, causal, scale)
    else:
        dqr, dkr, dv = masked.attention_bwd_masked(qr, kr, v, dout, causal, scale, window_left, window_right,
                                                   alibi_slopes, kv_ranges)
    dq = rotate(dqr, -qpos, theta, interleaved)
    dk = dkr if rotated_keys else rotate(dkr, -kpos, theta, interleaved)
    return dq, dk, dv


def kv_cache_write(k_cache, v_cache, k_new, v_new, pos: int, theta: float, interleaved: bool = False):
    """Copies of the caches with the new tokens (B,H_kv,n,D) at [pos, pos+n); each key rotated at its cache position."""
    k_new = _f64(k_new)
    kr = rotate(k_new, pos + np.arange(k_new.shape[2]), theta, interleaved)
    return oracle.kv_cache_write(_f64(k_cache), _f64(v_cache), kr, _f64(v_new), pos)


def decode(q, k_cache, v_cache, cache_len: int, scale: float, theta: float, interleaved: bool = False,
           window_left: int = -1, alibi_slopes=None):
    """One query per (b, h), rotated at cache_len - 1, over a cache of already rotated keys.

    q: (B,H_q,D); caches (B,H_kv,L,D).  Returns O (B,H_q,D), LSE (B,H_q).
    """
    q = _f64(q)
    qr = rotate(q[:, :, None, :], [cache_len - 1], theta, interleaved)[:, :, 0, :]
    if _plain(window_left, -1, alibi_slopes):
        return oracle.decode(qr, k_cache, v_cache, cache_len, scale)
    return masked.decode_masked(qr, k_cache, v_cache, cache_len, scale, window_left, alibi_slopes)


def kv_cache_write_paged(k_pages, v_pages, k_new, v_new, block_table, positions, theta: float,
                         interleaved: bool = False):
    """Paged cache write: token t of request b goes to position positions[b] + t, its key rotated there."""
    k_new = _f64(k_new)
    kr = np.empty_like(k_new)
    for b in range(k_new.shape[0]):
        kr[b] = rotate(k_new[b], int(positions[b]) + np.arange(k_new.shape[2]), theta, interleaved)
    return oracle.kv_cache_write_paged(_f64(k_pages), _f64(v_pages), kr, _f64(v_new), block_table, positions)


def decode_paged(q, k_pages, v_pages, block_table, cache_lens, scale: float, theta: float,
                 interleaved: bool = False, window_left: int = -1, alibi_slopes=None):
    """Request b's query rotated at cache_lens[b] - 1, then decode over its gathered (rotated) keys."""
    q = _f64(q)
    qr = np.empty_like(q)
    for b in range(q.shape[0]):
        qr[b] = rotate(q[b][:, None, :], [int(cache_lens[b]) - 1], theta, interleaved)[:, 0, :]
    return masked.decode_paged_masked(qr, k_pages, v_pages, block_table, cache_lens, scale, window_left,
                                      alibi_slopes)


def _packed_positions(cu, total):
    pos = np.zeros(total, dtype=np.int64)
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        pos[s:e] = np.arange(e - s)
    return pos


def prefill_varlen(q, k, v, cu_q, cu_k, causal: bool, scale: float, theta: float, interleaved: bool = False,
                   window_left: int = -1, window_right: int = -1, alibi_slopes=None):
    """Packed sequences: each row rotated at its position within its own sequence, then attention per sequence.

    q: (total_q,H_q,D); k, v: (total_k,H_kv,D).  Returns O (total_q,H_q,D), LSE (H_q,total_q).
    """
    q, k = _f64(q), _f64(k)
    pq = _packed_positions(cu_q, q.shape[0])
    pk = _packed_positions(cu_k, k.shape[0])
    qr = rotate(q.transpose(1, 0, 2), pq, theta, interleaved).transpose(1, 0, 2)
    kr = rotate(k.transpose(1, 0, 2), pk, theta, interleaved).transpose(1, 0, 2)
    return masked.prefill_varlen_masked(qr, kr, v, cu_q, cu_k, causal, scale, window_left, window_right,
                                        alibi_slopes)
