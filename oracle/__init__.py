"""CPU fp64 oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the CPU-baseline leg of the
benchmark may import this module.  The CUDA library never calls it and has no
fallback to it.  It shares no code with the CUDA path: the arithmetic lives in
``attn_oracle.c`` (plain C, fp64, one explicit score row per query), which this
wrapper compiles with gcc on first use and calls through ctypes.

Definitions followed (see the header of ``attn_oracle.c`` for the steps):

* ``attention``: "Skill: Write a Triton Attention Kernel", Required reasoning
  process steps 1-8 -- O = softmax(scale * Q K^T + causal mask) V with the KV
  head h // (H_q / H_kv), and LSE = m + ln(l) in natural log.
* ``decode``: "Triton-FlashAttention", Phase 2 -- one query token over a cache
  whose first ``cache_len`` positions are all valid (no causal mask).
* ``kv_cache_write``: "Triton-FlashAttention", Phase 2 (the preallocated-cache
  write helper kept apart from the attention math) -- a plain copy of the new
  tokens into positions [pos, pos + n) of the cache.
* ``prefill_varlen``: "Skill: Write a Triton Attention Kernel" (Inputs and
  Correctness requirements on variable-length batches) -- ``attention`` of
  each packed sequence on its own rows, masks and positions per sequence; a
  sequence with no keys gives O = 0, LSE = -inf.
* ``attention_bwd``: the gradients of ``attention`` for an incoming dO
  ("Skill: Write a Triton Attention Kernel" keeps m + log(l) so that a
  backward pass can rebuild the weights; "Triton-FlashAttention" defers the
  GQA backward that sums dK, dV over a group): with the explicit weights P,
  dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dO o O)), dQ = scale dS K,
  dK = scale dS^T Q, dK and dV summed over the q heads of each kv head.
* ``attention_bwd_dq_rows``, ``attention_bwd_dkv_rows``: selected rows of the
  same gradients, by the same definitions restricted to those rows (a query
  row's dQ needs only its own weights; a key row's dK, dV need the weights of
  every query row of every q head of the group, whose row sums are formed in
  blocks of query rows), for inputs too large for ``attention_bwd``.
* ``gather_pages``, ``decode_paged``, ``kv_cache_write_paged``: the paged,
  per-request-length decode that "Triton-FlashAttention" lists as deferred
  work (Deferred / explicitly out of scope).  Row t of request b's cache is row
  t % page_size of page block_table[b][t // page_size] of a shared pool;
  decode_paged is ``decode`` over each request's gathered rows, and a request
  of length 0 gives O = 0, LSE = -inf.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(hand-derived fixtures, closed forms, invariants and planted-mistake checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_int64_p = ctypes.POINTER(ctypes.c_int64)


def compile_source(src: str, out: str) -> str:
    """Compile a C oracle source into a shared library (gcc, -O2, IEEE arithmetic)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (if stale or missing)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_c_double_p)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64 = ctypes.c_int64
        lib.oracle_attention_fwd.restype = ctypes.c_int
        lib.oracle_attention_fwd.argtypes = [
            _c_double_p, _c_double_p, _c_double_p, _c_double_p, _c_double_p,
            i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [
            _c_double_p, _c_double_p, _c_double_p,
            i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
            _c_int64_p, i64, _c_double_p, _c_double_p, ctypes.c_int]
        self._lib = lib

    def attention(self, q, k, v, causal: bool, scale: float, nthreads: int | None = None):
        """Full attention forward.

        q: (B, H_q, N_q, D); k, v: (B, H_kv, N_kv, D) -- any real dtype, converted
        exactly to fp64.  Returns (O (B,H_q,N_q,D) fp64, LSE (B,H_q,N_q) fp64).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Nq, D = q.shape
        Bk, Hkv, Nkv, Dk = k.shape
        if v.shape != k.shape or Bk != B or Dk != D:
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        o = np.empty((B, Hq, Nq, D), dtype=np.float64)
        lse = np.empty((B, Hq, Nq), dtype=np.float64)
        rc = self._lib.oracle_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                            B, Hq, Hkv, Nq, Nkv, D, 1 if causal else 0, float(scale),
                                            nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention_fwd rejected the arguments (code {rc})")
        return o, lse

    def attention_rows(self, q, k, v, causal: bool, scale: float, rows, nthreads: int | None = None):
        """Attention for selected query rows only.

        rows: integer array (n, 3) of (b, h, i).  Returns (O (n, D), LSE (n,)).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Nq, D = q.shape
        _, Hkv, Nkv, _ = k.shape
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = sel.shape[0]
        o = np.empty((n, D), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        rc = self._lib.oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, D,
                                             1 if causal else 0, float(scale),
                                             sel.ctypes.data_as(_c_int64_p), n, _ptr(o), _ptr(lse),
                                             nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention_rows rejected the arguments (code {rc})")
        return o, lse

    def decode(self, q, k_cache, v_cache, cache_len: int, scale: float, nthreads: int | None = None):
        """One query token per (batch, q-head) over the first cache_len cache rows.

        q: (B, H_q, D) or (B, H_q, 1, D); caches: (B, H_kv, max_len, D).
        Returns (O (B, H_q, D), LSE (B, H_q)).
        """
        q = _f64(q)
        if q.ndim == 3:
            q = q[:, :, None, :]
        if cache_len < 1:
            raise ValueError("cache_len must be >= 1")
        kc = np.asarray(k_cache)[:, :, :cache_len, :]
        vc = np.asarray(v_cache)[:, :, :cache_len, :]
        o, lse = self.attention(q, kc, vc, causal=False, scale=scale, nthreads=nthreads)
        return o[:, :, 0, :], lse[:, :, 0]


_default = None


def _oracle() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def attention(q, k, v, causal: bool, scale: float, nthreads: int | None = None):
    return _oracle().attention(q, k, v, causal, scale, nthreads)


def attention_rows(q, k, v, causal: bool, scale: float, rows, nthreads: int | None = None):
    return _oracle().attention_rows(q, k, v, causal, scale, rows, nthreads)


def decode(q, k_cache, v_cache, cache_len: int, scale: float, nthreads: int | None = None):
    return _oracle().decode(q, k_cache, v_cache, cache_len, scale, nthreads)


attention.__doc__ = Oracle.attention.__doc__
attention_rows.__doc__ = Oracle.attention_rows.__doc__
decode.__doc__ = Oracle.decode.__doc__


def kv_cache_write(k_cache, v_cache, k_new, v_new, pos: int):
    """Copies of the caches with k_new/v_new (B, H_kv, n, D) placed at [pos, pos+n)."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    n = np.asarray(k_new).shape[2]
    if pos < 0 or pos + n > kc.shape[2]:
        raise ValueError("write outside the cache")
    kc[:, :, pos:pos + n, :] = k_new
    vc[:, :, pos:pos + n, :] = v_new
    return kc, vc


def attention_bwd_dq_rows(q, k, v, dout, causal: bool, scale: float, b: int, h: int, rows):
    """dQ[b, h, rows, :] of ``attention_bwd``, each row from its own weights, in fp64."""
    hk = h // (q.shape[1] // k.shape[1])
    q, k, v, dout = _f64(q[b, h]), _f64(k[b, hk]), _f64(v[b, hk]), _f64(dout[b, h])
    Nkv = k.shape[0]
    out = np.zeros((len(rows), q.shape[1]))
    for n, i in enumerate(rows):
        s = scale * (k @ q[i])
        if causal:
            s = np.where(np.arange(Nkv) > i, -np.inf, s)
        p = np.exp(s - s.max())
        p /= p.sum()
        dp = v @ dout[i]
        ds = p * (dp - dout[i] @ (p @ v))
        out[n] = scale * (ds @ k)
    return out


def attention_bwd_dkv_rows(q, k, v, dout, causal: bool, scale: float, b: int, hk: int, keys, block: int = 512):
    """dK[b, hk, keys, :] and dV[b, hk, keys, :] of ``attention_bwd`` (summed over the q heads of kv
    head hk), in fp64.  The weights P[i, keys] need every query row's full softmax; rows are taken
    ``block`` at a time."""
    keys = np.asarray(keys)
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    kk, vv = _f64(k[b, hk]), _f64(v[b, hk])
    Nq, Nkv, D = q.shape[2], kk.shape[0], kk.shape[1]
    dk = np.zeros((len(keys), D))
    dv = np.zeros((len(keys), D))
    for h in range(hk * g, (hk + 1) * g):
        qh, gh = _f64(q[b, h]), _f64(dout[b, h])
        for i0 in range(0, Nq, block):
            qb, gb = qh[i0:i0 + block], gh[i0:i0 + block]
            s = scale * (qb @ kk.T)
            if causal:
                s = np.where(np.arange(Nkv)[None, :] > np.arange(i0, i0 + len(qb))[:, None], -np.inf, s)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o = p @ vv
            pk = p[:, keys]
            dpk = gb @ vv[keys].T
            dsk = pk * (dpk - (gb * o).sum(axis=1, keepdims=True))
            dv += pk.T @ gb
            dk += scale * (dsk.T @ qb)
    return dk, dv


def gather_pages(pages, block_table_row, length: int):
    """Rows [0, length) of one request's paged cache, as (H_kv, length, D).

    pages: (num_pages, H_kv, page_size, D); row t of the request is row
    t % page_size of page block_table_row[t // page_size].
    """
    pages = np.asarray(pages)
    page_size = pages.shape[2]
    out = np.empty((pages.shape[1], length, pages.shape[3]), dtype=pages.dtype)
    for t in range(length):
        out[:, t, :] = pages[int(block_table_row[t // page_size]), :, t % page_size, :]
    return out


def decode_paged(q, k_pages, v_pages, block_table, cache_lens, scale: float, nthreads: int | None = None):
    """Decode of each request b over its own cache_lens[b] paged rows.

    q: (B, H_q, D); pages: (num_pages, H_kv, page_size, D); block_table (B, max_pages).
    Returns (O (B, H_q, D), LSE (B, H_q)); a request of length 0 gets O = 0, LSE = -inf.
    """
    q = _f64(q)
    B, Hq, D = q.shape
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        n = int(cache_lens[b])
        if n == 0:
            continue
        kc = gather_pages(k_pages, block_table[b], n)[None]
        vc = gather_pages(v_pages, block_table[b], n)[None]
        ob, lb = decode(q[b:b + 1], kc, vc, n, scale, nthreads)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def kv_cache_write_paged(k_pages, v_pages, k_new, v_new, block_table, positions):
    """Copies of the page pools with token t of request b (k_new[b, :, t]) at
    row (p % page_size) of page block_table[b][p // page_size], p = positions[b] + t."""
    kp = np.array(k_pages, copy=True)
    vp = np.array(v_pages, copy=True)
    k_new, v_new = np.asarray(k_new), np.asarray(v_new)
    page_size = kp.shape[2]
    for b in range(k_new.shape[0]):
        for t in range(k_new.shape[2]):
            pos = int(positions[b]) + t
            page = int(block_table[b][pos // page_size])
            kp[page, :, pos % page_size, :] = k_new[b, :, t, :]
            vp[page, :, pos % page_size, :] = v_new[b, :, t, :]
    return kp, vp


def prefill_varlen(q, k, v, cu_q, cu_k, causal: bool, scale: float, nthreads: int | None = None):
    """Attention of packed sequences: sequence b is rows [cu_q[b], cu_q[b+1]) of
    q (total_q, H_q, D) against rows [cu_k[b], cu_k[b+1]) of k, v (total_k, H_kv, D).

    Returns (O (total_q, H_q, D), LSE (H_q, total_q)).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    total_q, Hq, D = q.shape
    o = np.zeros((total_q, Hq, D))
    lse = np.full((Hq, total_q), -np.inf)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if qe == qs or ke == ks:
            continue
        qb = q[qs:qe].transpose(1, 0, 2)[None]
        kb = k[ks:ke].transpose(1, 0, 2)[None]
        vb = v[ks:ke].transpose(1, 0, 2)[None]
        ob, lb = attention(qb, kb, vb, causal, scale, nthreads)
        o[qs:qe] = ob[0].transpose(1, 0, 2)
        lse[:, qs:qe] = lb[0]
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float):
    """(dQ, dK, dV) of O = softmax(scale Q K^T + mask) V for the incoming gradient dout, in fp64.

    q, dout: (B, H_q, N_q, D); k, v: (B, H_kv, N_kv, D).  Plain dense matrices per (b, q head).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            s = scale * (q[b, h] @ k[b, hk].T)
            if causal:
                s = np.where(np.arange(Nkv)[None, :] > np.arange(Nq)[:, None], -np.inf, s)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[b, hk]
            dv[b, hk] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, hk].T
            ds = p * (dp - (dout[b, h] * o).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
    return dq, dk, dv
