"""Python binding of libattn_gb300.so -- the GB300 (sm_103a) fused attention forward.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the shared library, reached through its C ABI (``include/attn.h``).
PyTorch supplies device memory and streams.  If the library has not been
built, every call raises ``AttnLibraryMissing``; there is no fallback.

Low-level functions carry the C names (``attn_fwd_prefill``, ``attn_fwd_decode``,
``kv_cache_write``, ``attn_decode_workspace_size``, ``attn_get_device_error``,
``attn_status_string``) and take raw pointers, sizes and strides.  The
tensor-level helpers ``prefill``, ``decode`` and ``write_kv_cache`` fill those
arguments from PyTorch tensors.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGNMENT = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_DEVICE_TIMEOUT = 6
ATTN_ERR_DEVICE_INDEX = 7

ATTN_F16 = 0
ATTN_BF16 = 1

# Every function that include/attn.h declares.
EXPORTS = ("attn_fwd_prefill", "attn_fwd_prefill_ex", "attn_fwd_prefill_host", "attn_fwd_prefill_host_workspace_size",
           "attn_fwd_prefill_varlen", "attn_fwd_prefill_varlen_ex",
           "attn_fwd_decode_ex", "attn_fwd_decode_paged_ex", "attn_decode_workspace_size", "attn_decode_splits", "attn_fwd_decode",
           "attn_fwd_decode_noalloc", "kv_cache_write", "kv_cache_write_ex", "attn_fwd_decode_paged",
           "kv_cache_write_paged", "kv_cache_write_paged_ex",
           "attn_bwd_workspace_size", "attn_bwd_ex_workspace_size", "attn_bwd", "attn_bwd_ex",
           "attn_get_device_error", "attn_selftest_wait_timeout", "attn_status_string", "attn_version")


class AttnLibraryMissing(RuntimeError):
    pass


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} ({status})")


class AttnOptions(ctypes.Structure):
    """attn_options_t: sliding-window bounds (-1: none), ALiBi slopes (device fp32 pointer or None),
    rotary embedding base (0: none) and pairing, the decode split count (0: automatic), key ranges and the
    prefill kernel (0 automatic, 1 one-CTA, 2 CTA pair)."""
    _fields_ = [("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
                ("alibi_slopes", ctypes.c_void_p), ("rope_theta", ctypes.c_float),
                ("rope_interleaved", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("rope_rotated_keys", ctypes.c_int32), ("kv_ranges", ctypes.c_void_p),
                ("prefill_kernel", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None
_I64x4 = ctypes.c_int64 * 4


def lib() -> ctypes.CDLL:
    """The loaded C library (built in-tree by ``attention_fa2_fwd_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise AttnLibraryMissing(
                    f"{LIB_PATH} is missing: build it with `python -m attention_fa2_fwd_gb300.build` "
                    "(or __graft_entry__.build()); there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.attn_fwd_prefill.restype = i32
            L.attn_fwd_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                           i64p, i64p, i64p, i64p, i32, f32, vp]
            L.attn_fwd_prefill_varlen.restype = i32
            L.attn_fwd_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, i32,
                                                  i32, i32, i64p, i64p, i64p, i64p, i32, f32, vp]
            optp = ctypes.POINTER(AttnOptions)
            L.attn_fwd_prefill_ex.restype = i32
            L.attn_fwd_prefill_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                              i64p, i64p, i64p, i64p, i32, f32, optp, vp]
            L.attn_fwd_prefill_varlen_ex.restype = i32
            L.attn_fwd_prefill_varlen_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, i32,
                                                     i32, i32, i64p, i64p, i64p, i64p, i32, f32, optp, vp]
            L.attn_fwd_decode_ex.restype = i32
            L.attn_fwd_decode_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                             i64p, i64p, i64p, i64p, f32, vp, ctypes.c_size_t, optp, vp]
            L.attn_fwd_decode_paged_ex.restype = i32
            L.attn_fwd_decode_paged_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                                   vp, i32, ctypes.c_int64, vp, i32, i64p, i64p, i64p, i64p, f32, vp,
                                                   ctypes.c_size_t, optp, vp]
            L.attn_fwd_prefill_host_workspace_size.restype = ctypes.c_size_t
            L.attn_fwd_prefill_host_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.attn_fwd_prefill_host.restype = i32
            L.attn_fwd_prefill_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                                optp, vp, ctypes.c_size_t, vp]
            L.attn_decode_workspace_size.restype = ctypes.c_size_t
            L.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32]
            L.attn_decode_splits.restype = i32
            L.attn_decode_splits.argtypes = [i32, i32, i32, i32, i32]
            L.attn_fwd_decode.restype = i32
            L.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                          i64p, i64p, i64p, i64p, f32, vp, ctypes.c_size_t, vp]
            L.attn_fwd_decode_noalloc.restype = i32
            L.attn_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                  i64p, i64p, i64p, i64p, f32, vp]
            L.kv_cache_write.restype = i32
            L.kv_cache_write.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                         i64p, i64p, i64p, i64p, vp]
            L.kv_cache_write_ex.restype = i32
            L.kv_cache_write_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                            i64p, i64p, i64p, i64p, optp, vp]
            i64 = ctypes.c_int64
            L.attn_fwd_decode_paged.restype = i32
            L.attn_fwd_decode_paged.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                                vp, i32, i64, vp, i32, i64p, i64p, i64p, i64p, f32, vp,
                                                ctypes.c_size_t, vp]
            L.kv_cache_write_paged.restype = i32
            L.kv_cache_write_paged.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, i32, i64,
                                               vp, i64p, i64p, i64p, i64p, vp]
            L.kv_cache_write_paged_ex.restype = i32
            L.kv_cache_write_paged_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, i32, i64,
                                                  vp, i64p, i64p, i64p, i64p, optp, vp]
            L.attn_bwd_workspace_size.restype = ctypes.c_size_t
            L.attn_bwd_workspace_size.argtypes = [i32, i32, i32]
            L.attn_bwd_ex_workspace_size.restype = ctypes.c_size_t
            L.attn_bwd_ex_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, optp]
            L.attn_bwd.restype = i32
            L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                   i64p, i64p, i64p, i64p, i64p, i64p, i64p, i64p, i32, f32, vp, ctypes.c_size_t, vp]
            L.attn_bwd_ex.restype = i32
            L.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                      i64p, i64p, i64p, i64p, i64p, i64p, i64p, i64p, i32, f32, vp, vp,
                                      ctypes.c_size_t, vp]
            L.attn_get_device_error.restype = i32
            L.attn_get_device_error.argtypes = [vp]
            L.attn_selftest_wait_timeout.restype = i32
            L.attn_selftest_wait_timeout.argtypes = [vp]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_status_string.argtypes = [i32]
            L.attn_version.restype = i32
            L.attn_version.argtypes = []
            _lib = L
    return _lib


def _strides(s):
    return _I64x4(*[int(x) for x in s])


# ------------------------------------------------------------------ C names

def attn_fwd_prefill(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str,
                     causal, scale, stream) -> int:
    return lib().attn_fwd_prefill(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, _strides(q_str),
                                  _strides(k_str), _strides(v_str), _strides(o_str), int(causal), float(scale),
                                  stream)


def _opts(opts):
    return ctypes.byref(opts) if opts is not None else None


def attn_fwd_prefill_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str,
                        causal, scale, opts, stream) -> int:
    return lib().attn_fwd_prefill_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, _strides(q_str),
                                     _strides(k_str), _strides(v_str), _strides(o_str), int(causal), float(scale),
                                     _opts(opts), stream)


def attn_fwd_prefill_varlen_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, D, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                               max_seqlen_k, total_q, total_k, q_str, k_str, v_str, o_str, causal, scale, opts,
                               stream) -> int:
    s3 = ctypes.c_int64 * 3
    return lib().attn_fwd_prefill_varlen_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, D, cu_seqlens_q, cu_seqlens_k,
                                            max_seqlen_q, max_seqlen_k, total_q, total_k, s3(*q_str), s3(*k_str),
                                            s3(*v_str), s3(*o_str), int(causal), float(scale), _opts(opts), stream)


def attn_fwd_decode_ex(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str, vc_str, o_str,
                       scale, workspace, workspace_bytes, opts, stream) -> int:
    return lib().attn_fwd_decode_ex(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D,
                                    _strides(q_str), _strides(kc_str), _strides(vc_str), _strides(o_str),
                                    float(scale), workspace, workspace_bytes, _opts(opts), stream)


def attn_fwd_decode_paged_ex(q, k_pages, v_pages, o, lse, dtype, B, H_q, H_kv, D, num_pages, page_size, block_table,
                             max_pages, bt_stride, cache_lens, max_cache_len, q_str, kp_str, vp_str, o_str, scale,
                             workspace, workspace_bytes, opts, stream) -> int:
    return lib().attn_fwd_decode_paged_ex(q, k_pages, v_pages, o, lse, dtype, B, H_q, H_kv, D, num_pages,
                                          page_size, block_table, max_pages, bt_stride, cache_lens, max_cache_len,
                                          _strides(q_str), _strides(kp_str), _strides(vp_str), _strides(o_str),
                                          float(scale), workspace, workspace_bytes, _opts(opts), stream)


def attn_fwd_prefill_host_workspace_size(dtype, B, H_q, H_kv, N_q, N_kv, D) -> int:
    return lib().attn_fwd_prefill_host_workspace_size(dtype, B, H_q, H_kv, N_q, N_kv, D)


def attn_fwd_prefill_host(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, causal, scale, opts, workspace,
                          workspace_bytes, stream) -> int:
    return lib().attn_fwd_prefill_host(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, int(causal), float(scale),
                                       _opts(opts), workspace, workspace_bytes, stream)


def make_options(window_left: int = -1, window_right: int = -1, alibi_slopes=None, rope_theta: float = 0.0,
                 rope_interleaved: bool = False, num_splits: int = 0, rope_rotated_keys: bool = False,
                 kv_ranges=None, prefill_kernel: int = 0):
    """An AttnOptions for the *_ex calls (None when nothing is set).

    alibi_slopes: fp32 CUDA tensor (H_q); rope_theta: base of the rotary embedding (0: none);
    rope_interleaved: pairs (2c, 2c+1) instead of (c, c+D/2); num_splits: decode split count (0: automatic);
    rope_rotated_keys: prefill keys already rotated (only the queries are rotated);
    kv_ranges: int32 CUDA tensor of per-query-row key ranges [lo, hi), (B, N_q, 2) or packed (total_q, 2);
    prefill_kernel: 0 automatic, 1 the one-CTA kernel, 2 the CTA-pair kernel (D = 128, no masks or RoPE).
    """
    if (window_left == -1 and window_right == -1 and alibi_slopes is None and not rope_theta
            and not num_splits and kv_ranges is None and not prefill_kernel):
        return None
    if kv_ranges is not None:
        import torch
        if kv_ranges.dtype != torch.int32 or not kv_ranges.is_cuda or not kv_ranges.is_contiguous() \
                or kv_ranges.shape[-1] != 2:
            raise TypeError("kv_ranges must be a contiguous int32 CUDA tensor of [lo, hi) pairs")
    if alibi_slopes is not None:
        import torch
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda:
            raise TypeError("alibi_slopes must be an fp32 CUDA tensor")
    return AttnOptions(int(window_left), int(window_right),
                       alibi_slopes.data_ptr() if alibi_slopes is not None else None, float(rope_theta),
                       1 if rope_interleaved else 0, int(num_splits), 1 if rope_rotated_keys else 0,
                       kv_ranges.data_ptr() if kv_ranges is not None else None, int(prefill_kernel))


def attn_fwd_prefill_varlen(q, k, v, o, lse, dtype, B, H_q, H_kv, D, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                            max_seqlen_k, total_q, total_k, q_str, k_str, v_str, o_str, causal, scale,
                            stream) -> int:
    s3 = ctypes.c_int64 * 3
    return lib().attn_fwd_prefill_varlen(q, k, v, o, lse, dtype, B, H_q, H_kv, D, cu_seqlens_q, cu_seqlens_k,
                                         max_seqlen_q, max_seqlen_k, total_q, total_k, s3(*q_str), s3(*k_str),
                                         s3(*v_str), s3(*o_str), int(causal), float(scale), stream)


def attn_decode_workspace_size(B, H_q, H_kv, D) -> int:
    return int(lib().attn_decode_workspace_size(B, H_q, H_kv, D))


def attn_decode_splits(B, H_q, H_kv, cache_len, D) -> int:
    return int(lib().attn_decode_splits(B, H_q, H_kv, cache_len, D))


def attn_fwd_decode(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str, vc_str, o_str,
                    scale, workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_decode(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, _strides(q_str),
                                 _strides(kc_str), _strides(vc_str), _strides(o_str), float(scale), workspace,
                                 workspace_bytes, stream)


def attn_fwd_decode_noalloc(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str, vc_str,
                            o_str, scale, stream) -> int:
    """attn_fwd_decode without a workspace argument, for callers that may not allocate device memory.

    The split partials go to a 4 MiB scratch array inside the library (shared
    by every call on the device; overlapping calls race on it).  Returns
    ATTN_ERR_WORKSPACE if the call would need more than 4 MiB of scratch.
    """
    return lib().attn_fwd_decode_noalloc(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D,
                                         _strides(q_str), _strides(kc_str), _strides(vc_str), _strides(o_str),
                                         float(scale), stream)


def kv_cache_write(k_cache, v_cache, k_new, v_new, dtype, B, H_kv, n_new, D, pos, max_len, kc_str, vc_str, kn_str,
                   vn_str, stream) -> int:
    return lib().kv_cache_write(k_cache, v_cache, k_new, v_new, dtype, B, H_kv, n_new, D, pos, max_len,
                                _strides(kc_str), _strides(vc_str), _strides(kn_str), _strides(vn_str), stream)


def kv_cache_write_ex(k_cache, v_cache, k_new, v_new, dtype, B, H_kv, n_new, D, pos, max_len, kc_str, vc_str, kn_str,
                      vn_str, opts, stream) -> int:
    return lib().kv_cache_write_ex(k_cache, v_cache, k_new, v_new, dtype, B, H_kv, n_new, D, pos, max_len,
                                   _strides(kc_str), _strides(vc_str), _strides(kn_str), _strides(vn_str), _opts(opts),
                                   stream)


def kv_cache_write_paged_ex(k_pages, v_pages, k_new, v_new, dtype, B, H_kv, n_new, D, num_pages, page_size,
                            block_table, max_pages, bt_stride, positions, kp_str, vp_str, kn_str, vn_str, opts,
                            stream) -> int:
    return lib().kv_cache_write_paged_ex(k_pages, v_pages, k_new, v_new, dtype, B, H_kv, n_new, D, num_pages,
                                         page_size, block_table, max_pages, bt_stride, positions, _strides(kp_str),
                                         _strides(vp_str), _strides(kn_str), _strides(vn_str), _opts(opts), stream)


def attn_fwd_decode_paged(q, k_pages, v_pages, o, lse, dtype, B, H_q, H_kv, D, num_pages, page_size, block_table,
                          max_pages, bt_stride, cache_lens, max_cache_len, q_str, kp_str, vp_str, o_str, scale,
                          workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_decode_paged(q, k_pages, v_pages, o, lse, dtype, B, H_q, H_kv, D, num_pages, page_size,
                                       block_table, max_pages, bt_stride, cache_lens, max_cache_len,
                                       _strides(q_str), _strides(kp_str), _strides(vp_str), _strides(o_str),
                                       float(scale), workspace, workspace_bytes, stream)


def kv_cache_write_paged(k_pages, v_pages, k_new, v_new, dtype, B, H_kv, n_new, D, num_pages, page_size,
                         block_table, max_pages, bt_stride, positions, kp_str, vp_str, kn_str, vn_str,
                         stream) -> int:
    return lib().kv_cache_write_paged(k_pages, v_pages, k_new, v_new, dtype, B, H_kv, n_new, D, num_pages,
                                      page_size, block_table, max_pages, bt_stride, positions, _strides(kp_str),
                                      _strides(vp_str), _strides(kn_str), _strides(vn_str), stream)


def attn_bwd_workspace_size(B, H_q, N_q) -> int:
    return int(lib().attn_bwd_workspace_size(B, H_q, N_q))


def attn_bwd_ex_workspace_size(B, H_q, H_kv, N_q, N_kv, D, opts) -> int:
    return int(lib().attn_bwd_ex_workspace_size(B, H_q, H_kv, N_q, N_kv, D, _opts(opts)))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str,
             do_str, dq_str, dk_str, dv_str, causal, scale, workspace, workspace_bytes, stream) -> int:
    return lib().attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, dtype, B, H_q, H_kv, N_q, N_kv, D, _strides(q_str),
                          _strides(k_str), _strides(v_str), _strides(o_str), _strides(do_str), _strides(dq_str),
                          _strides(dk_str), _strides(dv_str), int(causal), float(scale), workspace, workspace_bytes,
                          stream)


def attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str,
                do_str, dq_str, dk_str, dv_str, causal, scale, opts, workspace, workspace_bytes, stream) -> int:
    return lib().attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, dtype, B, H_q, H_kv, N_q, N_kv, D, _strides(q_str),
                             _strides(k_str), _strides(v_str), _strides(o_str), _strides(do_str), _strides(dq_str),
                             _strides(dk_str), _strides(dv_str), int(causal), float(scale), _opts(opts), workspace,
                             workspace_bytes, stream)


def attn_get_device_error(stream=None) -> int:
    return lib().attn_get_device_error(stream)


def attn_selftest_wait_timeout(stream=None) -> int:
    """Enqueue the bounded-wait self-test kernel (see include/attn.h); returns its launch status."""
    return lib().attn_selftest_wait_timeout(stream)


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_version() -> int:
    return lib().attn_version()


# ------------------------------------------------------------------ tensor helpers

def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_F16
    raise TypeError(f"unsupported dtype {t.dtype}: fp16 or bf16 only")


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def prefill(q, k, v, causal: bool = False, scale: float | None = None, return_lse: bool = True, out=None,
            lse_out=None, stream=None, window=(-1, -1), alibi_slopes=None, rope_theta: float = 0.0,
            rope_interleaved: bool = False, rope_rotated_keys: bool = False, kv_ranges=None,
            prefill_kernel: int = 0):
    """Fused attention forward.  q (B,H_q,N_q,D); k, v (B,H_kv,N_kv,D) CUDA tensors.

    Any (b, h, n) strides are accepted (16-byte multiples, d stride 1), so a
    (B,N,H,D) tensor passed as its permuted (B,H,N,D) view works directly.
    Returns (O, LSE) with O shaped like q (contiguous unless ``out`` is given)
    and LSE (B,H_q,N_q) fp32, or None when ``return_lse`` is False.
    """
    import torch
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    st = attn_fwd_prefill_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr() if lse is not None else None, _dtype_code(q), B, Hq, Hkv, Nq, Nkv, D,
                             q.stride(), k.stride(), v.stride(), o.stride(), 1 if causal else 0, scale,
                             make_options(window[0], window[1], alibi_slopes, rope_theta, rope_interleaved,
                                          rope_rotated_keys=rope_rotated_keys, kv_ranges=kv_ranges,
                                          prefill_kernel=prefill_kernel),
                             _stream_handle(stream))
    _check(st, "attn_fwd_prefill")
    return o, lse


def prefill_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse_out=None,
                 workspace=None, stream=None, window=(-1, -1), alibi_slopes=None, rope_theta: float = 0.0,
                 rope_interleaved: bool = False, kv_ranges=None, prefill_kernel: int = 0):
    """Prefill on host tensors (contiguous, ideally pinned) with copies pipelined against the compute.

    q (B,H_q,N_q,D), k, v (B,H_kv,N_kv,D) CPU tensors; returns host (O, LSE).  The results are complete
    once ``stream`` (default: the current CUDA stream) has finished; this helper synchronises it.
    """
    import torch
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    lse = lse_out if lse_out is not None else torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=True)
    code = _dtype_code(q)
    need = attn_fwd_prefill_host_workspace_size(code, B, Hq, Hkv, Nq, Nkv, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = attn_fwd_prefill_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), code, B, Hq,
                               Hkv, Nq, Nkv, D, causal, scale,
                               make_options(window[0], window[1], alibi_slopes, rope_theta, rope_interleaved,
                                            kv_ranges=kv_ranges, prefill_kernel=prefill_kernel),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream))
    _check(st, "attn_fwd_prefill_host")
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return o, lse


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                   causal: bool = False, scale: float | None = None, return_lse: bool = True, out=None,
                   lse_out=None, stream=None, window=(-1, -1), alibi_slopes=None, rope_theta: float = 0.0,
                   rope_interleaved: bool = False, rope_rotated_keys: bool = False, kv_ranges=None):
    """Attention over packed sequences of different lengths.

    q (total_q, H_q, D); k, v (total_k, H_kv, D); cu_seqlens_q / cu_seqlens_k int32 CUDA tensors (B + 1).
    Returns (O (total_q, H_q, D), LSE (H_q, total_q) fp32 or None).
    """
    import torch
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    cq = _int32_cuda(cu_seqlens_q, "cu_seqlens_q")
    ck = _int32_cuda(cu_seqlens_k, "cu_seqlens_k")
    B = cq.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty((total_q, Hq, D), dtype=q.dtype, device=q.device)
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    st = attn_fwd_prefill_varlen_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, _dtype_code(q), B, Hq, Hkv, D,
                                    cq.data_ptr(), ck.data_ptr(), int(max_seqlen_q), int(max_seqlen_k), total_q,
                                    total_k, q.stride(), k.stride(), v.stride(), o.stride(), 1 if causal else 0, scale,
                                    make_options(window[0], window[1], alibi_slopes, rope_theta, rope_interleaved,
                                                 rope_rotated_keys=rope_rotated_keys, kv_ranges=kv_ranges),
                                    _stream_handle(stream))
    _check(st, "attn_fwd_prefill_varlen")
    return o, lse


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, workspace=None, stream=None,
             window=(-1, -1), alibi_slopes=None, kv_ranges=None, rope_theta: float = 0.0,
             rope_interleaved: bool = False, rope_rotated_keys: bool = False):
    """Gradients (dQ, dK, dV) of attn_fwd_prefill from its output O and LSE and the incoming dO.

    Shapes as for prefill; dK, dV are summed over each GQA group.  window, alibi_slopes, kv_ranges and the
    rope_* options must be those of the forward call (with rope_rotated_keys, dK is the gradient with respect
    to the rotated keys passed in).  Returns new contiguous tensors.
    """
    import torch
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
    dk = torch.empty((B, Hkv, Nkv, D), dtype=q.dtype, device=q.device)
    dv = torch.empty((B, Hkv, Nkv, D), dtype=q.dtype, device=q.device)
    opts = make_options(window[0], window[1], alibi_slopes, kv_ranges=kv_ranges, rope_theta=rope_theta,
                        rope_interleaved=rope_interleaved, rope_rotated_keys=rope_rotated_keys)
    n = attn_bwd_ex_workspace_size(B, Hq, Hkv, Nq, Nkv, D, opts)
    if workspace is None:
        workspace = torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device=q.device)
    st = attn_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), _dtype_code(q), B, Hq, Hkv, Nq, Nkv, D, q.stride(),
                     k.stride(), v.stride(), o.stride(), dout.stride(), dq.stride(), dk.stride(), dv.stride(),
                     1 if causal else 0, scale, opts, workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def decode_workspace(B, H_q, H_kv, D, device=None, num_splits: int = 0):
    """A workspace tensor for attn_fwd_decode (None when it needs 0 bytes): attn_decode_workspace_size bytes,
    or -- for a forced split count num_splits above the automatic one -- the 4 B H_q n (D + 1) bytes it needs."""
    import torch
    n = attn_decode_workspace_size(B, H_q, H_kv, D)
    if num_splits > 1:
        n = max(n, 4 * B * H_q * num_splits * (D + 1))
    if n == 0:
        return None
    return torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device=device or "cuda")


def decode(q, k_cache, v_cache, cache_len: int, scale: float | None = None, return_lse: bool = True, out=None,
           lse_out=None, workspace=None, stream=None, window_left: int = -1, alibi_slopes=None,
           num_splits: int = 0, rope_theta: float = 0.0, rope_interleaved: bool = False):
    """One query token per (batch, q-head) over the first cache_len cache rows.

    q (B,H_q,D) or (B,H_q,1,D); caches (B,H_kv,max_len,D).  Returns (O (B,H_q,D), LSE (B,H_q)).
    num_splits: 0 automatic, n >= 1 at most n KV splits (a workspace for more splits than the automatic
    choice must be passed in).
    """
    import torch
    q4 = q if q.dim() == 4 else q.unsqueeze(2)
    B, Hq, _, D = q4.shape
    _, Hkv, max_len, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty((B, Hq, D), dtype=q.dtype, device=q.device)
    o4 = o.unsqueeze(2) if o.dim() == 3 else o
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, D, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = attn_fwd_decode_ex(q4.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o4.data_ptr(),
                            lse.data_ptr() if lse is not None else None, _dtype_code(q), B, Hq, Hkv, int(cache_len), D,
                            q4.stride(), k_cache.stride(), v_cache.stride(), o4.stride(), scale, ws_ptr, ws_bytes,
                            make_options(window_left, -1, alibi_slopes, rope_theta, rope_interleaved, num_splits),
                            _stream_handle(stream))
    _check(st, "attn_fwd_decode")
    return o, lse


def write_kv_cache(k_cache, v_cache, k_new, v_new, pos: int, stream=None, rope_theta: float = 0.0,
                   rope_interleaved: bool = False):
    """Copy k_new/v_new (B,H_kv,n,D) into cache rows [pos, pos+n) in place (keys rotated at their
    positions when rope_theta > 0)."""
    B, Hkv, max_len, D = k_cache.shape
    n = k_new.shape[2]
    st = kv_cache_write_ex(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                           _dtype_code(k_cache), B, Hkv, n, D, int(pos), max_len, k_cache.stride(), v_cache.stride(),
                           k_new.stride(), v_new.stride(), make_options(rope_theta=rope_theta,
                                                                        rope_interleaved=rope_interleaved),
                           _stream_handle(stream))
    _check(st, "kv_cache_write")


def _int32_cuda(t, name):
    import torch
    if t.dtype != torch.int32 or not t.is_cuda:
        raise TypeError(f"{name} must be an int32 CUDA tensor")
    return t


def decode_paged(q, k_pages, v_pages, block_table, cache_lens, max_cache_len: int, scale: float | None = None,
                 return_lse: bool = True, out=None, lse_out=None, workspace=None, stream=None,
                 window_left: int = -1, alibi_slopes=None, rope_theta: float = 0.0, rope_interleaved: bool = False,
                 num_splits: int = 0):
    """Decode over paged caches with per-request lengths.

    q (B,H_q,D); k_pages, v_pages (num_pages,H_kv,page_size,D); block_table int32 (B,max_pages) and
    cache_lens int32 (B) on the device; max_cache_len a host upper bound of cache_lens.
    Returns (O (B,H_q,D), LSE (B,H_q)).
    """
    import torch
    q4 = q if q.dim() == 4 else q.unsqueeze(2)
    B, Hq, _, D = q4.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    bt = _int32_cuda(block_table, "block_table")
    cl = _int32_cuda(cache_lens, "cache_lens")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty((B, Hq, D), dtype=q.dtype, device=q.device)
    o4 = o.unsqueeze(2) if o.dim() == 3 else o
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, D, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = attn_fwd_decode_paged_ex(q4.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), o4.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, _dtype_code(q), B, Hq, Hkv, D,
                                  num_pages, page_size, bt.data_ptr(), bt.shape[1], bt.stride(0), cl.data_ptr(),
                                  int(max_cache_len), q4.stride(), k_pages.stride(), v_pages.stride(), o4.stride(),
                                  scale, ws_ptr, ws_bytes,
                                  make_options(window_left, -1, alibi_slopes, rope_theta, rope_interleaved, num_splits),
                                  _stream_handle(stream))
    _check(st, "attn_fwd_decode_paged")
    return o, lse


def write_kv_cache_paged(k_pages, v_pages, k_new, v_new, block_table, positions, stream=None,
                         rope_theta: float = 0.0, rope_interleaved: bool = False):
    """Write k_new/v_new (B,H_kv,n,D) at positions[b] + t of each request's paged cache (in place; keys
    rotated at their positions when rope_theta > 0)."""
    num_pages, Hkv, page_size, D = k_pages.shape
    B, _, n, _ = k_new.shape
    bt = _int32_cuda(block_table, "block_table")
    pos = _int32_cuda(positions, "positions")
    st = kv_cache_write_paged_ex(k_pages.data_ptr(), v_pages.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                 _dtype_code(k_pages), B, Hkv, n, D, num_pages, page_size, bt.data_ptr(), bt.shape[1],
                                 bt.stride(0), pos.data_ptr(), k_pages.stride(), v_pages.stride(), k_new.stride(),
                                 v_new.stride(), make_options(rope_theta=rope_theta, rope_interleaved=rope_interleaved),
                                 _stream_handle(stream))
    _check(st, "kv_cache_write_paged")


def check_device_error(stream=None):
    """Synchronise and raise if a kernel recorded a failure (clears the record)."""
    _check(attn_get_device_error(_stream_handle(stream)), "device")
