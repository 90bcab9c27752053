"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

* the shared library loads and exports every function include/attn.h declares;
* every argument error is reported synchronously with its status code.  Each
  call below fails validation, which runs before any CUDA call, so the fake
  (never dereferenced) pointers are never seen by a kernel.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import attention_fa2_fwd_gb300 as A
from attention_fa2_fwd_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "attn.h")
P = 0x7F0000000000  # 16-byte aligned fake device address
BAD = P + 8         # misaligned


@pytest.fixture(scope="module")
def lib():
    build()
    return A.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_expected_functions():
    assert declared_functions() == sorted(A.EXPORTS)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert A.attn_version() >= 100


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_UNSUPPORTED"),
                       (3, "ATTN_ERR_ALIGNMENT"), (4, "ATTN_ERR_WORKSPACE"), (5, "ATTN_ERR_CUDA"),
                       (6, "ATTN_ERR_DEVICE_TIMEOUT"), (7, "ATTN_ERR_DEVICE_INDEX")]:
        assert A.attn_status_string(code) == name
    assert A.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


def contig(B, H, N, D):
    return (H * N * D, N * D, D, 1)


def prefill(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, dtype=A.ATTN_BF16, B=2, H_q=8, H_kv=2, N_q=64, N_kv=64, D=128,
             q_str=contig(2, 8, 64, 128), k_str=contig(2, 2, 64, 128), v_str=contig(2, 2, 64, 128),
             o_str=contig(2, 8, 64, 128), causal=1, scale=0.088, stream=None)
    a.update(kw)
    return A.attn_fwd_prefill(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(o=None), A.ATTN_ERR_INVALID_ARG),
    (dict(B=0), A.ATTN_ERR_INVALID_ARG),
    (dict(N_q=0), A.ATTN_ERR_INVALID_ARG),
    (dict(N_kv=0), A.ATTN_ERR_INVALID_ARG),
    (dict(H_kv=3), A.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), A.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=7), A.ATTN_ERR_UNSUPPORTED),
    (dict(q=BAD), A.ATTN_ERR_ALIGNMENT),
    (dict(v=BAD), A.ATTN_ERR_ALIGNMENT),
    (dict(lse=P + 2), A.ATTN_ERR_ALIGNMENT),
    (dict(q_str=(8 * 64 * 128, 64 * 128, 128, 2)), A.ATTN_ERR_ALIGNMENT),
    (dict(k_str=(2 * 64 * 128, 64 * 128, 132, 1)), A.ATTN_ERR_ALIGNMENT),
    (dict(o_str=(8 * 64 * 128, 64 * 128, -128, 1)), A.ATTN_ERR_INVALID_ARG),
])
def test_prefill_argument_errors(lib, kw, code):
    assert prefill(**kw) == code


def decode(**kw):
    a = dict(q=P, k_cache=P, v_cache=P, o=P, lse=None, dtype=A.ATTN_BF16, B=2, H_q=32, H_kv=8, cache_len=100,
             D=128, q_str=contig(2, 32, 1, 128), kc_str=contig(2, 8, 256, 128), vc_str=contig(2, 8, 256, 128),
             o_str=contig(2, 32, 1, 128), scale=0.088, workspace=P, workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return A.attn_fwd_decode(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(k_cache=None), A.ATTN_ERR_INVALID_ARG),
    (dict(cache_len=0), A.ATTN_ERR_INVALID_ARG),
    (dict(H_q=30), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), A.ATTN_ERR_INVALID_ARG),
    (dict(D=80), A.ATTN_ERR_UNSUPPORTED),
    (dict(k_cache=BAD), A.ATTN_ERR_ALIGNMENT),
    (dict(kc_str=(8 * 256 * 128, 256 * 128, 128, 3)), A.ATTN_ERR_ALIGNMENT),
])
def test_decode_argument_errors(lib, kw, code):
    assert decode(**kw) == code


def cache_write(**kw):
    a = dict(k_cache=P, v_cache=P, k_new=P, v_new=P, dtype=A.ATTN_BF16, B=2, H_kv=8, n_new=1, D=128, pos=10,
             max_len=256, kc_str=contig(2, 8, 256, 128), vc_str=contig(2, 8, 256, 128),
             kn_str=contig(2, 8, 1, 128), vn_str=contig(2, 8, 1, 128), stream=None)
    a.update(kw)
    return A.kv_cache_write(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(k_new=None), A.ATTN_ERR_INVALID_ARG),
    (dict(pos=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(pos=256), A.ATTN_ERR_INVALID_ARG),
    (dict(pos=250, n_new=7), A.ATTN_ERR_INVALID_ARG),
    (dict(n_new=0), A.ATTN_ERR_INVALID_ARG),
    (dict(D=32), A.ATTN_ERR_UNSUPPORTED),
    (dict(v_cache=BAD), A.ATTN_ERR_ALIGNMENT),
])
def test_cache_write_argument_errors(lib, kw, code):
    assert cache_write(**kw) == code


def test_workspace_size_rejects_bad_arguments(lib):
    assert A.attn_decode_workspace_size(0, 32, 8, 128) == 0
    assert A.attn_decode_workspace_size(2, 30, 8, 128) == 0
    assert A.attn_decode_workspace_size(2, 32, 8, 96) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(A, "_lib", None)
    monkeypatch.setattr(A, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(A.AttnLibraryMissing):
        A.lib()


def decode_paged(**kw):
    a = dict(q=P, k_pages=P, v_pages=P, o=P, lse=None, dtype=A.ATTN_BF16, B=2, H_q=32, H_kv=8, D=128,
             num_pages=100, page_size=16, block_table=P, max_pages=64, bt_stride=64, cache_lens=P,
             max_cache_len=1000, q_str=contig(2, 32, 1, 128), kp_str=contig(100, 8, 16, 128),
             vp_str=contig(100, 8, 16, 128), o_str=contig(2, 32, 1, 128), scale=0.088, workspace=P,
             workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return A.attn_fwd_decode_paged(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(block_table=None), A.ATTN_ERR_INVALID_ARG),
    (dict(cache_lens=None), A.ATTN_ERR_INVALID_ARG),
    (dict(max_cache_len=0), A.ATTN_ERR_INVALID_ARG),
    (dict(max_cache_len=64 * 16 + 1), A.ATTN_ERR_INVALID_ARG),
    (dict(bt_stride=10), A.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), A.ATTN_ERR_INVALID_ARG),
    (dict(page_size=24), A.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(block_table=P + 2), A.ATTN_ERR_ALIGNMENT),
    (dict(cache_lens=P + 1), A.ATTN_ERR_ALIGNMENT),
    (dict(D=80), A.ATTN_ERR_UNSUPPORTED),
    (dict(H_q=30), A.ATTN_ERR_INVALID_ARG),
])
def test_decode_paged_argument_errors(lib, kw, code):
    assert decode_paged(**kw) == code


def cache_write_paged(**kw):
    a = dict(k_pages=P, v_pages=P, k_new=P, v_new=P, dtype=A.ATTN_BF16, B=2, H_kv=8, n_new=1, D=128,
             num_pages=100, page_size=16, block_table=P, max_pages=64, bt_stride=64, positions=P,
             kp_str=contig(100, 8, 16, 128), vp_str=contig(100, 8, 16, 128), kn_str=contig(2, 8, 1, 128),
             vn_str=contig(2, 8, 1, 128), stream=None)
    a.update(kw)
    return A.kv_cache_write_paged(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(positions=None), A.ATTN_ERR_INVALID_ARG),
    (dict(block_table=None), A.ATTN_ERR_INVALID_ARG),
    (dict(n_new=0), A.ATTN_ERR_INVALID_ARG),
    (dict(page_size=8), A.ATTN_ERR_UNSUPPORTED),
    (dict(positions=P + 2), A.ATTN_ERR_ALIGNMENT),
    (dict(k_new=P + 8), A.ATTN_ERR_ALIGNMENT),
])
def test_cache_write_paged_argument_errors(lib, kw, code):
    assert cache_write_paged(**kw) == code


def prefill_varlen(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, dtype=A.ATTN_BF16, B=3, H_q=8, H_kv=2, D=128, cu_seqlens_q=P,
             cu_seqlens_k=P, max_seqlen_q=100, max_seqlen_k=100, total_q=200, total_k=200,
             q_str=(8 * 128, 128, 1), k_str=(2 * 128, 128, 1), v_str=(2 * 128, 128, 1), o_str=(8 * 128, 128, 1),
             causal=1, scale=0.088, stream=None)
    a.update(kw)
    return A.attn_fwd_prefill_varlen(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_seqlens_q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(max_seqlen_q=0), A.ATTN_ERR_INVALID_ARG),
    (dict(max_seqlen_k=300), A.ATTN_ERR_INVALID_ARG),
    (dict(total_q=0), A.ATTN_ERR_INVALID_ARG),
    (dict(H_kv=3), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(cu_seqlens_k=P + 2), A.ATTN_ERR_ALIGNMENT),
    (dict(q_str=(8 * 128, 128, 2)), A.ATTN_ERR_ALIGNMENT),
    (dict(k_str=(2 * 128 + 4, 128, 1)), A.ATTN_ERR_ALIGNMENT),
])
def test_prefill_varlen_argument_errors(lib, kw, code):
    assert prefill_varlen(**kw) == code


def bwd(**kw):
    s4 = contig(2, 8, 64, 128)
    k4 = contig(2, 2, 64, 128)
    a = dict(q=P, k=P, v=P, o=P, dout=P, lse=P, dq=P, dk=P, dv=P, dtype=A.ATTN_BF16, B=2, H_q=8, H_kv=2, N_q=64,
             N_kv=64, D=128, q_str=s4, k_str=k4, v_str=k4, o_str=s4, do_str=s4, dq_str=s4, dk_str=k4, dv_str=k4,
             causal=1, scale=0.088, workspace=P, workspace_bytes=1 << 20, stream=None)
    a.update(kw)
    return A.attn_bwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(dout=None), A.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), A.ATTN_ERR_INVALID_ARG),
    (dict(H_kv=3), A.ATTN_ERR_INVALID_ARG),
    (dict(N_kv=0), A.ATTN_ERR_INVALID_ARG),
    (dict(D=32), A.ATTN_ERR_UNSUPPORTED),
    (dict(dq=P + 8), A.ATTN_ERR_ALIGNMENT),
    (dict(lse=P + 2), A.ATTN_ERR_ALIGNMENT),
    (dict(workspace=None), A.ATTN_ERR_WORKSPACE),
    (dict(workspace_bytes=16), A.ATTN_ERR_WORKSPACE),
    (dict(dk_str=(2 * 64 * 128, 64 * 128, 128, 2)), A.ATTN_ERR_ALIGNMENT),
])
def test_bwd_argument_errors(lib, kw, code):
    assert bwd(**kw) == code


def test_bwd_workspace_size():
    assert A.attn_bwd_workspace_size(2, 8, 64) == 2 * 8 * 64 * 4
    assert A.attn_bwd_workspace_size(1, 1, 3) == 16
    assert A.attn_bwd_workspace_size(0, 8, 64) == 0


def test_bwd_ex_workspace_size(lib):
    """Without rotary embeddings the plain size; with them room for the rotated Q (and K unless given rotated)."""
    plain = A.attn_bwd_workspace_size(2, 8, 64)
    assert A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 96, 128, None) == plain
    assert A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 96, 128, A.make_options(window_left=5)) == plain
    rope = A.make_options(rope_theta=10000.0)
    assert A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 96, 128, rope) == plain + 2 * 8 * 64 * 128 * 2 + 2 * 2 * 96 * 128 * 2
    rk = A.make_options(rope_theta=10000.0, rope_rotated_keys=True)
    assert A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 96, 64, rk) == plain + 2 * 8 * 64 * 64 * 2
    for args in ((0, 8, 2, 64, 96, 128), (2, 8, 3, 64, 96, 128), (2, 8, 2, 64, 0, 128), (2, 8, 2, 64, 96, 80)):
        assert A.attn_bwd_ex_workspace_size(*args, rope) == 0
    assert A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 96, 128, A.AttnOptions(-1, -1, None, -1.0, 0, 0, 0)) == 0


def test_bwd_rope_needs_the_larger_workspace(lib):
    """A workspace of the plain size is too small once rotary embeddings are on (checked before any CUDA call)."""
    rope = A.make_options(rope_theta=10000.0)
    n = A.attn_bwd_ex_workspace_size(2, 8, 2, 64, 64, 128, rope)
    assert A.attn_bwd_ex(P, P, P, P, P, P, P, P, P, A.ATTN_BF16, 2, 8, 2, 64, 64, 128, contig(2, 8, 64, 128),
                         contig(2, 2, 64, 128), contig(2, 2, 64, 128), contig(2, 8, 64, 128), contig(2, 8, 64, 128),
                         contig(2, 8, 64, 128), contig(2, 2, 64, 128), contig(2, 2, 64, 128), 1, 0.088, rope, P,
                         A.attn_bwd_workspace_size(2, 8, 64), None) == A.ATTN_ERR_WORKSPACE
    assert A.attn_bwd_ex(P, P, P, P, P, P, P, P, P, A.ATTN_BF16, 2, 8, 2, 64, 64, 128, contig(2, 8, 64, 128),
                         contig(2, 2, 64, 128), contig(2, 2, 64, 128), contig(2, 8, 64, 128), contig(2, 8, 64, 128),
                         contig(2, 8, 64, 128), contig(2, 2, 64, 128), contig(2, 2, 64, 128), 1, 0.088, rope, P,
                         n - 1, None) == A.ATTN_ERR_WORKSPACE


OPTION_CALLS = {
    "prefill": lambda o: A.attn_fwd_prefill_ex(
        P, P, P, P, None, A.ATTN_BF16, 2, 8, 2, 64, 64, 128, contig(2, 8, 64, 128), contig(2, 2, 64, 128),
        contig(2, 2, 64, 128), contig(2, 8, 64, 128), 1, 0.088, o, None),
    "prefill_varlen": lambda o: A.attn_fwd_prefill_varlen_ex(
        P, P, P, P, None, A.ATTN_BF16, 3, 8, 2, 128, P, P, 100, 100, 200, 200, (8 * 128, 128, 1),
        (2 * 128, 128, 1), (2 * 128, 128, 1), (8 * 128, 128, 1), 1, 0.088, o, None),
    "decode": lambda o: A.attn_fwd_decode_ex(
        P, P, P, P, None, A.ATTN_BF16, 2, 32, 8, 100, 128, contig(2, 32, 1, 128), contig(2, 8, 256, 128),
        contig(2, 8, 256, 128), contig(2, 32, 1, 128), 0.088, P, 1 << 30, o, None),
    "decode_paged": lambda o: A.attn_fwd_decode_paged_ex(
        P, P, P, P, None, A.ATTN_BF16, 2, 32, 8, 128, 100, 16, P, 64, 64, P, 1000, contig(2, 32, 1, 128),
        contig(100, 8, 16, 128), contig(100, 8, 16, 128), contig(2, 32, 1, 128), 0.088, P, 1 << 30, o, None),
    "bwd": lambda o: A.attn_bwd_ex(
        P, P, P, P, P, P, P, P, P, A.ATTN_BF16, 2, 8, 2, 64, 64, 128, contig(2, 8, 64, 128), contig(2, 2, 64, 128),
        contig(2, 2, 64, 128), contig(2, 8, 64, 128), contig(2, 8, 64, 128), contig(2, 8, 64, 128),
        contig(2, 2, 64, 128), contig(2, 2, 64, 128), 1, 0.088, o, P, 1 << 20, None),
    "cache_write": lambda o: A.kv_cache_write_ex(
        P, P, P, P, A.ATTN_BF16, 2, 8, 1, 128, 10, 256, contig(2, 8, 256, 128), contig(2, 8, 256, 128),
        contig(2, 8, 1, 128), contig(2, 8, 1, 128), o, None),
    "cache_write_paged": lambda o: A.kv_cache_write_paged_ex(
        P, P, P, P, A.ATTN_BF16, 2, 8, 1, 128, 100, 16, P, 64, 64, P, contig(100, 8, 16, 128),
        contig(100, 8, 16, 128), contig(2, 8, 1, 128), contig(2, 8, 1, 128), o, None),
}


@pytest.mark.parametrize("call", sorted(OPTION_CALLS))
@pytest.mark.parametrize("opts,code", [
    ((-2, -1, None), A.ATTN_ERR_INVALID_ARG),
    ((-1, -5, None), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, P + 2), A.ATTN_ERR_ALIGNMENT),
    ((3, 4, P + 1), A.ATTN_ERR_ALIGNMENT),
    ((-1, -1, None, -1.0, 0, 0), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, float("nan"), 0, 0), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, float("inf"), 0, 0), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 10000.0, 2, 0), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 0.0, 0, -1), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 0.0, 0, 65), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 10000.0, 0, 0, 2), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 10000.0, 0, 0, -1), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 0.0, 0, 0, 0, P + 4), A.ATTN_ERR_ALIGNMENT),
    ((-1, -1, None, 0.0, 0, 0, 0, None, 3), A.ATTN_ERR_INVALID_ARG),
    ((-1, -1, None, 0.0, 0, 0, 0, None, -1), A.ATTN_ERR_INVALID_ARG),
])
def test_option_errors(lib, call, opts, code):
    """Options are validated with the other arguments, before any CUDA call."""
    assert OPTION_CALLS[call](A.AttnOptions(*opts)) == code


@pytest.mark.parametrize("call", sorted(set(OPTION_CALLS) - {"prefill"}))
@pytest.mark.parametrize("kernel", [1, 2])
def test_prefill_kernel_choice_only_where_offered(lib, call, kernel):
    """Only the dense prefill (and the host-buffer call) take a kernel choice; the others accept only 0."""
    assert OPTION_CALLS[call](A.AttnOptions(-1, -1, None, 0.0, 0, 0, 0, None, kernel)) == A.ATTN_ERR_INVALID_ARG


def test_option_argument_errors_still_checked_first(lib):
    """With valid options the ordinary argument checks still apply."""
    assert A.attn_fwd_prefill_ex(None, P, P, P, None, A.ATTN_BF16, 2, 8, 2, 64, 64, 128, contig(2, 8, 64, 128),
                                 contig(2, 2, 64, 128), contig(2, 2, 64, 128), contig(2, 8, 64, 128), 1, 0.088,
                                 A.AttnOptions(16, -1, None), None) == A.ATTN_ERR_INVALID_ARG


def test_make_options():
    assert A.make_options() is None
    o = A.make_options(5, 7)
    assert (o.window_left, o.window_right, o.alibi_slopes) == (5, 7, None)
    import torch
    with pytest.raises(TypeError):
        A.make_options(alibi_slopes=torch.zeros(4))  # a CPU tensor is not a device pointer


def prefill_host(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=None, dtype=A.ATTN_BF16, B=2, H_q=8, H_kv=2, N_q=64, N_kv=64, D=128, causal=1,
             scale=0.088, opts=None, workspace=P, workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return A.attn_fwd_prefill_host(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(o=None), A.ATTN_ERR_INVALID_ARG),
    (dict(H_kv=3), A.ATTN_ERR_INVALID_ARG),
    (dict(N_kv=0), A.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), A.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(workspace=None), A.ATTN_ERR_WORKSPACE),
    (dict(workspace_bytes=1024), A.ATTN_ERR_WORKSPACE),
    (dict(workspace=P + 16), A.ATTN_ERR_ALIGNMENT),
    (dict(opts=A.AttnOptions(-3, -1, None)), A.ATTN_ERR_INVALID_ARG),
])
def test_prefill_host_argument_errors(lib, kw, code):
    assert prefill_host(**kw) == code


def test_prefill_host_workspace_size():
    n = A.attn_fwd_prefill_host_workspace_size(A.ATTN_BF16, 2, 8, 2, 64, 64, 128)
    q = 2 * 8 * 64 * 128 * 2
    kv = 2 * 2 * 64 * 128 * 2
    lse = 2 * 8 * 64 * 4
    assert n == 2 * q + 2 * kv + lse  # every region a multiple of 256 bytes here
    assert A.attn_fwd_prefill_host_workspace_size(A.ATTN_BF16, 2, 8, 3, 64, 64, 128) == 0
    assert A.attn_fwd_prefill_host_workspace_size(A.ATTN_BF16, 2, 8, 2, 64, 64, 80) == 0


def test_noalloc_decode_checks_arguments_before_the_scratch_size(lib):
    """A call that is both malformed and too large for the fixed scratch array
    reports the malformed argument, in the order attn_fwd_decode checks them;
    nothing is launched (the pointers are never used)."""
    B, Hq, Hkv, D, L = 64, 32, 8, 128, 8192
    q_s, c_s = (Hq * D, D, D, 1), (Hkv * L * D, L * D, D, 1)
    args = dict(q=P, k_cache=P, v_cache=P, o=P, lse=None, dtype=A.ATTN_BF16, B=B, H_q=Hq, H_kv=Hkv, cache_len=L,
                D=D, q_str=q_s, kc_str=c_s, vc_str=c_s, o_str=q_s, scale=0.088, stream=None)
    cases = [(dict(q=None), A.ATTN_ERR_INVALID_ARG), (dict(cache_len=0), A.ATTN_ERR_INVALID_ARG),
             (dict(scale=0.0), A.ATTN_ERR_INVALID_ARG), (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
             (dict(k_cache=BAD), A.ATTN_ERR_ALIGNMENT), (dict(lse=P + 2), A.ATTN_ERR_ALIGNMENT),
             (dict(kc_str=(Hkv * L * D, L * D, D, 2)), A.ATTN_ERR_ALIGNMENT),
             (dict(o_str=(Hq * D, -D, D, 1)), A.ATTN_ERR_INVALID_ARG)]
    for kw, code in cases:
        a = {**args, **kw}
        assert A.attn_fwd_decode_noalloc(**a) == code, kw
        ws = {k: v for k, v in a.items()}
        assert A.attn_fwd_decode(**ws, workspace=P, workspace_bytes=1 << 30) == code, kw


def test_make_options_rope_and_splits():
    o = A.make_options(rope_theta=10000.0, rope_interleaved=True, num_splits=3, rope_rotated_keys=True)
    assert (o.window_left, o.window_right, o.alibi_slopes) == (-1, -1, None)
    assert (o.rope_theta, o.rope_interleaved, o.num_splits, o.rope_rotated_keys) == (10000.0, 1, 3, 1)
    assert A.make_options(num_splits=0, rope_theta=0.0) is None


def test_options_struct_matches_the_header():
    """The ctypes struct has the fields, order and size of attn_options_t."""
    import ctypes
    names = [f[0] for f in A.AttnOptions._fields_]
    assert names == ["window_left", "window_right", "alibi_slopes", "rope_theta", "rope_interleaved", "num_splits",
                     "rope_rotated_keys", "kv_ranges", "prefill_kernel"]
    text = open(HEADER).read()
    body = text[text.index("typedef struct {"):text.index("} attn_options_t;")]
    declared = re.findall(r"\b([a-z_]+);", body)
    assert declared == names
    assert ctypes.sizeof(A.AttnOptions) == 48  # 4 + 4 + 8 + 4 + 4 + 4 + 4 + 8 + 4 (+ 4 padding) on LP64


def test_key_ranges_are_a_prefill_mask(lib):
    """Decode calls refuse key ranges with ATTN_ERR_UNSUPPORTED; the option checks run before any CUDA call."""
    opts = A.AttnOptions(-1, -1, None, 0.0, 0, 0, 0, P)
    assert OPTION_CALLS["decode"](opts) == A.ATTN_ERR_UNSUPPORTED
    assert OPTION_CALLS["decode_paged"](opts) == A.ATTN_ERR_UNSUPPORTED
