"""A decode serving step captured once in a CUDA graph and replayed per token.

The paged calls take the per-request positions and lengths from device memory
and allocate nothing, so one captured step -- write the new token at
positions[b], lengths = positions + 1, decode, positions += 1 -- serves every
token: between replays only the staging buffers (new K/V, queries) are
refilled.  Each replay must match, bit for bit, the same calls made eagerly on
a second copy of the page pool, and the last step must match the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
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


def test_paged_decode_step_replayed_from_a_cuda_graph():
    import attention_fa2_fwd_gb300 as A
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, D, ps = 4, 32, 8, 128, 64
    start = torch.tensor([100, 37, 250, 0], dtype=torch.int32)
    steps, max_len = 12, 320
    max_pages = (max_len + ps - 1) // ps
    num_pages = B * max_pages + 3
    g = torch.Generator().manual_seed(31)
    table = torch.randperm(num_pages, generator=g)[:B * max_pages].view(B, max_pages).to(torch.int32)
    kp0 = torch.randn((num_pages, Hkv, ps, D), generator=g).to(torch.bfloat16)
    vp0 = torch.randn((num_pages, Hkv, ps, D), generator=g).to(torch.bfloat16)
    k_new = torch.randn((steps, B, Hkv, 1, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((steps, B, Hkv, 1, D), generator=g).to(torch.bfloat16)
    q_all = torch.randn((steps, B, Hq, D), generator=g).to(torch.bfloat16)

    def state():
        return {"kp": kp0.to(dev), "vp": vp0.to(dev), "pos": start.to(dev), "lens": torch.zeros(B, dtype=torch.int32, device=dev),
                "kn": torch.empty((B, Hkv, 1, D), dtype=torch.bfloat16, device=dev),
                "vn": torch.empty((B, Hkv, 1, D), dtype=torch.bfloat16, device=dev),
                "q": torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev),
                "o": torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty((B, Hq), dtype=torch.float32, device=dev),
                "ws": A.decode_workspace(B, Hq, Hkv, D, dev)}

    td = table.to(dev)

    def step(s):
        A.write_kv_cache_paged(s["kp"], s["vp"], s["kn"], s["vn"], td, s["pos"])
        torch.add(s["pos"], 1, out=s["lens"])
        A.decode_paged(s["q"], s["kp"], s["vp"], td, s["lens"], max_len, out=s["o"], lse_out=s["lse"],
                       workspace=s["ws"])
        s["pos"].add_(1)

    eager, graphed = state(), state()
    # one eager call first: the library's per-device setup happens outside the capture
    side = state()
    side["kn"].zero_(), side["vn"].zero_(), side["q"].zero_()
    step(side)
    torch.cuda.synchronize()

    capture_stream = torch.cuda.Stream()
    capture_stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(capture_stream):
        with torch.cuda.graph(graph, stream=capture_stream):
            step(graphed)
    torch.cuda.current_stream().wait_stream(capture_stream)
    torch.cuda.synchronize()
    # capturing ran nothing: reset the graphed state's positions
    graphed["pos"].copy_(start.to(dev))

    for t in range(steps):
        for s in (eager, graphed):
            s["kn"].copy_(k_new[t].to(dev))
            s["vn"].copy_(v_new[t].to(dev))
            s["q"].copy_(q_all[t].to(dev))
        step(eager)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(graphed["o"], eager["o"]), f"step {t}: O differs between graph and eager"
        assert torch.equal(graphed["lse"], eager["lse"]), f"step {t}: LSE differs between graph and eager"
    assert torch.equal(graphed["kp"], eager["kp"]) and torch.equal(graphed["vp"], eager["vp"])

    # the last step against the fp64 oracle, from the host copy of the pool
    kp_h, vp_h = np64(graphed["kp"]), np64(graphed["vp"])
    lens = (start + steps).numpy()
    o_ref, lse_ref = oracle.decode_paged(np64(q_all[steps - 1]), kp_h, vp_h, table.numpy(), lens, 1 / math.sqrt(D))
    assert_close(graphed["o"], o_ref, graphed["lse"], lse_ref, "graph replay vs oracle")


def test_backward_replayed_from_a_cuda_graph():
    """attn_bwd captured into a CUDA graph (after an earlier call on the device): its dK/dV kernel runs on the
    library's second stream, joined to the captured stream by events, and every replay reproduces the eager
    gradients bit for bit (the backward is deterministic); new inputs copied into the captured buffers give
    their own gradients."""
    import attention_fa2_fwd_gb300 as A
    from attention_fa2_fwd_gb300 import inputs as I
    B, Hq, Hkv, N, D = 1, 8, 2, 640, 128
    q, k, v = (t.cuda() for t in I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=90))
    dout = torch.randn_like(q)
    o, lse = A.prefill(q, k, v, causal=True)  # the first call on the device happens before the capture
    n = A.attn_bwd_workspace_size(B, Hq, N)
    ws = torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device="cuda")
    eager = A.backward(q, k, v, o, lse, dout, causal=True, workspace=ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            captured = A.backward(q, k, v, o, lse, dout, causal=True, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    A.check_device_error()
    for x, y in zip(captured, eager):
        assert torch.equal(x, y)
    # new inputs in the captured buffers
    q2, k2, v2 = (t.cuda() for t in I.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=91))
    o2, lse2 = A.prefill(q2, k2, v2, causal=True)
    g2 = torch.randn_like(q2)
    ref = A.backward(q2, k2, v2, o2, lse2, g2, causal=True)
    for dst, src in ((q, q2), (k, k2), (v, v2), (o, o2), (lse, lse2), (dout, g2)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    A.check_device_error()
    for x, y in zip(captured, ref):
        assert torch.equal(x, y)
