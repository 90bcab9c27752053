"""Calls on several CUDA streams at once share no hidden state.

Two different prefill problems, two decodes with their own workspaces and a
backward are enqueued on three streams without synchronising in between; each
result must equal, bit for bit, the same call made alone.
"""
from __future__ import annotations

import pytest
import torch

from attention_fa2_fwd_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fa2_fwd_gb300 as A
    A.lib()
    yield
    A.check_device_error()


def test_concurrent_streams_match_serial_calls():
    import attention_fa2_fwd_gb300 as A
    dev = torch.device("cuda", 0)
    p1 = [t.to(dev) for t in I.prefill_inputs(2, 16, 4, 1500, 1500, 128, "bf16", seed=1)]
    p2 = [t.to(dev) for t in I.prefill_inputs(1, 8, 8, 700, 2100, 64, "f16", seed=2)]
    kd, vd = (t.to(dev) for t in I.decode_stream(4, 8, 3000, 128, "bf16", seed=3))
    qd = I.decode_queries(4, 32, 128, [2999], "bf16", seed=3)[:, :, 0].to(dev)
    kd2, vd2 = (t.to(dev) for t in I.decode_stream(2, 8, 5000, 128, "bf16", seed=4))
    qd2 = I.decode_queries(2, 32, 128, [4999], "bf16", seed=4)[:, :, 0].to(dev)
    dout = torch.randn(p1[0].shape, generator=torch.Generator(device=dev).manual_seed(5), device=dev).to(torch.bfloat16)

    def run_all(streams):
        s1, s2, s3 = streams
        out = {}
        with torch.cuda.stream(s1):
            out["pre1"] = A.prefill(*p1, causal=True)
            out["dec1"] = A.decode(qd, kd, vd, 3000, workspace=A.decode_workspace(4, 32, 8, 128, dev))
        with torch.cuda.stream(s2):
            out["pre2"] = A.prefill(*p2, causal=False)
            out["dec2"] = A.decode(qd2, kd2, vd2, 4321, workspace=A.decode_workspace(2, 32, 8, 128, dev))
        with torch.cuda.stream(s3):
            o, lse = A.prefill(*p1, causal=True)
            out["bwd"] = A.backward(*p1, o, lse, dout, causal=True)
        torch.cuda.synchronize()
        return out

    main = torch.cuda.current_stream()
    serial = run_all((main, main, main))
    side = [torch.cuda.Stream() for _ in range(3)]
    for s in side:
        s.wait_stream(main)
    concurrent = run_all(side)
    for key in serial:
        for a, b in zip(serial[key], concurrent[key]):
            assert torch.equal(a, b), f"{key}: concurrent result differs from the serial one"
