"""Run one kernel of the library on one synthetic case, for profiling and timing.

    python -m attention_fa2_fwd_gb300.run_case prefill [--B 2 --Hq 32 --Hkv 8 --N 8192 --D 128 --causal 1]
    python -m attention_fa2_fwd_gb300.run_case decode  [--B 64 --Hq 32 --Hkv 8 --L 8192 --D 128]
    python -m attention_fa2_fwd_gb300.run_case decode_paged [--page-size 16 --ragged 1 ...]
    python -m attention_fa2_fwd_gb300.run_case bwd     [prefill sizes; FLOPs counted as 2.5 x the forward]
    python -m attention_fa2_fwd_gb300.run_case varlen  [--B 16 --N 8192: B packed sequences, lengths uniform in
                                                        [N/8, N] (seeded), H_q=32 H_kv=8, causal by default]
    python -m attention_fa2_fwd_gb300.run_case cross   [--D 64|128: the cross-attention workload, B=4 H_q=16
                                                        H_kv=4 N_q=1024 N_kv=4096, (B,N,H,D) memory, non-causal]
    prefill / decode / decode_paged also take --window-left W and --alibi 1 (sliding window, ALiBi slopes)
    prefill / varlen / cross / decode / decode_paged / bwd take --rope THETA [--rope-interleaved 1] (rotary
    embeddings; prefill and bwd also --rope-rotated-keys 1)
    decode / decode_paged take --graph 1: the step (cache write of one token + decode) captured once in a
    CUDA graph and replayed, against the same calls launched one by one

Inputs are seeded N(0,1) bf16 tensors drawn on the device.  Each iteration is
timed with CUDA events on the launching stream (L2 flushed by a 256 MiB write
before each); the per-iteration times and the derived TFLOPS or GB/s are
printed.  Exits non-zero if a call or the device error word reports a failure.
"""
from __future__ import annotations

import argparse
import statistics

import torch

import attention_fa2_fwd_gb300 as A


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=("prefill", "decode", "decode_paged", "bwd", "cross", "varlen"))
    ap.add_argument("--B", type=int)
    ap.add_argument("--Hq", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--L", type=int, default=8192)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--causal", type=int, default=1)
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--dtype", choices=("bf16", "f16"), default="bf16")
    ap.add_argument("--page-size", type=int, default=16)
    ap.add_argument("--ragged", type=int, default=0, help="decode_paged: lengths uniform in [L/2, L]")
    ap.add_argument("--window-left", type=int, default=-1, help="sliding window: keys i - W .. i (-1: none)")
    ap.add_argument("--alibi", type=int, default=0, help="ALiBi slopes 2^(-8 (h + 1) / H_q)")
    ap.add_argument("--graph", type=int, default=0, help="decode: time a one-token serving step, eager vs CUDA graph")
    ap.add_argument("--rope", type=float, default=0.0, help="rotary embeddings of this base (0: none)")
    ap.add_argument("--rope-interleaved", type=int, default=0, help="rotary pairs (2c, 2c+1) instead of (c, c+D/2)")
    ap.add_argument("--rope-rotated-keys", type=int, default=0, help="prefill, bwd: keys given already rotated")
    ap.add_argument("--num-splits", type=int, default=0, help="decode: force at most this many KV splits (0: auto)")
    ap.add_argument("--prefill-kernel", type=int, default=0,
                    help="prefill / cross: 0 automatic, 1 one-CTA kernel, 2 CTA-pair kernel")
    a = ap.parse_args()
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(42)

    def randn(*s):
        return torch.randn(s, generator=g, device=dev, dtype=torch.float32).to(dt)

    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    wl = a.window_left
    rope = dict(rope_theta=a.rope, rope_interleaved=bool(a.rope_interleaved))
    rope_pre = dict(rope, rope_rotated_keys=bool(a.rope_rotated_keys), prefill_kernel=a.prefill_kernel)
    slopes = (torch.tensor([2.0 ** (-8.0 * (h + 1) / a.Hq) for h in range(a.Hq)], dtype=torch.float32, device=dev)
              if a.alibi else None)
    if a.kind == "prefill":
        B = a.B or 2
        q, k, v = randn(B, a.Hq, a.N, a.D), randn(B, a.Hkv, a.N, a.D), randn(B, a.Hkv, a.N, a.D)
        o = torch.empty_like(q)
        lse = torch.empty((B, a.Hq, a.N), dtype=torch.float32, device=dev)
        # FLOPs of the visible (query, key) pairs: 4 D per pair (Q K^T and P V)
        i = torch.arange(a.N, dtype=torch.float64)
        hi = i if a.causal else torch.full_like(i, a.N - 1)
        lo = torch.clamp(i - wl, min=0) if wl >= 0 else torch.zeros_like(i)
        pairs = float((hi - lo + 1).sum()) if (a.causal or wl >= 0) else float(a.N) * a.N
        work = 4.0 * B * a.Hq * a.D * pairs if (a.causal or wl >= 0) else 4.0 * B * a.Hq * a.N * a.N * a.D

        def call():
            A.prefill(q, k, v, causal=bool(a.causal), out=o, lse_out=lse, window=(wl, -1), alibi_slopes=slopes,
                      **rope_pre)
        unit, scale = "TFLOPS", 1e12
    elif a.kind == "varlen":
        B = a.B or 16
        lens = torch.randint(a.N // 8, a.N + 1, (B,), generator=torch.Generator().manual_seed(11)).tolist()
        tq = sum(lens)
        q, k, v = randn(tq, a.Hq, a.D), randn(tq, a.Hkv, a.D), randn(tq, a.Hkv, a.D)
        cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((a.Hq, tq), dtype=torch.float32, device=dev)
        pairs = sum(n * (n + 1) // 2 if a.causal else n * n for n in lens)
        work = 4.0 * a.Hq * a.D * pairs
        print(f"varlen: {B} sequences, {tq} tokens, lengths {min(lens)}..{max(lens)}")

        def call():
            A.prefill_varlen(q, k, v, cu, cu, max(lens), max(lens), causal=bool(a.causal), out=o, lse_out=lse,
                             window=(a.window_left, -1), alibi_slopes=slopes, **rope)
        unit, scale = "TFLOPS", 1e12
    elif a.kind == "cross":
        import attention_fa2_fwd_gb300.inputs as I
        w = I.CROSS[a.D]
        g2 = torch.Generator(device=dev).manual_seed(42)
        # the workload's distributions (Q ~ N(0,1), K ~ N(0,2), V ~ U(-1,1)), drawn on the device, in its layout
        q = I.to_layout(torch.randn((w.B, w.Hq, w.Nq, w.D), generator=g2, device=dev).to(dt), w.layout)
        k = I.to_layout((torch.randn((w.B, w.Hkv, w.Nkv, w.D), generator=g2, device=dev) * 2 ** 0.5).to(dt), w.layout)
        v = I.to_layout((torch.rand((w.B, w.Hkv, w.Nkv, w.D), generator=g2, device=dev) * 2 - 1).to(dt), w.layout)
        o = I.to_layout(torch.empty_like(q), w.layout)
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        work = w.flops

        def call():
            A.prefill(q, k, v, causal=False, out=o, lse_out=lse, prefill_kernel=a.prefill_kernel, **rope)
        unit, scale = "TFLOPS", 1e12
    elif a.kind == "bwd":
        B = a.B or 2
        q, k, v = randn(B, a.Hq, a.N, a.D), randn(B, a.Hkv, a.N, a.D), randn(B, a.Hkv, a.N, a.D)
        dout = randn(B, a.Hq, a.N, a.D)
        # the forward's masks and rotary embedding, passed to the backward too
        mk = dict(window=(wl, -1), alibi_slopes=slopes, rope_theta=a.rope, rope_interleaved=bool(a.rope_interleaved),
                  rope_rotated_keys=bool(a.rope_rotated_keys))
        o, lse = A.prefill(q, k, v, causal=bool(a.causal), **mk)
        nbytes = A.attn_bwd_ex_workspace_size(B, a.Hq, a.Hkv, a.N, a.N, a.D,
                                              A.make_options(rope_theta=a.rope, rope_rotated_keys=bool(a.rope_rotated_keys)))
        ws = torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32, device=dev)
        # five matrix products of the forward's size (S, dP, dV, dK, dQ) over the visible pairs: 2.5 x its FLOPs
        i = torch.arange(a.N, dtype=torch.float64)
        hi = i if a.causal else torch.full_like(i, a.N - 1)
        lo = torch.clamp(i - wl, min=0) if wl >= 0 else torch.zeros_like(i)
        work = 2.5 * 4.0 * B * a.Hq * a.D * float((hi - lo + 1).sum())

        def call():
            A.backward(q, k, v, o, lse, dout, causal=bool(a.causal), workspace=ws, **mk)
        unit, scale = "TFLOPS", 1e12
    elif a.kind == "decode_paged":
        B = a.B or 64
        ps = a.page_size
        max_pages = (a.L + ps - 1) // ps
        num_pages = B * max_pages
        kp, vp = randn(num_pages, a.Hkv, ps, a.D), randn(num_pages, a.Hkv, ps, a.D)
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(7)).to(torch.int32)
        table = perm.view(B, max_pages).to(dev)
        if a.ragged:
            lens = torch.randint(a.L // 2, a.L + 1, (B,), generator=torch.Generator().manual_seed(8))
        else:
            lens = torch.full((B,), a.L)
        lens = lens.to(torch.int32).to(dev)
        qd = randn(B, a.Hq, a.D)
        od = torch.empty_like(qd)
        lsed = torch.empty((B, a.Hq), dtype=torch.float32, device=dev)
        ws = A.decode_workspace(B, a.Hq, a.Hkv, a.D, dev)
        span = lens.clamp(max=wl + 1) if wl >= 0 else lens
        work = 2.0 * a.Hkv * a.D * 2 * float(span.sum())

        def call():
            A.decode_paged(qd, kp, vp, table, lens, a.L, out=od, lse_out=lsed, workspace=ws, window_left=wl,
                           alibi_slopes=slopes, **rope)
        unit, scale = "GB/s", 1e9
    else:
        B = a.B or 64
        kc, vc = randn(B, a.Hkv, a.L, a.D), randn(B, a.Hkv, a.L, a.D)
        qd = randn(B, a.Hq, a.D)
        od = torch.empty_like(qd)
        lsed = torch.empty((B, a.Hq), dtype=torch.float32, device=dev)
        ws = A.decode_workspace(B, a.Hq, a.Hkv, a.D, dev)
        if a.num_splits:
            ws = torch.empty(B * a.Hq * a.num_splits * (a.D + 1), dtype=torch.float32, device=dev)
        work = 2.0 * B * a.Hkv * (min(a.L, wl + 1) if wl >= 0 else a.L) * a.D * 2

        def call():
            A.decode(qd, kc, vc, a.L, out=od, lse_out=lsed, workspace=ws, window_left=wl, alibi_slopes=slopes,
                     num_splits=a.num_splits, **rope)
        unit, scale = "GB/s", 1e9
    if a.graph and a.kind in ("decode", "decode_paged"):
        # one serving step: write one new token per request, then decode
        kn = randn(B, a.Hkv, 1, a.D)
        vn = randn(B, a.Hkv, 1, a.D)
        if a.kind == "decode":
            pos = a.L - 1

            def serve():
                A.write_kv_cache(kc, vc, kn, vn, pos, **rope)
                call()
        else:
            positions = (lens - 1).clamp(min=0)

            def serve():
                A.write_kv_cache_paged(kp, vp, kn, vn, table, positions, **rope)
                call()
        serve()
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                serve()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        reps = 50
        for label, fn in (("eager", serve), ("graph", graph.replay)):
            meds = []
            for _ in range(a.iters):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
                meds.append(e0.elapsed_time(e1) / reps)
            print(f"{a.kind} step ({label}, {reps} back to back): median_ms={statistics.median(meds):.4f}")
        A.check_device_error()
        return
    times = []
    for _ in range(a.iters):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    A.check_device_error()
    med = statistics.median(times)
    print(f"{a.kind}: times_ms={[round(t, 4) for t in times]} median_ms={med:.4f} "
          f"{unit}={work / (med * 1e-3) / scale:.1f}")


if __name__ == "__main__":
    main()
