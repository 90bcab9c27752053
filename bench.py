"""Benchmark of the fused attention forward hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * prefill: causal GQA attention, B=2, H_q=32, H_kv=8, N=8192, D=128, bf16,
    with LSE (attn_fwd_prefill);
  * one decode step: B=64, H_q=32, H_kv=8, D=128, bf16 -- the new token is
    written to the preallocated cache (kv_cache_write) and attends to the
    8192 cached positions (attn_fwd_decode).

Every kernel is timed with CUDA events on the stream it is launched on; the
L2 cache (129 MB) is flushed by a 256 MiB write between timed kernels, outside
the event pairs.  The JSON line reports prefill TFLOPS (4*B*H_q*N^2*D / 2 per
forward) as ``value`` and decode K/V bytes per second (2*B*H_kv*L*D*2 bytes
per step) beside it, each against the measured peaks in MEASURED_PEAKS.json.

``--impl reference`` times the CPU fp64 oracle instead (host cores, a bounded
sample of query rows of the same prefill workload per step).

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path needs no exchange between GPUs); times are reduced with a MAX over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill TFLOPS & decode KV GB/s on 1 GB300 (fraction of peak), oracle-matched"
FLUSH_BYTES = 256 << 20
PREFILL = dict(B=2, Hq=32, Hkv=8, N=8192, D=128, causal=True)
DECODE = dict(B=64, Hq=32, Hkv=8, L=8192, D=128)
WORKLOAD = ("gqa_causal_prefill_b2_hq32_hkv8_n8192_d128_bf16"
            " + decode_step_b64_hq32_hkv8_l8192_d128_bf16 (kv_cache_write + attn_fwd_decode)")
PROFILES = os.path.join(ROOT, "profiles")


def prefill_flops(B, Hq, N, D, causal, **_):
    f = 4.0 * B * Hq * N * N * D
    return f / 2 if causal else f


def decode_bytes(B, Hkv, L, D, **_):
    return 2 * B * Hkv * L * D * 2


def prefill_exps(B, Hq, N, causal, **_):
    """Exponentials the softmax needs: one per attended (query, key) pair."""
    return B * Hq * (N * (N + 1) / 2 if causal else N * N)


# ex2.approx.f32 lanes per clock per SM on this part (a stand-alone issue-rate
# micro-benchmark); times the SM count and the SM clock it is the exp peak.
EX2_LANES_PER_CLK_SM = 32


def nvtx_ranges():
    """(push, pop) for NVTX ranges that name the bench's phases in a timeline
    profiler; no-ops where NVTX is unavailable.  They cost the host ~1 us and
    do not touch the device."""
    try:
        from torch.cuda import nvtx
        nvtx.range_push("probe")
        nvtx.range_pop()
        return nvtx.range_push, nvtx.range_pop
    except Exception:  # noqa: BLE001 -- any failure just disables the ranges
        return (lambda _name: None), (lambda: None)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    import hashlib
    path = os.path.join(PROFILES, "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel]
        src = os.path.join(ROOT, "attention_fa2_fwd_gb300", "csrc", t["source"])
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != t["source_sha256"]:
                return None
        return float(t["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def reduce_max(values, world, device):
    """Element-wise MAX of per-rank timings over all ranks (identity for one process)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_throughput(units_per_rank, world, steps, max_ms_total):
    """Whole-job rate: units every rank processed in `steps` steps over the slowest rank's time (ms)."""
    return world * units_per_rank * steps / (max_ms_total * 1e-3)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CUDA arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import attention_fa2_fwd_gb300 as A

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    A.lib()
    stream = torch.cuda.current_stream(dev)
    P, Dc = PREFILL, DECODE
    gen = torch.Generator(device=dev).manual_seed(42 + rank)

    def randn(*shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    q = randn(P["B"], P["Hq"], P["N"], P["D"])
    k = randn(P["B"], P["Hkv"], P["N"], P["D"])
    v = randn(P["B"], P["Hkv"], P["N"], P["D"])
    o = torch.empty_like(q)
    lse = torch.empty((P["B"], P["Hq"], P["N"]), dtype=torch.float32, device=dev)
    # Decode: a cache holding L-1 tokens; each step writes token L-1 and attends to all L.
    kc = randn(Dc["B"], Dc["Hkv"], Dc["L"], Dc["D"])
    vc = randn(Dc["B"], Dc["Hkv"], Dc["L"], Dc["D"])
    kn = randn(Dc["B"], Dc["Hkv"], 1, Dc["D"])
    vn = randn(Dc["B"], Dc["Hkv"], 1, Dc["D"])
    qd = randn(Dc["B"], Dc["Hq"], Dc["D"])
    od = torch.empty_like(qd)
    lsed = torch.empty((Dc["B"], Dc["Hq"]), dtype=torch.float32, device=dev)
    ws = A.decode_workspace(Dc["B"], Dc["Hq"], Dc["Hkv"], Dc["D"], dev)
    splits = A.attn_decode_splits(Dc["B"], Dc["Hq"], Dc["Hkv"], Dc["L"], Dc["D"])
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def do_prefill():
        A.prefill(q, k, v, causal=True, out=o, lse_out=lse)

    def do_decode():
        A.write_kv_cache(kc, vc, kn, vn, Dc["L"] - 1)
        A.decode(qd, kc, vc, Dc["L"], out=od, lse_out=lsed, workspace=ws)

    range_push, range_pop = nvtx_ranges()

    R = args.passes_per_step

    def one_pass(evs=None):
        flush.zero_()
        if evs:
            evs[0].record(stream)
        range_push("prefill")
        do_prefill()
        range_pop()
        if evs:
            evs[1].record(stream)
        flush.zero_()
        if evs:
            evs[2].record(stream)
        range_push("decode_step")
        do_decode()
        range_pop()
        if evs:
            evs[3].record(stream)

    def step(evs=None):
        # One step: R passes of the whole path over the same batch, the L2 cache
        # flushed before every timed kernel group.
        for r in range(R):
            one_pass(evs[r] if evs else None)

    for _ in range(args.warmup):
        step()
    A.check_device_error()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
        for _ in range(max(args.warmup, 10)):  # keep the GPU busy while the sampler starts
            step()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(R)] for _ in range(args.steps)]
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    r0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    r1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    A.check_device_error()
    pre_ms = [e[0].elapsed_time(e[1]) for se in evs for e in se]
    dec_ms = [e[2].elapsed_time(e[3]) for se in evs for e in se]
    region_ms = r0.elapsed_time(r1)
    sum_pre, sum_dec, region_ms = reduce_max([sum(pre_ms), sum(dec_ms), region_ms], world, dev)

    flops = prefill_flops(**P)
    kvb = decode_bytes(**Dc)
    n_pass = args.steps * R
    value = aggregate_throughput(flops, world, n_pass, sum_pre) / 1e12
    decode_gbs = aggregate_throughput(kvb, world, n_pass, sum_dec) / 1e9

    # End to end through the public API with host buffers (pinned), copies inside the timed region:
    # attn_fwd_prefill_host pipelines the host-to-device copies, the compute and the copies back.
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    code = A.ATTN_BF16
    ws_bytes = A.attn_fwd_prefill_host_workspace_size(code, P["B"], P["Hq"], P["Hkv"], P["N"], P["N"], P["D"])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(P["D"])

    def host_call():
        st = A.attn_fwd_prefill_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr(),
                                     code, P["B"], P["Hq"], P["Hkv"], P["N"], P["N"], P["D"], 1, scale, None,
                                     ws.data_ptr(), ws_bytes, stream.cuda_stream)
        if st != A.ATTN_OK:
            raise RuntimeError(f"attn_fwd_prefill_host failed: {A.attn_status_string(st)}")
    n_e2e = max(3, min(args.steps, 10))
    for _ in range(2):
        host_call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        host_call()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max([e0.elapsed_time(e1) / n_e2e], world, dev)[0]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    e2e = {"value": round(aggregate_throughput(flops, world, 1, e2e_ms) / 1e12, 2), "unit": "TFLOPS",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_call": round(e2e_ms, 4),
           "path": "pinned host Q,K,V -> attn_fwd_prefill_host (copies pipelined with the compute) -> host O,LSE"}

    if rank != 0:
        return None, None
    peaks = load_peaks()
    pre_avg = sum_pre / n_pass
    dec_avg = sum_dec / n_pass
    ach = flops / (pre_avg * 1e-3) / 1e12
    ach_d = kvb / (dec_avg * 1e-3) / 1e9
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    exp_rate = prefill_exps(**P) / (pre_avg * 1e-3)
    exp_peak = EX2_LANES_PER_CLK_SM * sms * clk_mhz * 1e6
    tr = profiled_traffic("prefill_fwd")
    tr_d = profiled_traffic("decode_split")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round((sum_pre + sum_dec) / args.steps, 4),
        "passes_per_step": R,
        "ms_per_pass": round((sum_pre + sum_dec) / n_pass, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, generated on device)",
        "config": {"workload": WORKLOAD, "prefill": P, "decode": Dc,
                   "l2": "flushed by a 256 MiB write before every timed kernel group (outside the event pairs)",
                   "step": f"{R} passes of the whole path (prefill + decode step) over the same batch",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "decode_splits": splits},
        "prefill_ms": round(pre_avg, 4),
        "prefill_ms_median": round(statistics.median(pre_ms), 4) if world == 1 else None,
        "prefill_ms_std": round(statistics.pstdev(pre_ms), 4) if world == 1 else None,
        "decode_ms_std": round(statistics.pstdev(dec_ms), 4) if world == 1 else None,
        "exp_rate": {"value": round(exp_rate / 1e12, 3), "unit": "Texp/s", "exps_per_step": prefill_exps(**P),
                     "peak": round(exp_peak / 1e12, 3), "frac": round(exp_rate / exp_peak, 4),
                     "peak_source": f"ex2 {EX2_LANES_PER_CLK_SM} lanes/clk/SM x {sms} SMs x {clk_mhz:.0f} MHz (secondary: the tensor pipe bounds the prefill)"},
        "decode": {"value": round(decode_gbs, 1), "unit": "GB/s", "ms_per_step": round(dec_avg, 4),
                   "kv_bytes_per_step": kvb, "kernels": "kv_cache_write + decode_split" + (" + decode_merge" if splits > 1 else "")},
        "region_ms_incl_flush": round(region_ms, 3),
        # time x median SM clock under load (ms x MHz = thousands of SM cycles): comparable across clocks
        "sm_kcycles": {"prefill": round(pre_avg * clk_mhz, 1), "decode_step": round(dec_avg * clk_mhz, 1),
                       "per_step": round((sum_pre + sum_dec) / args.steps * clk_mhz, 1), "sm_mhz": clk_mhz},
        "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": tr,
                     "peak_source": f"{peaks['source']} bf16 dense (burst)", "kernel": "prefill_fwd"},
        "roofline_decode": {"bound": "hbm", "achieved": round(ach_d, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(ach_d / peaks["hbm_gbs"], 4), "traffic": tr_d,
                            "peak_source": f"{peaks['source']} HBM copy", "kernel": "decode_split"},
        "e2e": e2e,
        "gpu_launches": n_pass * (1 + 1 + (2 if splits > 1 else 1)),
        "clocks": clocks,
    }
    if args.also and world == 1:
        sampler2 = ClockSampler(local_rank)
        sampler2.start()
        line["also_measured"] = {"results": measure_also(A, dev, stream, flush, peaks),
                                 "how": "CUDA events on the launching stream, 3 warm-ups, median of 10 "
                                        "(backward 5), L2 flushed before each timed call",
                                 "clocks": sampler2.stop()}
    data = {"prefill": (q, k, v, o, lse), "decode": (qd, kc, vc, od, lsed, Dc["L"])}
    return line, data


# --------------------------------------------------------------------------- secondary workloads

def measure_also(A, dev, stream, flush, peaks, reps=10):
    """Event-timed secondary measurements of the same library (rank 0, one GPU):
    the D=64 causal prefill, the cross-attention workload at D=128 and 64,
    the headline prefill on the CTA-pair kernel, the causal prefill with rotary embeddings (keys given rotated, and rotated
    in the kernel), the backward pass, and the B=2 one-token decode step
    replayed from a CUDA graph.  Each kernel is timed with CUDA events on the
    launching stream after 3 warm-ups, the L2 flushed before every timed call;
    the median is reported against the measured peaks.  Returns a dict."""
    import torch

    import attention_fa2_fwd_gb300.inputs as I

    g = torch.Generator(device=dev).manual_seed(7)

    def randn(*shape, std=1.0):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std).to(torch.bfloat16)

    def timed(fn, n=reps):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def tf_line(name, flops, ms):
        v = flops / (ms * 1e-3) / 1e12
        return {"workload": name, "value": round(v, 1), "unit": "TFLOPS", "ms": round(ms, 4),
                "frac": round(v / peaks["bf16_tflops"], 4)}

    out = []
    P = PREFILL
    # D=64 causal prefill, otherwise the headline sizes
    q, k, v = randn(P["B"], P["Hq"], P["N"], 64), randn(P["B"], P["Hkv"], P["N"], 64), randn(P["B"], P["Hkv"], P["N"], 64)
    o = torch.empty_like(q)
    ms = timed(lambda: A.prefill(q, k, v, causal=True, out=o))
    out.append(tf_line("gqa_causal_prefill_b2_hq32_hkv8_n8192_d64_bf16", prefill_flops(P["B"], P["Hq"], P["N"], 64, True), ms))
    del q, k, v, o
    # cross-attention workload: (B,N,H,D) memory, K variance 2, V ~ U(-1,1)
    for D in (128, 64):
        w = I.CROSS[D]
        q = I.to_layout(randn(w.B, w.Hq, w.Nq, D), w.layout)
        k = I.to_layout(randn(w.B, w.Hkv, w.Nkv, D, std=2 ** 0.5), w.layout)
        v = I.to_layout(((torch.rand((w.B, w.Hkv, w.Nkv, D), generator=g, device=dev) * 2 - 1).to(torch.bfloat16)),
                        w.layout)
        o = I.to_layout(torch.empty_like(q), w.layout)
        ms = timed(lambda: A.prefill(q, k, v, causal=False, out=o))
        out.append(tf_line(w.name, w.flops, ms))
    # rotary embeddings on the headline workload
    q, k, v = randn(P["B"], P["Hq"], P["N"], P["D"]), randn(P["B"], P["Hkv"], P["N"], P["D"]), randn(P["B"], P["Hkv"], P["N"], P["D"])
    o = torch.empty_like(q)
    lse = torch.empty((P["B"], P["Hq"], P["N"]), dtype=torch.float32, device=dev)
    fl = prefill_flops(**P)
    # the CTA-pair kernel on the headline workload (the library's automatic choice is the one-CTA kernel)
    ms = timed(lambda: A.prefill(q, k, v, causal=True, out=o, lse_out=lse, prefill_kernel=2))
    out.append(tf_line("gqa_causal_prefill_n8192_d128, CTA-pair kernel", fl, ms))
    ms = timed(lambda: A.prefill(q, k, v, causal=True, out=o, lse_out=lse, rope_theta=10000.0, rope_rotated_keys=True))
    out.append(tf_line("gqa_causal_prefill_n8192_d128 + RoPE (keys given rotated)", fl, ms))
    ms = timed(lambda: A.prefill(q, k, v, causal=True, out=o, lse_out=lse, rope_theta=10000.0))
    out.append(tf_line("gqa_causal_prefill_n8192_d128 + RoPE (keys rotated in the kernel)", fl, ms))
    # backward of the headline workload (2.5x the forward's FLOPs: S, dP, dV, dK, dQ products)
    A.prefill(q, k, v, causal=True, out=o, lse_out=lse)
    dout = randn(P["B"], P["Hq"], P["N"], P["D"])
    ws = torch.empty((A.attn_bwd_workspace_size(P["B"], P["Hq"], P["N"]) + 3) // 4, dtype=torch.float32, device=dev)
    ms = timed(lambda: A.backward(q, k, v, o, lse, dout, causal=True, workspace=ws), n=max(3, reps // 2))
    out.append(tf_line("gqa_causal_backward_b2_hq32_hkv8_n8192_d128_bf16 (2.5x forward FLOPs)", 2.5 * fl, ms))
    # the same backward with rotary embeddings (Q and K rotated into the workspace, dQ and dK turned back)
    A.prefill(q, k, v, causal=True, out=o, lse_out=lse, rope_theta=10000.0)
    nb = A.attn_bwd_ex_workspace_size(P["B"], P["Hq"], P["Hkv"], P["N"], P["N"], P["D"], A.make_options(rope_theta=10000.0))
    ws = torch.empty((nb + 15) // 16 * 4, dtype=torch.float32, device=dev)
    ms = timed(lambda: A.backward(q, k, v, o, lse, dout, causal=True, workspace=ws, rope_theta=10000.0),
               n=max(3, reps // 2))
    out.append(tf_line("gqa_causal_backward_n8192_d128 + RoPE (2.5x forward FLOPs)", 2.5 * fl, ms))
    del q, k, v, o, lse, dout, ws
    # variable-length prefill: 16 packed causal sequences, lengths uniform in [N/8, N] (seeded)
    lens = torch.randint(P["N"] // 8, P["N"] + 1, (16,), generator=torch.Generator().manual_seed(11)).tolist()
    tq = sum(lens)
    q, k, v = randn(tq, P["Hq"], P["D"]), randn(tq, P["Hkv"], P["D"]), randn(tq, P["Hkv"], P["D"])
    cu = torch.tensor([0] + torch.tensor(lens).cumsum(0).tolist(), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ms = timed(lambda: A.prefill_varlen(q, k, v, cu, cu, max(lens), max(lens), causal=True, out=o,
                                        return_lse=False))
    pairs = sum(n * (n + 1) // 2 for n in lens)
    out.append(tf_line(f"varlen_causal_prefill_16_seqs_{min(lens)}..{max(lens)}_tokens_hq32_hkv8_d128 "
                       f"(FLOPs over the visible pairs)", 4.0 * P["Hq"] * P["D"] * pairs, ms))
    del q, k, v, o
    # paged decode: B=64 requests of 8192 cached tokens in 16-token pages of a shuffled pool
    Dc = DECODE
    ps = 16
    max_pages = Dc["L"] // ps
    kp, vp = randn(Dc["B"] * max_pages, Dc["Hkv"], ps, Dc["D"]), randn(Dc["B"] * max_pages, Dc["Hkv"], ps, Dc["D"])
    table = torch.randperm(Dc["B"] * max_pages, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    table = table.view(Dc["B"], max_pages).to(dev)
    lens_d = torch.full((Dc["B"],), Dc["L"], dtype=torch.int32, device=dev)
    qd = randn(Dc["B"], Dc["Hq"], Dc["D"])
    od = torch.empty_like(qd)
    wsd = A.decode_workspace(Dc["B"], Dc["Hq"], Dc["Hkv"], Dc["D"], dev)
    ms = timed(lambda: A.decode_paged(qd, kp, vp, table, lens_d, Dc["L"], out=od, return_lse=False, workspace=wsd))
    kvb = decode_bytes(Dc["B"], Dc["Hkv"], Dc["L"], Dc["D"])
    out.append({"workload": "paged_decode_b64_hq32_hkv8_l8192_d128_bf16, 16-token pages, shuffled pool",
                "value": round(kvb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms": round(ms, 4),
                "frac": round(kvb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)})
    del kp, vp, table, lens_d, qd, od, wsd
    # B=2 one-token decode step (cache write + decode) replayed from a CUDA graph
    Dc = dict(DECODE, B=2)
    kc, vc = randn(2, Dc["Hkv"], Dc["L"], Dc["D"]), randn(2, Dc["Hkv"], Dc["L"], Dc["D"])
    kn, vn = randn(2, Dc["Hkv"], 1, Dc["D"]), randn(2, Dc["Hkv"], 1, Dc["D"])
    qd = randn(2, Dc["Hq"], Dc["D"])
    od = torch.empty_like(qd)
    wsd = A.decode_workspace(2, Dc["Hq"], Dc["Hkv"], Dc["D"], dev)

    def step():
        A.write_kv_cache(kc, vc, kn, vn, Dc["L"] - 1)
        A.decode(qd, kc, vc, Dc["L"], out=od, return_lse=False, workspace=wsd)
    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    n_rep = 50
    ms = timed(lambda: [graph.replay() for _ in range(n_rep)]) / n_rep
    kvb = decode_bytes(2, Dc["Hkv"], Dc["L"], Dc["D"])
    out.append({"workload": "decode_step_b2_hq32_hkv8_l8192_d128_bf16, CUDA graph replay (50 steps back to back)",
                "value": round(kvb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "us_per_step": round(ms * 1e3, 2),
                "frac": round(kvb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)})
    # the same step replayed once per rep with L2 flushed before it (the 67 MB cache read from HBM)
    ms = timed(graph.replay)
    out.append({"workload": "decode_step_b2_hq32_hkv8_l8192_d128_bf16, CUDA graph replay, L2 flushed before each step",
                "value": round(kvb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "us_per_step": round(ms * 1e3, 2),
                "frac": round(kvb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)})
    A.check_device_error()
    return out


# --------------------------------------------------------------------------- oracle (CPU)

def oracle_sample(rows_per_step: int, seed: int):
    """A bounded sample of the prefill workload for the CPU oracle: query rows of one (b, h)."""
    import numpy as np
    import torch

    P = PREFILL
    g = torch.Generator().manual_seed(seed)
    # One (b, h) of the workload: Q rows of head h and K/V of its kv head, N(0,1) bf16.
    q = torch.randn((1, 1, P["N"], P["D"]), generator=g).to(torch.bfloat16).float().numpy()
    k = torch.randn((1, 1, P["N"], P["D"]), generator=g).to(torch.bfloat16).float().numpy()
    v = torch.randn((1, 1, P["N"], P["D"]), generator=g).to(torch.bfloat16).float().numpy()
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, P["N"], size=rows_per_step)
    sel = np.stack([np.zeros_like(rows), np.zeros_like(rows), rows], axis=1)
    flops = float(np.sum(4.0 * P["D"] * (rows + 1)))  # causal: row i attends to i+1 keys
    return q, k, v, sel, flops


def cpu_baseline_leg(target_s: float, data, seed=0):
    """The CPU-baseline leg: the oracle, as it stands, timed on the host cores on
    a bounded sample of the bench's own prefill workload -- growing batches of
    query rows of single (b, h) heads of the very Q, K, V the GPU was timed on,
    until about target_s seconds.  The oracle rows are then also compared with
    the O and LSE the timed kernels wrote (and a few batch entries of the decode
    step with its O and LSE), so the bench line says whether the outputs it
    timed match the oracle.  Returns the cpu_baseline record."""
    import numpy as np
    import torch

    import oracle
    cores = oracle.default_threads()
    P = PREFILL
    q, k, v, o, lse = data["prefill"]
    g = P["Hq"] // P["Hkv"]
    scale = 1 / math.sqrt(P["D"])
    rng = np.random.default_rng(seed)

    def f64(t):
        return t.detach().double().cpu().numpy()

    rows, total_f, total_t, total_rows = 64, 0.0, 0.0, 0
    o_err, l_err, o_sum, n_el, heads = 0.0, 0.0, 0.0, 0, 0
    while total_t < target_s:
        b, h = int(rng.integers(P["B"])), int(rng.integers(P["Hq"]))
        qh, kh, vh = (f64(t[b:b + 1, x:x + 1]) for t, x in ((q, h), (k, h // g), (v, h // g)))
        sel_i = rng.integers(0, P["N"], size=rows)
        sel = np.stack([np.zeros_like(sel_i), np.zeros_like(sel_i), sel_i], axis=1)
        t0 = time.perf_counter()
        o_ref, l_ref = oracle.attention_rows(qh, kh, vh, True, scale, sel, nthreads=cores)
        total_t += time.perf_counter() - t0
        total_f += float(np.sum(4.0 * P["D"] * (sel_i + 1)))
        total_rows += rows
        heads += 1
        idx = torch.as_tensor(sel_i, dtype=torch.long, device=o.device)
        og = f64(o[b, h].index_select(0, idx))
        lg = f64(lse[b, h].index_select(0, idx))
        e = np.abs(og - o_ref)
        o_err = max(o_err, float(e.max()))
        o_sum += float(e.sum())
        n_el += e.size
        l_err = max(l_err, float(np.abs(lg - l_ref).max()))
        rows = min(rows * 2, 1 << 16)
    qd, kc, vc, od, lsed, L = data["decode"]
    d_err, dl_err = 0.0, 0.0
    for b in (0, qd.shape[0] - 1):
        o_ref, l_ref = oracle.decode(f64(qd[b:b + 1]), f64(kc[b:b + 1]), f64(vc[b:b + 1]), L, scale, nthreads=cores)
        d_err = max(d_err, float(np.abs(f64(od[b:b + 1]) - o_ref).max()))
        dl_err = max(dl_err, float(np.abs(f64(lsed[b:b + 1]) - l_ref).max()))
    ok = (o_err <= 2e-2 and o_sum / max(n_el, 1) <= 2e-3 and l_err <= 1e-3 and d_err <= 2e-2 and dl_err <= 1e-3)
    return {"value": total_f / total_t / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": (f"{total_rows} random query rows of {heads} single (b, h) heads of the bench's own causal "
                       f"prefill inputs (N=8192, D=128), {total_t:.1f} s on the host cores; FLOPs 4*D*(i+1) per "
                       f"row i"),
            "check": {"ok": ok, "prefill_rows": total_rows, "o_max_abs": o_err, "o_mean_abs": o_sum / max(n_el, 1),
                      "lse_max_abs": l_err, "decode_batches": [0, int(qd.shape[0]) - 1],
                      "decode_o_max_abs": d_err, "decode_lse_max_abs": dl_err,
                      "bounds": "O max 2e-2, mean 2e-3; LSE max 1e-3 (fp64 oracle)"}}


def run_reference(args, rank, world):
    """The oracle as the reference arm: host cores, bounded row samples of the prefill workload per step."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    rows_per_step = 512
    for i in range(args.warmup):
        q, k, v, sel, _ = oracle_sample(rows_per_step, 1000 + i)
        oracle.attention_rows(q, k, v, True, 1 / math.sqrt(PREFILL["D"]), sel, nthreads=cores)
    tot_f, tot_t = 0.0, 0.0
    for i in range(args.steps):
        q, k, v, sel, f = oracle_sample(rows_per_step, i)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, True, 1 / math.sqrt(PREFILL["D"]), sel, nthreads=cores)
        tot_t += time.perf_counter() - t0
        tot_f += f
    val = tot_f / tot_t / 1e12
    sample = (f"{rows_per_step} random query rows of one (b, h) of the causal prefill workload per step "
              f"(N=8192, D=128; FLOPs counted as 4*D*(i+1) per row i)")
    return {
        "impl": "reference",
        "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": WORKLOAD, "prefill": PREFILL, "decode": DECODE},
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def oracle_config_table():
    """Wall time of the fp64 oracle on each parity configuration, on this host's cores.

    All cores for every configuration, one core as well for the small MHA case
    and the cross-attention; the N=8192 causal prefill on sampled rows (its
    full run is hours), extrapolated by FLOPs.  Prints one JSON line per entry.
    """
    import numpy as np
    import torch

    import oracle
    from attention_fa2_fwd_gb300 import inputs as I
    oracle.build()
    cores = oracle.default_threads()
    model = ""
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True).stdout
        model = next((l.split(":", 1)[1].strip() for l in out.splitlines() if l.startswith("Model name")), "")
    except OSError:
        pass

    def f64(t):
        return t.to(torch.float64).numpy()

    def emit(config, what, seconds, threads, flops=None):
        rec = {"oracle_config": config, "what": what, "seconds": round(seconds, 4), "threads": threads,
               "host": model, "nproc": os.cpu_count()}
        if flops:
            rec["tflops"] = round(flops / seconds / 1e12, 5)
        print(json.dumps(rec), flush=True)

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    c = I.MHA_256
    q, k, v = (f64(t) for t in c.make())
    for th in (cores, 1):
        emit(1, c.name, timed(lambda: oracle.attention(q, k, v, c.causal, c.scale, nthreads=th)), th, c.flops)
    for n in (2048, 4096):
        c = I.GQA_CAUSAL[n]
        q, k, v = (f64(t) for t in c.make())
        emit(2, c.name, timed(lambda: oracle.attention(q, k, v, c.causal, c.scale, nthreads=cores)), cores, c.flops)
    c = I.GQA_CAUSAL[8192]
    q, k, v = (f64(t) for t in c.make())
    rng = np.random.default_rng(0)
    sel = np.stack([rng.integers(0, c.B, 4096), rng.integers(0, c.Hq, 4096), rng.integers(0, c.Nq, 4096)], 1)
    sec = timed(lambda: oracle.attention_rows(q, k, v, True, c.scale, sel, nthreads=cores))
    f = float(sum(4 * c.D * (int(i) + 1) for i in sel[:, 2]))
    emit(2, c.name + " (4096 sampled rows; full run extrapolated by FLOPs: %.0f s)" % (sec * c.flops / f), sec,
         cores, f)
    tot, fl = 0.0, 0.0
    for c in I.sweep_cases():
        q, k, v = (f64(t) for t in c.make())
        tot += timed(lambda: oracle.attention(q, k, v, c.causal, c.scale, nthreads=cores))
        fl += c.flops
    emit(3, "sweep, 160 cases", tot, cores, fl)
    for B in I.DECODE_B:
        kk, vv = (f64(t) for t in I.decode_stream(B, 8, max(I.DECODE_LENS), 128, "bf16"))
        qs = f64(I.decode_queries(B, 32, 128, [L - 1 for L in I.DECODE_LENS], "bf16"))
        tot = 0.0
        for j, L in enumerate(I.DECODE_LENS):
            tot += timed(lambda: oracle.decode(qs[:, :, j], kk, vv, L, 1 / math.sqrt(128), nthreads=cores))
        emit(4, f"decode B={B}, one step at each of L={list(I.DECODE_LENS)}", tot, cores)
    for D in sorted(I.CROSS):
        c = I.CROSS[D]
        q, k, v = (f64(t.contiguous()) for t in c.make())
        for th in (cores, 1):
            emit(5, c.name, timed(lambda: oracle.attention(q, k, v, c.causal, c.scale, nthreads=th)), th, c.flops)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--passes-per-step", type=int, default=20,
                    help="passes of the whole path per timed step (keeps the timed region long enough for the "
                         "clock sampler: 20 steps x 20 passes is about 0.45 s)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--no-also", dest="also", action="store_false",
                    help="skip the secondary measurements (D=64, cross-attention, RoPE, backward, B=2 decode step)")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="with --impl reference: time the oracle on every parity configuration (a few minutes)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference" and args.oracle_configs:
        if rank == 0:
            oracle_config_table()
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line, data = run_ours(args, rank, world, local_rank)
        if line is not None:
            if world == 1:
                line["cpu_baseline"] = cpu_baseline_leg(args.cpu_baseline_seconds, data)
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
