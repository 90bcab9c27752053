"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random tensors and names workloads; it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU from a
``torch.Generator`` seeded with 42 by default ("Triton-FlashAttention",
Phase 3: fixed seed 42), in fp32, then cast to the workload's dtype, so the
GPU path and the oracle see the same rounded values.

Distributions follow the workloads' descriptions: i.i.d. N(0, 1) for Q, K, V;
the cross-attention workload draws K with variance 2 (std sqrt(2)) -- and, as
a second reading of its "N(0, 2)", with standard deviation 2 -- and V from
U(-1, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _draw(shape, gen, dist):
    kind, a = dist
    if kind == "normal":  # N(0, a) with a the variance
        return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(a)
    if kind == "uniform":  # U(-a, a)
        return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * a
    if kind == "zeros":
        return torch.zeros(shape, dtype=torch.float32)
    raise ValueError(kind)


def to_layout(x: torch.Tensor, layout: str) -> torch.Tensor:
    """Return a (B,H,N,D)-indexed view whose memory is laid out as ``layout``.

    ``bhnd``: contiguous (B,H,N,D).  ``bnhd``: memory (B,N,H,D), returned as the
    permuted (B,H,N,D) view, so strides are (N*H*D, D, H*D, 1).
    """
    if layout == "bhnd":
        return x.contiguous()
    if layout == "bnhd":
        return x.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    raise ValueError(layout)


def prefill_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype="bf16", layout="bhnd", seed=42,
                   q_dist=("normal", 1.0), k_dist=("normal", 1.0), v_dist=("normal", 1.0)):
    """Q (B,Hq,Nq,D), K, V (B,Hkv,Nkv,D) on the CPU in ``dtype`` and ``layout``."""
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    q = _draw((B, Hq, Nq, D), gen, q_dist).to(dt)
    k = _draw((B, Hkv, Nkv, D), gen, k_dist).to(dt)
    v = _draw((B, Hkv, Nkv, D), gen, v_dist).to(dt)
    return to_layout(q, layout), to_layout(k, layout), to_layout(v, layout)


def decode_stream(B, Hkv, L, D, dtype="bf16", seed=42):
    """Key/value token streams K, V (B,H_kv,L,D): token t's key and value are K[:, :, t], V[:, :, t]."""
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    k = _draw((B, Hkv, L, D), gen, ("normal", 1.0)).to(dt)
    v = _draw((B, Hkv, L, D), gen, ("normal", 1.0)).to(dt)
    return k, v


def decode_queries(B, Hq, D, steps, dtype="bf16", seed=42):
    """Queries (B,H_q,len(steps),D) of the given decode steps, N(0,1).

    Step t's query is drawn from its own generator (seeded from seed and t),
    so a step's query does not depend on which other steps are requested.
    """
    dt = DTYPES[dtype]
    out = torch.empty((B, Hq, len(steps), D), dtype=dt)
    for j, t in enumerate(steps):
        gen = torch.Generator().manual_seed(seed * 1_000_003 + 7919 * int(t) + 1)
        out[:, :, j] = _draw((B, Hq, D), gen, ("normal", 1.0)).to(dt)
    return out


@dataclass(frozen=True)
class Prefill:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    D: int
    causal: bool
    dtype: str
    layout: str = "bhnd"
    q_dist: tuple = ("normal", 1.0)
    k_dist: tuple = ("normal", 1.0)
    v_dist: tuple = ("normal", 1.0)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H_q*N_q*N_kv*D per forward, halved for causal (two GEMMs)."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nkv * self.D
        return f / 2.0 if self.causal else f

    def make(self, seed=42):
        return prefill_inputs(self.B, self.Hq, self.Hkv, self.Nq, self.Nkv, self.D, self.dtype,
                              self.layout, seed, self.q_dist, self.k_dist, self.v_dist)


@dataclass(frozen=True)
class Decode:
    name: str
    B: int
    Hq: int
    Hkv: int
    cache_len: int
    D: int
    dtype: str = "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def kv_bytes(self) -> int:
        """K and V bytes read once per kv head: 2 * B * H_kv * L * D * 2."""
        return 2 * self.B * self.Hkv * self.cache_len * self.D * 2


# Workload 1: small MHA prefill, the case the oracle finishes in well under a second.
MHA_256 = Prefill("mha_prefill_b1_h4_n256_d64_f16", 1, 4, 4, 256, 256, 64, False, "f16")

# Workload 2: GQA causal prefill, bf16, B=2, H_q=32, H_kv=8, D=128.
GQA_CAUSAL = {n: Prefill(f"gqa_causal_prefill_b2_hq32_hkv8_n{n}_d128_bf16", 2, 32, 8, n, n, 128, True,
                         "bf16") for n in (2048, 4096, 8192)}

# Workload 3: GQA/MQA ratio and boundary sweep, fp16, B=2, H_q=16.
SWEEP_N = (1, 31, 33, 63, 65, 127, 257, 1024)
SWEEP_HKV = (16, 8, 4, 2, 1)
SWEEP_D = (64, 128)


def sweep_cases():
    for D in SWEEP_D:
        for hkv in SWEEP_HKV:
            for causal in (False, True):
                for n in SWEEP_N:
                    yield Prefill(f"sweep_hkv{hkv}_d{D}_{'c' if causal else 'nc'}_n{n}", 2, 16, hkv, n, n, D,
                                  causal, "f16")


# Workload 4: KV-cache decode, bf16, H_q=32, H_kv=8, D=128.
DECODE_LENS = (1, 33, 257, 1024, 4097, 8192)
DECODE_B = (2, 64)

# Workload 5: cross-attention, bf16, (B,N,H,D) memory layout, unequal lengths.
# "K ~ N(0, 2)" is read as variance 2 (CROSS); the standard-deviation reading,
# K = 2 * N(0, 1) (variance 4), is run as well (CROSS_STD2).
CROSS = {D: Prefill(f"cross_b4_hq16_hkv4_nq1024_nkv4096_d{D}_bnhd_bf16", 4, 16, 4, 1024, 4096, D, False,
                    "bf16", "bnhd", ("normal", 1.0), ("normal", 2.0), ("uniform", 1.0)) for D in (64, 128)}
CROSS_STD2 = {D: Prefill(f"cross_b4_hq16_hkv4_nq1024_nkv4096_d{D}_bnhd_bf16_kstd2", 4, 16, 4, 1024, 4096, D, False,
                         "bf16", "bnhd", ("normal", 1.0), ("normal", 4.0), ("uniform", 1.0)) for D in (64, 128)}
