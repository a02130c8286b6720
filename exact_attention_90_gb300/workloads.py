"""Workload shapes and the bench's work accounting.

The shapes follow the pages' workloads: the single-head benchmark sweep of the
yelogs.com Flash Attention2/Triton tutorial (section "基準測試設置": dtype in
{fp32, bf16}, d in {16, 32, 64, 128}, T in {256, 1024, 4096}, B in {1, 64},
[B, T, d] randn, causal), the GPT-2 124M attention layer of "Flash Attention
Memory Optimization Explained" (section "Performance and Benefits": 12 heads of
64, T = 1024), long sequences, and the multi-query variant of the tutorial's
section "2. 多查詢注意力（MQA）" with its grouped generalisation.

Work accounting (metric conventions, not the method):
  flops  = 4 * B * Hq * T^2 * d, halved when causal (two contractions of
           2*T*T*d each per head; causal keeps about half of the scores);
  bytes  = e * d * T * (2*B*Hq + 2*B*Hkv) + 4*B*Hq*T   (Q, K, V read once,
           O written once in the input dtype of e bytes, LSE written in fp32);
  scores = B * Hq * T^2, halved when causal (one exponential each).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    d: int
    dtype: str          # "f32", "bf16" or "f16"
    causal: bool
    scale: float
    mult: float = 1.0   # Q, K, V = N(0,1) * mult before rounding to dtype
    seed: int = 0
    tags: tuple = field(default_factory=tuple)

    @property
    def flops(self) -> float:
        f = 4.0 * self.B * self.Hq * self.T * self.T * self.d
        return f / 2 if self.causal else f

    @property
    def bytes(self) -> float:
        e = ELEM_BYTES[self.dtype]
        return (e * self.d * self.T * (2 * self.B * self.Hq + 2 * self.B * self.Hkv)
                + 4 * self.B * self.Hq * self.T)

    @property
    def scores(self) -> float:
        s = float(self.B * self.Hq * self.T * self.T)
        return s / 2 if self.causal else s

    def describe(self) -> str:
        return (f"B={self.B} Hq={self.Hq} Hkv={self.Hkv} T={self.T} d={self.d} "
                f"{self.dtype} {'causal' if self.causal else 'non-causal'}")


def _sweep():
    out = []
    for dtype in ("f32", "bf16"):
        for d in (16, 32, 64, 128):
            for T in (256, 1024, 4096):
                for B in (1, 64):
                    out.append(Workload(
                        name=f"sweep_B{B}_T{T}_d{d}_{dtype}", B=B, Hq=1, Hkv=1, T=T,
                        d=d, dtype=dtype, causal=True, scale=1.0 / math.sqrt(d),
                        seed=1001, tags=("sweep",)))
    return out


def all_workloads():
    """Every workload shape, grouped by the configuration it belongs to."""
    w = []
    for causal in (True, False):
        w.append(Workload(name=f"tiny_T64_d16_f32_{'causal' if causal else 'full'}",
                          B=1, Hq=1, Hkv=1, T=64, d=16, dtype="f32", causal=causal,
                          scale=0.25, seed=1000, tags=("tiny",)))
    w += _sweep()
    w.append(Workload(name="gpt2_B16_H12_T1024_d64_bf16", B=16, Hq=12, Hkv=12, T=1024,
                      d=64, dtype="bf16", causal=True, scale=0.125, mult=0.5,
                      seed=1002, tags=("gpt2",)))
    for T in (8192, 16384):
        for causal in (True, False):
            w.append(Workload(name=f"long_B1_H16_T{T}_d128_bf16_{'causal' if causal else 'full'}",
                              B=1, Hq=16, Hkv=16, T=T, d=128, dtype="bf16",
                              causal=causal, scale=1.0 / math.sqrt(128), seed=1003,
                              tags=("long",)))
    for Hkv in (1, 8):
        w.append(Workload(name=f"{'mqa' if Hkv == 1 else 'gqa'}_B8_Hq32_Hkv{Hkv}_T4096_d128_bf16",
                          B=8, Hq=32, Hkv=Hkv, T=4096, d=128, dtype="bf16", causal=True,
                          scale=1.0 / math.sqrt(128), seed=1004, tags=("shared_kv",)))
    return w


def by_name(name: str) -> Workload:
    for w in all_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


# The bench's default (headline) workload: the sweep's causal bf16 d=128 T=4096
# point at B=64, the shape the throughput target is stated on.
HEADLINE = "sweep_B64_T4096_d128_bf16"
