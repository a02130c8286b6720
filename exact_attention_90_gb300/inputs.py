"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws Q, K, V.  Values are
i.i.d. N(0, 1) drawn in fp32 from a CPU ``torch.Generator``, optionally
multiplied by a constant, then rounded to the requested dtype, so the device
path and the fp64 oracle see identical bits.  The pages' benchmark draws
``torch.randn`` tensors of shape [B, T, d] (yelogs.com Flash Attention2/Triton
tutorial, section "基準測試設置"); multi-head inputs use [B, H, T, d].
"""

from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def make_qkv(B: int, Hq: int, Hkv: int, T: int, d: int, dtype: str = "bf16",
             seed: int = 0, mult: float = 1.0, device: str = "cpu"):
    """Q [B,Hq,T,d], K and V [B,Hkv,T,d], contiguous, in ``dtype`` ("f32"/"bf16"/"f16").

    Q, K and V are drawn in that order from one generator seeded with ``seed``.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    tdt = DTYPES[dtype]
    out = []
    for H in (Hq, Hkv, Hkv):
        x = torch.randn((B, H, T, d), generator=g, dtype=torch.float32)
        if mult != 1.0:
            x = x * mult
        out.append(x.to(tdt).contiguous().to(device))
    return tuple(out)


def make_structured_qkv(B: int, H: int, T: int, d: int, dtype: str = "bf16",
                        seed: int = 0, ramp: float = 4.0, device: str = "cpu"):
    """Inputs whose row maximum keeps growing along the keys.

    K rows carry a component that grows linearly with the key index and Q rows
    a matching positive component, so the running maximum of a row rises from
    block to block; a kernel that rescales its accumulator lazily is exercised
    on every block.  Still i.i.d. noise plus a deterministic ramp: no
    arithmetic of the method.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, T, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, T, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, T, d), generator=g, dtype=torch.float32)
    q[..., 0] = q[..., 0].abs() + 1.0
    k[..., 0] = torch.linspace(-ramp, ramp, T).expand(B, H, T) * (d ** 0.5)
    tdt = DTYPES[dtype]
    return tuple(x.to(tdt).contiguous().to(device) for x in (q, k, v))


def make_grad_out(B: int, H: int, T: int, d: int, dtype: str = "bf16", seed: int = 0,
                  device: str = "cpu"):
    """An upstream gradient dO [B,H,T,d] for the backward pass: i.i.d. N(0, 1)
    drawn in fp32 from a generator seeded with ``seed`` + 7919 (so that it is
    not a copy of the Q drawn with the same seed), rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    x = torch.randn((B, H, T, d), generator=g, dtype=torch.float32)
    return x.to(DTYPES[dtype]).contiguous().to(device)
