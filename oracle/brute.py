"""Scalar restatement of naive attention with pure-Python loops (tiny inputs).

TEST INFRASTRUCTURE ONLY (see the package docstring).

This is a second, independent transcription of the four naive steps named in
"Flash Attention Memory Optimization Explained" (lzwjava.github.io, section
"What is Flash Attention?") and printed as code in the yelogs.com Flash
Attention2/Triton tutorial (section "內存牆：注意力機制的阿喀琉斯之踵"):
scores, scale and mask, softmax, weighted sum; plus the per-row log-sum-exp
of the tutorial's kernel (section "核心 Kernel 實現").  It uses no array
library at all: every score is a ``math.fsum`` of products, the softmax uses
``math.exp`` on the max-shifted score and the sums are ``math.fsum`` (exactly
rounded).  It exists to pin ``attention_ref``: a dropped term, a transposed
operand, a wrong head index or an off-by-one in the causal mask in either
would make them disagree.  Only for T <= 8, d <= 8.
"""

from __future__ import annotations

import math


def _to_nested(x):
    if hasattr(x, "detach"):
        import torch

        return x.detach().to(device="cpu", dtype=torch.float64).tolist()
    if hasattr(x, "tolist"):
        return x.tolist()
    return x


def attention_brute(q, k, v, scale: float, causal: bool, window=None, global_tokens=None):
    """Returns (O, LSE) as nested Python lists [B][Hq][T][d] and [B][Hq][T].

    window = (wl, wr) keeps, in addition, only keys i - wl <= j <= i + wr
    (-1 = unbounded side), the band form of the tutorial's sliding window.
    global_tokens lists keys kept for every row in addition to that band (the
    tutorial's local-global mask: band OR key in the list), still subject to
    the causal rule.
    """
    q, k, v = _to_nested(q), _to_nested(k), _to_nested(v)
    B, Hq, T, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    if T > 8 or d > 8:
        raise ValueError("attention_brute is for tiny inputs only (T, d <= 8)")
    group = Hq // Hkv
    O = [[[[0.0] * d for _ in range(T)] for _ in range(Hq)] for _ in range(B)]
    L = [[[0.0] * T for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            for i in range(T):
                keys = []
                for j in range(T):
                    if causal and j > i:
                        continue
                    is_global = global_tokens is not None and j in list(global_tokens)
                    if window is not None and not is_global:
                        if window[0] >= 0 and j < i - window[0]:
                            continue
                        if window[1] >= 0 and j > i + window[1]:
                            continue
                    keys.append(j)
                scores = {}
                for j in keys:
                    dot = math.fsum(q[b][h][i][c] * k[b][hk][j][c] for c in range(d))
                    scores[j] = scale * dot
                mx = max(scores[j] for j in keys)
                w = {j: math.exp(scores[j] - mx) for j in keys}
                den = math.fsum(w[j] for j in keys)
                for c in range(d):
                    O[b][h][i][c] = math.fsum(w[j] * v[b][hk][j][c] for j in keys) / den
                L[b][h][i] = mx + math.log(den)
    return O, L
