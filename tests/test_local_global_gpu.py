"""GPU parity of the local-global mask (fa_fwd_local_global) against the
fp64 oracle, through the C ABI, with the global keys packed into dense tiles
(the default of the 16-bit path) and visited as whole key tiles.

The yelogs.com Flash Attention2/Triton tutorial, section "1. 稀疏注意力支持",
keeps key j for query i when |i - j| <= local_window or j is a global token
(isin over the key index); with causal the union is intersected with j <= i.
Tolerances are the forward's (tests/parity_util.py).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import make_qkv
from parity_util import TOL

pytestmark = pytest.mark.gpu


def global_set(kind, T, seed):
    rng = np.random.default_rng(seed)
    if kind == "none":
        return []
    if kind == "sink":
        return [0]
    if kind == "sinks4":
        return [0, 1, 2, 3]
    if kind == "last":
        return [T - 1]
    if kind == "strided":
        return list(range(5, T, 97))
    if kind == "random":
        # unsorted, with repeats and entries outside [0, T)
        g = rng.integers(-20, T + 20, size=37).tolist()
        return g + g[:5]
    if kind == "dense":
        # more than 128 distinct tokens: several packed tiles, many of them
        # inside the rows' bands
        return rng.permutation(T)[: min(T, 300)].tolist()
    if kind == "near":
        # clustered around the middle: inside the band of the middle rows,
        # outside it for the others
        return list(range(T // 2 - 20, T // 2 + 20, 3))
    raise ValueError(kind)


def run_lg(fa, B, Hq, Hkv, T, d, w, kind, causal, dtype, seed, pack=True):
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=seed)
    g = global_set(kind, T, seed)
    gt = torch.tensor(g, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, window=(w, w),
                    global_tokens=gt, pack_global=pack)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal, window=(w, w), global_tokens=g)
    tol_o, tol_l = TOL[dtype]
    eo = float(np.max(np.abs(oracle.as_f64(o) - O_ref)))
    el = float(np.max(np.abs(oracle.as_f64(lse) - L_ref)))
    assert eo <= tol_o and el <= tol_l, \
        f"T={T} d={d} w={w} {kind} causal={causal} {dtype}: |dO|={eo:.3g} |dL|={el:.3g}"


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind,w", [("none", 3), ("sink", 0), ("sinks4", 64), ("last", 5),
                                    ("strided", 1), ("random", 200), ("dense", 40),
                                    ("near", 30)])
@pytest.mark.parametrize("T,d", [(129, 32), (640, 128), (1000, 64), (2500, 128)])
def test_local_global_parity(cuda_lib, T, d, kind, w, causal, dtype):
    """Band tiles plus global keys below, inside or above the band, ragged T,
    repeats and out-of-range entries; the 16-bit path packs the global keys."""
    run_lg(cuda_lib, 1, 2, 1, T, d, w, kind, causal, dtype, seed=T + d + w)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind,w", [("sinks4", 64), ("strided", 1), ("random", 200),
                                    ("dense", 40), ("near", 30)])
@pytest.mark.parametrize("T,d", [(640, 128), (1000, 64)])
def test_local_global_parity_whole_tiles(cuda_lib, T, d, kind, w, causal, dtype):
    """The same mask with the global keys visited as whole key tiles (the
    smaller workspace)."""
    run_lg(cuda_lib, 1, 2, 1, T, d, w, kind, causal, dtype, seed=T + d + w, pack=False)


@pytest.mark.parametrize("causal", [False, True])
def test_local_global_packed_many_tokens_and_heads(cuda_lib, causal):
    """Three packed tiles (300 distinct tokens), GQA heads, d = 16."""
    run_lg(cuda_lib, 2, 4, 2, 1777, 16, 9, "dense", causal, "bf16", seed=11)
    run_lg(cuda_lib, 2, 6, 3, 900, 128, 0, "dense", causal, "f16", seed=12)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_local_global_grouped_heads_and_d16(cuda_lib, dtype):
    run_lg(cuda_lib, 2, 4, 2, 777, 16, 7, "random", True, dtype, seed=5)
    run_lg(cuda_lib, 1, 8, 1, 513, 64, 0, "strided", False, dtype, seed=6)


def test_local_global_extremes_match_plain_masks(cuda_lib):
    """Every key global is no mask; no global key is the symmetric band;
    a window wider than T is no mask."""
    fa = cuda_lib
    T, d = 700, 128
    q, k, v = (x.cuda() for x in make_qkv(1, 2, 2, T, d, dtype="bf16", seed=9))
    every = torch.arange(T, dtype=torch.int32, device="cuda")
    none = torch.empty(0, dtype=torch.int32, device="cuda")
    o1, l1 = fa.fwd(q, k, v, causal=True, window=(0, 0), global_tokens=every)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    o3, l3 = fa.fwd(q, k, v, window=(9, 9), global_tokens=none)
    o4, l4 = fa.fwd(q, k, v, window=(9, 9))
    o5, l5 = fa.fwd(q, k, v, window=(5000, 5000), global_tokens=none)
    o6, l6 = fa.fwd(q, k, v)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    tol_o, tol_l = TOL["bf16"]
    for a, b in ((o1, o2), (o3, o4), (o5, o6)):
        assert (a.float() - b.float()).abs().max().item() <= tol_o
    for a, b in ((l1, l2), (l3, l4), (l5, l6)):
        assert (a - b).abs().max().item() <= tol_l
