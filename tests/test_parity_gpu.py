"""Parity of fa_fwd (through the C ABI) with the fp64 oracle, on the GPU.

Small and medium shapes are compared element by element with the full
oracle; they span several 128-row tiles and ragged tails (T not a multiple of
the tile), every head dimension, causal and not, MHA/GQA/MQA, and the
degenerate cases (T = 1, zero and negative scale, one dominant key).  The
workload shapes themselves (full sizes, the same launch as the bench) are
compared on sampled rows, which the oracle evaluates exactly one by one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import make_qkv, make_structured_qkv
from exact_attention_90_gb300.workloads import all_workloads
from parity_util import TOL, check_full, check_sampled, spread_pairs

pytestmark = pytest.mark.gpu

DS = [16, 32, 64, 128]


def run(fa, q, k, v, causal, scale=None, kernel="auto"):
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale, kernel=kernel)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0, "a kernel wait timed out"
    return o, lse


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", DS)
@pytest.mark.parametrize("T", [1, 5, 64, 127, 129, 200, 257, 640, 1000])
def test_full_parity_ragged(cuda_lib, T, d, causal, dtype):
    q, k, v = make_qkv(2, 4, 2, T, d, dtype=dtype, seed=T * 7 + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = run(cuda_lib, q, k, v, causal, scale)
    check_full(o, lse, q, k, v, scale, causal, what=f"T={T} d={d} causal={causal} {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (8, 2), (8, 8), (6, 3)])
def test_full_parity_grouped_heads(cuda_lib, Hq, Hkv, dtype):
    for causal in (False, True):
        q, k, v = make_qkv(2, Hq, Hkv, 300, 64, dtype=dtype, seed=Hq * 10 + Hkv, device="cuda")
        o, lse = run(cuda_lib, q, k, v, causal, 0.125)
        check_full(o, lse, q, k, v, 0.125, causal, what=f"Hq={Hq} Hkv={Hkv} {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", DS)
def test_full_parity_many_units_per_cta(cuda_lib, d, dtype):
    """More work units than SMs (8 x 32 heads x 2 row blocks = 512 units), so
    every CTA of the persistent grid runs several units and the barrier phase
    counters carry across unit boundaries (including units whose second Q
    tile is empty: T = 300); every row against the oracle."""
    for causal in (False, True):
        q, k, v = make_qkv(8, 32, 8, 300, d, dtype=dtype, seed=600 + d, device="cuda")
        scale = 1.0 / math.sqrt(d)
        o, lse = run(cuda_lib, q, k, v, causal, scale)
        check_full(o, lse, q, k, v, scale, causal, what=f"many units d={d} {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("scale", [0.0, -0.09, 0.7])
def test_full_parity_scale_edge_cases(cuda_lib, scale, dtype):
    for causal in (False, True):
        q, k, v = make_qkv(1, 2, 2, 333, 32, dtype=dtype, seed=77, device="cuda")
        o, lse = run(cuda_lib, q, k, v, causal, scale)
        check_full(o, lse, q, k, v, scale, causal, what=f"scale={scale} {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", DS)
@pytest.mark.parametrize("ramp", [40.0, 200.0])
def test_full_parity_row_max_jumps(cuda_lib, ramp, d, dtype):
    """Row maxima that jump from one 128-key tile to the next by ~30 (ramp 40)
    or ~150 (ramp 200) in log2 units: a tile exponentiated against the
    previous reference gives P sums far above 2^15, finite or infinite, and
    the kernel has to take the maximum, rescale and exponentiate again."""
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_structured_qkv(1, 2, 1024, d, dtype=dtype, seed=17, ramp=ramp, device="cuda")
    for causal in (False, True):
        o, lse = run(cuda_lib, q, k, v, causal, scale)
        check_full(o, lse, q, k, v, scale, causal, what=f"jumps ramp={ramp} d={d} {dtype}")


def fp32_lse_bound(q, k, scale):
    """Per-row bound on the LSE error of any fp32 evaluation (a stress-input
    tolerance, not a target one): each score is an fp32 dot product of d
    terms, off by at most scale * gamma_d * sum_c |q_c k_c| with
    gamma_d = d u / (1 - d u), u = 2^-24 (recursive summation); LSE is
    1-Lipschitz in the max norm of its score row; add a few roundings of
    |LSE| itself."""
    qa, ka = oracle.as_f64(q).__abs__(), oracle.as_f64(k).__abs__()
    d = qa.shape[-1]
    u = 2.0 ** -24
    gamma = d * u / (1 - d * u)
    B, Hq, T, _ = qa.shape
    g = Hq // ka.shape[1]
    worst = np.empty((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            worst[b, h] = (qa[b, h] @ ka[b, h // g].T).max(axis=1)
    return abs(scale) * gamma * worst


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_full_parity_growing_row_max(cuda_lib, d, dtype):
    """Row maxima that keep rising along the keys: the accumulator has to be
    rescaled many times (exercises the lazy rescale of the bf16 kernel).
    The scores reach |s| ~ 60 through one dot-product term of ~500, so for
    fp32 the LSE tolerance is the larger of 1e-5 and the fp32 error bound
    of the scores (fp32_lse_bound); O keeps its 1e-4 and bf16 its targets."""
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_structured_qkv(2, 2, 1024, d, dtype=dtype, seed=5, ramp=12.0, device="cuda")
    for causal in (False, True):
        o, lse = run(cuda_lib, q, k, v, causal, scale)
        O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
        tol_o, tol_l = TOL[dtype]
        eo = np.max(np.abs(oracle.as_f64(o) - O_ref))
        el = np.abs(oracle.as_f64(lse) - L_ref)
        if dtype == "f32":
            bound = np.maximum(tol_l, fp32_lse_bound(q, k, scale) + 4 * 2.0 ** -24 * np.abs(L_ref))
        else:
            bound = tol_l
        assert eo <= tol_o, f"ramp d={d} {dtype}: max|dO|={eo:.3g}"
        assert np.all(el <= bound), f"ramp d={d} {dtype}: max|dL|={el.max():.3g}"


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("window", [(0, 0), (3, 3), (64, 64), (100, 0), (0, 200), (-1, 50),
                                    (300, -1), (127, 128), (2000, 2000)])
@pytest.mark.parametrize("T,d", [(129, 32), (640, 128), (1000, 64)])
def test_window_parity(cuda_lib, T, d, window, dtype):
    """Band masks (the tutorial's sliding window |i - j| <= w and one-sided
    bands) against the oracle, with ragged T and tiles skipped outside the
    band."""
    fa = cuda_lib
    q, k, v = make_qkv(1, 4, 2, T, d, dtype=dtype, seed=T + d + window[0], device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, False, window=window)
    tol_o, tol_l = TOL[dtype]
    eo = float(np.max(np.abs(oracle.as_f64(o) - O_ref)))
    el = float(np.max(np.abs(oracle.as_f64(lse) - L_ref)))
    assert eo <= tol_o and el <= tol_l, f"window {window}: |dO|={eo:.3g} |dL|={el:.3g}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_window_causal_intersection(cuda_lib, dtype):
    """causal + window (w, w) is the band (w, 0), and (-1, 0) is plain causal."""
    fa = cuda_lib
    q, k, v = make_qkv(2, 2, 2, 700, 128, dtype=dtype, seed=5, device="cuda")
    o1, l1 = fa.fwd(q, k, v, causal=True, window=(90, 90))
    o2, l2 = fa.fwd(q, k, v, window=(90, 0))
    o3, l3 = fa.fwd(q, k, v, window=(-1, 0))
    o4, l4 = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o3, o4) and torch.equal(l3, l4)
    O_ref, L_ref = oracle.attention_ref(q, k, v, 1 / math.sqrt(128), True, window=(90, 90))
    assert float(np.max(np.abs(oracle.as_f64(o1) - O_ref))) <= TOL[dtype][0]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T,d,splits", [(1000, 128, 2), (1000, 64, 3), (777, 32, 5),
                                        (4096, 128, 8), (300, 16, 4), (129, 128, 2),
                                        (2048, 64, 64)])
def test_split_kv_parity(cuda_lib, T, d, splits, causal, dtype):
    """Split-KV forward (partials merged by log-sum-exp weights) against the
    oracle, including more splits than KV tiles (empty splits) and ragged T."""
    fa = cuda_lib
    q, k, v = make_qkv(1, 4, 2, T, d, dtype=dtype, seed=T + d + splits, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    check_full(o, lse, q, k, v, scale, causal, what=f"split={splits} T={T} d={d} {dtype}")


def test_split_count_with_a_mask_that_has_no_split_is_refused(cuda_lib):
    """The band and local-global paths have no KV split: asking for one with
    them is an error, not a silently unsplit run."""
    fa = cuda_lib
    q, k, v = make_qkv(1, 2, 2, 300, 64, dtype="bf16", seed=5, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, causal=True, window=(64, 0), num_splits=2)
    g = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, causal=True, global_tokens=g, num_splits=3)
    # num_splits = 1 (or None) with a window is an ordinary banded call
    o, lse = fa.fwd(q, k, v, causal=True, window=(64, 0), num_splits=1)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0


def test_split_heuristic_path_matches_unsplit(cuda_lib):
    """A shape the heuristic splits (one head of T = 4096) gives the oracle's
    result and agrees with the unsplit kernel."""
    fa = cuda_lib
    q, k, v = make_qkv(1, 1, 1, 4096, 128, dtype="bf16", seed=21, device="cuda")
    assert fa.fa_fwd_split_heuristic(1, 1, 1, 4096, 128, 1) > 1
    o1, l1 = run(fa, q, k, v, True)
    o2, l2 = fa.fwd(q, k, v, causal=True, num_splits=1)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 2e-3
    check_full(o1, l1, q, k, v, 1 / math.sqrt(128), True, what="heuristic split")


def test_causal_row0_and_zero_query_closed_forms(cuda_lib):
    """Closed forms on the device: causal row 0 returns V[0] (exactly, up to
    output rounding) and Q = 0 gives LSE[i] = ln(i+1)."""
    fa = cuda_lib
    for dtype in ("bf16", "f32", "f16"):
        q, k, v = make_qkv(2, 2, 2, 500, 64, dtype=dtype, seed=3, device="cuda")
        o, lse = run(fa, q, k, v, True, 0.125)
        assert torch.equal(o[:, :, 0, :], v[:, :, 0, :])
        qz = torch.zeros_like(q)
        o, lse = run(fa, qz, k, v, True, 0.125)
        want = torch.log(torch.arange(1, 501, dtype=torch.float64))
        err = (lse.double().cpu() - want).abs().max().item()
        assert err <= TOL[dtype][1]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [129, 200, 257])
def test_full_parity_simt_wide_ctas(cuda_lib, T, d, causal):
    """The CUDA-core kernel with 128-row CTAs: it takes them for d >= 64 once
    the grid gives every SM a CTA (here 2 x 76 heads x 2 row blocks = 304),
    and 64-row CTAs below that, which the small shapes above exercise.  GQA
    heads and a ragged last block of rows."""
    q, k, v = make_qkv(2, 76, 38, T, d, dtype="f32", seed=T + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = run(cuda_lib, q, k, v, causal, scale)
    check_full(o, lse, q, k, v, scale, causal, what=f"wide T={T} d={d} causal={causal}")


def test_simt_wide_ctas_window_and_16bit(cuda_lib):
    """128-row CTAs with a band window, and on bf16 inputs (fp32 arithmetic)."""
    fa = cuda_lib
    q, k, v = make_qkv(2, 76, 76, 300, 128, dtype="f32", seed=12, device="cuda")
    scale = 1.0 / math.sqrt(128)
    o, lse = fa.fwd(q, k, v, causal=False, scale=scale, window=(70, 20))
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, False, window=(70, 20))
    assert float(np.max(np.abs(oracle.as_f64(o) - O_ref))) <= TOL["f32"][0]
    assert float(np.max(np.abs(oracle.as_f64(lse) - L_ref))) <= TOL["f32"][1]
    qb, kb, vb = q.bfloat16(), k.bfloat16(), v.bfloat16()
    o2, l2 = run(fa, qb, kb, vb, True, scale, kernel="simt")
    check_full(o2, l2, qb, kb, vb, scale, True, what="wide bf16 via the CUDA-core kernel")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tensor_core_agrees_with_fp32_simt(cuda_lib, dtype):
    """The tcgen05 kernel and the CUDA-core kernel on the same 16-bit inputs."""
    fa = cuda_lib
    q, k, v = make_qkv(2, 4, 4, 777, 128, dtype=dtype, seed=9, device="cuda")
    for causal in (False, True):
        o1, l1 = run(fa, q, k, v, causal)
        o2, l2 = run(fa, q, k, v, causal, kernel="simt")
        assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
        assert (l1 - l2).abs().max().item() <= 2e-3


def test_deterministic_and_no_stray_writes(cuda_lib):
    """Two runs give identical bits, and nothing outside O and LSE changes
    (guard regions around both outputs)."""
    fa = cuda_lib
    B, H, T, d = 2, 3, 333, 128
    for dtype in ("bf16", "f32", "f16"):
        q, k, v = make_qkv(B, H, H, T, d, dtype=dtype, seed=4, device="cuda")
        tdt = q.dtype
        pad_o, pad_l = 4096, 1024
        for causal in (False, True):
            obuf = torch.full((B * H * T * d + 2 * pad_o,), 7.0, dtype=tdt, device="cuda")
            lbuf = torch.full((B * H * T + 2 * pad_l,), 7.0, dtype=torch.float32, device="cuda")
            o = obuf[pad_o:pad_o + B * H * T * d].view(B, H, T, d)
            lse = lbuf[pad_l:pad_l + B * H * T].view(B, H, T)
            outs = []
            for _ in range(2):
                fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
                torch.cuda.synchronize()
                outs.append((o.clone(), lse.clone()))
            assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
            for buf, pad in ((obuf, pad_o), (lbuf, pad_l)):
                assert torch.all(buf[:pad] == 7.0) and torch.all(buf[-pad:] == 7.0)
            check_full(o, lse, q, k, v, 1 / math.sqrt(d), causal, what=f"guarded {dtype}")


def test_inputs_unchanged(cuda_lib):
    fa = cuda_lib
    q, k, v = make_qkv(1, 4, 2, 256, 64, dtype="bf16", seed=8, device="cuda")
    q0, k0, v0 = q.clone(), k.clone(), v.clone()
    run(fa, q, k, v, True)
    assert torch.equal(q, q0) and torch.equal(k, k0) and torch.equal(v, v0)


def test_streams_are_honoured(cuda_lib):
    fa = cuda_lib
    q, k, v = make_qkv(2, 2, 2, 512, 64, dtype="bf16", seed=12, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.fwd(q, k, v, causal=True)
    s.synchronize()
    check_full(o, lse, q, k, v, 0.125, True, what="side stream")


# ---------------------------------------------------------------- workloads
WORKLOADS = all_workloads()


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(cuda_lib, w):
    """Every workload shape at full size, as the bench launches it; sampled
    rows of several (b, h) against the oracle (all rows for the small ones)."""
    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.T, w.d, dtype=w.dtype, seed=w.seed, mult=w.mult,
                       device="cuda")
    if w.dtype == "bf16":
        assert v.abs().max().item() < 8.0  # |O| < 8: bf16 half-ulp of O stays below 2e-2
    o, lse = run(cuda_lib, q, k, v, w.causal, w.scale)
    small = w.B * w.Hq * w.T * w.T * w.d <= 2 ** 28
    if small:
        check_full(o, lse, q, k, v, w.scale, w.causal, what=w.name)
    else:
        pairs = spread_pairs(w.B, w.Hq, n=4, seed=w.seed)
        check_sampled(o, lse, q, k, v, w.scale, w.causal, pairs, n_rows=40, what=w.name,
                      seed=w.seed)
