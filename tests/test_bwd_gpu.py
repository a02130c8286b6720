"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 oracle,
through the C ABI (fa_bwd).

The oracle differentiates the forward by the chain rule
(``oracle.attention_bwd_ref``; pinned in test_oracle_bwd.py).  The backward
kernels recompute P from the forward's log-sum-exp ("Flash Attention Memory
Optimization Explained", section "Key Mechanisms", item "Backward
Checkpointing").  Unless a test says otherwise, O and LSE come from the
oracle's forward (rounded to the dtype and to fp32), so that a case checks the
backward kernels alone.

Tolerance (no target is stated for gradients): max |g - g_ref| over a
gradient tensor <= tol * max(max |g_ref|, 0.1), with tol = 1e-4 for fp32
inputs (fp32 FFMA everywhere) and 2e-2 for bf16 / fp16 (P and dS are
rounded to the input type, relative 2^-9 for bf16, before the tensor-core
products, and the gradients are rounded to it on output: a few times 2^-9
of the tensor's scale; the bound leaves about a 5x margin).  The floor 0.1
covers gradients that vanish exactly: when a row keeps a single key, dS =
P (dP - D) is the difference of two fp32 roundings of the same dot product
dO . v (D is formed as sum dO * O), about u sqrt(d) |dO| |O| ~ 1e-5, which
times scale |k| leaves up to ~3e-6 in dQ against an exact 0.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import DTYPES, make_grad_out, make_qkv

pytestmark = pytest.mark.gpu

BWD_TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-2}


def oracle_fwd_outputs(q, k, v, scale, causal, window, dtype):
    O, L = oracle.attention_ref(q, k, v, scale, causal, window=window)
    o = torch.from_numpy(O).to(DTYPES[dtype]).contiguous()
    lse = torch.from_numpy(L).to(torch.float32).contiguous()
    return o, lse


def check_grads(got, ref, dtype, what):
    worst = []
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        G = oracle.as_f64(g)
        assert np.all(np.isfinite(G)), f"{what}: non-finite {name}"
        err = float(np.max(np.abs(G - r))) if r.size else 0.0
        bound = BWD_TOL[dtype] * max(float(np.max(np.abs(r))) if r.size else 0.0, 0.1)
        assert err <= bound, f"{what}: max|{name} err|={err:.3g} > {bound:.3g}"
        worst.append(err / bound)
    return worst


def run_bwd(fa, B, Hq, Hkv, T, d, dtype, causal, window=None, scale=None, seed=0,
            library_fwd=False):
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=seed)
    do = make_grad_out(B, Hq, T, d, dtype=dtype, seed=seed)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    if library_fwd:
        o, lse = fa.fwd(qc, kc, vc, causal=causal, scale=scale, window=window)
    else:
        o, lse = oracle_fwd_outputs(q, k, v, scale, causal, window, dtype)
        o, lse = o.cuda(), lse.cuda()
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    ref = oracle.attention_bwd_ref(q, k, v, do, scale, causal, window=window)
    return (dq, dk, dv), ref


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("T", [1, 5, 64, 127, 129, 200, 257, 640])
def test_bwd_parity(cuda_lib, T, d, causal, dtype):
    """Every head dimension, ragged T spanning several 64/128-row tiles,
    causal or not, grouped heads (2 query heads on 1 KV head)."""
    got, ref = run_bwd(cuda_lib, 1, 2, 1, T, d, dtype, causal, seed=T * 7 + d)
    check_grads(got, ref, dtype, f"T={T} d={d} causal={causal} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B,Hq,Hkv,T,d", [(2, 4, 2, 300, 64), (1, 8, 1, 200, 128),
                                          (1, 3, 3, 129, 32), (2, 6, 3, 513, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_grouped_heads(cuda_lib, B, Hq, Hkv, T, d, causal, dtype):
    """dK and dV of a KV head sum the contributions of every query head that
    reads it (MQA, GQA and MHA)."""
    got, ref = run_bwd(cuda_lib, B, Hq, Hkv, T, d, dtype, causal, seed=B + Hq + T)
    check_grads(got, ref, dtype, f"B={B} Hq={Hq} Hkv={Hkv} T={T} d={d} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("window", [(0, 0), (3, 3), (64, 64), (100, 0), (0, 200), (-1, 50),
                                    (300, -1), (127, 128)])
@pytest.mark.parametrize("T,d", [(129, 64), (640, 128)])
def test_bwd_window(cuda_lib, T, d, window, dtype):
    """Band masks: only the blocks inside the band are visited."""
    got, ref = run_bwd(cuda_lib, 1, 2, 1, T, d, dtype, False, window=window,
                       seed=T + window[0] + 3 * window[1])
    check_grads(got, ref, dtype, f"window={window} T={T} d={d} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [0.0, -0.09, 0.7])
def test_bwd_scales(cuda_lib, scale, dtype):
    """Zero, negative and large scales (scale 0: uniform P, dS from dP - D)."""
    got, ref = run_bwd(cuda_lib, 1, 2, 2, 300, 64, dtype, True, scale=scale, seed=11)
    check_grads(got, ref, dtype, f"scale={scale} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_after_library_forward(cuda_lib, causal, dtype):
    """The usual call sequence: O and LSE from this library's forward."""
    got, ref = run_bwd(cuda_lib, 2, 4, 2, 700, 128, dtype, causal, seed=3, library_fwd=True)
    check_grads(got, ref, dtype, f"library forward causal={causal} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_is_deterministic_and_leaves_inputs(cuda_lib, dtype):
    """No gradient is accumulated by atomics: two calls agree bit for bit;
    inputs are unchanged; nothing is written around the outputs."""
    fa = cuda_lib
    B, Hq, Hkv, T, d = 2, 4, 1, 333, 64
    q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=4))
    do = make_grad_out(B, Hq, T, d, dtype=dtype, seed=4).cuda()
    o, lse = fa.fwd(q, k, v, causal=True)
    snap = [x.clone() for x in (q, k, v, o, lse, do)]
    pad = 4096
    bufs = [torch.full((x.numel() + 2 * pad,), 7.0, dtype=x.dtype, device="cuda")
            for x in (q, k, v)]
    dq, dk, dv = (b[pad:pad + x.numel()].view(x.shape) for b, x in zip(bufs, (q, k, v)))
    fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    first = [x.clone() for x in (dq, dk, dv)]
    fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    for a, b in zip(first, (dq, dk, dv)):
        assert torch.equal(a, b)
    for a, b in zip(snap, (q, k, v, o, lse, do)):
        assert torch.equal(a, b)
    for b in bufs:
        assert bool((b[:pad] == 7.0).all()) and bool((b[-pad:] == 7.0).all())


def test_bwd_on_a_side_stream(cuda_lib):
    fa = cuda_lib
    q, k, v = (x.cuda() for x in make_qkv(1, 2, 2, 256, 128, dtype="bf16", seed=6))
    do = make_grad_out(1, 2, 256, 128, dtype="bf16", seed=6).cuda()
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        got = fa.bwd(q, k, v, o, lse, do, causal=True, stream=s.cuda_stream)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,T,d,causal", [(64, 1, 4096, 128, True), (16, 12, 1024, 64, True),
                                            (1, 16, 8192, 128, False)])
def test_bwd_full_size_sampled_heads(cuda_lib, B, H, T, d, causal):
    """Workload sizes (the causal d=128 T=4096 sweep point, the GPT-2 layer,
    a long sequence): the whole launch runs; two (b, h) heads are compared in
    full with the oracle (a head's gradients depend only on that head)."""
    fa = cuda_lib
    q, k, v = make_qkv(B, H, H, T, d, dtype="bf16", seed=B + T)
    do = make_grad_out(B, H, T, d, dtype="bf16", seed=B + T)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    for b, h in ((0, 0), (B - 1, H - 1)):
        ref = oracle.attention_bwd_head_ref(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
        check_grads((dq[b, h], dk[b, h], dv[b, h]), ref, "bf16", f"head ({b},{h}) T={T}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T,d,w,tokens", [(129, 32, 0, [0]), (640, 128, 5, [0, 1, 2, 3]),
                                          (1000, 64, 64, [999, 17, 17, -4, 1500, 300]),
                                          (777, 16, 2, []), (2500, 128, 100, "strided")])
def test_bwd_local_global(cuda_lib, T, d, w, tokens, causal, dtype):
    """Backward of the local-global mask: key tiles holding a global key are
    visited by every query step (dK, dV) and by every row tile (dQ)."""
    fa = cuda_lib
    g = list(range(7, T, 113)) if tokens == "strided" else tokens
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(1, 2, 1, T, d, dtype=dtype, seed=T + w)
    do = make_grad_out(1, 2, T, d, dtype=dtype, seed=T + w)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    gt = torch.tensor(g, dtype=torch.int32, device="cuda")
    O, L = oracle.attention_ref(q, k, v, scale, causal, window=(w, w), global_tokens=g)
    o = torch.from_numpy(O).to(DTYPES[dtype]).cuda()
    lse = torch.from_numpy(L).to(torch.float32).cuda()
    grads = fa.bwd(qc, kc, vc, o, lse, doc, causal=causal, scale=scale, window=(w, w),
                   global_tokens=gt)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    ref = oracle.attention_bwd_ref(q, k, v, do, scale, causal, window=(w, w), global_tokens=g)
    check_grads(grads, ref, dtype, f"local-global T={T} d={d} w={w} causal={causal} {dtype}")
