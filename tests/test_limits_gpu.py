"""Sizes at the edges: very long sequences and very many heads.

At these sizes the full oracle would take too long, so rows are sampled
(a row of O, LSE and dQ depends only on that query row) and the key-side
gradients are checked through properties that hold at any size:
sum_j dK_j = 0 (every row of dS sums to zero) and sum_j dV_j = sum_i dO_i
(every row of P sums to one), per KV head.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import make_grad_out, make_qkv
from parity_util import TOL, sample_rows

pytestmark = pytest.mark.gpu


def test_forward_long_sequence_131072(cuda_lib):
    fa = cuda_lib
    B, H, T, d = 1, 2, 131072, 128
    q, k, v = make_qkv(B, H, H, T, d, dtype="bf16", seed=41)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    oc, lc = o.cpu(), lse.cpu()
    for h in range(H):
        rows = sample_rows(T, 24, seed=h)
        O_ref, L_ref = oracle.attention_rows_ref(q, k, v, scale, True, 0, h, rows)
        assert float(np.max(np.abs(oracle.as_f64(oc[0, h, rows]) - O_ref))) <= TOL["bf16"][0]
        assert float(np.max(np.abs(oracle.as_f64(lc[0, h, rows]) - L_ref))) <= TOL["bf16"][1]


def test_forward_many_heads(cuda_lib):
    """8192 (b, h) heads of a short sequence: unit indexing over a long grid."""
    fa = cuda_lib
    B, Hq, Hkv, T, d = 512, 16, 4, 200, 64
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype="bf16", seed=42)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=False, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    oc, lc = o.cpu(), lse.cpu()
    for b, h in ((0, 0), (B - 1, Hq - 1), (257, 9)):
        rows = np.arange(T)
        O_ref, L_ref = oracle.attention_rows_ref(q, k, v, scale, False, b, h, rows)
        assert float(np.max(np.abs(oracle.as_f64(oc[b, h]) - O_ref))) <= TOL["bf16"][0]
        assert float(np.max(np.abs(oracle.as_f64(lc[b, h]) - L_ref))) <= TOL["bf16"][1]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_long_sequence_32768(cuda_lib, dtype):
    fa = cuda_lib
    B, Hq, Hkv, T, d = 1, 2, 1, 32768, 64
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=43)
    do = make_grad_out(B, Hq, T, d, dtype=dtype, seed=43)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    o, lse = fa.fwd(qc, kc, vc, causal=True, scale=scale)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    tol = {"bf16": 2e-2, "f32": 1e-4}[dtype]
    dqc = oracle.as_f64(dq.cpu())
    for h in range(Hq):
        rows = sample_rows(T, 16, seed=10 + h)
        ref = oracle.attention_bwd_dq_rows_ref(q, k, v, do, scale, True, 0, h, rows)
        err = float(np.max(np.abs(dqc[0, h, rows] - ref)))
        assert err <= tol * max(float(np.max(np.abs(ref))), 0.1), f"dQ rows head {h}: {err:.3g}"
    # key-side properties, per KV head (in fp64 of the returned values)
    dkc, dvc = oracle.as_f64(dk.cpu()), oracle.as_f64(dv.cpu())
    do64 = oracle.as_f64(do)
    ksum = dkc[0, 0].sum(axis=0)
    vsum = dvc[0, 0].sum(axis=0)
    vref = do64[0].sum(axis=(0, 1))  # both query heads share KV head 0
    kscale = np.abs(dkc[0, 0]).sum(axis=0)
    # the sums cancel exactly in exact arithmetic; what remains is the
    # rounding of the T summands (bf16: about 2^-9 each, fp32: 2^-24 each)
    rel = {"bf16": 2e-2, "f32": 1e-4}[dtype]
    assert np.all(np.abs(ksum) <= rel * kscale + 1e-6), "sum_j dK_j is not ~0"
    assert np.all(np.abs(vsum - vref) <= rel * np.abs(dvc[0, 0]).sum(axis=0) + 1e-6), \
        "sum_j dV_j differs from sum_i dO_i"
