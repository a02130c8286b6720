"""fa_fwd_host: host buffers in and out, batch chunks pipelined over two
streams.  The chunks run the same kernels on the same per-head data as one
device call, so the results are the device call's bits."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import make_qkv
from parity_util import TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("chunks", [1, 2, 3, 64])
def test_host_forward_matches_device_forward(cuda_lib, chunks, dtype):
    fa = cuda_lib
    B, Hq, Hkv, T, d = 5, 4, 2, 333, 64
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=51)
    qp, kp, vp = (x.pin_memory() for x in (q, k, v))
    o, lse = fa.fwd_host(qp, kp, vp, causal=True, chunks=chunks)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    od, ld = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
    O_ref, L_ref = oracle.attention_ref(q, k, v, 1 / math.sqrt(d), True)
    assert float(np.max(np.abs(oracle.as_f64(o) - O_ref))) <= TOL[dtype][0]
    assert float(np.max(np.abs(oracle.as_f64(lse) - L_ref))) <= TOL[dtype][1]


def test_host_forward_pageable_memory_and_side_stream(cuda_lib):
    """Pageable host buffers work (without overlap); the call orders after
    the given stream and the stream after it."""
    fa = cuda_lib
    B, H, T, d = 3, 2, 500, 128
    q, k, v = make_qkv(B, H, H, T, d, dtype="bf16", seed=52)
    s = torch.cuda.Stream()
    o, lse = fa.fwd_host(q, k, v, chunks=2, stream=s.cuda_stream,
                         out=torch.empty(q.shape, dtype=q.dtype),
                         lse=torch.empty((B, H, T), dtype=torch.float32))
    s.synchronize()
    assert fa.fa_debug_sync_check(s.cuda_stream) == 0
    od, ld = fa.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_host_forward_rejects_bad_arguments(cuda_lib):
    fa = cuda_lib
    q, k, v = make_qkv(2, 2, 2, 64, 64, dtype="bf16", seed=53)
    o = torch.empty_like(q)
    lse = torch.empty((2, 2, 64), dtype=torch.float32)
    need = fa.fa_fwd_host_workspace_size(2, 2, 2, 64, 64, fa.FA_DTYPE_BF16, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (q, k, v, o, lse, 2, 2, 2, 64, 64, 0.125, 0, fa.FA_DTYPE_BF16)
    assert fa.fa_fwd_host(*args, 0, ws, need) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_host(*args, 2, ws, need - 16) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_host(*args, 2, 0, need) == fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("chunks,window", [(1, None), (2, (40, 0)), (3, None), (8, (16, 16))])
def test_host_backward_matches_device_backward(cuda_lib, chunks, window, dtype):
    from exact_attention_90_gb300.inputs import make_grad_out

    fa = cuda_lib
    B, Hq, Hkv, T, d = 5, 4, 2, 300, 64
    q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype=dtype, seed=54)
    do = make_grad_out(B, Hq, T, d, dtype=dtype, seed=54)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    o, lse = fa.fwd(qc, kc, vc, causal=True, window=window)
    ref = fa.bwd(qc, kc, vc, o, lse, doc, causal=True, window=window)
    torch.cuda.synchronize()
    pinned = [x.pin_memory() for x in (q, k, v, o.cpu(), lse.cpu(), do)]
    got = fa.bwd_host(*pinned, causal=True, window=window, chunks=chunks)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b.cpu())
