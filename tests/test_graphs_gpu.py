"""fa_fwd, fa_bwd, fa_fwd_split and fa_fwd_local_global under CUDA-graph capture.

These calls allocate, free and synchronise nothing, so a sequence of them is
captured once and replayed: the replay must give the same bits as direct
calls, and the same results as the fp64 oracle.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_90_gb300.inputs import make_grad_out, make_qkv
from parity_util import TOL

pytestmark = pytest.mark.gpu


def test_forward_and_backward_replay_from_a_graph(cuda_lib):
    fa = cuda_lib
    B, Hq, Hkv, T, d = 2, 4, 2, 700, 128
    q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, T, d, dtype="bf16", seed=31))
    do = make_grad_out(B, Hq, T, d, dtype="bf16", seed=31).cuda()
    scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, Hq, T), dtype=torch.uint8, device="cuda")
    code = fa.FA_DTYPE_BF16

    def step(stream):
        assert fa.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, 1, code, stream) == 0
        assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, T, d, scale, 1, -1, -1, code,
                         ws, ws.numel(), stream) == 0

    # direct calls first (the first call of an instantiation sets its attributes)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s.cuda_stream)
    torch.cuda.synchronize()
    ref = [x.clone() for x in (o, lse, dq, dk, dv)]
    for x in (o, lse, dq, dk, dv):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream().cuda_stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    for a, b in zip(ref, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b)
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, True)
    assert float(np.max(np.abs(oracle.as_f64(o) - O_ref))) <= TOL["bf16"][0]
    assert float(np.max(np.abs(oracle.as_f64(lse) - L_ref))) <= TOL["bf16"][1]


def test_split_and_local_global_replay_from_a_graph(cuda_lib):
    """The paths with a caller workspace and several launches per call."""
    fa = cuda_lib
    B, H, T, d = 1, 2, 2048, 64
    q, k, v = (x.cuda() for x in make_qkv(B, H, H, T, d, dtype="bf16", seed=32))
    scale = 1.0 / math.sqrt(d)
    code = fa.FA_DTYPE_BF16
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    splits = 4
    ws1 = torch.empty(fa.fa_fwd_split_workspace_size(B, H, T, d, splits), dtype=torch.uint8,
                      device="cuda")
    gt = torch.tensor([0, 1, 2, 3, 1500], dtype=torch.int32, device="cuda")
    ws2 = torch.empty(fa.fa_fwd_local_global_workspace_size(T), dtype=torch.uint8, device="cuda")

    def step(stream):
        assert fa.fa_fwd_split(q, k, v, o1, l1, B, H, H, T, d, scale, 1, code, splits, ws1,
                               ws1.numel(), stream) == 0
        assert fa.fa_fwd_local_global(q, k, v, o2, l2, B, H, H, T, d, scale, 1, 16, gt,
                                      gt.numel(), code, ws2, ws2.numel(), stream) == 0

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s.cuda_stream)
    torch.cuda.synchronize()
    ref = [x.clone() for x in (o1, l1, o2, l2)]
    for x in (o1, l1, o2, l2):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream().cuda_stream)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    for a, b in zip(ref, (o1, l1, o2, l2)):
        assert torch.equal(a, b)
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, True, window=(16, 16),
                                        global_tokens=gt.cpu().tolist())
    assert float(np.max(np.abs(oracle.as_f64(o2) - O_ref))) <= TOL["bf16"][0]
    assert float(np.max(np.abs(oracle.as_f64(l2) - L_ref))) <= TOL["bf16"][1]
