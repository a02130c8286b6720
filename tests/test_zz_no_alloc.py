"""The split-KV entry point for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: a plugin hosted by an
application that hands out all device memory through its own pool, or a
latency-critical path that cannot afford cudaMalloc's implicit device-wide
synchronisation.  fa_fwd_split_static serves them with a fixed scratch array
inside the library.  This file is collected last on purpose: a run that stops
at the first failure has run every other test before this one.
"""

import math

import pytest
import torch

from exact_attention_90_gb300.inputs import make_qkv
from parity_util import check_full

pytestmark = pytest.mark.gpu


def _split_with_workspace(fa, q, k, v, causal, scale, splits):
    """The existing entry point, fa_fwd_split, with a torch-allocated workspace."""
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    nbytes = fa.fa_fwd_split_workspace_size(B, Hq, T, d, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    code = fa.FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else fa.FA_DTYPE_F16
    assert fa.fa_fwd_split(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, int(causal), code, splits,
                           ws, nbytes) == 0
    torch.cuda.synchronize()
    return o, lse


def _split_static(fa, q, k, v, causal, scale, splits):
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    code = fa.FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else fa.FA_DTYPE_F16
    assert fa.fa_fwd_split_static(q, k, v, o, lse, B, Hq, Hkv, T, d, scale, int(causal), code,
                                  splits) == 0
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    return o, lse


def test_static_scratch_matches_caller_workspace_on_two_calls_in_a_row(cuda_lib):
    """Both entry points run the same kernels with the same split count on the
    same inputs, and the kernels are deterministic: the results must agree bit
    for bit.  A tolerance would hide a partial read of stale scratch left by
    the first call in the one shared array.  Each result is also checked
    against the fp64 oracle."""
    fa = cuda_lib
    cases = [  # two calls in a row, different shapes and inputs on the one array;
        # the second needs less scratch than the first, so stale partials of
        # the first call lie where a wrong offset of the second would read
        (1, 2, 1, 4096, 128, True, 8, 31),
        (1, 1, 1, 3000, 64, False, 5, 32),
    ]
    for (B, Hq, Hkv, T, d, causal, splits, seed) in cases:
        q, k, v = make_qkv(B, Hq, Hkv, T, d, dtype="bf16", seed=seed, device="cuda")
        scale = 1.0 / math.sqrt(d)
        o_ref, l_ref = _split_with_workspace(fa, q, k, v, causal, scale, splits)
        o, lse = _split_static(fa, q, k, v, causal, scale, splits)
        assert torch.equal(o, o_ref), "static-scratch O differs from fa_fwd_split's"
        assert torch.equal(lse, l_ref), "static-scratch LSE differs from fa_fwd_split's"
        check_full(o, lse, q, k, v, scale, causal, what=f"static scratch T{T} d{d}")


def test_static_scratch_rejects_shapes_beyond_its_size(cuda_lib):
    """More partial results than the 64 MiB array holds: refused up front
    with FA_ERR_WORKSPACE, nothing launched."""
    fa = cuda_lib
    B, Hq, T, d, splits = 4, 8, 4096, 128, 8
    assert fa.fa_fwd_split_workspace_size(B, Hq, T, d, splits) > 64 << 20
    q, k, v = make_qkv(B, Hq, Hq, T, d, dtype="bf16", seed=1, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_split_static(q, k, v, o, lse, B, Hq, Hq, T, d, 0.1, 1, fa.FA_DTYPE_BF16,
                                splits)
    assert st == fa.FA_ERR_WORKSPACE
