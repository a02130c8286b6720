"""Gradients of exact attention by the chain rule, fp64 (the backward oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Sources (cited by page and section):
  [en]  "Flash Attention Memory Optimization Explained", section "Key
        Mechanisms", item "Backward Checkpointing": the backward pass
        recomputes the forward's intermediates instead of storing them.
  [zh]  the Chinese twin of [en], "核心运行机制", item "反向传播检查点".
  [tri] yelogs.com Flash Attention2/Triton tutorial, "核心 Kernel 實現": the
        forward writes the per-row log-sum-exp L that the recomputation uses.

The pages name the backward pass but print no formula for it.  What it must
compute is fixed by the forward: the gradient of O = softmax(S) V with
S = scale * Q K^T (masked entries excluded) with respect to Q, K and V, for an
upstream gradient dO of O (the LSE output carries no gradient).  Written out
by the chain rule, for one (b, h) with KV head hk:

    P      = softmax of the masked, scaled score rows       (the forward's P)
    dV    += P^T dO                       (O = P V)
    dP     = dO V^T
    dS_ij  = P_ij * (dP_ij - sum_k P_ik dP_ik)   (Jacobian of a softmax row)
    dQ     = scale * dS K
    dK    += scale * dS^T Q

dK and dV of a KV head sum the contributions of every query head that reads
it (the grouped-head map of [tri] "2. 多查詢注意力（MQA）").  Masked entries
have P_ij = 0 and so contribute nothing.  The recomputation of [en] ("rebuild
P from the saved L") is an implementation choice of the fast path; the oracle
simply rebuilds P by the forward's definition.
"""

from __future__ import annotations

import numpy as np

from .attention_ref import _check_shapes, as_f64, kv_head_of, valid_keys


def attention_bwd_head_ref(qh, kh, vh, doh, scale: float, causal: bool, window=None,
                           row_chunk: int = 256, global_tokens=None):
    """The chain-rule gradients for one query head (2-D [T, d] fp64 arrays).

    Returns (dQ_h [T, d], dK_h [T, d], dV_h [T, d]): dQ of this query head and
    this head's contributions to the gradients of its KV head.  Rows are
    processed in chunks of ``row_chunk`` (only a grouping of independent query
    rows; every sum over keys is a plain product).
    """
    qh, kh, vh, doh = as_f64(qh), as_f64(kh), as_f64(vh), as_f64(doh)
    T, d = qh.shape
    dq = np.zeros((T, d))
    dk = np.zeros((T, d))
    dv = np.zeros((T, d))
    for r0 in range(0, T, row_chunk):
        rows = np.arange(r0, min(T, r0 + row_chunk))
        s = (qh[rows] @ kh.T) * scale
        valid = valid_keys(rows, T, causal, window, global_tokens)
        s = np.where(valid, s, -np.inf)
        m = s.max(axis=1)
        e = np.where(valid, np.exp(s - m[:, None]), 0.0)
        p = e / e.sum(axis=1)[:, None]                      # P rows (forward's)
        dv += p.T @ doh[rows]                               # dV += P^T dO
        dp = doh[rows] @ vh.T                               # dP = dO V^T
        ds = p * (dp - (p * dp).sum(axis=1)[:, None])       # softmax Jacobian
        dq[rows] = scale * (ds @ kh)                        # dQ = scale dS K
        dk += scale * (ds.T @ qh[rows])                     # dK += scale dS^T Q
    return dq, dk, dv


def attention_bwd_ref(q, k, v, do, scale: float, causal: bool, window=None,
                      row_chunk: int = 256, global_tokens=None):
    """Gradients of the attention forward with respect to Q, K and V (fp64).

    Args:
      q: [B, Hq, T, d]; k, v: [B, Hkv, T, d]; do: [B, Hq, T, d], the
        upstream gradient of O (any real dtype, numpy or torch).
      scale, causal, window, global_tokens: as for ``attention_ref``.

    Returns:
      (dQ [B, Hq, T, d], dK [B, Hkv, T, d], dV [B, Hkv, T, d]) in fp64.
    """
    q, k, v, do = as_f64(q), as_f64(k), as_f64(v), as_f64(do)
    B, Hq, Hkv, T, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError(f"do{do.shape} must have the shape of q{q.shape}")
    dQ = np.zeros((B, Hq, T, d))
    dK = np.zeros((B, Hkv, T, d))
    dV = np.zeros((B, Hkv, T, d))
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            dq, dk, dv = attention_bwd_head_ref(q[b, h], k[b, hk], v[b, hk], do[b, h], scale,
                                                causal, window, row_chunk, global_tokens)
            dQ[b, h] = dq
            dK[b, hk] += dk
            dV[b, hk] += dv
    return dQ, dK, dV


def attention_bwd_dq_rows_ref(q, k, v, do, scale: float, causal: bool, b: int, h: int, rows,
                              window=None, global_tokens=None):
    """dQ for selected query rows of one (b, h) only (fp64).

    Exact for those rows: dQ_i = scale * sum_j dS_ij k_j needs only row i of
    P and dP (and so only row i of Q and dO), which makes full-size checks
    of dQ affordable.  Returns dQ_rows [len(rows), d].
    """
    q, k, v, do = as_f64(q), as_f64(k), as_f64(v), as_f64(do)
    B, Hq, Hkv, T, d = _check_shapes(q, k, v)
    rows = np.asarray(rows, dtype=np.int64)
    hk = kv_head_of(h, Hq, Hkv)
    kh, vh = k[b, hk], v[b, hk]
    s = (q[b, h][rows] @ kh.T) * scale
    valid = valid_keys(rows, T, causal, window, global_tokens)
    s = np.where(valid, s, -np.inf)
    e = np.where(valid, np.exp(s - s.max(axis=1)[:, None]), 0.0)
    p = e / e.sum(axis=1)[:, None]
    dp = do[b, h][rows] @ vh.T
    ds = p * (dp - (p * dp).sum(axis=1)[:, None])
    return scale * (ds @ kh)
