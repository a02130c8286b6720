"""Naive four-step attention in fp64: the oracle's definition of the method.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Sources (web pages; cited by page and section):
  [en]  "Flash Attention Memory Optimization Explained",
        lzwjava.github.io/flash-attention-memory-en
  [zh]  "Flash Attention内存优化原理解析", lzwjava.github.io/flash-attention-memory-zh
        (Chinese twin of [en])
  [tri] yelogs.com tutorial "Flash Attention2 ... Triton" (Traditional Chinese),
        yelogs.com/u/u_17583190/story/499f2d6e-1697-42a6-83e0-56a4579cb114

What the method computes.  [en] "What is Flash Attention?" (and [zh] "什么是
Flash Attention？") states that FlashAttention is an *exact* implementation of
scaled dot-product attention and lists the naive pipeline it replaces: scores
Q@K^T, scale and mask, softmax, weighted sum attention@V.  [tri] section
"內存牆：注意力機制的阿喀琉斯之踵" prints the same pipeline as code (scores by a
dot over d, divide by sqrt(d_model), masked_fill, softmax, dot with V).  The
kernel in [tri] "核心 Kernel 實現" additionally writes, per query row, the
log-sum-exp L = m + log(l) of the scaled, masked score row.  Because the method
reaches the naive result exactly (up to rounding order), the oracle is that
definition written out, in fp64:

  for every batch b, query head h (KV head hk = h // (Hq // Hkv)):
    S[i, j]  = scale * sum_c Q[b,h,i,c] * K[b,hk,j,c]
    valid    = { j : j < T }                      (non-causal)
             = { j : j <= i }                     (causal, top-left aligned)
    m_i      = max_{j valid} S[i, j]
    l_i      = sum_{j valid} exp(S[i, j] - m_i)
    P[i, j]  = exp(S[i, j] - m_i) / l_i   for valid j, 0 otherwise
    O[i, :]  = sum_j P[i, j] * V[b,hk,j,:]
    LSE[i]   = m_i + ln(l_i)

Readings of points the pages leave open or print inconsistently:
  * causal keeps j <= i: the kernel's mask in [tri] "核心 Kernel 實現" keeps
    offs_q >= offs_k.  Masked entries are excluded from the softmax, which is
    the common limit of the -1e9 fill of the naive listing and the -inf fill
    of the kernel (every causal row keeps j = i, so the two agree).
  * LSE uses the natural log and no epsilon: the kernel's `log(l + eps)` with
    eps ~ 1e-6 ([tri] "常見問題及解決方案") only guards l = 0, which cannot
    happen because l >= 1 (the maximal term contributes exp(0) = 1).
  * scale multiplies the fp64 score; the naive listing divides scores by
    sqrt(d) and the kernel multiplies Q by the scale before the dot: both are
    the same real number, the oracle takes the plain definition.
  * sliding windows: [tri] "1. 稀疏注意力支持" keeps key j for query i when
    |i - j| <= window_size.  The oracle takes a band window = (wl, wr): keep j
    when i - wl <= j <= i + wr, -1 meaning unbounded on that side; the page's
    window is (w, w), causal attention is (-1, 0), and `causal` combines with
    a window by intersection.
  * local-global: the same passage keeps key j for query i when
    |i - j| <= local_window OR j is one of the listed global tokens
    (torch.isin over the key index): global tokens are keys every query
    attends to.  The oracle takes global_tokens as a list of key indices;
    entries outside [0, T) and repeats select nothing more (isin semantics);
    with `causal` the union is intersected with j <= i.
  * MQA/GQA: [tri] "2. 多查詢注意力（MQA）" broadcasts a single KV head to all
    query heads; the grouped generalisation maps query head h to KV head
    h // (Hq // Hkv) (equivalently repeat_interleave of K, V along heads).
"""

from __future__ import annotations

import numpy as np


def as_f64(x) -> np.ndarray:
    """Exact conversion of a NumPy array or a (CPU or CUDA) torch tensor to fp64.

    bf16 and fp32 values are exactly representable in fp64, so the oracle sees
    the very same numbers as the device path.
    """
    if hasattr(x, "detach"):  # torch tensor, imported lazily
        import torch

        return x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """KV head read by query head ``h``: all heads share one KV head for MQA
    ([tri] "2. 多查詢注意力（MQA）": K, V broadcast over query heads); groups of
    Hq // Hkv consecutive query heads share one for GQA."""
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} must be a positive multiple of Hkv={Hkv}")
    return h // (Hq // Hkv)


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, T, d]")
    B, Hq, T, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != T or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} is not a multiple of Hkv={Hkv}")
    return B, Hq, Hkv, T, d


def valid_keys(rows, T, causal, window=None, global_tokens=None):
    """Boolean [len(rows), T]: key j is kept for query row i (the mask).

    With ``global_tokens`` (the local-global mask of [tri] "1. 稀疏注意力支持")
    the band ``window`` is the local part and the listed keys are kept for
    every row as well: (band | isin(j, global_tokens)) & causal.
    """
    j = np.arange(T)[None, :]
    i = np.asarray(rows)[:, None]
    band = np.ones((len(rows), T), dtype=bool)
    if window is not None:
        wl, wr = window
        if wl >= 0:
            band &= j >= i - wl
        if wr >= 0:
            band &= j <= i + wr
    if global_tokens is not None:
        band |= np.isin(j, np.asarray(global_tokens, dtype=np.int64))
    if causal:
        band &= j <= i                                # keep j <= i
    return band


def _rows_of_head(qh, kh, vh, rows, scale, causal, window=None, global_tokens=None):
    """The four naive steps for the query rows ``rows`` of one head (fp64).

    Step 1 (scores) and step 4 (weighted sum) are dense products; steps 2 and 3
    (scale + mask, softmax with the row maximum subtracted) follow the naive
    listing in [tri] "內存牆" and the max-subtracted softmax of [tri]
    "核心思想：分塊計算與在線更新" (traditional_softmax).
    """
    T = kh.shape[0]
    s = (qh[rows] @ kh.T) * scale                     # step 1 + scale
    valid = valid_keys(rows, T, causal, window, global_tokens)
    s = np.where(valid, s, -np.inf)                   # step 2: mask (excluded)
    m = s.max(axis=1)                                 # row maximum
    e = np.where(valid, np.exp(s - m[:, None]), 0.0)  # step 3: softmax numerator
    l = e.sum(axis=1)                                 # normaliser
    o = (e @ vh) / l[:, None]                         # step 4: weighted sum
    lse = m + np.log(l)                               # L = m + ln l
    return o, lse, e / l[:, None]


def attention_ref(q, k, v, scale: float, causal: bool, row_chunk: int = 256, window=None,
                  global_tokens=None):
    """Exact attention forward by its definition, fp64.

    Args:
      q: [B, Hq, T, d]; k, v: [B, Hkv, T, d] (any real dtype, numpy or torch).
      scale: multiplies every score (1/sqrt(d) in the pages' workloads).
      causal: keep key j for query i iff j <= i.
      row_chunk: rows of S formed at once (memory O(row_chunk * T)); only the
        grouping of independent rows, no reordering of any sum.
      window: optional band (wl, wr): keep key j for query i iff
        i - wl <= j <= i + wr (-1 = unbounded side); every row must keep at
        least one key (true whenever wl, wr are -1 or >= 0).
      global_tokens: optional key indices kept for every row in addition to
        the band (the local-global mask; the page's local window is
        window = (w, w)).

    Returns:
      (O, LSE): O [B, Hq, T, d] fp64, LSE [B, Hq, T] fp64 (natural log).
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, Hkv, T, d = _check_shapes(q, k, v)
    O = np.empty((B, Hq, T, d), dtype=np.float64)
    L = np.empty((B, Hq, T), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            for r0 in range(0, T, row_chunk):
                rows = np.arange(r0, min(T, r0 + row_chunk))
                o, lse, _ = _rows_of_head(q[b, h], k[b, hk], v[b, hk], rows, scale, causal,
                                          window, global_tokens)
                O[b, h, rows] = o
                L[b, h, rows] = lse
    return O, L


def attention_rows_ref(q, k, v, scale: float, causal: bool, b: int, h: int, rows, window=None,
                       global_tokens=None):
    """The definition evaluated for selected query rows of one (b, h) only.

    Used for parity at full workload sizes, where the whole oracle would take
    too long: the result for a row depends only on that row of Q and on the
    KV head, so sampling rows is exact.

    Returns (O_rows [len(rows), d], LSE_rows [len(rows)]) in fp64.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, Hkv, T, d = _check_shapes(q, k, v)
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= T):
        raise ValueError("row index out of range")
    hk = kv_head_of(h, Hq, Hkv)
    o, lse, _ = _rows_of_head(q[b, h], k[b, hk], v[b, hk], rows, scale, causal, window,
                              global_tokens)
    return o, lse


def attention_probs_ref(q, k, v, scale: float, causal: bool, window=None, global_tokens=None):
    """The full probability matrix P [B, Hq, T, T] (fp64); small cases only."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, Hkv, T, d = _check_shapes(q, k, v)
    P = np.zeros((B, Hq, T, T), dtype=np.float64)
    rows = np.arange(T)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            _, _, p = _rows_of_head(q[b, h], k[b, hk], v[b, hk], rows, scale, causal, window,
                                    global_tokens)
            P[b, h] = p
    return P


def naive_score_bytes(T: int, elem_bytes: int) -> int:
    """Bytes of the T x T attention matrix that the naive path materialises per
    (batch, head): the memory table of [tri] "性能瓶頸的量化分析" (fp16, 2 bytes
    per element) and the "huge matrix" of [en] "What is Flash Attention?"."""
    return int(T) * int(T) * int(elem_bytes)
