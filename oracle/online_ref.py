"""The online-softmax recurrence in fp64 over an arbitrary key partition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the yelogs.com Flash Attention2/Triton tutorial: the state update of
section "核心思想：分塊計算與在線更新" (online_softmax_update), the equations of
section "Softmax 的在線計算"

    m_new = max(m_old, max(s_new))
    l_new = exp(m_old - m_new) * l_old + sum exp(s_new - m_new)

and, for the output, the per-block steps of section "核心 Kernel 實現": the
accumulator is rescaled by exp(m_old - m_new) before the block's weighted sum
is added, the result is divided by l at the end, and L = m + log(l).  The state
starts at m = -inf, l = 0, O = 0 (the flowchart of section "算法流程圖").

Its only use is to pin the statement of section "Softmax 的在線計算" that the
recurrence reproduces the batch softmax exactly: the tests run it over many
different partitions of the keys and compare with ``attention_ref``.
(The running-state formula printed in "Flash Attention Memory Optimization
Explained", section "Key Mechanisms", swaps the roles of the max and the
log-sum-exp and does not define a valid recurrence; the tutorial's version,
which matches the definition, is the one restated here.)
"""

from __future__ import annotations

import numpy as np

from .attention_ref import as_f64, kv_head_of


def attention_online_ref(q, k, v, scale: float, causal: bool, block_sizes, window=None):
    """O and LSE by the block recurrence.

    Args:
      block_sizes: positive ints; the keys are split into consecutive blocks
        of these sizes, cycling through the list until all T keys are covered.
    Returns (O [B,Hq,T,d], LSE [B,Hq,T]) in fp64.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    sizes = [int(s) for s in block_sizes]
    if not sizes or min(sizes) <= 0:
        raise ValueError("block sizes must be positive")
    O = np.empty((B, Hq, T, d))
    L = np.empty((B, Hq, T))
    rows = np.arange(T)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, Hq, Hkv)
            qh, kh, vh = q[b, h], k[b, hk], v[b, hk]
            m = np.full(T, -np.inf)   # running maximum
            l = np.zeros(T)           # running normaliser
            acc = np.zeros((T, d))    # unnormalised output
            c0, n = 0, 0
            while c0 < T:
                c1 = min(T, c0 + sizes[n % len(sizes)])
                cols = np.arange(c0, c1)
                s = (qh @ kh[c0:c1].T) * scale
                keep = np.ones(s.shape, dtype=bool)
                if causal:
                    keep &= rows[:, None] >= cols[None, :]
                if window is not None:
                    if window[0] >= 0:
                        keep &= cols[None, :] >= rows[:, None] - window[0]
                    if window[1] >= 0:
                        keep &= cols[None, :] <= rows[:, None] + window[1]
                s = np.where(keep, s, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                # a row that has seen only masked keys keeps m = -inf; its
                # correction factor and probabilities are then 0 by definition
                finite = np.isfinite(m_new)
                shift = np.where(finite, m_new, 0.0)
                alpha = np.where(finite, np.exp(m - shift), 1.0)
                p = np.exp(s - shift[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ vh[c0:c1]
                m = m_new
                c0, n = c1, n + 1
            O[b, h] = acc / l[:, None]
            L[b, h] = m + np.log(l)
    return O, L
