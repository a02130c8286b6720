"""CPU oracle for the exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
anything in this package: only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it, to check
and to time the CUDA path.  It shares no code with the CUDA path; the seeded
input generators live in ``exact_attention_90_gb300.inputs`` and hold none of
the method's arithmetic.

Contents (each function cites the passage it follows):

* ``attention_ref``      -- the naive four-step definition in fp64 (scores,
                            scale + mask, softmax, weighted sum) plus the
                            per-row log-sum-exp.  This is the oracle.
* ``attention_rows_ref`` -- the same definition evaluated for a chosen set of
                            query rows only (full-size parity by sampling).
* ``attention_probs_ref``-- the full probability matrix, small cases only.
* ``attention_online_ref`` -- the online-softmax recurrence in fp64 over an
                            arbitrary partition of the keys; used only to pin
                            the statement that the recurrence reproduces the
                            batch softmax.
* ``attention_brute``    -- scalar pure-Python loops with ``math.fsum``, tiny
                            inputs only; an independent restatement used to pin
                            ``attention_ref``.
* ``attention_bwd_ref``  -- the gradients of the forward with respect to Q, K
                            and V for an upstream gradient dO, by the chain
                            rule in fp64 (the backward oracle);
                            ``attention_bwd_head_ref`` is its one-head step,
                            ``attention_bwd_dq_rows_ref`` dQ for chosen rows.
* ``naive_score_bytes``  -- bytes of the T x T score matrix that the naive path
                            materialises (the pages' memory table).

Parity status: every function above is pinned by ``tests/test_oracle.py``
(closed forms, brute force, a library special case, invariants, and the pages'
printed memory table); the backward by ``tests/test_oracle_bwd.py`` (finite
differences of the forward, torch autograd, invariants, closed forms).  Nothing here is "parity unpinned".
"""

from .attention_ref import (
    as_f64,
    attention_probs_ref,
    attention_ref,
    attention_rows_ref,
    kv_head_of,
    naive_score_bytes,
    valid_keys,
)
from .attention_bwd_ref import attention_bwd_dq_rows_ref, attention_bwd_head_ref, attention_bwd_ref
from .brute import attention_brute
from .online_ref import attention_online_ref

__all__ = [
    "as_f64",
    "attention_ref",
    "attention_rows_ref",
    "attention_probs_ref",
    "attention_online_ref",
    "attention_brute",
    "attention_bwd_ref",
    "attention_bwd_head_ref",
    "attention_bwd_dq_rows_ref",
    "kv_head_of",
    "naive_score_bytes",
    "valid_keys",
]
