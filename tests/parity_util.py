"""Helpers shared by the GPU parity tests: tolerances, sampled-row checks."""

import numpy as np
import torch

import oracle

# Tolerances on max-abs error against the fp64 oracle (the stated targets):
#   fp32 inputs:                 O <= 1e-4, LSE <= 1e-5
#   bf16 inputs, fp32 accumulate: O <= 2e-2, LSE <= 2e-3
#   fp16 inputs (the pages' other tensor-core precision; no target stated):
#     the bf16 tolerances -- fp16 carries 3 more mantissa bits, so every
#     rounding in the path (P before the second product, O on output) is at
#     least as precise, and P <= 2^8, |O| < 8 stay far inside fp16's range.
TOL = {"f32": (1e-4, 1e-5), "bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3)}


def dtype_name(t: torch.Tensor) -> str:
    return {torch.bfloat16: "bf16", torch.float16: "f16"}.get(t.dtype, "f32")


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def check_full(o, lse, q, k, v, scale, causal, what=""):
    """Element-by-element comparison with the full oracle."""
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
    tol_o, tol_l = TOL[dtype_name(q)]
    O = oracle.as_f64(o)
    L = oracle.as_f64(lse)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), f"{what}: non-finite output"
    eo, el = max_abs(O, O_ref), max_abs(L, L_ref)
    assert eo <= tol_o and el <= tol_l, f"{what}: max|dO|={eo:.3g} (tol {tol_o}), max|dL|={el:.3g} (tol {tol_l})"
    return eo, el


def sample_rows(T: int, n_random: int, seed: int):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, T // 2, T - 1, min(T - 1, 127), min(T - 1, 128), min(T - 1, 255),
             min(T - 1, 256)}
    rand = set(rng.integers(0, T, size=min(n_random, T)).tolist())
    return np.array(sorted(fixed | rand), dtype=np.int64)


def check_sampled(o, lse, q, k, v, scale, causal, bh_pairs, n_rows=48, what="", seed=0):
    """Compare selected rows of selected (b, h) with the oracle evaluated row
    by row (exact for those rows: a row depends only on its own query)."""
    B, Hq, T, d = q.shape
    tol_o, tol_l = TOL[dtype_name(q)]
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    oc, lc = o.cpu(), lse.cpu()
    worst_o = worst_l = 0.0
    for i, (b, h) in enumerate(bh_pairs):
        rows = sample_rows(T, n_rows, seed + i)
        O_ref, L_ref = oracle.attention_rows_ref(qc, kc, vc, scale, causal, b, h, rows)
        O = oracle.as_f64(oc[b, h, rows])
        L = oracle.as_f64(lc[b, h, rows])
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), f"{what}: non-finite output"
        worst_o = max(worst_o, max_abs(O, O_ref))
        worst_l = max(worst_l, max_abs(L, L_ref))
    assert worst_o <= tol_o and worst_l <= tol_l, \
        f"{what}: max|dO|={worst_o:.3g} (tol {tol_o}), max|dL|={worst_l:.3g} (tol {tol_l})"
    return worst_o, worst_l


def spread_pairs(B, Hq, n=6, seed=0):
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (B - 1, Hq - 1), (B // 2, Hq // 2)}
    while len(pairs) < min(n, B * Hq):
        pairs.add((int(rng.integers(0, B)), int(rng.integers(0, Hq))))
    return sorted(pairs)
