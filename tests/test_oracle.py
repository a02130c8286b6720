"""Pins for the fp64 CPU oracle (no GPU).

The oracle is pinned to things other than itself: brute force on tiny inputs,
closed forms, the library routine of the API the pages use
(torch's scaled_dot_product_attention, CPU, float64), invariants of the
definition, the online recurrence's stated equality with the batch softmax,
and the memory table the tutorial prints.  The last test plants plausible
mistakes in a copy of the oracle and checks that every one of them trips at
least one pin.

Sources: "Flash Attention Memory Optimization Explained" (lzwjava.github.io),
sections "What is Flash Attention?" and "How to Use It in Code"; yelogs.com
Flash Attention2/Triton tutorial, sections "內存牆：注意力機制的阿喀琉斯之踵",
"性能瓶頸的量化分析", "核心思想：分塊計算與在線更新", "核心 Kernel 實現",
"Softmax 的在線計算", "2. 多查詢注意力（MQA）".
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import importlib

ar_mod = importlib.import_module("oracle.attention_ref")
from exact_attention_90_gb300.inputs import make_qkv, make_structured_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(B, Hq, Hkv, T, d, seed, mult=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, T, d)) * mult
    k = rng.standard_normal((B, Hkv, T, d)) * mult
    v = rng.standard_normal((B, Hkv, T, d)) * mult
    return q, k, v


# --------------------------------------------------------------------------
# pins, written as functions of an oracle callable ref(q, k, v, scale, causal)
# so that the planted-mistake test can run them against mutated copies
# --------------------------------------------------------------------------

def pin_brute(ref):
    """ref equals the scalar pure-Python restatement for every tiny shape."""
    for T in range(1, 9):
        for d in (1, 2, 4):
            for causal in (False, True):
                for Hq, Hkv in ((2, 2), (2, 1), (4, 2)):
                    q, k, v = _rand(2, Hq, Hkv, T, d, seed=T * 100 + d * 10 + Hq + Hkv)
                    scale = 0.7
                    O, L = ref(q, k, v, scale, causal)
                    Ob, Lb = oracle.attention_brute(q, k, v, scale, causal)
                    np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-13)
                    np.testing.assert_allclose(L, np.array(Lb), rtol=0, atol=1e-13)


def pin_library_sdpa(ref):
    """ref equals torch's scaled_dot_product_attention (CPU, float64), the
    routine the pages call (section "How to Use It in Code"), and its LSE
    equals torch.logsumexp of the masked, scaled score rows."""
    for (B, H, T, d, causal, scale) in ((2, 3, 17, 8, True, 0.3), (1, 2, 33, 16, False, 0.25),
                                        (2, 2, 64, 32, True, 1 / math.sqrt(32))):
        q, k, v = _rand(B, H, H, T, d, seed=T + d)
        O, L = ref(q, k, v, scale, causal)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        Ot = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=None, dropout_p=0.0, is_causal=causal, scale=scale)
        np.testing.assert_allclose(O, Ot.numpy(), rtol=0, atol=1e-12)
        s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
        if causal:
            s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def pin_causal_row0(ref):
    """Causal row 0 sees key 0 only: O[0] = V[0] and LSE[0] = scale * q0.k0."""
    q, k, v = _rand(2, 4, 2, 19, 8, seed=7)
    scale = 0.37
    O, L = ref(q, k, v, scale, True)
    for b in range(2):
        for h in range(4):
            hk = h // 2
            assert np.array_equal(O[b, h, 0], v[b, hk, 0])
            want = scale * math.fsum(q[b, h, 0, c] * k[b, hk, 0, c] for c in range(8))
            assert abs(L[b, h, 0] - want) <= 1e-13


def pin_zero_query(ref):
    """Q = 0 makes every valid score 0: O[i] is the mean of V over the valid
    keys and LSE[i] = ln(#valid) (ln(i+1) causal, ln T otherwise)."""
    T, d = 23, 4
    _, k, v = _rand(1, 2, 2, T, d, seed=11)
    q = np.zeros((1, 2, T, d))
    for causal in (True, False):
        O, L = ref(q, k, v, 0.9, causal)
        for i in range(T):
            n = i + 1 if causal else T
            np.testing.assert_allclose(O[0, :, i], v[0, :, :n].mean(axis=1), rtol=0, atol=1e-14)
            np.testing.assert_allclose(L[0, :, i], math.log(n), rtol=0, atol=1e-14)


def pin_constant_values(ref):
    """V identical in every row gives O = that row, whatever the scores."""
    q, k, _ = _rand(1, 2, 1, 31, 8, seed=12)
    c = np.linspace(-2, 2, 8)
    v = np.broadcast_to(c, (1, 1, 31, 8)).copy()
    for causal in (True, False):
        O, _ = ref(q, k, v, 0.5, causal)
        np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), rtol=0, atol=1e-14)


def pin_key_shift(ref):
    """Adding u to every K row adds scale*q_i.u to every score of row i: O is
    unchanged and LSE[i] moves by scale*q_i.u."""
    q, k, v = _rand(1, 2, 2, 29, 8, seed=13)
    u = np.random.default_rng(5).standard_normal(8)
    for causal in (True, False):
        O0, L0 = ref(q, k, v, 0.4, causal)
        O1, L1 = ref(q, k + u, v, 0.4, causal)
        np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L1 - L0, 0.4 * (q @ u), rtol=0, atol=1e-12)


def pin_dominant_key(ref):
    """With huge scores the max-subtracted softmax must not overflow: each row
    puts all its weight on its largest valid score (no ties w.p. 1)."""
    T, d = 12, 4
    q, k, v = _rand(1, 1, 1, T, d, seed=14)
    scale = 1.0e5  # scores of order 1e5: exp() without the max shift overflows
    for causal in (True, False):
        O, L = ref(q, k, v, scale, causal)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
        s = scale * (q[0, 0] @ k[0, 0].T)
        for i in range(T):
            n = i + 1 if causal else T
            j = int(np.argmax(s[i, :n]))
            if n > 1:  # the runner-up is far enough below to carry no weight
                assert np.sort(s[i, :n])[-2] < s[i, j] - 60.0
            np.testing.assert_allclose(O[0, 0, i], v[0, 0, j], rtol=0, atol=1e-9)
            np.testing.assert_allclose(L[0, 0, i], s[i, j], rtol=1e-15, atol=1e-9)


def pin_grouped_heads(ref):
    """Grouped / multi-query KV equals plain multi-head attention on K, V
    repeated over each group of query heads (the broadcast of section
    "2. 多查詢注意力（MQA）")."""
    for Hq, Hkv in ((4, 1), (8, 2), (6, 3)):
        q, k, v = _rand(2, Hq, Hkv, 21, 8, seed=Hq * 10 + Hkv)
        g = Hq // Hkv
        kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
        for causal in (True, False):
            O, L = ref(q, k, v, 0.35, causal)
            Or, Lr = ref(q, kr, vr, 0.35, causal)
            np.testing.assert_array_equal(O, Or)
            np.testing.assert_array_equal(L, Lr)


def pin_head_mapping_brute(ref):
    """Head mapping h -> h // (Hq/Hkv) against the scalar restatement."""
    q, k, v = _rand(1, 6, 2, 5, 3, seed=15)
    for causal in (True, False):
        O, L = ref(q, k, v, 0.8, causal)
        Ob, Lb = oracle.attention_brute(q, k, v, 0.8, causal)
        np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-13)
        np.testing.assert_allclose(L, np.array(Lb), rtol=0, atol=1e-13)


def pin_window_library_sdpa(ref):
    """Band windows against torch's scaled_dot_product_attention (CPU,
    float64) with the explicit boolean mask |i - j| <= w of the tutorial's
    sliding_window_mask, and asymmetric bands, causal or not."""
    for (T, d, window, causal) in ((40, 8, (3, 3), False), (40, 8, (5, 0), False),
                                   (33, 16, (7, 2), True), (64, 8, (0, 10), False),
                                   (50, 4, (-1, 4), False), (50, 4, (6, -1), True)):
        q, k, v = _rand(1, 2, 2, T, d, seed=T + d + window[0])
        O, L = ref(q, k, v, 0.4, causal, window=window)
        i = torch.arange(T)[:, None]
        j = torch.arange(T)[None, :]
        keep = torch.ones(T, T, dtype=torch.bool)
        if causal:
            keep &= j <= i
        if window[0] >= 0:
            keep &= j >= i - window[0]
        if window[1] >= 0:
            keep &= j <= i + window[1]
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        Ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=keep, scale=0.4)
        np.testing.assert_allclose(O, Ot.numpy(), rtol=0, atol=1e-12)
        sc = (torch.einsum("bhid,bhjd->bhij", tq, tk) * 0.4).masked_fill(~keep, float("-inf"))
        np.testing.assert_allclose(L, torch.logsumexp(sc, dim=-1).numpy(), rtol=0, atol=1e-12)


def pin_window_closed_forms(ref):
    """Window (0, 0): each row attends only to itself, so O[i] = V[i] and
    LSE[i] = scale * q_i . k_i; a window wider than T is no window."""
    q, k, v = _rand(1, 2, 2, 17, 8, seed=71)
    O, L = ref(q, k, v, 0.3, False, window=(0, 0))
    np.testing.assert_array_equal(O, v)
    np.testing.assert_allclose(L, 0.3 * np.einsum("bhid,bhid->bhi", q, k), rtol=0, atol=1e-13)
    O1, L1 = ref(q, k, v, 0.3, True, window=(100, 100))
    O2, L2 = ref(q, k, v, 0.3, True)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def pin_window_brute(ref):
    """Windows against the scalar restatement on tiny shapes."""
    for T in (3, 6, 8):
        for window in ((0, 1), (2, 2), (1, -1), (-1, 1)):
            for causal in (False, True):
                q, k, v = _rand(1, 2, 1, T, 3, seed=T * 11 + window[0] + 2 * window[1])
                O, L = ref(q, k, v, 0.8, causal, window=window)
                Ob, Lb = oracle.attention_brute(q, k, v, 0.8, causal, window=window)
                np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-13)
                np.testing.assert_allclose(L, np.array(Lb), rtol=0, atol=1e-13)


def _lg_mask(T, w, g, causal):
    """The tutorial's local_global_mask written with torch ops: |i - j| <= w
    OR torch.isin(j, global_tokens), then intersected with causal."""
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    keep = (i - j).abs() <= w
    keep = keep | torch.isin(j, torch.tensor(g, dtype=torch.long))
    if causal:
        keep &= j <= i
    return keep


LG_CASES = ((40, 8, 3, [0], False), (40, 8, 2, [0, 1, 2, 3], True), (37, 16, 0, [5, 30], False),
            (50, 4, 6, [49, 0, 17, 17, -3, 77], True), (33, 8, 1, [], False),
            (45, 8, 4, list(range(0, 45, 7)), True))


def pin_local_global_library_sdpa(ref):
    """Local-global masks against torch's scaled_dot_product_attention (CPU,
    float64) with the explicit mask of the tutorial's local_global_mask:
    sinks at the start, tokens at the end, repeats and out-of-range entries
    (selecting nothing), no global token, causal or not."""
    for (T, d, w, g, causal) in LG_CASES:
        q, k, v = _rand(1, 2, 2, T, d, seed=T + d + w)
        O, L = ref(q, k, v, 0.4, causal, window=(w, w), global_tokens=g)
        keep = _lg_mask(T, w, g, causal)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        Ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=keep, scale=0.4)
        np.testing.assert_allclose(O, Ot.numpy(), rtol=0, atol=1e-12)
        sc = (torch.einsum("bhid,bhjd->bhij", tq, tk) * 0.4).masked_fill(~keep, float("-inf"))
        np.testing.assert_allclose(L, torch.logsumexp(sc, dim=-1).numpy(), rtol=0, atol=1e-12)


def pin_local_global_brute(ref):
    """Local-global masks against the scalar restatement on tiny shapes."""
    for T in (4, 7):
        for w, g in ((0, [0]), (1, [T - 1]), (0, [1, 1, 3])):
            for causal in (False, True):
                q, k, v = _rand(1, 2, 1, T, 3, seed=T * 13 + w + len(g))
                O, L = ref(q, k, v, 0.7, causal, window=(w, w), global_tokens=g)
                Ob, Lb = oracle.attention_brute(q, k, v, 0.7, causal, window=(w, w),
                                                global_tokens=g)
                np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-13)
                np.testing.assert_allclose(L, np.array(Lb), rtol=0, atol=1e-13)


def pin_local_global_closed_forms(ref):
    """Local window 0 with global token 0: row 0 sees only key 0 (O = V[0]);
    row i > 0 sees exactly keys {0, i}, a two-way softmax; every key global
    is no mask at all."""
    T = 12
    q, k, v = _rand(1, 1, 1, T, 4, seed=81)
    O, L = ref(q, k, v, 0.5, True, window=(0, 0), global_tokens=[0])
    np.testing.assert_array_equal(O[0, 0, 0], v[0, 0, 0])
    for i in range(1, T):
        s0 = 0.5 * q[0, 0, i] @ k[0, 0, 0]
        si = 0.5 * q[0, 0, i] @ k[0, 0, i]
        m = max(s0, si)
        e0, ei = math.exp(s0 - m), math.exp(si - m)
        np.testing.assert_allclose(O[0, 0, i], (e0 * v[0, 0, 0] + ei * v[0, 0, i]) / (e0 + ei),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(L[0, 0, i], m + math.log(e0 + ei), rtol=0, atol=1e-13)
    O1, L1 = ref(q, k, v, 0.5, False, window=(0, 0), global_tokens=list(range(T)))
    O2, L2 = ref(q, k, v, 0.5, False)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-15)


ALL_PINS = [pin_brute, pin_library_sdpa, pin_causal_row0, pin_zero_query,
            pin_constant_values, pin_key_shift, pin_dominant_key, pin_grouped_heads,
            pin_head_mapping_brute, pin_window_library_sdpa, pin_window_closed_forms,
            pin_window_brute, pin_local_global_library_sdpa, pin_local_global_brute,
            pin_local_global_closed_forms]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.attention_ref)


# --------------------------------------------------------------------------
# further pins of the other oracle functions
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [[1], [7], [64], [200], [3, 5, 11], [128, 1]])
def test_online_recurrence_equals_batch(causal, blocks):
    """Section "Softmax 的在線計算": the running (m, l) recurrence gives the
    same result as the batch softmax, whatever the block partition."""
    q, k, v = _rand(2, 2, 1, 150, 16, seed=21)
    O, L = oracle.attention_ref(q, k, v, 0.25, causal)
    Oo, Lo = oracle.attention_online_ref(q, k, v, 0.25, causal, blocks)
    np.testing.assert_allclose(Oo, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lo, L, rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [(5, 5), (20, 0), (0, 30), (-1, 7)])
def test_online_recurrence_equals_batch_with_window(window):
    q, k, v = _rand(1, 2, 2, 120, 8, seed=23)
    for causal in (False, True):
        O, L = oracle.attention_ref(q, k, v, 0.25, causal, window=window)
        Oo, Lo = oracle.attention_online_ref(q, k, v, 0.25, causal, [16, 9], window=window)
        np.testing.assert_allclose(Oo, O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Lo, L, rtol=0, atol=1e-12)


def test_online_recurrence_growing_max():
    """Rows whose maximum keeps rising across blocks (every block rescales)."""
    q, k, v = make_structured_qkv(1, 2, 300, 16, dtype="f32", seed=3, ramp=8.0)
    for causal in (False, True):
        O, L = oracle.attention_ref(q, k, v, 0.25, causal)
        Oo, Lo = oracle.attention_online_ref(q, k, v, 0.25, causal, [32])
        np.testing.assert_allclose(Oo, O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Lo, L, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_are_a_softmax(causal):
    """Each row of P is non-negative, zero on masked keys and sums to 1
    (the softmax definition of section "Softmax 的在線計算"), and O = P V."""
    q, k, v = _rand(2, 2, 2, 40, 8, seed=31)
    P = oracle.attention_probs_ref(q, k, v, 0.5, causal)
    assert np.all(P >= 0)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(P[..., np.triu_indices(40, 1)[0], np.triu_indices(40, 1)[1]] == 0)
    O, _ = oracle.attention_ref(q, k, v, 0.5, causal)
    np.testing.assert_allclose(O, np.einsum("bhij,bhjd->bhid", P, v), rtol=0, atol=1e-12)
    # convexity: O lies within the range of the values it averages
    assert np.all(O <= v.max(axis=2, keepdims=True) + 1e-12)
    assert np.all(O >= v.min(axis=2, keepdims=True) - 1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_ref_matches_full(causal):
    q, k, v = _rand(2, 4, 2, 300, 16, seed=41)
    O, L = oracle.attention_ref(q, k, v, 0.25, causal, row_chunk=64)
    rows = np.array([0, 1, 63, 64, 150, 299])
    for b, h in ((0, 0), (1, 3)):
        o, l = oracle.attention_rows_ref(q, k, v, 0.25, causal, b, h, rows)
        np.testing.assert_allclose(o, O[b, h, rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l, L[b, h, rows], rtol=0, atol=1e-13)


def test_row_chunking_is_only_grouping():
    q, k, v = _rand(1, 2, 2, 130, 8, seed=42)
    for causal in (False, True):
        O1, L1 = oracle.attention_ref(q, k, v, 0.3, causal, row_chunk=1000)
        O2, L2 = oracle.attention_ref(q, k, v, 0.3, causal, row_chunk=7)
        np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-13)


def test_bf16_inputs_are_read_exactly():
    """The oracle sees the exact bf16 values the device sees."""
    q, k, v = make_qkv(1, 1, 1, 8, 4, dtype="bf16", seed=5)
    assert oracle.as_f64(q).dtype == np.float64
    assert np.array_equal(oracle.as_f64(q), q.float().double().numpy())
    O, L = oracle.attention_ref(q, k, v, 0.5, True)
    Ob, Lb = oracle.attention_brute(q, k, v, 0.5, True)
    np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-13)


def test_golden_naive_memory_table():
    """The tutorial's memory table (fp16 bytes of the naive T x T matrix)."""
    rows = []
    with open(os.path.join(GOLDEN, "naive_score_matrix_fp16.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                T, mb = line.split()
                rows.append((int(T), int(mb)))
    assert len(rows) == 4
    for T, mb in rows:
        assert oracle.naive_score_bytes(T, 2) == mb * 2 ** 20
    assert oracle.naive_score_bytes(4096, 1) == 16 * 2 ** 20  # "16M floats" at n = 4096


def test_rejects_bad_heads():
    q, k, v = _rand(1, 3, 2, 4, 2, seed=1)
    with pytest.raises(ValueError):
        oracle.attention_ref(q, k, v, 1.0, False)


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

def _make_rows_fn(mistake):
    """A copy of the oracle's per-head step with one planted mistake."""

    def rows_fn(qh, kh, vh, rows, scale, causal, window=None, global_tokens=None):
        T = kh.shape[0]
        kk, vv = (vh, kh) if mistake == "swap_kv" else (kh, vh)
        sc = 1.0 if mistake == "drop_scale" else scale
        s = (qh[rows] @ kk.T) * sc
        if mistake == "transpose_q":
            s = (qh[rows][:, ::-1] @ kk.T) * sc
        if window is not None and mistake in ("window_off_by_one", "window_swapped"):
            wl, wr = window if mistake == "window_off_by_one" else (window[1], window[0])
            jj, ii = np.arange(T)[None, :], rows[:, None]
            off = 1 if mistake == "window_off_by_one" else 0
            wvalid = np.ones((len(rows), T), dtype=bool)
            if wl >= 0:
                wvalid &= jj >= ii - wl + off
            if wr >= 0:
                wvalid &= jj <= ii + wr
        else:
            wvalid = ar_mod.valid_keys(rows, T, False, window)
        if global_tokens is not None:
            g = np.asarray(global_tokens, dtype=np.int64)
            if mistake == "global_as_queries":
                wvalid = wvalid | np.isin(rows, g)[:, None]
            elif mistake != "global_dropped":
                wvalid = wvalid | np.isin(np.arange(T), g)[None, :]
        if causal:
            if mistake == "strict_mask":
                valid = np.arange(T)[None, :] < rows[:, None]
            elif mistake == "loose_mask":
                valid = np.arange(T)[None, :] <= rows[:, None] + 1
            elif mistake == "flipped_mask":
                valid = np.arange(T)[None, :] >= rows[:, None]
            else:
                valid = np.arange(T)[None, :] <= rows[:, None]
        else:
            valid = np.ones((len(rows), T), dtype=bool)
        valid = valid & wvalid
        if mistake == "global_ignores_causal" and global_tokens is not None:
            valid = valid | np.isin(np.arange(T), np.asarray(global_tokens))[None, :]
        s = np.where(valid, s, -np.inf)
        m = s.max(axis=1)
        if mistake == "no_max_shift":
            e = np.where(valid, np.exp(s), 0.0)
        else:
            e = np.where(valid, np.exp(s - m[:, None]), 0.0)
        l = e.sum(axis=1)
        o = (e @ vv) / (l[:, None] if mistake != "no_normalise" else 1.0)
        if mistake == "log2_lse":
            lse = m + np.log2(l)
        elif mistake == "lse_without_max":
            lse = np.log(l)
        else:
            lse = m + np.log(l)
        return o, lse, e / l[:, None]

    return rows_fn


MISTAKES = ["swap_kv", "drop_scale", "transpose_q", "strict_mask", "loose_mask",
            "flipped_mask", "no_max_shift", "no_normalise", "log2_lse",
            "lse_without_max", "head_modulo", "window_off_by_one", "window_swapped",
            "global_dropped", "global_as_queries", "global_ignores_causal"]


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake, monkeypatch):
    if mistake == "head_modulo":
        monkeypatch.setattr(ar_mod, "kv_head_of", lambda h, Hq, Hkv: h % Hkv)
    else:
        monkeypatch.setattr(ar_mod, "_rows_of_head", _make_rows_fn(mistake))
    caught = []
    with np.errstate(all="ignore"):
        for pin in ALL_PINS:
            try:
                pin(ar_mod.attention_ref)
            except (AssertionError, FloatingPointError, ValueError):
                caught.append(pin.__name__)
    assert caught, f"planted mistake {mistake!r} passed every pin"
