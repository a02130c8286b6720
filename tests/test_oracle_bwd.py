"""Pins for the backward oracle (no GPU).

``oracle.attention_bwd_ref`` is pinned to things other than itself:

* finite differences of the forward oracle (directional, medium shapes) and
  of the scalar brute-force forward (every element, tiny shapes): the
  gradient is whatever the forward's derivative is, independent of the
  chain-rule formula;
* torch autograd through scaled_dot_product_attention in float64 on the CPU
  (the API of "Flash Attention Memory Optimization Explained", section "How
  to Use It in Code"), with the band as an explicit boolean mask;
* invariants of the definition: the key gradients sum to zero, the value
  gradients sum to the summed upstream gradient, a common shift of all keys
  changes no gradient, constant values give zero query and key gradients;
* closed forms: T = 1 and the first causal row.

The last test plants plausible mistakes in a copy of the per-head step and
checks that each trips at least one pin.

The pages name the backward pass ("Key Mechanisms", item "Backward
Checkpointing") without a formula; the gradient is fixed by the forward.
"""

import numpy as np
import pytest
import torch

import oracle


def _rand(B, Hq, Hkv, T, d, seed, mult=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, T, d)) * mult
    k = rng.standard_normal((B, Hkv, T, d)) * mult
    v = rng.standard_normal((B, Hkv, T, d)) * mult
    do = rng.standard_normal((B, Hq, T, d))
    return q, k, v, do


def _objective(fwd, q, k, v, do, scale, causal, window):
    """sum(O * dO): its gradient with respect to (q, k, v) is the backward."""
    O, _ = fwd(q, k, v, scale, causal, window=window)
    return float(np.sum(np.asarray(O) * do))


# --------------------------------------------------------------------------
# pins, written as functions of a backward callable
# bwd(q, k, v, do, scale, causal, window=None) -> (dQ, dK, dV)
# --------------------------------------------------------------------------

def pin_bwd_directional_fd(bwd):
    """<grad, delta> equals the central difference of sum(O * dO) along a
    random direction delta, for each of q, k and v."""
    cases = ((1, 2, 2, 17, 4, False, None), (1, 2, 1, 17, 4, True, None),
             (2, 4, 2, 12, 3, False, (3, 2)), (1, 3, 3, 20, 5, True, (4, -1)))
    for n, (B, Hq, Hkv, T, d, causal, window) in enumerate(cases):
        q, k, v, do = _rand(B, Hq, Hkv, T, d, seed=40 + n)
        scale = 0.6
        grads = bwd(q, k, v, do, scale, causal, window=window)
        rng = np.random.default_rng(90 + n)
        h = 1e-5
        for which in range(3):
            args = [q, k, v]
            delta = rng.standard_normal(args[which].shape)
            plus = list(args)
            minus = list(args)
            plus[which] = args[which] + h * delta
            minus[which] = args[which] - h * delta
            fd = (_objective(oracle.attention_ref, *plus, do, scale, causal, window)
                  - _objective(oracle.attention_ref, *minus, do, scale, causal, window)) / (2 * h)
            an = float(np.sum(grads[which] * delta))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (n, which, fd, an)


def pin_bwd_elementwise_fd_brute(bwd):
    """Every element of every gradient equals the central difference of the
    scalar pure-Python forward (tiny shapes, all masks)."""
    for n, (Hq, Hkv, T, d, causal, window) in enumerate(
            ((2, 1, 3, 2, False, None), (2, 2, 4, 2, True, None), (1, 1, 4, 2, False, (1, 0)),
             (2, 1, 3, 3, True, (0, -1)))):
        q, k, v, do = _rand(1, Hq, Hkv, T, d, seed=70 + n)
        scale = 0.9
        grads = bwd(q, k, v, do, scale, causal, window=window)

        def f(qq, kk, vv):
            O, _ = oracle.attention_brute(qq, kk, vv, scale, causal, window=window)
            return float(np.sum(np.array(O) * do))

        h = 1e-6
        for which in range(3):
            base = [q, k, v]
            num = np.zeros_like(base[which])
            for idx in np.ndindex(base[which].shape):
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[which][idx] += h
                minus[which][idx] -= h
                num[idx] = (f(*plus) - f(*minus)) / (2 * h)
            np.testing.assert_allclose(grads[which], num, rtol=0, atol=1e-8)


def pin_bwd_library_autograd(bwd):
    """torch autograd through F.scaled_dot_product_attention (CPU, float64),
    grouped heads by repeat_interleave, band windows as a boolean mask."""
    cases = ((2, 4, 2, 33, 8, False, None), (1, 4, 1, 40, 16, True, None),
             (1, 2, 2, 37, 8, False, (5, 5)), (2, 2, 1, 29, 4, True, (7, 0)),
             (1, 3, 3, 31, 8, False, (-1, 3)))
    for n, (B, Hq, Hkv, T, d, causal, window) in enumerate(cases):
        q, k, v, do = _rand(B, Hq, Hkv, T, d, seed=10 + n)
        scale = 0.35
        dQ, dK, dV = bwd(q, k, v, do, scale, causal, window=window)
        qt = torch.tensor(q, requires_grad=True)
        kt = torch.tensor(k, requires_grad=True)
        vt = torch.tensor(v, requires_grad=True)
        g = Hq // Hkv
        kr = kt.repeat_interleave(g, dim=1)
        vr = vt.repeat_interleave(g, dim=1)
        mask = torch.ones(T, T, dtype=torch.bool)
        i = torch.arange(T)[:, None]
        j = torch.arange(T)[None, :]
        if causal:
            mask &= j <= i
        if window is not None:
            if window[0] >= 0:
                mask &= j >= i - window[0]
            if window[1] >= 0:
                mask &= j <= i + window[1]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kr, vr, attn_mask=mask,
                                                             scale=scale)
        o.backward(torch.tensor(do))
        np.testing.assert_allclose(dQ, qt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dK, kt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dV, vt.grad.numpy(), rtol=0, atol=1e-12)


def pin_bwd_local_global_autograd(bwd):
    """Local-global masks (band OR global key, then causal) against torch
    autograd through SDPA with the tutorial's mask written out."""
    for n, (T, w, g, causal) in enumerate(((30, 2, [0, 1], True), (27, 0, [26, 5, 5, -1], False),
                                           (33, 3, [], True))):
        q, k, v, do = _rand(1, 2, 1, T, 8, seed=60 + n)
        scale = 0.45
        dQ, dK, dV = bwd(q, k, v, do, scale, causal, window=(w, w), global_tokens=g)
        qt = torch.tensor(q, requires_grad=True)
        kt = torch.tensor(k, requires_grad=True)
        vt = torch.tensor(v, requires_grad=True)
        i = torch.arange(T)[:, None]
        j = torch.arange(T)[None, :]
        mask = ((i - j).abs() <= w) | torch.isin(j, torch.tensor(g, dtype=torch.long))
        if causal:
            mask &= j <= i
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.repeat_interleave(2, dim=1), vt.repeat_interleave(2, dim=1), attn_mask=mask,
            scale=scale)
        o.backward(torch.tensor(do))
        np.testing.assert_allclose(dQ, qt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dK, kt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dV, vt.grad.numpy(), rtol=0, atol=1e-12)


def pin_bwd_invariants(bwd):
    """Key gradients sum to 0 over the keys; value gradients sum to the
    group's summed dO; shifting all keys by one vector changes no gradient;
    constant V gives dQ = dK = 0."""
    for causal, window in ((False, None), (True, None), (False, (4, 6))):
        B, Hq, Hkv, T, d = 2, 4, 2, 24, 6
        q, k, v, do = _rand(B, Hq, Hkv, T, d, seed=5 + int(causal))
        dQ, dK, dV = bwd(q, k, v, do, 0.5, causal, window=window)
        np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
        do_group = do.reshape(B, Hkv, Hq // Hkv, T, d).sum(axis=2)
        np.testing.assert_allclose(dV.sum(axis=2), do_group.sum(axis=2), rtol=0, atol=1e-12)
        u = np.random.default_rng(3).standard_normal(d)
        dQs, dKs, dVs = bwd(q, k + u, v, do, 0.5, causal, window=window)
        np.testing.assert_allclose(dQs, dQ, rtol=0, atol=1e-11)
        np.testing.assert_allclose(dKs, dK, rtol=0, atol=1e-11)
        np.testing.assert_allclose(dVs, dV, rtol=0, atol=1e-11)
        vc = np.broadcast_to(np.random.default_rng(4).standard_normal(d), v.shape).copy()
        dQc, dKc, _ = bwd(q, k, vc, do, 0.5, causal, window=window)
        np.testing.assert_allclose(dQc, 0.0, atol=1e-12)
        np.testing.assert_allclose(dKc, 0.0, atol=1e-12)


def pin_bwd_closed_forms(bwd):
    """T = 1: dQ = dK = 0 and dV = dO (summed over the group); causal row 0
    sees only key 0, so its dQ is 0."""
    q, k, v, do = _rand(2, 4, 2, 1, 5, seed=8)
    dQ, dK, dV = bwd(q, k, v, do, 0.7, False)
    np.testing.assert_array_equal(dQ, 0.0)
    np.testing.assert_array_equal(dK, 0.0)
    np.testing.assert_allclose(dV, do.reshape(2, 2, 2, 1, 5).sum(axis=2), rtol=0, atol=1e-15)
    q, k, v, do = _rand(1, 2, 2, 9, 4, seed=9)
    dQ, _, _ = bwd(q, k, v, do, 0.7, True)
    np.testing.assert_array_equal(dQ[:, :, 0], 0.0)


PINS = [pin_bwd_directional_fd, pin_bwd_elementwise_fd_brute, pin_bwd_library_autograd,
        pin_bwd_local_global_autograd, pin_bwd_invariants, pin_bwd_closed_forms]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_bwd_oracle_pin(pin):
    pin(oracle.attention_bwd_ref)


def test_bwd_row_chunking_is_only_grouping():
    q, k, v, do = _rand(1, 2, 1, 50, 8, seed=12)
    a = oracle.attention_bwd_ref(q, k, v, do, 0.3, True, row_chunk=7)
    b = oracle.attention_bwd_ref(q, k, v, do, 0.3, True, row_chunk=256)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)


def test_bwd_rejects_bad_shapes():
    q, k, v, do = _rand(1, 2, 1, 5, 4, seed=1)
    with pytest.raises(ValueError):
        oracle.attention_bwd_ref(q, k, v, do[:, :1], 0.5, False)


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

def _mutant_head(mistake):
    """A copy of the per-head chain-rule step with one planted mistake."""
    from oracle.attention_ref import valid_keys

    def head(qh, kh, vh, doh, scale, causal, window=None, global_tokens=None):
        T, d = qh.shape
        rows = np.arange(T)
        s = (qh @ kh.T) * scale
        valid = valid_keys(rows, T, causal, window, global_tokens)
        if mistake == "mask_dropped":
            valid = np.ones_like(valid)
        s = np.where(valid, s, -np.inf)
        e = np.where(valid, np.exp(s - s.max(axis=1)[:, None]), 0.0)
        p = e / e.sum(axis=1)[:, None]
        dv = (p if mistake == "dv_untransposed" else p.T) @ doh
        dp = (vh @ doh.T) if mistake == "dp_transposed" else (doh @ vh.T)
        if mistake == "drop_d_term":
            ds = p * dp
        elif mistake == "d_without_p":
            ds = p * (dp - dp.sum(axis=1)[:, None])
        else:
            ds = p * (dp - (p * dp).sum(axis=1)[:, None])
        dq = (ds @ kh) * (1.0 if mistake == "dq_no_scale" else scale)
        if mistake == "dq_uses_v":
            dq = scale * (ds @ vh)
        dk = scale * ((ds @ qh) if mistake == "dk_untransposed" else (ds.T @ qh))
        return dq, dk, dv

    def bwd(q, k, v, do, scale, causal, window=None, global_tokens=None):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        B, Hq, T, d = q.shape
        Hkv = k.shape[1]
        dQ = np.zeros_like(q)
        dK = np.zeros_like(k)
        dV = np.zeros_like(v)
        for b in range(B):
            for h in range(Hq):
                hk = h // (Hq // Hkv) if mistake != "head_modulo" else h % Hkv
                dq, dk, dv = head(q[b, h], k[b, hk], v[b, hk], do[b, h], scale, causal, window,
                                  global_tokens)
                dQ[b, h] = dq
                if mistake == "no_group_sum":
                    dK[b, hk] = dk
                    dV[b, hk] = dv
                else:
                    dK[b, hk] += dk
                    dV[b, hk] += dv
        return dQ, dK, dV

    return bwd


MISTAKES = ["mask_dropped", "dv_untransposed", "dp_transposed", "drop_d_term", "d_without_p",
            "dq_no_scale", "dq_uses_v", "dk_untransposed", "head_modulo", "no_group_sum"]


def test_mutant_harness_is_faithful():
    """With no mistake the mutant harness passes every pin (so a failure
    below is the planted mistake, not the harness)."""
    bwd = _mutant_head("none")
    for pin in PINS:
        pin(bwd)


@pytest.mark.parametrize("mistake", MISTAKES)
def test_bwd_planted_mistake_is_caught(mistake):
    bwd = _mutant_head(mistake)
    caught = []
    for pin in PINS:
        try:
            pin(bwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {mistake!r} passed every pin"


def test_bwd_dq_rows_equal_the_full_backward():
    """The rows-only dQ is the full backward's dQ for those rows (every mask)."""
    q, k, v, do = _rand(2, 4, 2, 37, 8, seed=17)
    for causal, window, g in ((False, None, None), (True, None, None), (False, (3, 5), None),
                              (True, (2, 2), [0, 30])):
        dQ, _, _ = oracle.attention_bwd_ref(q, k, v, do, 0.3, causal, window=window, global_tokens=g)
        rows = [0, 5, 36, 17]
        got = oracle.attention_bwd_dq_rows_ref(q, k, v, do, 0.3, causal, 1, 3, rows, window=window,
                                               global_tokens=g)
        np.testing.assert_allclose(got, dQ[1, 3, rows], rtol=0, atol=1e-13)
