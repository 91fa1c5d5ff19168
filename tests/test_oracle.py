"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

None of these compares the oracle with itself.  Each checks a closed form, an
invariant, an independent brute force, finite differences, or the worked
example one page prints, chosen so that a dropped term, a wrong sign or index,
a missing scale or a transposed operand fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import (
    attention_bwd_preprocess_ref,
    attention_bwd_ref,
    attention_fwd_ref,
    attention_probs_ref,
    online_softmax_ref,
    recompute_probs_from_lse_ref,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# worked example printed by datarekha.com "FlashAttention",
# section "The online softmax - why it's exact"
# --------------------------------------------------------------------------
def test_worked_example_online_equals_full():
    with open(os.path.join(GOLDEN, "datarekha_online_softmax_example.json")) as f:
        g = json.load(f)
    n, d, tile = g["N"], g["d"], g["tile"]
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    scale = 1.0 / math.sqrt(d)
    o_full, _ = attention_fwd_ref(q, k, v, scale)
    o_online, _ = online_softmax_ref(q, k, v, scale, tile=tile)
    diff = np.abs(o_full - o_online).max()
    # the page prints 1.11e-16; equal up to fp64 rounding (a few ulps)
    assert diff <= 10 * g["printed_max_abs_difference"]
    # the example is not degenerate: the output is a real mix of the values
    assert np.abs(o_full).max() > 0.05


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_two_query_closed_form_orientation_and_scale():
    # d = 1; q = [1, 0], k = [0, 1], v = [0, 1], scale s
    # S = s * [[0, 1], [0, 0]] ->
    #   row 0: P = [1, e^s] / (1 + e^s)  -> O_0 = e^s / (1 + e^s)
    #   row 1: P = [1/2, 1/2]            -> O_1 = 1/2
    # LSE_0 = log(1 + e^s), LSE_1 = log 2.  Using P^T V instead of P V, or
    # dropping the scale, gives other numbers.
    s = 0.7
    q = np.array([[1.0], [0.0]])
    k = np.array([[0.0], [1.0]])
    v = np.array([[0.0], [1.0]])
    o, lse = attention_fwd_ref(q, k, v, s)
    es = math.exp(s)
    assert o[0, 0] == pytest.approx(es / (1 + es), abs=1e-15)
    assert o[1, 0] == pytest.approx(0.5, abs=1e-15)
    assert lse[0] == pytest.approx(math.log(1 + es), abs=1e-15)
    assert lse[1] == pytest.approx(math.log(2.0), abs=1e-15)
    # causal: row 0 only sees key 0
    oc, lsec = attention_fwd_ref(q, k, v, s, causal=True)
    assert oc[0, 0] == 0.0 and lsec[0] == pytest.approx(0.0, abs=1e-15)
    assert oc[1, 0] == pytest.approx(0.5, abs=1e-15)


def test_single_key_gives_v_and_scaled_dot():
    q, k, v = rand((2, 3, 1, 8), 1), rand((2, 3, 1, 8), 2), rand((2, 3, 1, 8), 3)
    scale = 0.37
    for causal in (False, True):
        o, lse = attention_fwd_ref(q, k, v, scale, causal)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, scale * (q * k).sum(-1), rtol=0, atol=1e-14)


def test_constant_values_give_that_value():
    n, d = 37, 16
    q, k = rand((2, n, d), 4), rand((2, n, d), 5)
    row = rand((d,), 6)
    v = np.broadcast_to(row, (2, n, d)).copy()
    for causal in (False, True):
        o, _ = attention_fwd_ref(q, k, v, 0.25, causal)
        np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), rtol=0, atol=1e-14)


def test_equal_scores_give_mean_and_log_count():
    n, d = 50, 8
    q = np.zeros((n, d))
    k, v = rand((n, d), 7), rand((n, d), 8)
    o, lse = attention_fwd_ref(q, k, v, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(n), atol=1e-14)
    # causal, top-left: row i averages v_0..v_i and LSE_i = log(i + 1)
    oc, lsec = attention_fwd_ref(q, k, v, 1.0, causal=True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(oc, prefix, atol=1e-14)
    np.testing.assert_allclose(lsec, np.log(np.arange(1, n + 1)), atol=1e-14)


def test_causal_row_zero_sees_only_key_zero():
    q, k, v = rand((33, 8), 9), rand((33, 8), 10), rand((33, 8), 11)
    o, lse = attention_fwd_ref(q, k, v, 0.5, causal=True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert lse[0] == pytest.approx(0.5 * q[0] @ k[0], abs=1e-14)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k = rand((2, 2, 40, 16), 12), rand((2, 2, 40, 16), 13)
    p = attention_probs_ref(q, k, 0.3, causal)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-14)
    assert (p >= 0).all()
    if causal:
        assert np.all(np.triu(p[0, 0], 1) == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_lse_is_log_sum_exp_of_scaled_scores(causal):
    n, d, scale = 29, 8, 0.4
    q, k, v = rand((n, d), 14), rand((n, d), 15), rand((n, d), 16)
    _, lse = attention_fwd_ref(q, k, v, scale, causal)
    for i in range(n):
        s = scale * (k @ q[i])
        if causal:
            s = s[: i + 1]
        assert lse[i] == pytest.approx(np.logaddexp.reduce(s), abs=1e-13)


def test_key_shift_invariance():
    n, d, scale = 31, 8, 0.6
    q, k, v = rand((n, d), 17), rand((n, d), 18), rand((n, d), 19)
    u = rand((d,), 20)
    for causal in (False, True):
        o0, l0 = attention_fwd_ref(q, k, v, scale, causal)
        o1, l1 = attention_fwd_ref(q, k + u, v, scale, causal)
        np.testing.assert_allclose(o1, o0, atol=1e-13)
        np.testing.assert_allclose(l1, l0 + scale * (q @ u), atol=1e-12)


def _bruteforce_fwd(q, k, v, scale, causal):
    """Pure-Python loops straight from the definition (tiny inputs only)."""
    n, d = len(q), len(q[0])
    dv = len(v[0])
    o = [[0.0] * dv for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        js = [j for j in range(len(k)) if not (causal and j > i)]
        s = {j: scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in js}
        mx = max(s.values())
        den = sum(math.exp(s[j] - mx) for j in js)
        for c in range(dv):
            o[i][c] = sum(math.exp(s[j] - mx) / den * v[j][c] for j in js)
        lse[i] = mx + math.log(den)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_matches_pure_python_bruteforce(causal):
    q, k, v = rand((2, 6, 5), 21), rand((2, 6, 5), 22), rand((2, 6, 3), 23)
    o, lse = attention_fwd_ref(q, k, v, 0.45, causal)
    for h in range(2):
        ob, lb = _bruteforce_fwd(q[h].tolist(), k[h].tolist(), v[h].tolist(), 0.45, causal)
        np.testing.assert_allclose(o[h], np.array(ob), atol=1e-14)
        np.testing.assert_allclose(lse[h], np.array(lb), atol=1e-14)


def test_row_chunking_does_not_change_results():
    q, k, v, do = (rand((1, 2, 45, 8), s) for s in (24, 25, 26, 27))
    for causal in (False, True):
        a = attention_fwd_ref(q, k, v, 0.3, causal, row_chunk=4)
        b = attention_fwd_ref(q, k, v, 0.3, causal, row_chunk=1000)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, atol=1e-14)
        a = attention_bwd_ref(q, k, v, do, 0.3, causal, row_chunk=7)
        b = attention_bwd_ref(q, k, v, do, 0.3, causal, row_chunk=1000)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, atol=1e-13)


# --------------------------------------------------------------------------
# online softmax (the streaming update) against the full-row softmax
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 7, 128, 300, 512])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_equals_full_row(n, causal):
    d = 16
    q, k, v = rand((n, d), 30 + n), rand((n, d), 31 + n), rand((n, d), 32 + n)
    k = 3.0 * k  # wide score range so the running max moves
    o_ref, lse_ref = attention_fwd_ref(q, k, v, 0.25, causal)
    for tile in sorted({1, 2, 3, 128, n}):
        for thr in (None, 0.0, 8 * math.log(2.0)):
            o, lse = online_softmax_ref(q, k, v, 0.25, tile, causal, rescale_threshold=thr)
            np.testing.assert_allclose(o, o_ref, atol=1e-12)
            np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_online_softmax_when_max_rises_every_tile():
    # scores increase along the row, so every tile raises the maximum and the
    # correction factor e^{m - m'} is exercised on every step
    n, d = 64, 1
    q = np.ones((3, d))
    k = np.linspace(-4.0, 4.0, n)[:, None]
    v = rand((n, 5), 33)
    o_ref, lse_ref = attention_fwd_ref(q, k, v, 1.0)
    for thr in (None, 0.0, 8 * math.log(2.0), 50.0):
        o, lse = online_softmax_ref(q, k, v, 1.0, tile=4, rescale_threshold=thr)
        np.testing.assert_allclose(o, o_ref, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (5, 3), (16, 8)])
def test_backward_matches_central_finite_differences(causal, n, d):
    scale = 0.5
    q, k, v, do = (rand((n, d), s) for s in (40 + n, 41 + n, 42 + n, 43 + n))

    def loss(qq, kk, vv):
        o, _ = attention_fwd_ref(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    dq, dk, dv = attention_bwd_ref(q, k, v, do, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v, name: xp}
            args_m = {"q": q, "k": k, "v": v, name: xm}
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                        - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-3)
        assert err <= 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    q, k, v, do = (rand((2, 40, 8), s) for s in (50, 51, 52, 53))
    dq, dk, dv = attention_bwd_ref(q, k, v, do, 0.35, causal)
    # rows of dS sum to zero -> sum over keys of dK vanishes
    np.testing.assert_allclose(dk.sum(-2), 0.0, atol=1e-12)
    # rows of P sum to one -> sum over keys of dV equals sum over queries of dO
    np.testing.assert_allclose(dv.sum(-2), do.sum(-2), atol=1e-12)
    # a key the causal mask hides from every query gets no gradient:
    # in the square top-left case only the last key is seen by one row only
    if causal:
        p = attention_probs_ref(q, k, 0.35, True)
        np.testing.assert_allclose(dv[:, -1], p[:, -1, -1, None] * do[:, -1], atol=1e-13)


def test_delta_equals_rowsum_of_dout_times_out():
    q, k, v, do = (rand((3, 20, 6), s) for s in (60, 61, 62, 63))
    for causal in (False, True):
        o, _ = attention_fwd_ref(q, k, v, 0.4, causal)
        p = attention_probs_ref(q, k, 0.4, causal)
        dp = do @ np.swapaxes(v, -1, -2)
        np.testing.assert_allclose(attention_bwd_preprocess_ref(o, do), (p * dp).sum(-1), atol=1e-13)
    # a hand example: O = [[1, 2]], dO = [[3, -1]] -> 3 - 2 = 1
    assert attention_bwd_preprocess_ref(np.array([[1.0, 2.0]]), np.array([[3.0, -1.0]]))[0] == 1.0


@pytest.mark.parametrize("causal", [False, True])
def test_probs_recomputed_from_lse_equal_forward_probs(causal):
    q, k, v = rand((2, 30, 8), 70), rand((2, 30, 8), 71), rand((2, 30, 8), 72)
    _, lse = attention_fwd_ref(q, k, v, 0.6, causal)
    np.testing.assert_allclose(recompute_probs_from_lse_ref(q, k, lse, 0.6, causal),
                               attention_probs_ref(q, k, 0.6, causal), atol=1e-14)
