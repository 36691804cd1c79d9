"""Pins of the sampling-constraint step (temperature, top-k, top-p) against
a brute-force O(V^2) definition written independently here, and against the
closed form p = softmax(l / T) when nothing is cut."""
import math

import numpy as np
import pytest

import oracle


def brute_keep(l, T, k, P):
    """Keep-set by definition: top-k on raw logits (ties kept), then token j
    survives top-p iff the renormalised mass of surviving tokens with a
    strictly larger logit is < P. Returns (keep, margin of the top-p test)."""
    V = len(l)
    keep = [True] * V
    if 0 < k < V:
        kth = sorted(l, reverse=True)[k - 1]
        keep = [x >= kth for x in l]
    m = max(l)
    e = [math.exp((x - m) / T) if keep[j] else 0.0 for j, x in enumerate(l)]
    Z = math.fsum(e)
    margin = math.inf
    if P < 1.0:
        out = []
        for j in range(V):
            if not keep[j]:
                out.append(False)
                continue
            above = math.fsum(e[i] for i in range(V) if keep[i] and l[i] > l[j]) / Z
            margin = min(margin, abs(above - P) / P)
            out.append(above < P)
        keep = out
    return keep, margin


@pytest.mark.parametrize("seed", range(40))
def test_keep_sets_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(1, 17))
    # integer-valued logits make ties common; half the cases use continuous values
    if seed % 2 == 0:
        l = rng.integers(-4, 5, size=V).astype(np.float64)
    else:
        l = rng.normal(0, 2, size=V)
    T = float(rng.choice([0.3, 0.7, 1.0, 1.5]))
    k = int(rng.choice([0, 1, 2, 3, V, V + 3]))
    P = float(rng.choice([1.0, 0.5, 0.8, 0.9, 0.95, 0.3]))
    keep, margin = brute_keep(list(l), T, k, P)
    if margin < 1e-9:
        pytest.skip("boundary within rounding of top_p")
    p, info = oracle.target_probs(l, T, k, P)
    assert info["status"] == 0
    assert [bool(x > 0) for x in p] == keep
    # on the kept set p is proportional to exp(l / T) and sums to 1
    kept = np.array(keep)
    ref = np.exp((l[kept] - l.max()) / T)
    np.testing.assert_allclose(p[kept], ref / ref.sum(), rtol=1e-12)
    assert abs(p.sum() - 1.0) < 1e-12


def test_no_filter_is_softmax():
    rng = np.random.default_rng(1)
    l = rng.normal(0, 3, size=1000)
    for T in (0.25, 1.0, 2.0):
        p, info = oracle.target_probs(l, T)
        z = np.exp((l - l.max()) / T)
        np.testing.assert_allclose(p, z / z.sum(), rtol=1e-12)
        assert info["theta"] == -math.inf and info["n_kept"] == 1000
        assert info["argmax"] == int(np.argmax(l))


def test_top_k_keeps_ties():
    l = np.array([3.0, 1.0, 2.0, 2.0, 2.0, 0.0])
    p, info = oracle.target_probs(l, 1.0, top_k=2)
    assert (p > 0).tolist() == [True, False, True, True, True, False]
    assert info["theta"] == 2.0


def test_top_p_small_example_by_hand():
    # p = [.5, .25, .15, .07, .03]; top_p = .8: mass above .15 is .75 < .8 -> kept,
    # mass above .07 is .90 >= .8 -> dropped.
    l = np.log([0.5, 0.25, 0.15, 0.07, 0.03])
    p, info = oracle.target_probs(l, 1.0, top_p=0.8)
    np.testing.assert_allclose(p, np.array([0.5, 0.25, 0.15, 0, 0]) / 0.9, rtol=1e-12)
    assert info["n_kept"] == 3
    # margins: kept side (.8 - .75) / .8, dropped side (.90 - .8) / .8
    assert abs(info["topp_margin"] - 0.0625) < 1e-9


def test_top_p_keeps_at_least_the_max():
    l = np.array([0.0, 5.0, 1.0])
    p, info = oracle.target_probs(l, 1.0, top_p=0.01)
    assert (p > 0).tolist() == [False, True, False] and p[1] == 1.0


def test_argmax_lowest_index():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([-math.inf, -math.inf]) == 0


def test_nonfinite_rows_are_flagged():
    _, info = oracle.target_probs([0.0, math.nan], 1.0)
    assert info["status"] == 1
    _, info = oracle.target_probs([0.0, math.inf], 1.0)
    assert info["status"] == 1
    _, info = oracle.target_probs([-math.inf, -math.inf], 1.0)
    assert info["status"] == 2
    p, info = oracle.target_probs([-math.inf, 0.0], 1.0)
    assert info["status"] == 0 and p.tolist() == [0.0, 1.0]
