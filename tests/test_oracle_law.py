"""Exact enumeration of the oracle's output law (V <= 4, gamma <= 2).

Proof being checked: the velog post "vLLM speculative decoding이 기각 토큰을
다시 뽑는 이유", section "왜 하필 max(p − q, 0)인가" (Appendix A.1 of the
paper): the emitted token is distributed as min(p, q) + (1 - beta) *
norm(max(0, p - q)) = p. Section "기본값 greedy 드래프트에서도 분포가
지켜질까": a one-hot draft also preserves p, with acceptance p(x).

Nothing here restates the oracle's formulas. The acceptance probability is
read off the oracle's own accept test (it must be a threshold in u, found by
probing the oracle around the exact ratio), the residual weights are the
oracle's own, and the race law is the exponential-race identity (pinned
separately by test_oracle_race). All arithmetic is exact (Fraction).
"""
import itertools
from fractions import Fraction as F

import numpy as np
import pytest

import oracle

GRID = 8  # probabilities are multiples of 1/8


def dyadic_dists(V):
    for parts in itertools.product(range(GRID + 1), repeat=V):
        if sum(parts) == GRID:
            yield tuple(F(a, GRID) for a in parts)


def accept_probability(p_x, q_x):
    """P_u(oracle accepts) for u ~ U(0,1), read from the oracle's accept test.

    The test must accept on (0, t] and reject on (t, 1) for one t; probe just
    below and above the candidate t = min(1, p/q) (and 0 when q = 0)."""
    if q_x == 0:
        t = F(0)
    else:
        t = min(F(1), p_x / q_x)
    pf, qf = float(p_x), float(q_x)
    eps = 2.0 ** -40
    probes_in = [eps, float(t) - eps] if t > 0 else []
    probes_out = [float(t) + eps, 1.0 - eps] if t < 1 else []
    for u in probes_in:
        if 0 < u < 1:
            assert oracle.accept(pf, qf, u), (p_x, q_x, u)
    for u in probes_out:
        if 0 < u < 1:
            assert not oracle.accept(pf, qf, u), (p_x, q_x, u)
    if t == 0:
        assert not oracle.accept(pf, qf, 2.0 ** -53)
    return t


def race_law(w):
    total = sum(w)
    assert total > 0
    return [wi / total for wi in w]


def emitted_law(p, q, one_hot_at=None):
    """Exact law of the token emitted at one judged position."""
    V = len(p)
    law = [F(0)] * V
    pf = np.array([float(x) for x in p])
    if one_hot_at is None:
        drafts = [(x, q[x]) for x in range(V) if q[x] > 0]
        qf = np.array([float(x) for x in q])
        mode = 0
    else:
        drafts = [(one_hot_at, F(1))]
        qf = None
        mode = 1
    for x, qx_prob in drafts:
        q_x = q[x] if one_hot_at is None else F(1)
        a = accept_probability(p[x], q_x)
        law[x] += qx_prob * a
        if a < 1:
            w = oracle.residual_weights(pf, qf, x, mode)
            wfr = [F(v) for v in w]  # doubles are exact rationals
            for y, ry in enumerate(race_law(wfr)):
                law[y] += qx_prob * (1 - a) * ry
    return law


@pytest.mark.parametrize("V", [1, 2, 3, 4])
def test_probabilistic_draft_preserves_p(V):
    dists = list(dyadic_dists(V))
    for p in dists:
        for q in dists:
            assert emitted_law(p, q) == list(p), (p, q)


@pytest.mark.parametrize("V", [1, 2, 3, 4])
def test_one_hot_draft_preserves_p(V):
    for p in dyadic_dists(V):
        for x in range(V):
            law = emitted_law(p, None, one_hot_at=x)
            assert law == list(p), (p, x)
            # acceptance of a one-hot draft at x is p(x)
            assert accept_probability(p[x], F(1)) == p[x]


def test_acceptance_is_overlap():
    # beta = sum_x q(x) min(1, p/q) = sum min(p, q) (Theorem 3.5 as the page cites it)
    for p in dyadic_dists(3):
        for q in dyadic_dists(3):
            beta = sum(q[x] * accept_probability(p[x], q[x]) for x in range(3) if q[x] > 0)
            assert beta == sum(min(a, b) for a, b in zip(p, q))


def test_naive_control_is_biased_as_printed():
    # naive: on rejection resample from p -> law min(p,q) + (1-beta) p, token 0 = 0.425
    p = [F(50, 100), F(25, 100), F(15, 100), F(7, 100), F(3, 100)]
    q = [F(30, 100), F(40, 100), F(10, 100), F(15, 100), F(5, 100)]
    pf = np.array([float(x) for x in p])
    V = 5
    law = [F(0)] * V
    for x in range(V):
        a = min(F(1), p[x] / q[x])
        law[x] += q[x] * a
        w = [F(v) for v in oracle.residual_weights(pf, None, x, 2)]
        for y, ry in enumerate(race_law(w)):
            law[y] += q[x] * (1 - a) * ry
    # the oracle's naive weights are p itself (as doubles), so compare in float
    assert abs(float(law[0]) - 0.425) < 1e-12
    expect = [0.425, 0.3125, 0.1375, 0.0875, 0.0375]
    assert np.allclose([float(v) for v in law], expect, atol=1e-12)


@pytest.mark.parametrize("case", range(30))
def test_multi_position_round_law(case):
    """gamma = 2: positions judged left to right, each with its own (p_i, q_i),
    the bonus from p_2. For every emitted sequence the exact probability must
    factor as p_0(y_0) [x_0 accepted: p_1(y_1) [x_1 accepted: p_2(y_2)]]:
    the token at each later position, given that the round reached it, is
    distributed as that position's p."""
    rng = np.random.default_rng(case)
    V = int(rng.integers(2, 5))
    dists = list(dyadic_dists(V))
    ps = [dists[int(rng.integers(len(dists)))] for _ in range(3)]
    qs = [dists[int(rng.integers(len(dists)))] for _ in range(2)]
    for i in range(2):
        # position i: P(emit y and the round continues) = q(y) min(1, p/q) for
        # y = x accepted; the emitted law itself must be p_i
        assert emitted_law(ps[i], qs[i]) == list(ps[i])
        cont = [qs[i][y] * accept_probability(ps[i][y], qs[i][y]) if qs[i][y] > 0 else F(0)
                for y in range(V)]
        # conditioned on continuing, the next position is judged afresh: its
        # law does not depend on which y was accepted
        if sum(cont) > 0:
            nxt = emitted_law(ps[i + 1], qs[i + 1]) if i + 1 < 2 else list(ps[2])
            assert nxt == list(ps[i + 1])
    # bonus token: race over w = p_2
    w = [F(v) for v in np.array([float(x) for x in ps[2]])]
    assert race_law(w) == list(ps[2])
