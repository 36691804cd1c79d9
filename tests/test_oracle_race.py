"""Pins of the oracle's exponential race (velog post "vLLM speculative
decoding이 기각 토큰을 다시 뽑는 이유", section "vLLM 커널은 이 규칙을 어떻게
옮겼나": argmax of w_j / E_j with E_j ~ Exp(1) is a draw proportional to w)."""
import math

import numpy as np

import oracle


def test_race_law_chi_square():
    w = np.array([0.0, 3.0, 1.0, 0.5, 0.25, 2.0, 0.0, 1.25])
    n = 200_000
    counts = np.zeros(w.size)
    for r in range(n):
        j, _ = oracle.race(w, 2024, r, r % 7)
        counts[j] += 1
    assert counts[0] == 0 and counts[6] == 0
    expect = w / w.sum() * n
    nz = expect > 0
    chi2 = ((counts[nz] - expect[nz]) ** 2 / expect[nz]).sum()
    assert chi2 < 22.46  # 6 dof, 1e-3


def test_zero_weights_never_win_and_all_zero_gives_minus_one():
    w = np.zeros(10)
    assert oracle.race(w, 1, 2, 3)[0] == -1
    w[7] = 1e-300
    for r in range(100):
        assert oracle.race(w, 1, r, 0)[0] == 7


def test_exact_tie_goes_to_lowest_index():
    seed, req, pos = 5, 11, 1
    E = [-math.log(oracle.race_uniform(seed, req, pos, j)) for j in range(5)]
    # w_j = E_j makes the score exactly 1.0 for j = 2 and j = 4
    w = np.array([0.0, 0.0, E[2], 0.0, E[4]])
    j, margin = oracle.race(w, seed, req, pos)
    assert j == 2 and margin == 0.0


def test_race_is_scale_free():
    rng = np.random.default_rng(3)
    w = rng.random(50)
    for r in range(200):
        assert oracle.race(w, 9, r, 0)[0] == oracle.race(w * 1e-30, 9, r, 0)[0]


def test_zero_residual_mass_draws_from_p():
    """Draft probabilities of 1 at every token: p <= q everywhere, so after a
    rejection the residual max(p - q, 0) has zero mass; the reading is that
    the token is then drawn from p (the race on w = p) and the request is
    flagged (status bit 3). With the draft drawn uniformly over the 5 toy
    tokens, acceptance is mean p(x) = 1/5 and the first emitted token
    follows p exactly: P(j) = p_j / 5 (accepted) + (4/5) p_j (drawn from p)."""
    import synth
    rounds = 400_000
    b = synth.toy_batch("prob", rounds, seed=17, q=[1.0] * 5)
    o = oracle.verify(b)
    acc = o["num_accepted"].astype(np.float64)
    assert abs(acc.mean() - 0.2) < 5 * math.sqrt(0.2 * 0.8 / rounds)
    rejected = acc < 1
    flagged = (o["req_status"] & 0x8) != 0
    assert np.array_equal(flagged, rejected)
    first = o["out_tokens"].reshape(-1, 2)[:, 0]
    p = np.asarray(synth.TOY_P)
    expect = p * rounds
    counts = np.bincount(first, minlength=5)
    assert ((counts - expect) ** 2 / expect).sum() < 18.47  # 4 dof, 1e-3
    # and the tokens drawn after a rejection alone follow p too
    counts_r = np.bincount(first[rejected], minlength=5)
    expect_r = p * rejected.sum()
    assert ((counts_r - expect_r) ** 2 / expect_r).sum() < 18.47
