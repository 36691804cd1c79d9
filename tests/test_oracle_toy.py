"""The 5-token worked example, run through the oracle's whole verify call.

Page: velog "vLLM speculative decoding이 기각 토큰을 다시 뽑는 이유", section
"Java로 규칙을 재현해 본 결과" (tests/golden/toy_table.txt). 2,000,000 rounds
per mode, one request per round, gamma = 1.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines

ROUNDS = 2_000_000
CHI2_4DOF_1E3 = 18.47


def _table():
    t = {}
    for row in golden_lines("toy_table.txt"):
        t[row[0]] = [float(x) for x in row[1:]]
    return t


@pytest.fixture(scope="module")
def runs():
    out = {}
    for mode in ("prob", "greedy", "naive"):
        b = synth.toy_batch(mode, ROUNDS)
        out[mode] = (b, oracle.verify(b))
    return out


def _stats(b, o):
    acc = o["num_accepted"].astype(np.float64).mean()
    first = o["out_tokens"].reshape(-1, 2)[:, 0]
    freq = np.bincount(first, minlength=5) / first.size
    return acc, freq, first


def chi2(freq, law, n):
    e = np.asarray(law) * n
    return float(((freq * n - e) ** 2 / e).sum())


@pytest.mark.slow
def test_acceptance_rates(runs):
    t = _table()
    sd = np.sqrt(0.75 * 0.25 / ROUNDS)
    for mode, exact in (("prob", t["exact_accept_prob"][0]),
                        ("greedy", t["exact_accept_greedy"][0]),
                        ("naive", t["exact_accept_prob"][0])):
        acc, _, _ = _stats(*runs[mode])
        assert abs(acc - exact) < 5 * sd, (mode, acc)
        # and within sampling error of the page's own printed sample value
        printed = t[mode][0]
        assert abs(acc - printed) < 5 * np.sqrt(2) * sd + 5e-5, (mode, acc, printed)


@pytest.mark.slow
def test_output_law_is_p(runs):
    t = _table()
    p = np.array(t["p"])
    for mode in ("prob", "greedy"):
        _, freq, first = _stats(*runs[mode])
        assert chi2(freq, p, first.size) < CHI2_4DOF_1E3, mode
        sd = np.sqrt(p * (1 - p) / ROUNDS)
        printed = np.array(t[mode][1:6])
        assert np.all(np.abs(freq - printed) < 5 * np.sqrt(2) * sd + 5e-5), mode


@pytest.mark.slow
def test_naive_control_is_rejected(runs):
    t = _table()
    p = np.array(t["p"])
    _, freq, first = _stats(*runs["naive"])
    # biased law min(p,q) + 0.25 p: token 0 at 0.425 as the page computes
    naive_law = np.minimum(p, np.array(t["q"])) + 0.25 * p
    assert abs(naive_law[0] - t["exact_naive_f0"][0]) < 1e-12
    assert chi2(freq, naive_law, first.size) < CHI2_4DOF_1E3
    assert chi2(freq, p, first.size) > 1e4  # expected about 6.8e4
    printed = np.array(t["naive"][1:6])
    sd = np.sqrt(naive_law * (1 - naive_law) / ROUNDS)
    assert np.all(np.abs(freq - printed) < 5 * np.sqrt(2) * sd + 5e-5)


@pytest.mark.slow
def test_bonus_token_law_is_p(runs):
    p = np.array(_table()["p"])
    b, o = runs["prob"]
    toks = o["out_tokens"].reshape(-1, 2)
    accepted = o["num_accepted"] == 1
    bonus = toks[accepted, 1]
    freq = np.bincount(bonus, minlength=5) / bonus.size
    assert chi2(freq, p, bonus.size) < CHI2_4DOF_1E3
    assert np.all(toks[~accepted, 1] == -1)
