"""Pins of the oracle's sampler-match acceptance.

Page: mlxcel "투기적 디코딩", section "mlxcel의 프롬프트 조회": a proposed token
is accepted only when it equals the token the target's sampler freshly draws
at that position; for one-hot proposals the rule is lossless and accepts as
often as the rejection rule. What fixes the oracle here, independently of its
own code:

* with top_k = 1 the target's sampler is deterministic (p is one-hot at the
  argmax), so the rule must reproduce temperature-0 verification exactly;
* acceptance of a one-hot draft x is p(x): drafts x ~ q give sum_x q(x) p(x),
  drafts at argmax q give p(argmax q) = 0.25, the value the velog page prints
  for the one-hot draft of its 5-token example (tests/golden/toy_table.txt);
* every emitted token follows p (chi-square), and the tokens per round of
  i.i.d. positions follow the truncated geometric law of cortexys 식 1;
* a mismatch emits the sampler's token, never the draft, and only kept
  tokens (top-k / top-p) are ever emitted.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines

CHI2_4DOF_1E3 = 18.47


def _sm(batch):
    b = dict(batch)
    b["flags"] = oracle.FLAG_SAMPLER_MATCH
    return b


def _small_batch(seed, B=120, V=64, top_k=None, top_p=None, T=1.0, draft="mixed"):
    rng = np.random.default_rng(seed)
    gam = rng.integers(0, 5, size=B)
    cu = np.concatenate([[0], np.cumsum(gam)]).astype(np.int32)
    N = int(cu[-1])
    R = N + B
    # distinct values per row: no ties, so argmax and top-k = 1 are unique
    logits = np.stack([rng.permutation(V).astype(np.float32) * 0.25 - 4.0 for _ in range(R)])
    ids = np.empty(N, np.int32)
    for r in range(B):
        for i in range(int(gam[r])):
            row = cu[r] + r + i
            if draft == "argmax" or (draft == "mixed" and rng.random() < 0.7):
                ids[cu[r] + i] = int(np.argmax(logits[row]))
            else:
                ids[cu[r] + i] = int(rng.integers(0, V))
    return dict(B=B, V=V, cu_num_draft=cu, draft_token_ids=ids, target_logits=logits,
                logits_dtype="f32", draft_probs=None, temperature=np.full(B, T, np.float32),
                top_k=None if top_k is None else np.full(B, top_k, np.int32),
                top_p=None if top_p is None else np.full(B, top_p, np.float32),
                seed=11, request_base=0, flags=0)


def test_top_k_one_reduces_to_argmax_match():
    b = _small_batch(3, top_k=1)
    sm = oracle.verify(_sm(b))
    g = dict(b)
    g["temperature"] = np.zeros(b["B"], np.float32)
    ref = oracle.verify(g)
    assert np.array_equal(sm["num_accepted"], ref["num_accepted"])
    assert np.array_equal(sm["out_tokens"], ref["out_tokens"])
    assert 0 < sm["num_accepted"].sum() < len(b["draft_token_ids"])


def test_draft_probs_are_not_read():
    b = synth.toy_batch("prob", 20000, seed=5, gamma=3)
    with_q = oracle.verify(_sm(b))
    nq = dict(b)
    nq["draft_probs"] = None
    without_q = oracle.verify(_sm(nq))
    assert np.array_equal(with_q["out_tokens"], without_q["out_tokens"])
    assert np.array_equal(with_q["num_accepted"], without_q["num_accepted"])


def test_mismatch_emits_the_sampled_token_and_only_kept_tokens():
    for kw in (dict(top_k=5), dict(top_p=0.6), dict()):
        b = _small_batch(7, draft="mixed", T=0.7, **kw)
        o = oracle.verify(_sm(b))
        cu = b["cu_num_draft"]
        for r in range(b["B"]):
            c0, c1 = int(cu[r]), int(cu[r + 1])
            g = c1 - c0
            row0 = c0 + r
            k = int(o["num_accepted"][r])
            t = o["out_tokens"][row0:row0 + g + 1]
            assert np.array_equal(t[:k], b["draft_token_ids"][c0:c0 + k])
            if k < g:
                assert t[k] != b["draft_token_ids"][c0 + k]
            assert np.all(t[k + 1:] == -1)
            p, _ = oracle.target_probs(b["target_logits"][row0 + k], 0.7, **kw)
            assert p[t[k]] > 0.0
            # the race behind each emitted token is logged with a finite margin
            assert np.all(np.isfinite(o["row_race_margin"][row0:row0 + k + 1]))
            assert np.all(np.isinf(o["row_race_margin"][row0 + k + 1:row0 + g + 1]))


@pytest.fixture(scope="module")
def toy_runs():
    n = 1_000_000
    return {mode: oracle.verify(_sm(synth.toy_batch(mode, n, seed=9))) for mode in ("prob", "greedy")}


def _toy_table():
    return {row[0]: [float(x) for x in row[1:]] for row in golden_lines("toy_table.txt")}


@pytest.mark.slow
def test_acceptance_of_one_hot_drafts(toy_runs):
    p, q = synth.TOY_P, synth.TOY_Q
    n = 1_000_000
    # drafts x ~ q, judged one-hot: P(accept) = sum_x q(x) p(x)
    alpha = float((p * q).sum())
    acc = toy_runs["prob"]["num_accepted"].mean()
    assert abs(acc - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / n), (acc, alpha)
    # drafts at argmax q: the page's one-hot acceptance p(argmax q) = 0.25
    exact = _toy_table()["exact_accept_greedy"][0]
    acc = toy_runs["greedy"]["num_accepted"].mean()
    assert abs(acc - exact) < 5 * np.sqrt(exact * (1 - exact) / n), (acc, exact)


@pytest.mark.slow
def test_first_token_follows_p(toy_runs):
    p = synth.TOY_P
    for mode, o in toy_runs.items():
        first = o["out_tokens"].reshape(-1, 2)[:, 0]
        n = first.size
        f = np.bincount(first, minlength=5)
        chi2 = float(((f - p * n) ** 2 / (p * n)).sum())
        assert chi2 < CHI2_4DOF_1E3, (mode, chi2)


@pytest.mark.slow
def test_tokens_per_round_truncated_geometric():
    p, q = synth.TOY_P, synth.TOY_Q
    gamma, n = 3, 400_000
    o = oracle.verify(_sm(synth.toy_batch("prob", n, seed=13, gamma=gamma)))
    alpha = float((p * q).sum())
    law = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    tokens = o["num_accepted"].astype(np.float64) + 1.0
    mean = float((law * np.arange(1, gamma + 2)).sum())
    assert np.isclose(mean, (1 - alpha ** (gamma + 1)) / (1 - alpha))
    var = float((law * (np.arange(1, gamma + 2) - mean) ** 2).sum())
    assert abs(tokens.mean() - mean) < 5 * np.sqrt(var / n), (tokens.mean(), mean)
    # every emitted position (accepted or sampled) follows p
    out = o["out_tokens"].reshape(n, gamma + 1)
    em = out[out >= 0]
    f = np.bincount(em, minlength=5)
    chi2 = float(((f - p * em.size) ** 2 / (p * em.size)).sum())
    assert chi2 < CHI2_4DOF_1E3, chi2
