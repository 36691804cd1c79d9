"""Whole-round properties of the oracle's verify call.

* Expected tokens per round (1 - a^(g+1)) / (1 - a) under i.i.d. acceptance
  (cortexys.team "초안 모델로 생성 속도를 높이는 추측 디코딩", section "수락률 α와
  기대 속도 향상", 식 1; worked values in velog "vLLM speculative decoding이
  기각 토큰을 다시 뽑는 이유", section "수락률은 속도만 바꾸고 정답은 바꾸지
  않는다"), checked by simulation.
* Temperature 0 reproduces target-only argmax decoding exactly (cortexys,
  section 방법; mlxcel "투기적 디코딩", section 탐욕 디코딩 동등성).
* Structure of every emitted round: accepted prefix, one recovered or bonus
  token, -1 padding (mlxcel "투기적 디코딩", section 기본 라운드).
* End to end with sampling constraints: the first emitted token follows p
  after temperature / top-k / top-p (chi-square), with the filtered p taken
  from the brute-force definition in test_oracle_filters.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines
from test_oracle_filters import brute_keep


def closed_form(alpha, gamma):
    return (1 - alpha ** (gamma + 1)) / (1 - alpha)


def test_printed_expected_tokens_match_closed_form():
    for row in golden_lines("expected_tokens.txt"):
        if row[0] == "speedup":
            a, g, c, printed = float(row[1]), int(row[2]), float(row[3]), float(row[4])
            assert abs(closed_form(a, g) / (g * c + 1) - printed) < 0.005
            continue
        a, g, printed = float(row[0]), int(row[1]), float(row[2])
        assert abs(closed_form(a, g) - printed) < 0.0005 + 1e-9, row


@pytest.mark.slow
@pytest.mark.parametrize("mode,gamma,alpha", [("prob", 1, 0.75), ("greedy", 1, 0.25),
                                              ("prob", 3, 0.75), ("prob", 7, 0.75)])
def test_mean_tokens_per_round(mode, gamma, alpha):
    rounds = 200_000
    b = synth.toy_batch(mode, rounds, seed=100 + gamma, gamma=gamma)
    o = oracle.verify(b)
    tokens = o["num_accepted"].astype(np.float64) + 1
    # the number of tokens is a truncated geometric; its sd is below gamma / 2
    sd = tokens.std() / np.sqrt(rounds)
    assert abs(tokens.mean() - closed_form(alpha, gamma)) < 5 * sd


def _random_batch(seed, B=60, V=23, dtype="f32", probabilistic=True):
    rng = np.random.default_rng(seed)
    gam = rng.integers(0, 5, size=B).astype(np.int32)
    cu = np.zeros(B + 1, np.int32)
    np.cumsum(gam, out=cu[1:])
    N = int(cu[-1])
    logits = rng.normal(0, 2, size=(N + B, V)).astype(np.float32)
    logits[rng.random((N + B, V)) < 0.2] = 1.0  # ties
    q = rng.random((N, V)).astype(np.float32)
    q[rng.random((N, V)) < 0.3] = 0
    q /= np.maximum(q.sum(1, keepdims=True), 1e-30)
    ids = rng.integers(0, V, size=N).astype(np.int32)
    temp = rng.choice([0.0, 0.5, 1.0, 2.0], size=B).astype(np.float32)
    tk = rng.choice([0, 3, V], size=B).astype(np.int32)
    tp = rng.choice([1.0, 0.6, 0.9], size=B).astype(np.float32)
    if dtype == "bf16":
        logits = synth.f32_to_bf16_bits(logits)
    return dict(B=B, V=V, cu_num_draft=cu, draft_token_ids=ids, target_logits=logits,
                logits_dtype=dtype, draft_probs=q if probabilistic else None,
                temperature=temp, top_k=tk, top_p=tp, seed=seed, request_base=0, flags=0)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("probabilistic", [True, False])
def test_round_structure_and_decisions(seed, probabilistic):
    b = _random_batch(seed, probabilistic=probabilistic, dtype="bf16" if seed % 2 else "f32")
    o = oracle.verify(b)
    cu, V = b["cu_num_draft"], b["V"]
    logits = b["target_logits"]
    if b["logits_dtype"] == "bf16":
        logits = synth.bf16_bits_to_f32(logits)
    for r in range(b["B"]):
        g = cu[r + 1] - cu[r]
        row0 = cu[r] + r
        k = o["num_accepted"][r]
        toks = o["out_tokens"][row0:row0 + g + 1]
        assert 0 <= k <= g
        assert np.all(toks[:k] == b["draft_token_ids"][cu[r]:cu[r] + k])
        assert 0 <= toks[k] < V
        assert np.all(toks[k + 1:] == -1)
        T = b["temperature"][r]
        for i in range(k + (1 if k < g else 0)):
            x = b["draft_token_ids"][cu[r] + i]
            if T == 0:
                am = oracle.argmax(logits[row0 + i].astype(np.float64))
                assert (x == am) == (i < k)
                continue
            p_x = o["p_at_draft"][cu[r] + i]
            q_x = 1.0 if b["draft_probs"] is None else float(b["draft_probs"][cu[r] + i, x])
            u = oracle.accept_uniform(b["seed"], r, i)
            assert (q_x > 0 and p_x / q_x >= u) == (i < k)
        if T == 0:
            assert toks[k] == oracle.argmax(logits[row0 + k].astype(np.float64))


def test_temperature_zero_is_argmax_decoding():
    b = _random_batch(11)
    b["temperature"][:] = 0
    # drafts: the argmax at some positions, something else at others
    logits = b["target_logits"].astype(np.float64)
    cu = b["cu_num_draft"]
    rng = np.random.default_rng(0)
    for r in range(b["B"]):
        for i in range(cu[r + 1] - cu[r]):
            am = int(np.argmax(logits[cu[r] + r + i]))
            b["draft_token_ids"][cu[r] + i] = am if rng.random() < 0.7 else (am + 1) % b["V"]
    o = oracle.verify(b)
    for r in range(b["B"]):
        row0 = cu[r] + r
        k = o["num_accepted"][r]
        emitted = o["out_tokens"][row0:row0 + k + 1]
        greedy = [int(np.argmax(logits[row0 + i])) for i in range(k + 1)]
        assert emitted.tolist() == greedy


@pytest.mark.slow
@pytest.mark.parametrize("T,k,P,probabilistic", [(0.7, 4, 0.8, True), (1.3, 0, 0.6, False),
                                                  (1.0, 3, 1.0, True)])
def test_filtered_law_end_to_end(T, k, P, probabilistic):
    rounds = 300_000
    V = 7
    l = np.array([1.0, 2.5, 0.0, 2.5, -1.0, 0.5, 1.7], np.float32)
    keep, _ = brute_keep([float(x) for x in l], T, k, P)
    e = np.where(keep, np.exp((l.astype(np.float64) - l.max()) / T), 0.0)
    p = e / e.sum()
    q = np.array([0.05, 0.1, 0.3, 0.05, 0.2, 0.2, 0.1])
    B = rounds
    cu = np.arange(B + 1, dtype=np.int32)
    rng = np.random.default_rng(5)
    ids = (np.full(B, 2, np.int32) if not probabilistic
           else np.minimum(np.searchsorted(np.cumsum(q), rng.random(B)), V - 1).astype(np.int32))
    b = dict(B=B, V=V, cu_num_draft=cu, draft_token_ids=ids,
             target_logits=np.tile(l, (2 * B, 1)), logits_dtype="f32",
             draft_probs=np.tile(q.astype(np.float32), (B, 1)) if probabilistic else None,
             temperature=np.full(B, T, np.float32), top_k=np.full(B, k, np.int32),
             top_p=np.full(B, P, np.float32), seed=77, request_base=0, flags=0)
    o = oracle.verify(b)
    first = o["out_tokens"].reshape(-1, 2)[:, 0]
    counts = np.bincount(first, minlength=V)
    assert np.all(counts[p == 0] == 0)
    nz = p > 0
    chi2 = ((counts[nz] - p[nz] * B) ** 2 / (p[nz] * B)).sum()
    crit = {1: 10.83, 2: 13.82, 3: 16.27, 4: 18.47, 5: 20.52, 6: 22.46}[int(nz.sum()) - 1]
    assert chi2 < crit
