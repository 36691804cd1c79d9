"""Sampler-match acceptance on the GPU vs the oracle (mlxcel "투기적 디코딩",
section "mlxcel의 프롬프트 조회": a draft is accepted iff it equals the token
the target's sampler draws at its position), through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, check_structure, compare, full_batch, oracle_all, run_gpu

pytestmark = pytest.mark.gpu

CHI2_4DOF_1E3 = 18.47


def _sm(b):
    b = dict(b)
    b["flags"] = oracle.FLAG_SAMPLER_MATCH
    return b


@pytest.mark.parametrize("mode", ["prob", "greedy"])
def test_toy_workload(mode):
    b = _sm(synth.toy_batch(mode, 1_000_000, seed=9))
    gpu = run_gpu(b)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    assert_parity(compare(b, gpu, ref))
    p, q = synth.TOY_P, synth.TOY_Q
    alpha = float((p * q).sum()) if mode == "prob" else 0.25
    acc = gpu["num_accepted"].mean()
    assert abs(acc - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / b["B"]), acc
    first = gpu["out_tokens"].reshape(-1, 2)[:, 0]
    f = np.bincount(first, minlength=5)
    chi2 = float(((f - p * first.size) ** 2 / (p * first.size)).sum())
    assert chi2 < CHI2_4DOF_1E3, chi2


@pytest.mark.parametrize("name,B,V", [
    ("c2", None, None),
    ("c2", 6, 32001),            # misaligned fp32 rows, ragged tail
    ("c3", 27, 40003),           # every temperature/filter combination, odd V
    ("c4", 24, 50000),
    ("c5", 40, 70001),
    ("c5", 33, 65536),
])
def test_scaled_workloads(name, B, V):
    b = _sm(synth.make(name, B=B, V=V))
    gpu = run_gpu(b)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    rep = compare(b, gpu, ref)
    assert_parity(rep)
    assert rep["requests"] > 0


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_full_size_every_request(name):
    b = _sm(full_batch(name))
    gpu = run_gpu(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    rep = compare(b, gpu, oracle_all(b))
    assert rep["requests"] == b["B"]
    assert_parity(rep)


def test_top_k_one_equals_greedy_entry_point():
    # fp32 logits: no tied maxima, so top_k = 1 leaves one token per row
    b = synth.make("c2", B=24, V=30011)
    b["temperature"] = np.full(b["B"], 0.8, np.float32)
    b["top_k"] = np.ones(b["B"], np.int32)
    b["top_p"] = None
    # most drafts at the target argmax, so that rounds run past position 0
    cu, ids = b["cu_num_draft"], b["draft_token_ids"].copy()
    keep = np.random.default_rng(2).random(ids.size) < 0.8
    for r in range(b["B"]):
        for i in range(int(cu[r]), int(cu[r + 1])):
            if keep[i]:
                ids[i] = int(np.argmax(b["target_logits"][i + r]))
    b["draft_token_ids"] = ids
    sm = run_gpu(_sm(b))
    gr = run_gpu(b, greedy=True)
    assert sm["status"] == 0
    assert np.array_equal(sm["num_accepted"], gr["num_accepted"])
    assert np.array_equal(sm["out_tokens"], gr["out_tokens"])
    assert sm["num_accepted"].sum() > b["B"]


def test_mismatch_emits_a_token_other_than_the_draft():
    b = _sm(synth.make("c3", B=30, V=20000))
    gpu = run_gpu(b)
    cu, ids = b["cu_num_draft"], b["draft_token_ids"]
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        k = int(gpu["num_accepted"][r])
        if b["temperature"][r] > 0 and k < c1 - c0:
            assert gpu["out_tokens"][c0 + r + k] != ids[c0 + k], r
