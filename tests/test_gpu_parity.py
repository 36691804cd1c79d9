"""GPU verifier vs the CPU oracle, through the C ABI, on the five workloads:
scaled variants and the full sizes, every request of each."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, check_structure, compare, full_batch, oracle_all, run_gpu

pytestmark = pytest.mark.gpu

CHI2_4DOF_1E3 = 18.47


@pytest.mark.parametrize("mode", ["prob", "greedy", "naive"])
def test_toy_workload(mode):
    b = synth.toy_batch(mode, 2_000_000)
    gpu = run_gpu(b)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    rep = compare(b, gpu, ref)
    assert_parity(rep)
    p = synth.TOY_P
    acc = gpu["num_accepted"].mean()
    sd = np.sqrt(0.75 * 0.25 / b["B"])
    first = gpu["out_tokens"].reshape(-1, 2)[:, 0]
    freq = np.bincount(first, minlength=5) / first.size
    chi2 = float(((freq - p) ** 2 / p).sum() * first.size)
    if mode == "greedy":
        assert abs(acc - 0.25) < 5 * sd
    else:
        assert abs(acc - 0.75) < 5 * sd
    if mode == "naive":
        assert chi2 > 1e4
    else:
        assert chi2 < CHI2_4DOF_1E3


@pytest.mark.parametrize("name,B,V", [
    ("c2", None, None),          # the full fp32 workload
    ("c2", 6, 32001),            # misaligned fp32 rows, ragged tail
    ("c3", 27, 40003),           # all nine temperature/filter combinations, odd V
    ("c3", 18, 40000),
    ("c4", 24, 50000),
    ("c5", 40, 70001),
    ("c5", 33, 65536),
])
def test_scaled_workloads(name, B, V):
    b = synth.make(name, B=B, V=V)
    gpu = run_gpu(b)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    assert_parity(compare(b, gpu, ref))


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_full_size_every_request(name):
    """The full workload, every request against the oracle (run on every host
    core), and every temperature-0 request against numpy's argmax."""
    b = full_batch(name)
    gpu = run_gpu(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    ref = oracle_all(b)
    rep = compare(b, gpu, ref)
    assert rep["requests"] == b["B"]
    assert_parity(rep)
    # temperature-0 requests: the emitted tokens are the target argmax at each
    # emitted position (argmax decoding)
    cu = b["cu_num_draft"]
    logits = b["target_logits"]
    for r in np.nonzero(b["temperature"] == 0)[0]:
        row0 = int(cu[r]) + int(r)
        k = int(gpu["num_accepted"][r])
        rows = logits[row0:row0 + k + 1]
        if b["logits_dtype"] == "bf16":
            rows = synth.bf16_bits_to_f32(rows)
        assert np.array_equal(gpu["out_tokens"][row0:row0 + k + 1], np.argmax(rows, axis=1)), r


def test_greedy_entry_point():
    b = synth.make("c5", B=24, V=30011)
    gpu = run_gpu(b, greedy=True)
    b0 = dict(b)
    b0["temperature"] = np.zeros_like(b["temperature"])
    ref = oracle.verify(b0)
    assert np.array_equal(gpu["num_accepted"], ref["num_accepted"])
    assert np.array_equal(gpu["out_tokens"], ref["out_tokens"])
    assert np.array_equal(gpu["p_at_draft"], ref["p_at_draft"].astype(np.float32))


def test_request_base_split_equals_whole():
    b = synth.make("c3", B=20, V=20000)
    whole = run_gpu(b)
    cu = b["cu_num_draft"]
    h = 11
    parts = []
    for lo, hi in ((0, h), (h, b["B"])):
        n0, n1 = int(cu[lo]), int(cu[hi])
        part = dict(b)
        part.update(B=hi - lo, cu_num_draft=(cu[lo:hi + 1] - n0).astype(np.int32),
                    draft_token_ids=b["draft_token_ids"][n0:n1],
                    target_logits=b["target_logits"][n0 + lo:n1 + hi],
                    draft_probs=b["draft_probs"][n0:n1], temperature=b["temperature"][lo:hi],
                    top_k=b["top_k"][lo:hi], top_p=b["top_p"][lo:hi], request_base=lo)
        parts.append(run_gpu(part))
    assert np.array_equal(np.concatenate([p["out_tokens"] for p in parts]), whole["out_tokens"])
    assert np.array_equal(np.concatenate([p["num_accepted"] for p in parts]),
                          whole["num_accepted"])


def test_repeated_calls_are_identical():
    import speculative_decoding_rejection_02_gb300 as sv
    b = synth.make("c5", B=16, V=40000)
    R = b["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=16, max_rows=R, max_vocab=40000)
    first = run_gpu(b, verifier=ver)
    for _ in range(3):
        again = run_gpu(b, verifier=ver)
        assert np.array_equal(first["out_tokens"], again["out_tokens"])
        assert np.array_equal(first["p_at_draft"], again["p_at_draft"])
    ver.close()
