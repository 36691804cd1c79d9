"""Early-exit verification on the GPU (velog "드래프트가 제안하고 타깃이
판정한다": the first rejection ends the round), through the C ABI, against
the oracle under the same flag and against the GPU's own full pass. Four
schedules are run: rows read position by position through the work queue
and the full pass with early-exit judgement (each forced with a test-only
handle flag), the library's own choice between those two, and the cluster
kernel that keeps each judged row in shared memory and draws the token at
the stop from it (a handle flag; batches with top-k / top-p fall back to the
library's choice)."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, check_structure, compare, full_batch, oracle_all, run_gpu

pytestmark = pytest.mark.gpu

SCHEDULES = ["queue", "full", "auto", "resident"]


def _run(b, schedule, greedy=False):
    import speculative_decoding_rejection_02_gb300 as sv
    R = b["target_logits"].shape[0]
    flags = {"queue": sv.CONFIG_EARLY_QUEUE, "full": sv.CONFIG_EARLY_FULL_PASS,
             "auto": 0, "resident": sv.CONFIG_EARLY_RESIDENT}[schedule]
    ver = sv.Verifier(max_batch=max(b["B"], 1), max_rows=max(R, 1), max_vocab=b["V"],
                      config_flags=flags)
    try:
        return run_gpu(b, greedy=greedy, verifier=ver)
    finally:
        ver.close()


def _early(b):
    b = dict(b)
    b["flags"] = int(b.get("flags", 0)) | oracle.FLAG_EARLY_EXIT
    return b


def _unread_are_nan(b, out):
    cu = b["cu_num_draft"]
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        k = int(out["num_accepted"][r])
        assert np.all(np.isnan(out["p_at_draft"][c0 + k + 1:c1])), r


@pytest.mark.parametrize("name,B,V", [
    ("c2", None, None),      # fp32 rows, no filters
    ("c2", 6, 32008),        # fp32, ragged tail inside the last stage
    ("c2", 6, 32001),        # misaligned fp32 rows: always the full pass
    ("c3", 27, 40003),       # odd V with filters: the full pass and the exact filter kernel
    ("c3", 27, 40000),       # every temperature / filter combination
    ("c4", 24, 50000),       # one-hot drafts, top-p
    ("c5", 40, 70000),
    ("c5", 33, 65536),
])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_scaled_workloads(name, B, V, schedule):
    b = _early(synth.make(name, B=B, V=V))
    gpu = _run(b, schedule)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    assert_parity(compare(b, gpu, ref))
    _unread_are_nan(b, gpu)


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_same_round_as_the_full_pass(name, schedule):
    b = synth.make(name, B=64 if name != "c3" else None, V=None)
    full = run_gpu(b)
    early = _run(_early(b), schedule)
    assert early["status"] == 0
    assert np.array_equal(full["out_tokens"], early["out_tokens"])
    assert np.array_equal(full["num_accepted"], early["num_accepted"])
    cu = b["cu_num_draft"]
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        upto = min(int(full["num_accepted"][r]) + 1, c1 - c0)
        # a row split over several CTAs sums Z in another order: last bits
        assert np.allclose(full["p_at_draft"][c0:c0 + upto], early["p_at_draft"][c0:c0 + upto],
                           rtol=1e-5, atol=0)


@pytest.mark.parametrize("name,schedule", [
    ("c3", "auto"), ("c4", "auto"), ("c5", "auto"),  # the library's own choice
    ("c3", "queue"), ("c4", "queue"),                # the work queue at full size
    ("c5", "resident"),                              # rows held in clusters
])
def test_full_size_every_request(name, schedule):
    b = _early(full_batch(name))
    gpu = run_gpu(b) if schedule == "auto" else _run(b, schedule)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    rep = compare(b, gpu, oracle_all(b))
    assert rep["requests"] == b["B"]
    assert_parity(rep)
    _unread_are_nan(b, gpu)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_rows_after_the_stop_do_not_count(schedule):
    """NaN planted in the row after each stop: never read by the queue, read
    but without effect by the full pass."""
    b = synth.make("c3", B=36, V=4000)
    clean = run_gpu(b)
    cu = b["cu_num_draft"]
    t = b["target_logits"].copy()
    planted = []
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        k = int(clean["num_accepted"][r])
        if k + 1 <= c1 - c0:
            t[c0 + r + k + 1, 5] = 0x7FC0  # bf16 NaN in the first row after the stop
            planted.append(r)
    assert len(planted) > 5
    nb = dict(b)
    nb["target_logits"] = t
    early = _run(_early(nb), schedule)
    assert early["status"] == 0  # the NaN rows do not count
    assert np.array_equal(early["out_tokens"], clean["out_tokens"])
    assert np.array_equal(early["num_accepted"], clean["num_accepted"])
    full = run_gpu(nb)
    assert full["status"] & 0x1  # the full pass reads them


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_edge_rounds(schedule):
    # gamma = 0 requests, a long round, T = 0 and T > 0 mixed, unusable row at the stop
    rng = np.random.default_rng(5)
    V = 1024
    gam = np.array([0, 3, 40, 1, 0, 5, 2])
    B = gam.size
    cu = np.concatenate([[0], np.cumsum(gam)]).astype(np.int32)
    N = int(cu[-1])
    logits = rng.normal(0, 2, size=(N + B, V)).astype(np.float32)
    ids = np.empty(N, np.int32)
    for r in range(B):
        for i in range(int(gam[r])):
            ids[cu[r] + i] = int(np.argmax(logits[cu[r] + r + i]))  # argmax drafts: long rounds
    logits[cu[5] + 5 + 0, 3] = np.inf  # request 5 is voided at its first row
    b = dict(B=B, V=V, cu_num_draft=cu, draft_token_ids=ids,
             target_logits=synth.f32_to_bf16_bits(logits), logits_dtype="bf16", draft_probs=None,
             temperature=np.array([1, 0, 1, 0.7, 0, 1, 1], np.float32), top_k=None, top_p=None,
             seed=9, request_base=0, flags=oracle.FLAG_EARLY_EXIT)
    gpu = _run(b, schedule)
    ref = oracle.verify(b)
    assert gpu["status"] & 0x1
    assert_parity(compare(b, gpu, ref))
    assert gpu["num_accepted"][5] == 0 and np.all(gpu["out_tokens"][cu[5] + 5:cu[6] + 6] == -1)


def test_resident_bad_offsets_end_their_requests():
    """Cluster schedule: a request whose offsets are out of order is ended
    with SPEC_STATUS_BAD_OFFSETS and no rows read; the call still ends."""
    b = _early(synth.make("c5", B=12, V=4096))
    cu = b["cu_num_draft"].copy()
    cu[5], cu[6] = cu[6], cu[5]
    b["cu_num_draft"] = cu
    gpu = _run(b, "resident")
    assert gpu["status"] & 0x10
    assert gpu["num_accepted"][5] == 0


@pytest.mark.parametrize("case", ["host_q", "top_p", "misaligned"])
def test_resident_handle_falls_back_where_the_batch_needs_it(case):
    """A handle asking for the cluster schedule still verifies batches that
    schedule cannot take (draft_probs in page-locked host memory, top-p
    rows, rows that are not 16-byte aligned), with the same results as a
    default handle."""
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    if case == "top_p":
        b = _early(synth.make("c4", B=24, V=50000))
    elif case == "misaligned":
        b = _early(synth.make("c2", B=6, V=32001))
    else:
        b = _early(synth.make("c5", B=20, V=20008))
    R = b["target_logits"].shape[0]
    outs = []
    for flags in (0, sv.CONFIG_EARLY_RESIDENT):
        ver = sv.Verifier(max_batch=b["B"], max_rows=R, max_vocab=b["V"], config_flags=flags)
        db = sv.upload(b, "cuda:0")
        if case == "host_q":
            db.draft_probs = torch.from_numpy(b["draft_probs"]).pin_memory()
        ver.run(db)
        torch.cuda.synchronize()
        assert ver.status() == 0
        outs.append((db.out_tokens.cpu().numpy(), db.num_accepted.cpu().numpy()))
        ver.close()
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_naive_control_under_early_exit(schedule):
    """The negative control (a rejected position redrawn from p) combined
    with early exit, under every schedule, against the oracle."""
    b = _early(synth.make("c5", B=40, V=20008))
    b["flags"] = int(b["flags"]) | oracle.FLAG_NAIVE
    gpu = _run(b, schedule)
    ref = oracle.verify(b)
    assert gpu["status"] == 0
    check_structure(b, gpu)
    assert_parity(compare(b, gpu, ref))
