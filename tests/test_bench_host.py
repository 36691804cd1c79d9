"""Host-side logic of bench.py (no GPU): the algorithmic byte count of one
call and the all-cores oracle baseline."""
import os
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402


def test_algorithmic_bytes_by_hand():
    """Three requests (gamma 2, 0, 3), V = 10, bf16 logits, draft probs:
    request 0 (T > 0) rejects at position 1, request 1 (T > 0) has no draft
    tokens, request 2 is at temperature 0."""
    V = 10
    cu = np.array([0, 2, 2, 5], np.int32)
    batch = dict(B=3, V=V, cu_num_draft=cu, logits_dtype="bf16",
                 draft_probs=np.zeros((5, V), np.float32),
                 temperature=np.array([1.0, 0.5, 0.0], np.float32), flags=0)
    n_acc = np.array([1, 0, 3], np.int32)
    b = bench.algorithmic_bytes(batch, n_acc)
    R = 5 + 3
    assert b["row_pass"] == R * V * 2 == b["all_rows"]
    # one rejected request at T > 0 with a draft row: its q row is read
    assert b["race_q"] == V * 4
    # q(x) gathers of the judged positions at T > 0: min(n_acc + 1, gamma)
    assert b["q_gathers"] == (min(1 + 1, 2) + min(0 + 1, 0)) * 4
    # rows up to each request's first rejection: min(n_acc + 1, gamma + 1)
    assert b["rows_to_first_rejection"] == (2 + 1 + 4) * V * 2
    assert b["total"] == b["row_pass"] + b["race_q"] + b["small"]
    # early exit reads only those rows
    batch["flags"] = 4
    assert bench.algorithmic_bytes(batch, n_acc)["row_pass"] == (2 + 1 + 4) * V * 2


def test_parallel_oracle_calls_match_one_serial_call():
    """The all-cores baseline runs the unchanged oracle on disjoint request
    sets from several threads at once: the union of those results must be
    the single-threaded result."""
    batch = synth.make("c3", B=24, V=2003)
    whole = oracle.verify(batch)
    parts = [list(range(t, batch["B"], 4)) for t in range(4)]
    with ThreadPoolExecutor(4) as ex:
        outs = list(ex.map(lambda reqs: oracle.verify(batch, requests=reqs), parts))
    cu = batch["cu_num_draft"]
    for reqs, out in zip(parts, outs):
        for r in reqs:
            rows = slice(int(cu[r]) + r, int(cu[r + 1]) + r + 1)
            assert out["num_accepted"][r] == whole["num_accepted"][r]
            assert np.array_equal(out["out_tokens"][rows], whole["out_tokens"][rows])


def test_all_cores_baseline_reports_its_sample():
    batch = synth.make("c2", B=8, V=512)
    rate, desc, secs, threads = bench.cpu_oracle_rate_all_cores(batch, 0.05)
    assert rate > 0 and secs > 0
    assert 1 <= threads <= bench.host_cores()
    assert "threads on disjoint request sets" in desc


def test_race_issue_arithmetic_and_its_guards(monkeypatch):
    """The race's issue figure: warp instructions = instructions per entry x
    entries / 32 over the race phase, against SMs x 4 x the sampled clock;
    absent for other workloads, changed race sources or missing clocks."""
    import types

    import torch

    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda dev: types.SimpleNamespace(multi_processor_count=152))
    monkeypatch.setattr(bench, "RACE_SOURCES_SHA", bench.race_source_sha())
    args = types.SimpleNamespace(config="c5", accept="rejection", resident=False, V=None,
                                 top_p=None, top_k=None)
    batch = {"temperature": np.array([0.0, 0.8] * 8, np.float32), "V": 1000}
    r = bench.race_issue(batch, None, 0.5, args, {"sm_mhz": 2000.0}, None)
    want = bench.RACE_INSTR_PER_ENTRY * 8 * 1000 / 32 / 0.5e-3 / 1e9
    assert abs(r["achieved"] - want) < 1e-9 * want
    assert abs(r["peak"] - 152 * 4 * 2000e6 / 1e9) < 1e-9
    assert r["entries"] == 8000 and r["bound"] == "issue"
    assert bench.race_issue(batch, None, 0.5, args, None, None) is None
    for k, v in (("config", "c4"), ("accept", "sampler-match"), ("V", 5000)):
        other = types.SimpleNamespace(**{**vars(args), k: v})
        assert bench.race_issue(batch, None, 0.5, other, {"sm_mhz": 2000.0}, None) is None
    monkeypatch.setattr(bench, "RACE_SOURCES_SHA", "0" * 16)
    assert bench.race_issue(batch, None, 0.5, args, {"sm_mhz": 2000.0}, None) is None


def test_request_chunks_cover_the_batch_in_order():
    for B, k in ((1, 4), (5, 1), (7, 3), (1024, 4), (3, 8)):
        cu = np.arange(B + 1, dtype=np.int32) * 2
        ch = bench.request_chunks(cu, k)
        assert ch[0][0] == 0 and ch[-1][1] == B
        assert all(r1 > r0 for r0, r1 in ch)
        assert all(ch[i][1] == ch[i + 1][0] for i in range(len(ch) - 1))
        assert len(ch) == min(k, B)
