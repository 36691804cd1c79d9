"""Round-level metrics: the closed forms pinned to the values the pages print,
and the counters checked on oracle rounds whose acceptance law is known."""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines
from speculative_decoding_rejection_02_gb300 import metrics


def test_printed_expected_tokens_and_speedup():
    for row in golden_lines("expected_tokens.txt"):
        if row[0] == "speedup":
            a, g, c, printed = float(row[1]), int(row[2]), float(row[3]), float(row[4])
            assert abs(metrics.speedup(a, g, c) - printed) < 0.005
        else:
            a, g, printed = float(row[0]), int(row[1]), float(row[2])
            assert abs(metrics.expected_tokens(a, g) - printed) < 0.0005 + 1e-9


def test_gemma_upper_bound_as_printed():
    # cortexys, section 맥북 실측: the logged acceptance 0.901 put into 식 1
    # with c = 0 gives an upper bound of 3.44x at gamma = 3.
    assert abs(metrics.speedup(0.901, 3, 0.0) - 3.44) < 0.005


def test_speedup_with_verifier_reduces_to_theorem():
    assert metrics.speedup_with_verifier(0.8, 5, 0.05, 1.0, 0.0) == pytest.approx(
        metrics.speedup(0.8, 5, 0.05))
    assert metrics.speedup_with_verifier(0.8, 5, 0.0, 1.0, 0.1) < metrics.speedup(0.8, 5, 0.0)


def test_round_stats_on_iid_rounds():
    b = synth.toy_batch("prob", 100_000, seed=9, gamma=3)
    o = oracle.verify(b)
    st = metrics.round_stats(b["cu_num_draft"], o["num_accepted"])
    assert st["draft_rounds"] == 100_000 and st["draft_n"] == 300_000
    # every position accepts with probability sum min(p, q) = 0.75
    for a in st["acceptance_by_position"]:
        assert abs(a - 0.75) < 0.01
    assert abs(st["tokens_per_verification"] - metrics.expected_tokens(0.75, 3)) < 0.02
    assert st["mean_accepted_length"] == pytest.approx(st["tokens_per_verification"] - 1)


def test_round_stats_counts_by_hand():
    cu = [0, 2, 2, 5]
    k = [1, 0, 3]
    st = metrics.round_stats(cu, k)
    assert st["draft_n"] == 5 and st["draft_n_accepted"] == 4 and st["draft_rounds"] == 3
    # position 0 judged in requests 0 and 2 (both accept); position 1 judged
    # in 0 (reject) and 2 (accept); position 2 only in 2 (accept)
    assert st["acceptance_by_position"] == [1.0, 0.5, 1.0]
    assert st["all_accepted_fraction"] == pytest.approx(2 / 3)
