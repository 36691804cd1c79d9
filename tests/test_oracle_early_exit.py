"""Pins of the oracle's early-exit verification.

Page: velog "vLLM speculative decoding이 기각 토큰을 다시 뽑는 이유", section
"드래프트가 제안하고 타깃이 판정한다": the first rejection ends the round and
the later positions are discarded. Examining the rows in position order and
stopping there must change nothing that the round emits; it only leaves the
rows after the stop unread. Pinned here against the full-pass verification
(itself pinned by the exact law and the printed tables):

* same tokens, counts, accept and race margins; p(x) equal up to the stop
  and unset (NaN) after it, on workloads with every kind of request;
* rows after the stop are never read: NaN planted there voids the request
  in the full pass but leaves the early-exit result unchanged, while NaN
  planted at or before the stop voids it in both.
"""
import numpy as np
import pytest

import oracle
import synth


def _early(b):
    b = dict(b)
    b["flags"] = int(b.get("flags", 0)) | oracle.FLAG_EARLY_EXIT
    return b


@pytest.mark.parametrize("name,B,V", [("c2", None, None), ("c3", 27, 3001), ("c4", 20, 4000),
                                      ("c5", 30, 5003)])
def test_same_round_as_the_full_pass(name, B, V):
    b = synth.make(name, B=B, V=V)
    full = oracle.verify(b)
    early = oracle.verify(_early(b))
    assert np.array_equal(full["out_tokens"], early["out_tokens"])
    assert np.array_equal(full["num_accepted"], early["num_accepted"])
    assert np.array_equal(full["race_margin"], early["race_margin"], equal_nan=True)
    cu = b["cu_num_draft"]
    read = unread = 0
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        k = int(full["num_accepted"][r])
        upto = min(k + 1, c1 - c0)  # positions whose rows were examined
        assert np.array_equal(full["p_at_draft"][c0:c0 + upto], early["p_at_draft"][c0:c0 + upto])
        assert np.array_equal(full["accept_margin"][c0:c0 + upto],
                              early["accept_margin"][c0:c0 + upto], equal_nan=True)
        assert np.all(np.isnan(early["p_at_draft"][c0 + upto:c1]))
        read += upto
        unread += (c1 - c0) - upto
    assert read > 0 and unread > 0


def test_toy_rounds_unchanged():
    b = synth.toy_batch("prob", 50_000, seed=3, gamma=3)
    full = oracle.verify(b)
    early = oracle.verify(_early(b))
    assert np.array_equal(full["out_tokens"], early["out_tokens"])
    assert np.array_equal(full["num_accepted"], early["num_accepted"])


def _plant_nan(b, rows):
    b = dict(b)
    t = b["target_logits"].copy()
    for row in rows:
        if b["logits_dtype"] == "bf16":
            t[row, 7] = 0x7FC0  # bf16 NaN
        else:
            t[row, 7] = np.nan
    b["target_logits"] = t
    return b


def test_rows_after_the_stop_are_never_read():
    b = synth.make("c3", B=36, V=2000)
    clean = oracle.verify(b)
    cu = b["cu_num_draft"]
    T = b["temperature"]
    after, at = [], []
    for r in range(b["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        k = int(clean["num_accepted"][r])
        if k + 1 <= c1 - c0:
            after.append((r, c0 + r + k + 1))  # the first row after the stop
        at.append((r, c0 + r + k))             # the stop row itself
    assert len(after) > 5
    planted = _plant_nan(b, [row for _, row in after])
    full = oracle.verify(planted)
    early = oracle.verify(_early(planted))
    for r, _ in after:
        c0, c1 = int(cu[r]), int(cu[r + 1])
        row0 = c0 + r
        assert np.array_equal(early["out_tokens"][row0:c1 + r + 1],
                              clean["out_tokens"][row0:c1 + r + 1]), r
        assert early["num_accepted"][r] == clean["num_accepted"][r]
        assert early["req_status"][r] & 3 == 0
        if T[r] > 0:  # the full pass reads the planted row and voids the request
            assert full["req_status"][r] & 1
            assert full["num_accepted"][r] == 0 and np.all(full["out_tokens"][row0:c1 + r + 1] == -1)
    planted = _plant_nan(b, [row for _, row in at])
    early = oracle.verify(_early(planted))
    for r, _ in at:
        if T[r] > 0:
            c0, c1 = int(cu[r]), int(cu[r + 1])
            assert early["req_status"][r] & 1, r
            assert np.all(early["out_tokens"][c0 + r:c1 + r + 1] == -1)
