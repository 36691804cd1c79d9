"""GPU-vs-oracle comparison under the parity rules.

* argmax / temperature-0 outputs: identical.
* accepted counts and tokens: identical, except where the oracle's first
  differing decision has a relative margin below 1e-5 (|p/q - u| / u for an
  accept test, (s1 - s2) / s1 for a race, |mass above - top_p| / top_p for a
  top-p boundary); such excused decisions are counted. Under sampler-match
  acceptance the decision at a position is the race drawn on its row.
* p at the draft tokens: relative 1e-5 for fp32 logits, 2e-3 for bf16 (rows
  whose top-p boundary margin is below 1e-5 are skipped).
"""
import numpy as np

MARGIN = 1e-5


def run_gpu(batch, greedy=False, device="cuda:0", verifier=None):
    import torch

    import speculative_decoding_rejection_02_gb300 as sv

    B, V = batch["B"], batch["V"]
    R = batch["target_logits"].shape[0]
    ver = verifier or sv.Verifier(max_batch=max(B, 1), max_rows=max(R, 1), max_vocab=V)
    db = sv.upload(batch, device)
    (ver.greedy if greedy else ver.run)(db)
    torch.cuda.synchronize()
    out = dict(out_tokens=db.out_tokens.cpu().numpy(), num_accepted=db.num_accepted.cpu().numpy(),
               p_at_draft=db.p_at_draft.cpu().numpy(), status=ver.status())
    if verifier is None:
        ver.close()
    return out


def compare(batch, gpu, ref, requests=None, check_p=True):
    cu = batch["cu_num_draft"]
    B = batch["B"]
    temps = batch["temperature"]
    reqs = range(B) if requests is None else requests
    bf16 = batch["logits_dtype"] == "bf16"
    rtol = 2e-3 if bf16 else 1e-5
    sampler_match = bool(int(batch.get("flags", 0)) & 2)
    rep = dict(requests=0, decisions=0, excused=0, unexcused=[], p_checked=0, p_bad=[],
               p_max_rel=0.0)
    for r in reqs:
        r = int(r)
        if ref["req_status"][r] & 3:
            continue
        c0, c1 = int(cu[r]), int(cu[r + 1])
        g = c1 - c0
        row0 = c0 + r
        ko, kg = int(ref["num_accepted"][r]), int(gpu["num_accepted"][r])
        to = ref["out_tokens"][row0:row0 + g + 1]
        tg = gpu["out_tokens"][row0:row0 + g + 1]
        rep["requests"] += 1
        rep["decisions"] += ko + 1
        if ko != kg or not np.array_equal(to, tg):
            if ko != kg:
                d = min(ko, kg)
            else:
                d = int(np.nonzero(to != tg)[0][0])
            margins = [ref["topp_margin"][row0 + d]]
            if sampler_match:
                # the decision at position d is the race drawn on row d
                margins.append(ref["row_race_margin"][row0 + d])
            else:
                if d < g:
                    margins.append(ref["accept_margin"][c0 + d])
                if d == ko:
                    margins.append(ref["race_margin"][r])
            if temps[r] > 0 and np.nanmin(margins) < MARGIN:
                rep["excused"] += 1
            else:
                rep["unexcused"].append(dict(r=r, d=d, k_oracle=ko, k_gpu=kg,
                                             oracle=to.tolist(), gpu=tg.tolist(),
                                             margins=[float(x) for x in margins]))
        if check_p:
            for i in range(g):
                if ref["topp_margin"][row0 + i] < MARGIN:
                    continue
                po, pg = float(ref["p_at_draft"][c0 + i]), float(gpu["p_at_draft"][c0 + i])
                rep["p_checked"] += 1
                err = abs(pg - po)
                rel = err / po if po > 0 else err
                if po > 1e-30:
                    rep["p_max_rel"] = max(rep["p_max_rel"], rel)
                if err > rtol * abs(po) + 1e-30:
                    rep["p_bad"].append((r, i, po, pg))
    return rep


def assert_parity(rep, max_excused_frac=1e-4):
    assert not rep["unexcused"], rep["unexcused"][:5]
    assert not rep["p_bad"], rep["p_bad"][:5]
    allowed = max(1, int(max_excused_frac * rep["decisions"]))
    assert rep["excused"] <= allowed, rep


def check_structure(batch, gpu):
    """Properties of any emitted round, at any size: accepted prefix equal to
    the drafts, one token in [0, V), then -1."""
    cu = batch["cu_num_draft"]
    ids = batch["draft_token_ids"]
    V = batch["V"]
    for r in range(batch["B"]):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        g = c1 - c0
        row0 = c0 + r
        k = int(gpu["num_accepted"][r])
        t = gpu["out_tokens"][row0:row0 + g + 1]
        assert 0 <= k <= g, (r, k, g)
        assert np.array_equal(t[:k], ids[c0:c0 + k]), r
        assert 0 <= t[k] < V, (r, t)
        assert np.all(t[k + 1:] == -1), r
