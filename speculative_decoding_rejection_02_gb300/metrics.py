"""Round-level metrics of speculative verification (host side).

Summaries of what the verifier returns, in the terms the pages use:
* per-request counters as mlxcel reports them ("투기적 디코딩", section 응답에
  실리는 요청별 수락 통계: draft_n, draft_n_accepted, draft_rounds; mean
  accepted length = draft_n_accepted / draft_rounds) and its metric table
  (section 핵심 지표: token accept rate, mean accepted prefix length, tokens
  per verification);
* acceptance per position, which cortexys ("초안 모델로 생성 속도를 높이는
  추측 디코딩", section 맥북 실측) observed falling with depth (0.951, 0.889,
  0.852 at gamma = 3), unlike the i.i.d. assumption of its 식 1;
* the closed forms of cortexys section "수락률 α와 기대 속도 향상": expected
  tokens per round (1 - a^(g+1)) / (1 - a) (식 1) and the wall-time speedup
  (1 - a^(g+1)) / ((1 - a)(g c + 1)) (정리 3.8), plus the same model with a
  measured verification time added to each round.
"""
from __future__ import annotations

import numpy as np


def expected_tokens(alpha: float, gamma: int) -> float:
    """E[tokens per round] under i.i.d. acceptance with rate alpha."""
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def speedup(alpha: float, gamma: int, c: float) -> float:
    """Wall-time speedup with draft/target cost ratio c (Theorem 3.8)."""
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def speedup_with_verifier(alpha: float, gamma: int, t_draft: float, t_target: float,
                          t_verify: float) -> float:
    """The same model with the verification step's own time added to every
    round: tokens per round over the round's time (gamma drafts, one target
    pass, one verification), relative to one target pass per token."""
    return expected_tokens(alpha, gamma) * t_target / (gamma * t_draft + t_target + t_verify)


def round_stats(cu_num_draft, num_accepted) -> dict:
    """Counters and rates of one batch of verification rounds."""
    cu = np.asarray(cu_num_draft, dtype=np.int64)
    k = np.asarray(num_accepted, dtype=np.int64)
    gam = np.diff(cu)
    rounds = int(k.size)
    draft_n = int(gam.sum())
    accepted = int(k.sum())
    gmax = int(gam.max()) if rounds else 0
    reached = np.zeros(gmax, np.int64)
    passed = np.zeros(gmax, np.int64)
    for i in range(gmax):
        judged = (gam > i) & (k >= i)  # position i exists and was judged
        reached[i] = int(judged.sum())
        passed[i] = int((judged & (k > i)).sum())
    with np.errstate(invalid="ignore", divide="ignore"):
        per_pos = np.where(reached > 0, passed / np.maximum(reached, 1), np.nan)
    return {
        "draft_rounds": rounds,
        "draft_n": draft_n,
        "draft_n_accepted": accepted,
        "token_accept_rate": accepted / draft_n if draft_n else float("nan"),
        "mean_accepted_length": accepted / rounds if rounds else float("nan"),
        "tokens_per_verification": (accepted + rounds) / rounds if rounds else float("nan"),
        "all_accepted_fraction": float(np.mean(k == gam)) if rounds else float("nan"),
        "acceptance_by_position": per_pos.tolist(),
    }
