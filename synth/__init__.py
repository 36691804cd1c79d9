"""Seeded synthetic inputs for the speculative-sampling verifier.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests. It holds none of the verifier's arithmetic: it only draws target
logits, draft distributions and draft tokens (what a target model and a
draft model would have produced), row by row, from counter-style seeds so
that any single row can be regenerated on its own.

Recipes (the pages measure on public tasks; these seeded synthetic inputs
stand in for them, with the shapes and distributions of the five workloads):

* ``toy``  V=5, gamma=1, fixed p=[.50,.25,.15,.07,.03] and
  q=[.30,.40,.10,.15,.05] (the 5-token example of the velog post "vLLM
  speculative decoding이 기각 토큰을 다시 뽑는 이유", section "Java로 규칙을
  재현해 본 결과"); logits = ln p in fp32, temperature 1; one request per
  round; modes ``prob`` (x ~ q), ``greedy`` (x = argmax q, q one-hot, i.e.
  no draft_probs) and ``naive`` (prob with the resample-from-p control flag).
* ``c2``   B=8, gamma=3, V=32000, fp32 logits ~ N(0, 2^2), 3 random tokens per
  row +6; draft = target + N(0, 1); q = softmax(draft); x ~ q; T=1.
* ``c3``   B=64, gamma=5, V=128256, bf16 logits ~ N(0, 3^2) + Zipf(1.1) bias
  over a per-request random permutation; draft = target + N(0, 1.5^2);
  T by r mod 3 in {0, 0.7, 1}; filter by (r div 3) mod 3: none, top_k=50,
  top_p=0.9; T>0: q = softmax(draft / T), x ~ q; T=0: x = argmax(draft).
* ``c4``   B=256, gamma=4, V=151936, bf16 logits ~ N(0, 2.5^2) + Zipf(1.0);
  x = argmax(target + N(0, 1)), no draft_probs (one-hot draft); T=1,
  top_p=0.95.
* ``c5``   B=1024, gamma_r ~ U{1..7}, V=256000, bf16 logits ~ N(0, 2^2) +
  Zipf(1.2); sigma_r ~ U[0.5, 2]; draft = target + N(0, sigma_r^2); even r at
  T=0 with x = argmax(draft); odd r at T=0.8 with q = softmax(draft / 0.8),
  x ~ q.

Zipf(s) bias: the token at rank k (1-based) of a seeded random permutation
gets -s ln k, so softmax(bias) is proportional to k^-s.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

TOY_P = np.array([0.50, 0.25, 0.15, 0.07, 0.03])
TOY_Q = np.array([0.30, 0.40, 0.10, 0.15, 0.05])

_TAG_TARGET, _TAG_NOISE, _TAG_PERM, _TAG_BOOST = 1, 2, 3, 4
_TAG_SAMPLE, _TAG_GAMMA, _TAG_SIGMA = 5, 6, 7

CONFIGS = {
    "c2": dict(B=8, gamma=3, V=32000, dtype="f32", sigma=2.0, zipf=None, boost=(3, 6.0),
               draft_sigma=1.0, temps=(1.0,), filters=("none",), draft="prob", seed=1),
    "c3": dict(B=64, gamma=5, V=128256, dtype="bf16", sigma=3.0, zipf=1.1, boost=None,
               draft_sigma=1.5, temps=(0.0, 0.7, 1.0), filters=("none", "topk50", "topp0.9"),
               draft="prob", seed=3),
    "c4": dict(B=256, gamma=4, V=151936, dtype="bf16", sigma=2.5, zipf=1.0, boost=None,
               draft_sigma=1.0, temps=(1.0,), filters=("topp0.95",), draft="greedy", seed=4),
    "c5": dict(B=1024, gamma=(1, 7), V=256000, dtype="bf16", sigma=2.0, zipf=1.2, boost=None,
               draft_sigma=(0.5, 2.0), temps=("even0", 0.8), filters=("none",), draft="prob",
               seed=5),
}


def _rng(seed, *key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def _softmax64(x):
    z = x.astype(np.float64)
    z -= z.max()
    np.exp(z, out=z)
    z /= z.sum()
    return z


def _sample_inverse_cdf(prob, u):
    """Inverse-CDF draw from a (not necessarily normalised) probability row."""
    c = np.cumsum(prob, dtype=np.float64)
    idx = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(idx, prob.size - 1)


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


# ---------------------------------------------------------------------------
# The toy workload (5-token example)
# ---------------------------------------------------------------------------

def toy_batch(mode: str = "prob", rounds: int = 2_000_000, seed: int = 42, gamma: int = 1,
              p=TOY_P, q=TOY_Q):
    """One request per round; gamma positions, every position with the same
    p and q (i.i.d. positions, as the expected-length formula assumes)."""
    p = np.asarray(p, np.float64)
    q = np.asarray(q, np.float64)
    V = p.size
    B = rounds
    N = B * gamma
    cu = (np.arange(B + 1, dtype=np.int64) * gamma).astype(np.int32)
    logits = np.empty((N + B, V), np.float32)
    logits[:] = np.log(p).astype(np.float32)
    rng = _rng(seed, _TAG_SAMPLE)
    if mode == "greedy":
        ids = np.full(N, int(np.argmax(q)), np.int32)
        dprobs = None
    else:
        u = rng.random(N)
        ids = np.minimum(np.searchsorted(np.cumsum(q), u * q.sum(), side="right"),
                         V - 1).astype(np.int32)
        dprobs = np.empty((N, V), np.float32)
        dprobs[:] = q.astype(np.float32)
    return dict(name=f"toy-{mode}", B=B, V=V, cu_num_draft=cu, draft_token_ids=ids,
                target_logits=logits, logits_dtype="f32", draft_probs=dprobs,
                temperature=np.ones(B, np.float32), top_k=None, top_p=None,
                seed=seed, request_base=0, flags=1 if mode == "naive" else 0)


# ---------------------------------------------------------------------------
# The logit workloads (c2 .. c5) and scaled variants of them
# ---------------------------------------------------------------------------

def _filter_of(name):
    if name == "none":
        return 0, 1.0
    if name.startswith("topk"):
        return int(name[4:]), 1.0
    if name.startswith("topp"):
        return 0, float(name[4:])
    raise ValueError(name)


def make(name: str, B: int | None = None, V: int | None = None, seed: int | None = None,
         gamma=None, dtype: str | None = None, threads: int | None = None):
    """Generate workload ``name`` (c2..c5), optionally resized.

    Every row is drawn from its own seed (workload seed, tag, request,
    position), so a resized workload keeps the recipe and the per-request
    structure (temperature / filter cycle, gamma law) of the full one.
    """
    cfg = dict(CONFIGS[name])
    if B is not None:
        cfg["B"] = B
    if V is not None:
        cfg["V"] = V
    if seed is not None:
        cfg["seed"] = seed
    if gamma is not None:
        cfg["gamma"] = gamma
    if dtype is not None:
        cfg["dtype"] = dtype
    B, V, s = cfg["B"], cfg["V"], cfg["seed"]

    g = cfg["gamma"]
    if isinstance(g, tuple):
        gam = _rng(s, _TAG_GAMMA).integers(g[0], g[1] + 1, size=B).astype(np.int32)
    else:
        gam = np.full(B, g, np.int32)
    cu = np.zeros(B + 1, np.int32)
    np.cumsum(gam, out=cu[1:])
    N = int(cu[-1])

    temps = np.zeros(B, np.float32)
    tk = np.zeros(B, np.int32)
    tp = np.ones(B, np.float32)
    for r in range(B):
        t = cfg["temps"]
        if t == ("even0", 0.8):
            temps[r] = 0.0 if r % 2 == 0 else 0.8
        else:
            temps[r] = t[r % len(t)]
        f = cfg["filters"]
        tk[r], tp[r] = _filter_of(f[(r // 3) % len(f)] if len(f) > 1 else f[0])

    ds = cfg["draft_sigma"]
    if isinstance(ds, tuple):
        sig = _rng(s, _TAG_SIGMA).uniform(ds[0], ds[1], size=B)
    else:
        sig = np.full(B, ds)

    zipf_base = None
    if cfg["zipf"] is not None:
        zipf_base = (-cfg["zipf"] * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(
            np.float32)

    bf16 = cfg["dtype"] == "bf16"
    logits = np.empty((N + B, V), np.uint16 if bf16 else np.float32)
    prob_draft = cfg["draft"] == "prob"
    dprobs = np.zeros((N, V), np.float32) if prob_draft else None
    ids = np.zeros(N, np.int32)

    def one_request(r):
        bias = None
        if zipf_base is not None:
            perm = _rng(s, _TAG_PERM, r).permutation(V)
            bias = np.empty(V, np.float32)
            bias[perm] = zipf_base
        row0 = int(cu[r]) + r
        for i in range(int(gam[r]) + 1):
            x = _rng(s, _TAG_TARGET, r, i).standard_normal(V, dtype=np.float32)
            x *= np.float32(cfg["sigma"])
            if bias is not None:
                x += bias
            if cfg["boost"] is not None:
                n_b, amount = cfg["boost"]
                hot = _rng(s, _TAG_BOOST, r, i).choice(V, size=n_b, replace=False)
                x[hot] += np.float32(amount)
            logits[row0 + i] = f32_to_bf16_bits(x) if bf16 else x
            if i == gam[r]:
                break
            d = _rng(s, _TAG_NOISE, r, i).standard_normal(V, dtype=np.float32)
            d *= np.float32(sig[r])
            d += x
            n = int(cu[r]) + i
            if prob_draft and temps[r] > 0:
                qq = _softmax64(d / np.float32(temps[r])).astype(np.float32)
                dprobs[n] = qq
                u = _rng(s, _TAG_SAMPLE, r, i).random()
                ids[n] = _sample_inverse_cdf(qq, u)
            else:
                ids[n] = int(np.argmax(d))

    with ThreadPoolExecutor(max_workers=threads or _threads()) as ex:
        list(ex.map(one_request, range(B)))

    return dict(name=name, B=B, V=V, cu_num_draft=cu, draft_token_ids=ids,
                target_logits=logits, logits_dtype=cfg["dtype"], draft_probs=dprobs,
                temperature=temps, top_k=tk if np.any(tk > 0) else None,
                top_p=tp if np.any(tp < 1) else None, seed=s, request_base=0, flags=0)


def batch_bytes(batch) -> dict:
    """Sizes of the batch's arrays in bytes (for reporting)."""
    out = {}
    for k in ("cu_num_draft", "draft_token_ids", "target_logits", "draft_probs",
              "temperature", "top_k", "top_p"):
        a = batch.get(k)
        out[k] = 0 if a is None else int(a.nbytes)
    return out
