// Accept scan, one warp per request (velog "드래프트가 제안하고 타깃이
// 판정한다": positions are judged left to right with independent uniforms;
// x_i is accepted iff u_i <= p_i(x_i) / q_i(x_i), and the first rejection
// ends the round; "vLLM 커널은 이 규칙을 어떻게 옮겼나": the test is
// q > 0 and p / q >= u with float64 u; "기본값 greedy 드래프트에서도 분포가
// 지켜질까": no draft_probs means q(x) = 1, temperature 0 means argmax match).
//
// Lane i judges position i (chunks of 32 for longer rounds); the first
// rejection is a ballot. The warp writes the accepted prefix, num_accepted,
// -1 padding and, at temperature 0, the argmax at k*. For the other requests
// it appends the request to the race list and seeds the race's running best
// with the score of the row's argmax token (a valid candidate, so a lower
// bound of the winner's score that lets the race skip most entries).
#pragma once
#include "common.cuh"
#include "philox.cuh"
#include "race.cuh"

namespace sv {

constexpr int kAcceptWarps = 8;  // requests per CTA

// A request with an unusable target row emits nothing (the whole warp).
__device__ __forceinline__ void void_request(const Params& P, int r, int c0, int gamma,
                                             long long row0, const RaceDesc& d) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i <= gamma; i += 32) P.out_tokens[row0 + i] = -1;
  if (P.p_at_draft)
    for (int i = lane; i < gamma; i += 32) P.p_at_draft[c0 + i] = 0.f;
  if (lane == 0) {
    P.num_accepted[r] = 0;
    P.race[r] = d;
  }
}

// Sampler-match acceptance (mlxcel "투기적 디코딩", section "mlxcel의 프롬프트
// 조회"): the target's sampler draws y_i from p_i at every position
// i = 0 .. gamma and x_i is accepted iff it equals y_i. Each row of the
// request becomes one race over w = p_i keyed by position i (so y_gamma is the
// bonus draw of the rejection rule); the race writes y_i to the row's output
// slot and k_match finds the first mismatch. draft_probs is not read. Called
// by the whole warp for a usable temperature > 0 request.
__device__ __forceinline__ void enqueue_match_races(const Params& P, int r, int c0, int gamma,
                                                    long long row0, unsigned st) {
  const int lane = threadIdx.x & 31;
  unsigned bad_tok = 0;
  for (int base = 0; base <= gamma; base += 32) {
    const int i = base + lane;
    const bool on = i <= gamma;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, on);
    unsigned at = 0;
    if (lane == 0) at = atomicAdd(P.race_count, (unsigned)__popc(m));
    at = __shfl_sync(0xFFFFFFFFu, at, 0);
    if (on) {
      const long long row = row0 + i;
      const RowStats s = P.rows[row];
      if (i < gamma) {
        const int x = __ldg(P.ids + c0 + i);
        bad_tok |= (x >= 0 && x < P.V) ? 0u : 1u;
        if (P.p_at_draft) P.p_at_draft[c0 + i] = s.p_x;
      }
      RaceTask task;
      task.r = r;
      task.row = (int)row;
      task.qrow = c0 + i;
      task.kstar = i;
      task.mode = kRaceP;
      task.x = -1;
      task.m = s.m;
      task.c = s.c;
      task.inv_z = s.inv_z;
      task.theta = s.theta;
      task.z = s.z;
      task.slot = (int)row;
      const RaceView v = race_view(P, r, task.row, task.qrow, i, kRaceP, -1, s.m, s.c,
                                   s.inv_z, s.theta, s.z);
      P.race_best[row] = race_candidate(P, v, s.argmax);
      P.race_list[at + (unsigned)__popc(m & ((1u << lane) - 1u))] = task;
    }
  }
  if (__reduce_or_sync(0xFFFFFFFFu, bad_tok)) st |= SPEC_STATUS_BAD_TOKEN;
  if (lane == 0) {
    RaceDesc d;
    d.mode = kRaceMatch;
    d.kstar = 0;
    d.x = -1;
    d.row = (int)row0;
    d.qrow = c0;
    P.race[r] = d;
    if (st & SPEC_STATUS_BAD_TOKEN) atomicOr(P.status, SPEC_STATUS_BAD_TOKEN);
  }
}

__global__ void __launch_bounds__(kAcceptWarps * 32)
k_accept(Params P) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAcceptWarps + (threadIdx.x >> 5);
  if (r >= P.B) return;
  RaceDesc d;
  d.mode = kRaceNone;
  d.kstar = 0;
  d.x = -1;
  d.row = 0;
  d.qrow = 0;

  const int c0 = __ldg(P.cu + r), c1 = __ldg(P.cu + r + 1);
  bool bad = (c0 < 0 || c1 < c0 || c1 > P.N);
  if (r == 0 && c0 != 0) bad = true;
  if (r == P.B - 1 && c1 != P.N) bad = true;
  if (bad) {
    if (lane == 0) {
      atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
      P.num_accepted[r] = 0;
      P.race[r] = d;
    }
    return;
  }
  const int gamma = c1 - c0;
  const long long row0 = (long long)c0 + r;
  const bool greedy = P.greedy_call || !(__ldg(P.temp + r) > 0.f);
  // Early-exit semantics on the full pass (every row was read, but only the
  // rows up to the first rejection count): unusable rows and invalid draft
  // tokens after it are ignored, p_at_draft is NaN after it.
  const bool early_sem = (P.flags & SPEC_FLAG_EARLY_EXIT) != 0;
  constexpr unsigned kUnusable =
      SPEC_STATUS_NONFINITE | SPEC_STATUS_NO_FINITE | SPEC_STATUS_UNSETTLED;

  unsigned st = 0;
  for (int i = lane; i <= gamma; i += 32) st |= P.rows[row0 + i].status;
  st = __reduce_or_sync(0xFFFFFFFFu, st);
  if (!greedy && !early_sem && (st & kUnusable)) {
    void_request(P, r, c0, gamma, row0, d);
    return;
  }

  if (!greedy && (P.flags & SPEC_FLAG_SAMPLER_MATCH)) {
    enqueue_match_races(P, r, c0, gamma, row0, st);
    return;
  }

  const long long greq = P.req_base + r;
  int k = gamma;
  unsigned bad_tok = 0;
  for (int base = 0; base < gamma; base += 32) {
    const int i = base + lane;
    bool ok = true;
    if (i < gamma) {
      const int x = __ldg(P.ids + c0 + i);
      const bool valid = (x >= 0 && x < P.Vg);
      bad_tok |= valid ? 0u : 1u;
      const RowStats s = P.rows[row0 + i];
      float pa;
      if (greedy) {
        ok = (x == s.argmax);
        pa = ok ? 1.f : 0.f;
      } else {
        pa = s.p_x;
        // q(x): gathered here, or combined across the ranks of a sharded call
        const float qx = !P.q ? 1.f
                         : P.shard ? P.sh_qx[c0 + i]
                         : (valid ? __ldg(P.q + (long long)(c0 + i) * P.V + x) : 0.f);
        if (k == gamma) {
          const double u = accept_uniform(P.seed, greq, i);
          ok = (qx > 0.f) && ((double)pa / (double)qx >= u);
        }
      }
      if (P.p_at_draft) P.p_at_draft[c0 + i] = pa;
    }
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, !ok);
    if (k == gamma && rej) k = base + __ffs(rej) - 1;
  }
  bad_tok = __reduce_or_sync(0xFFFFFFFFu, bad_tok);
  if (early_sem) {
    // An invalid draft token is always rejected, so under early exit only
    // the one at the stop can be judged.
    const int xk = (k < gamma) ? __ldg(P.ids + c0 + k) : 0;
    bad_tok = (k < gamma && !(xk >= 0 && xk < P.Vg)) ? 1u : 0u;
  }
  if (bad_tok) st |= SPEC_STATUS_BAD_TOKEN;
  if (early_sem) {
    // Only the rows up to the stop count (a rejection always comes at or
    // before an unusable row: its p(x) is 0).
    unsigned st_k = 0;
    for (int i = lane; i <= k; i += 32) st_k |= P.rows[row0 + i].status;
    st_k = __reduce_or_sync(0xFFFFFFFFu, st_k);
    if (!greedy && (st_k & kUnusable)) {
      if (lane == 0) atomicOr(P.status, st_k & kUnusable);
      void_request(P, r, c0, gamma, row0, d);
      return;
    }
    if (P.p_at_draft)
      for (int i = k + 1 + lane; i < gamma; i += 32) P.p_at_draft[c0 + i] = __int_as_float(0x7FC00000);
  }

  for (int i = lane; i <= gamma; i += 32) {
    int t = -1;
    if (i < k) t = __ldg(P.ids + c0 + i);
    else if (i == k && greedy) t = P.rows[row0 + k].argmax;
    P.out_tokens[row0 + i] = t;
  }
  if (lane == 0) {
    P.num_accepted[r] = k;
    unsigned long long seed_best = 0ull;
    if (!greedy) {
      d.kstar = k;
      d.row = (int)(row0 + k);
      d.qrow = c0 + k;
      if (k < gamma) {
        const int x = __ldg(P.ids + c0 + k);
        d.x = x;
        if (P.flags & SPEC_FLAG_NAIVE) d.mode = kRaceP;
        else if (P.q) d.mode = kRaceResidual;
        else d.mode = (x >= 0 && x < P.Vg) ? kRaceMasked : kRaceP;
      } else {
        d.mode = kRaceP;
      }
      const RowStats s = P.rows[d.row];
      const RaceView v = race_view(P, r, d.row, d.qrow, d.kstar, d.mode, d.x, s.m, s.c,
                                   s.inv_z, s.theta, s.z);
      seed_best = race_candidate(P, v, s.argmax);
      RaceTask task;
      task.r = r;
      task.row = d.row;
      task.qrow = d.qrow;
      task.kstar = d.kstar;
      task.mode = d.mode;
      task.x = d.x;
      task.m = s.m;
      task.c = s.c;
      task.inv_z = s.inv_z;
      task.theta = s.theta;
      task.z = s.z;
      task.slot = r;
      P.race_list[atomicAdd(P.race_count, 1u)] = task;
    }
    P.race[r] = d;
    if (!greedy) {
      // Only requests with a race own slot r (under sampler-match the slots
      // are rows, and greedy requests must not touch them).
      P.race_best[r] = seed_best;
    }
    if (st & SPEC_STATUS_BAD_TOKEN) atomicOr(P.status, SPEC_STATUS_BAD_TOKEN);
  }
}

// After the races of a sampler-match batch: one warp per request finds the
// first position whose drawn token differs from the draft (the drawn tokens
// already sit in the output slots), pads the slots after it with -1 and
// writes num_accepted. Other requests were finished by k_accept.
__global__ void __launch_bounds__(kAcceptWarps * 32)
k_match(Params P) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAcceptWarps + (threadIdx.x >> 5);
  if (r >= P.B) return;
  const RaceDesc d = P.race[r];
  if (d.mode != kRaceMatch) return;
  const int c0 = d.qrow;
  const int gamma = __ldg(P.cu + r + 1) - c0;
  const long long row0 = d.row;
  int k = gamma;
  for (int base = 0; base < gamma; base += 32) {
    const int i = base + lane;
    const bool ok = (i >= gamma) || (P.out_tokens[row0 + i] == __ldg(P.ids + c0 + i));
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, !ok);
    if (rej) {
      k = base + __ffs(rej) - 1;
      break;
    }
  }
  for (int i = k + 1 + lane; i <= gamma; i += 32) P.out_tokens[row0 + i] = -1;
  if (lane == 0) P.num_accepted[r] = k;
}

}  // namespace sv
