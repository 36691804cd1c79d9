// Accept scan, one thread per request (velog "드래프트가 제안하고 타깃이
// 판정한다": positions are judged left to right with independent uniforms;
// x_i is accepted iff u_i <= p_i(x_i) / q_i(x_i), and the first rejection
// ends the round; "vLLM 커널은 이 규칙을 어떻게 옮겼나": the test is
// q > 0 and p / q >= u with float64 u; "기본값 greedy 드래프트에서도 분포가
// 지켜질까": no draft_probs means q(x) = 1, temperature 0 means argmax match).
//
// Writes the accepted prefix, num_accepted and -1 padding, emits the argmax
// at k* for temperature-0 requests, and leaves a race descriptor for the
// others (residual at the first rejection, or the bonus token from the last
// row).
#pragma once
#include "common.cuh"
#include "philox.cuh"

namespace sv {

__global__ void k_accept(Params P) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= P.B) return;
  RaceDesc d;
  d.mode = kRaceNone;
  d.kstar = 0;
  d.x = -1;
  d.row = 0;
  P.race_best[r] = 0ull;
  P.race_counter[r] = 0u;

  const int c0 = P.cu[r], c1 = P.cu[r + 1];
  bool bad = (c0 < 0 || c1 < c0 || c1 > P.N);
  if (r == 0 && c0 != 0) bad = true;
  if (r == P.B - 1 && c1 != P.N) bad = true;
  if (bad) {
    atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
    P.num_accepted[r] = 0;
    P.race[r] = d;
    return;
  }
  const int gamma = c1 - c0;
  const long long row0 = (long long)c0 + r;
  const bool greedy = P.greedy_call || !(P.temp[r] > 0.f);

  unsigned st = 0;
  for (int i = 0; i <= gamma; ++i) st |= P.rows[row0 + i].status;
  if (!greedy && (st & (SPEC_STATUS_NONFINITE | SPEC_STATUS_NO_FINITE))) {
    // Unusable target row: nothing is emitted for this request.
    for (int i = 0; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
    if (P.p_at_draft)
      for (int i = 0; i < gamma; ++i) P.p_at_draft[c0 + i] = 0.f;
    P.num_accepted[r] = 0;
    P.race[r] = d;
    return;
  }

  const long long greq = P.req_base + r;
  int k = gamma;
  for (int i = 0; i < gamma; ++i) {
    const int x = P.ids[c0 + i];
    const bool valid = (x >= 0 && x < P.V);
    if (!valid) st |= SPEC_STATUS_BAD_TOKEN;
    const RowStats s = P.rows[row0 + i];
    float pa;
    bool ok;
    if (greedy) {
      ok = (x == s.argmax);
      pa = ok ? 1.f : 0.f;
    } else {
      pa = s.p_x;
      if (k == gamma) {
        const float qx = P.q ? (valid ? __ldg(P.q + (long long)(c0 + i) * P.V + x) : 0.f) : 1.f;
        const double u = accept_uniform(P.seed, greq, i);
        ok = (qx > 0.f) && ((double)pa / (double)qx >= u);
      } else {
        ok = false;
      }
    }
    if (P.p_at_draft) P.p_at_draft[c0 + i] = pa;
    if (!ok && k == gamma) k = i;
  }

  for (int i = 0; i < k; ++i) P.out_tokens[row0 + i] = P.ids[c0 + i];
  for (int i = k + 1; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
  if (greedy) {
    P.out_tokens[row0 + k] = P.rows[row0 + k].argmax;
  } else {
    P.out_tokens[row0 + k] = -1;  // written by the race
    d.kstar = k;
    d.row = (int)(row0 + k);
    if (k < gamma) {
      const int x = P.ids[c0 + k];
      d.x = x;
      if (P.flags & SPEC_FLAG_NAIVE) d.mode = kRaceP;
      else if (P.q) d.mode = kRaceResidual;
      else d.mode = (x >= 0 && x < P.V) ? kRaceMasked : kRaceP;
    } else {
      d.mode = kRaceP;
    }
  }
  P.num_accepted[r] = k;
  P.race[r] = d;
  if (st & (SPEC_STATUS_BAD_TOKEN)) atomicOr(P.status, SPEC_STATUS_BAD_TOKEN);
}

}  // namespace sv
