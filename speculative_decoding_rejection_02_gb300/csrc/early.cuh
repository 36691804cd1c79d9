// Early-exit verification (velog "드래프트가 제안하고 타깃이 판정한다": the
// first rejection ends the round and the later positions are discarded, so
// their target rows need never be read).
//
// The row pass pulls its rows from a device work queue instead of walking
// all of them; a queue item is one part of a row (a row is split into up to
// kMaxParts parts streamed by different CTAs; the CTA that finishes a row's
// last part merges the parts' statistics and window histograms). The queue
// starts with row 0 of every request. When a CTA
// finishes a row, its consumer thread 0 judges that position at once (the
// same accept test as k_accept) and either queues the request's next row or
// ends the request: the outputs, num_accepted and, for temperature > 0, the
// race task of the token at k*. Each request has at most one row queued or
// streaming at a time, so the rows after the first rejection are never
// read. Readers take queue slots in order (one atomic ticket each) and wait,
// bounded, until the slot is filled or every request has ended.
#pragma once
#include "common.cuh"
#include "philox.cuh"
#include "pipe.cuh"
#include "race.cuh"

namespace sv {

constexpr uint32_t kQueueTryLimit = 1u << 19;  // polls of ~0.2-1 us: half a second at most
constexpr uint32_t kQueueTestTryLimit = 64;    // SPEC_CONFIG_TEST_WAIT_TIMEOUT

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Queue control words (P.queue_ctl).
enum : int { kQTaken = 0, kQFilled = 1, kQDone = 2 };

// Next item, (row << 3) | part; -1 once every request has ended (or on
// timeout, which also sets SPEC_STATUS_TIMEOUT). One thread. A reader takes
// the next slot in order (one atomic ticket) and waits until it is filled
// or every request has ended. Every slot is filled by a row part that is
// queued or streaming, or never (then every request ends), so no reader
// waits on another reader.
__device__ long long queue_pop(const Params& P) {
  unsigned* ctl = P.queue_ctl;
  const unsigned h = atomicAdd(ctl + kQTaken, 1u);
  if (h >= (unsigned)P.q_cap) return -1;
  const uint32_t limit = P.test_stall ? kQueueTestTryLimit : kQueueTryLimit;
  for (uint32_t it = 0; it < limit; ++it) {
    if (ld_acquire(&P.queue_ready[h])) return __ldcg(&P.queue[h]);
    if (ld_acquire(ctl + kQDone) >= (unsigned)P.B) return -1;
    __nanosleep(200);
  }
  atomicOr(P.status, SPEC_STATUS_TIMEOUT);
  return -1;
}

// Queue an item (one thread).
__device__ __forceinline__ void queue_push(const Params& P, long long item) {
  const unsigned t = atomicAdd(P.queue_ctl + kQFilled, 1u);
  if (t >= (unsigned)P.q_cap) {  // cannot happen: the queue holds every row part
    atomicOr(P.status, SPEC_STATUS_TIMEOUT);
    return;
  }
  P.queue[t] = item;
  st_release(&P.queue_ready[t], 1u);
}

__device__ __forceinline__ void request_done(const Params& P) {
  __threadfence();
  atomicAdd(P.queue_ctl + kQDone, 1u);
}

// Validate every request's offsets and queue the parts of its row 0 (one
// thread per request). Invalid requests end here, as in k_accept.
__global__ void k_early_init(Params P) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= P.B) return;
  const int c0 = __ldg(P.cu + r), c1 = __ldg(P.cu + r + 1);
  bool bad = (c0 < 0 || c1 < c0 || c1 > P.N);
  if (r == 0 && c0 != 0) bad = true;
  if (r == P.B - 1 && c1 != P.N) bad = true;
  if (bad) {
    RaceDesc d;
    d.mode = kRaceNone;
    d.kstar = 0;
    d.x = -1;
    d.row = 0;
    d.qrow = 0;
    atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
    P.num_accepted[r] = 0;
    P.race[r] = d;
    request_done(P);
    return;
  }
  // Test only: nothing is queued, so every reader's wait runs out.
  if (P.test_stall) return;
  for (int part = 0; part < P.parts; ++part) queue_push(P, (((long long)c0 + r) << 3) | part);
}

// Judge position `pos` of request r (rows of r start at row0 = c0 + r) once
// its row statistics are written, and queue the next row or end the
// request. Consumer thread 0 of the CTA that streamed the row.
__device__ __noinline__ void early_decide(const Params& P, int r, int pos, int gamma, int c0) {
  const long long row0 = (long long)c0 + r;
  const long long row = row0 + pos;
  const RowStats s = P.rows[row];
  const bool greedy = P.greedy_call || !(__ldg(P.temp + r) > 0.f);
  if (!greedy && (s.status & (SPEC_STATUS_NONFINITE | SPEC_STATUS_NO_FINITE))) {
    // Unusable target row: nothing is emitted for this request.
    atomicOr(P.status, s.status & (SPEC_STATUS_NONFINITE | SPEC_STATUS_NO_FINITE));
    for (int i = 0; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
    if (P.p_at_draft)
      for (int i = 0; i < gamma; ++i) P.p_at_draft[c0 + i] = 0.f;
    RaceDesc d;
    d.mode = kRaceNone;
    d.kstar = 0;
    d.x = -1;
    d.row = 0;
    d.qrow = 0;
    P.num_accepted[r] = 0;
    P.race[r] = d;
    request_done(P);
    return;
  }
  const long long greq = P.req_base + r;
  int k = gamma;
  if (pos < gamma) {
    const int x = __ldg(P.ids + c0 + pos);
    const bool valid = (x >= 0 && x < P.V);
    if (!valid) atomicOr(P.status, SPEC_STATUS_BAD_TOKEN);
    bool ok;
    float pa;
    if (greedy) {
      ok = (x == s.argmax);
      pa = ok ? 1.f : 0.f;
    } else {
      pa = s.p_x;
      const float qx =
          P.q ? (valid ? __ldg(P.q + (long long)(c0 + pos) * P.V + x) : 0.f) : 1.f;
      const double u = accept_uniform(P.seed, greq, pos);
      ok = (qx > 0.f) && ((double)pa / (double)qx >= u);
    }
    if (P.p_at_draft) P.p_at_draft[c0 + pos] = pa;
    if (ok) {
      P.out_tokens[row] = x;
      for (int part = 0; part < P.parts; ++part) queue_push(P, ((row + 1) << 3) | part);
      return;
    }
    k = pos;
  }
  // The round ends at k: the argmax, or a race task for the token at k.
  RaceDesc d;
  d.mode = kRaceNone;
  d.kstar = k;
  d.x = -1;
  d.row = (int)row;
  d.qrow = c0 + k;
  if (greedy) {
    P.out_tokens[row] = s.argmax;
  } else {
    if (k < gamma) {
      const int x = __ldg(P.ids + c0 + k);
      d.x = x;
      if (P.flags & SPEC_FLAG_NAIVE) d.mode = kRaceP;
      else if (P.q) d.mode = kRaceResidual;
      else d.mode = (x >= 0 && x < P.V) ? kRaceMasked : kRaceP;
    } else {
      d.mode = kRaceP;
    }
    const RaceView v = race_view(P, r, d.row, d.qrow, d.kstar, d.mode, d.x, s.m, s.c, s.inv_z,
                                 s.theta, s.z);
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
    P.race_best[r] = race_candidate(P, v, s.argmax);
    P.race_list[atomicAdd(P.race_count, 1u)] = task;
  }
  for (int i = k + 1; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
  if (P.p_at_draft)
    for (int i = k + 1; i < gamma; ++i) P.p_at_draft[c0 + i] = __int_as_float(0x7FC00000);
  P.num_accepted[r] = k;
  P.race[r] = d;
  request_done(P);
}

}  // namespace sv
