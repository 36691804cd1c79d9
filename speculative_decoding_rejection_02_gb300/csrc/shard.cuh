// Vocab-sharded (tensor-parallel) verification: the kernels between the
// caller's all-reduces (the protocol is stated in include/spec_verify.h).
//
// The row statistics of the method (velog "vLLM 커널은 이 규칙을 어떻게
// 옮겼나": temperature, top-k and top-p before the judgement) are a max, a
// sum of 2^((l - m) c) and, for top-k / top-p, a count histogram of values:
// each rank computes them over its columns (k_rows_tma<..., SHARD>), the
// maxima combine by MAX, the sums after rescaling to the global max
// (k_shard_rescale) by SUM, the histograms by SUM. k_shard_finish then
// reads off the thresholds, Z and p(x) exactly as the one-device pass does,
// the accept scan is k_accept, and the race runs over each rank's columns
// with the global column index in its Philox counter, so the winners
// combine by MAX into the one-device race's winner (exponential race:
// argmax_j w_j / E_j over all j is the max over the ranks' maxima).
#pragma once
#include "common.cuh"
#include "hist.cuh"
#include "pipe.cuh"
#include "race.cuh"
#include "rows.cuh"

namespace sv {

constexpr int kShardFinishThreads = 512;

// Rows: z to the global max, argmax kept only where the local max is the
// global one. Positions: q(x) of the local draft tokens. One thread per row
// and per position.
__global__ void k_shard_rescale(Params P) {
  const long long R = (long long)P.N + P.B;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < R) {
    int r = 0;
    if (locate_row(P, i, r)) {
      const int cls = row_class(P, r);
      const float ml = P.rows[i].m;  // this rank's max
      const float mg = P.sh_m[i];    // the global max
      if (cls != kArgmaxOnly) {
        const float c = kLog2e / __ldg(P.temp + r);
        float z = P.sh_z[i];
        z = (ml > -INFINITY) ? z * ex2(ml * c - mg * c) : 0.f;
        P.sh_z[i] = z;
      }
      if (!(ml == mg)) P.sh_arg[i] = 0x7FFFFFFF;
    }
  }
  if (P.sh_qx && i < P.N) {
    const int x = __ldg(P.ids + i);
    const int xl = x - P.v0;
    P.sh_qx[i] = (xl >= 0 && xl < P.V) ? __ldg(P.q + i * (long long)P.V + xl) : 0.f;
  }
}

// One row per block (kShardFinishThreads threads): thresholds, Z over the
// kept set and p(x) from the combined statistics, written as the row's
// RowStats. A top-k / top-p row reloads its combined window histogram into
// shared memory and runs the one-device row end on it.
__global__ void __launch_bounds__(kShardFinishThreads)
k_shard_finish(Params P) {
  extern __shared__ __align__(16) unsigned char shard_smem[];
  __shared__ float fscr[kShardFinishThreads / 32];
  __shared__ int iscr[kShardFinishThreads / 32];
  __shared__ int s_ok, s_req, s_cls;
  const long long row = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0) {
    int r = 0;
    s_ok = locate_row(P, row, r) ? 1 : 0;
    s_req = r;
    s_cls = s_ok ? row_class(P, r) : kArgmaxOnly;
  }
  __syncthreads();
  if (!s_ok) return;
  const int r = s_req, cls = s_cls;
  const float m = P.sh_m[row];
  const float z = P.sh_z[row];
  const int a = P.sh_arg[row];
  const float lx = P.sh_lx[row];
  const int x = draft_of_row(P, row, r);
  const float c = (cls != kArgmaxOnly) ? kLog2e / __ldg(P.temp + r) : 0.f;
  const int argmax = (a == 0x7FFFFFFF) ? 0 : a;
  if (cls != kFiltered) {
    if (tid == 0) finish_row_x(P, row, cls, m, argmax, cls == kSoftmax ? z : 0.f, -INFINITY, c,
                               x, lx);
    return;
  }
  WinHist* h = reinterpret_cast<WinHist*>(shard_smem);
  const int* hin = P.sh_hist + row * (long long)SPEC_SHARD_HIST_INTS;
  for (int i = tid; i < kWinSlots; i += kShardFinishThreads) h->cnt[i] = (unsigned)hin[i];
  if (tid < 2) h->tiny_w[tid] = P.sh_hist_w[2 * row + tid];
  __syncthreads();
  const int tk = P.top_k ? __ldg(P.top_k + r) : 0;
  const float tp = P.top_p ? __ldg(P.top_p + r) : 1.f;
  const HistResult hr =
      win_finish<kShardFinishThreads / 32>(h, m, c, tk, tp, P.Vg, tid, fscr, iscr);
  if (tid != 0) return;
  // (Z of a top-k / top-p row comes from its histogram: NaN if the row held one)
  if (hr.pending && m > -INFINITY && hr.zall == hr.zall && m < INFINITY) {
    // The window cannot settle this row and no rank holds it whole.
    RowStats s;
    s.m = m;
    s.c = c;
    s.inv_z = 0.f;
    s.theta = -INFINITY;
    s.argmax = argmax;
    s.p_x = 0.f;
    s.status = SPEC_STATUS_UNSETTLED;
    s.z = 0.f;
    P.rows[row] = s;
    atomicOr(P.status, SPEC_STATUS_UNSETTLED);
    return;
  }
  // NaN or +inf anywhere in the row: a NaN Z makes finish_row_x report it.
  const float zk = (hr.zall == hr.zall && m < INFINITY) ? hr.z : __int_as_float(0x7FC00000);
  finish_row_x(P, row, cls, m, argmax, zk, hr.theta, c, x, lx);
}

// Before the second race (on p, where the combined best is 0): clear those
// requests' race bests and slice counters. One thread per request.
__global__ void k_shard_race_reset(Params P) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= P.B) return;
  if (P.sh_skip[r] == 0ull) P.race_best[r] = 0ull;
}

// The recovered / bonus token of each request from the combined winners.
// One thread per request.
__global__ void k_shard_emit(Params P, const unsigned long long* best,
                             const unsigned long long* best_p) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= P.B) return;
  const RaceDesc d = P.race[r];
  if (d.mode == kRaceNone) return;
  unsigned long long packed = best[r];
  if (packed == 0ull) {
    // Every residual weight was 0 (rounding only): the race on p.
    atomicOr(P.status, SPEC_STATUS_EMPTY_RESIDUAL);
    packed = best_p[r];
  }
  P.out_tokens[d.row] = packed ? (int)(0xFFFFFFFFu - (uint32_t)(packed & 0xFFFFFFFFull)) : 0;
}

}  // namespace sv
