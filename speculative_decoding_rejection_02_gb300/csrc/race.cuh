// The recovered / bonus token: exponential race over one target row per
// request (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나": argmax_j w_j / E_j with
// E_j ~ Exp(1) is a draw proportional to w, no normalising sum needed;
// "왜 하필 max(p − q, 0)인가": w = max(p - q, 0) at the first rejection;
// "기본값 greedy 드래프트에서도 분포가 지켜질까": with a one-hot draft, w is p
// with the draft token masked; "드래프트가 제안하고 타깃이 판정한다": the bonus
// token comes from p of the last row).
//
// One CTA per task (race, slice of 8192 entries with draft probabilities,
// 16384 without, fewer for small batches), numbered slice-major so that
// later slices of a race start from the best score its earlier slices
// published (and from the argmax token's score seeded by the accept scan).
// A race is one request's k* row, or, under sampler-match acceptance, every
// row of a request (mlxcel "투기적 디코딩", section "mlxcel의 프롬프트 조회":
// the target's sampler draws a token at each position).
// The CTA pulls its slice of logits and draft probabilities into shared
// memory with two bulk copies, then scores it. Four consecutive entries share
// one Philox4x32-10 draw; E = -ln U, score = w / E, the lowest index wins
// ties. A group whose largest weight w satisfies w * kInvEMin <= best
// (kInvEMin above 1 / the smallest E a race uniform can give) cannot produce
// a winner and skips the draw: exact pruning. Since w <= p and p grows with
// the logit, the same bound (with a factor-2 margin for rounding) becomes a
// logit threshold, so most entries cost one compare. Groups that still need
// their draw are packed into a per-warp queue so the draws run on dense
// lanes; after the draw, -ln U >= 1 - U bounds every score by w / (1 - U),
// so the logarithm and the division run only for entries that can still
// win. Each warp raises its race's best with one 64-bit atomicMax of
// (score bits, ~index); k_race_token, launched next, writes each race's
// token to the race row's output slot.
#pragma once
#include "common.cuh"
#include "philox.cuh"
#include "pipe.cuh"

namespace sv {

constexpr int kRaceThreads = 256;
// Entries per task (multiples of 16 * kRaceThreads): 8192 when the call
// has draft probabilities (the slice's q is staged too), else 16384.
constexpr int kRaceSlice = 8192;
constexpr int kRaceSliceNoQ = 16384;
__host__ __device__ constexpr int race_slice(bool has_q) { return has_q ? kRaceSlice : kRaceSliceNoQ; }
// Calls with too few races to fill the GPU halve the slice down to this.
constexpr int kRaceSliceMin = 1024;
constexpr int kRaceGroups = 4;    // groups of 4 entries per thread per batch
// Above 1 / E_min, E_min = -ln(1 - 2^-24) ~ 5.96e-8 the smallest E a race
// uniform can give: no entry scores more than w * kInvEMin.
constexpr float kInvEMin = 1.7e7f;
// Units of 8 consecutive entries (two Philox groups) per thread of a staged
// slice, and the shared-memory queue of 16-bit group indices that holds up
// to two per unit.
__host__ __device__ constexpr int race_units(bool has_q) { return race_slice(has_q) / 8 / kRaceThreads; }
__host__ __device__ constexpr size_t race_queue_bytes(bool has_q) {
  return (size_t)kRaceThreads * 2 * race_units(has_q) * sizeof(uint16_t);
}
// Shared memory of the staged path: the slice's logits, when the race is
// on residual weights the slice's draft probabilities (fp32), and the queue.
__host__ __device__ constexpr size_t race_smem_bytes(int logit_bytes, bool has_q) {
  return has_q ? (size_t)kRaceSlice * (logit_bytes + 4) + race_queue_bytes(true)
               : (size_t)kRaceSliceNoQ * logit_bytes + race_queue_bytes(false);
}
// The largest of the above.
constexpr size_t kRaceSmemMax = race_smem_bytes(4, true) > race_smem_bytes(4, false)
                                    ? race_smem_bytes(4, true) : race_smem_bytes(4, false);

// What the scoring needs about the race row.
struct RaceView {
  int V, row, qrow, kstar, mode, x;  // V, x: local columns (x = -1: none)
  float c, mc, inv_z, theta, z;
  long long greq;
  int v0;        // global index of local column 0 (vocab-sharded calls; else 0)
  uint32_t g0;   // v0 / 4: the Philox draw of local group g is draw g0 + g
};

__device__ __forceinline__ RaceView race_view(const Params& P, int r, int row, int qrow,
                                              int kstar, int mode, int x, float m, float c,
                                              float inv_z, float theta, float z) {
  RaceView v;
  v.V = P.V;
  v.row = row;
  v.qrow = qrow;
  v.kstar = kstar;
  v.mode = mode;
  v.x = (x >= P.v0 && x - P.v0 < P.V) ? x - P.v0 : -1;
  v.v0 = P.v0;
  v.g0 = (uint32_t)P.v0 >> 2;
  v.c = c;
  v.mc = m * c;
  v.inv_z = inv_z;
  v.theta = theta;
  v.z = z;
  v.greq = P.req_base + r;
  return v;
}

// p of one entry of a race row (0 if cut by top-k / top-p).
__device__ __forceinline__ float race_p(float l, const RaceView& v) {
  return (l >= v.theta) ? ex2(fmaf(l, v.c, -v.mc)) * v.inv_z : 0.f;
}

// The race weight of entry j given p and q.
__device__ __forceinline__ float race_w(float p, float q, int j, int mode, int x) {
  if (mode == kRaceResidual) return fmaxf(p - q, 0.f);
  if (mode == kRaceMasked) return (j == x) ? 0.f : p;
  return p;
}

__device__ __forceinline__ float race_score(float w, uint32_t word) {
  const float E = -logf(race_uniform_from_word(word));
  return w / E;
}

__device__ __forceinline__ unsigned long long race_pack(float score, int j) {
  return ((unsigned long long)__float_as_uint(score) << 32) | (0xFFFFFFFFu - (uint32_t)j);
}

// A logit at or below the returned value has p * kInvEMin <= best / 2 (p
// is ex2(l c - m c) / Z), so neither its p nor its weight can reach `best`:
//   l <= (log2(best Z / (2 kInvEMin)) + m c) / c.
// The factor 2 absorbs every rounding of this bound and of p itself.
// Entries below theta have p = 0 and are always below the returned value.
__device__ __forceinline__ float race_logit_floor(const RaceView& v, float best) {
  float t = -INFINITY;
  if (best > 0.f && v.c > 0.f) t = (log2f(best * v.z / (2.f * kInvEMin)) + v.mc) / v.c;
  return fmaxf(t, nextafterf(v.theta, -INFINITY));
}

// One candidate entry, global index jg, scored exactly as the race scores
// it: the packed (score, ~jg), or 0 when it is not a local column or w = 0.
__device__ unsigned long long race_candidate(const Params& P, const RaceView& v, int jg) {
  const int j = jg - v.v0;
  if (j < 0 || j >= P.V || !(v.z > 0.f)) return 0ull;
  const float l = load_logit(P, v.row, j);
  const float q = (v.mode == kRaceResidual) ? __ldg(P.q + (long long)v.qrow * P.V + j) : 0.f;
  const float w = race_w(race_p(l, v), q, j, v.mode, v.x);
  if (!(w > 0.f)) return 0ull;
  const uint4 r = race_words(P.seed, v.greq, v.kstar, v.g0 + ((uint32_t)j >> 2));
  const uint32_t words[4] = {r.x, r.y, r.z, r.w};
  return race_pack(race_score(w, words[j & 3]), jg);
}

// A queued group (entries 4g .. 4g+3); its weights are recomputed from the
// group's logits when the queue is worked off, so an item is 4 bytes.
struct RaceItem {
  uint32_t g;
};

// The weights of group g (0 beyond the row), computed as race_batch's
// first pass computes them: fetch(g, l, q) supplies the logits and draft
// probabilities.
template <typename Fetch>
__device__ __forceinline__ void race_group_w(const RaceView& v, int mode, uint32_t g, Fetch& fetch,
                                             float w[4]) {
  float l[4], q[4];
  fetch(g, l, q);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = (int)(g * 4u) + e;
    w[e] = (j < v.V) ? race_w(race_p(l[e], v), q[e], j, mode, v.x) : 0.f;
  }
}

// Score one batch: this thread's kRaceGroups groups (group ids gk[k], their
// logits l[k][] and draft probabilities q[k][]; ids >= g1 are absent). All
// 32 lanes of the warp call it together. `qw` is the warp's queue of
// 32 * kRaceGroups items; fetch(g, l, q) gives any group's logits and draft
// probabilities again.
template <typename Fetch>
__device__ __forceinline__ void race_batch(const Params& P, const RaceView& v, int mode,
                                           const uint32_t gk[kRaceGroups], uint32_t g1,
                                           float l[kRaceGroups][4], float q[kRaceGroups][4],
                                           float& best, int& best_j, float& lthr,
                                           RaceItem* qw, Fetch fetch) {
  // Decide every group against one snapshot of the best (the best only
  // grows, so an older snapshot prunes less but never wrongly).
  const float cut = best;
  const int lane = threadIdx.x & 31;
  int n_items = 0;
#pragma unroll
  for (int k = 0; k < kRaceGroups; ++k) {
    const uint32_t g = gk[k];
    const float lmax = fmaxf(fmaxf(l[k][0], l[k][1]), fmaxf(l[k][2], l[k][3]));
    bool need = false;
    float w[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < g1 && lmax > lthr) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = (int)(g * 4u) + e;
        w[e] = (j < v.V) ? race_w(race_p(l[k][e], v), q[k][e], j, mode, v.x) : 0.f;
      }
      const float wmax = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
      need = (wmax > 0.f) && (wmax * kInvEMin > cut);
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, need);
    if (need) qw[n_items + __popc(m & ((1u << lane) - 1u))].g = g;
    n_items += __popc(m);
  }
  __syncwarp();
  for (int t = lane; t < n_items; t += 32) {
    const uint32_t gq = qw[t].g;
    float wq[4];
    race_group_w(v, mode, gq, fetch, wq);
    const uint4 r = race_words(P.seed, v.greq, v.kstar, v.g0 + gq);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // -ln U >= 1 - U, so w / (1 - U) bounds the score from above; 1 - U
      // is exact and the factor (1 + 2e-6) covers the roundings of the
      // score and of this test. Entries that fail cannot reach `cut`.
      const float v1 = 1.f - race_uniform_from_word(words[e]);
      if (wq[e] > 0.f && wq[e] * 1.000002f > cut * v1) {
        const float sc = race_score(wq[e], words[e]);
        const int j = (int)(gq * 4u) + e;
        if (sc > best || (sc == best && j < best_j)) {
          best = sc;
          best_j = j;
        }
      }
    }
  }
  __syncwarp();
  // One best for the whole warp: the next batch prunes against it.
  warp_argmax(best, best_j);
  if (best_j == kNoIndex) best = 0.f;
  if (best != cut) lthr = race_logit_floor(v, best);
}

// Groups [g0, g1) of the race row read straight from global memory (rows
// that are not 16-byte aligned, and the rare whole-row fallback).
__device__ void race_range_global(const Params& P, const RaceView& v, int mode, uint32_t g0,
                                  uint32_t g1, float& best, int& best_j, RaceItem* queue) {
  const int V = v.V;
  const uint32_t stride = blockDim.x;
  float lthr = race_logit_floor(v, best);
  RaceItem* qw = queue + (threadIdx.x >> 5) * (32 * kRaceGroups);
  const uint32_t span = stride * kRaceGroups;
  for (uint32_t gw = g0 + (threadIdx.x & ~31u); gw < g1; gw += span) {
    const uint32_t gb = gw + (threadIdx.x & 31u);
    float l[kRaceGroups][4], q[kRaceGroups][4];
    uint32_t gk[kRaceGroups];
#pragma unroll
    for (int k = 0; k < kRaceGroups; ++k) {
      gk[k] = gb + (uint32_t)k * stride;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = (int)(gk[k] * 4u) + e;
        const bool in = gk[k] < g1 && j < V;
        l[k][e] = in ? load_logit(P, v.row, j) : -INFINITY;
        q[k][e] = (in && mode == kRaceResidual) ? __ldg(P.q + (long long)v.qrow * V + j) : 0.f;
      }
    }
    race_batch(P, v, mode, gk, g1, l, q, best, best_j, lthr, qw,
               [&](uint32_t g, float* lf, float* qf) {
#pragma unroll
                 for (int e = 0; e < 4; ++e) {
                   const int j = (int)(g * 4u) + e;
                   const bool in = j < V;
                   lf[e] = in ? load_logit(P, v.row, j) : -INFINITY;
                   qf[e] = (in && mode == kRaceResidual)
                               ? __ldg(P.q + (long long)v.qrow * V + j) : 0.f;
                 }
               });
  }
}

// ---------------------------------------------------------------------------
// Scoring of a slice staged in shared memory
// ---------------------------------------------------------------------------
// The slice holds n entries (n a multiple of 4), logits at `lbuf` and, for a
// race on residual weights (HAS_Q), draft probabilities at `qbuf`. Thread t
// takes the units (8 entries, two Philox groups) t, t + blockDim.x, ...:
//  1. per group, the logit floor of the best so far, then the weights and
//     the kInvEMin bound decide whether the group needs its Philox draw;
//  2. the warp packs the groups that do into its queue (one prefix sum);
//  3. the lanes take the queued groups one each, recompute the weights,
//     draw, and score only entries whose bound w / (1 - U) can reach the
//     lane's best.
// The arithmetic of p and w is race_p / race_w's (packed in pairs, the same
// IEEE operations), so scores equal those of the global-memory path. A
// masked draft token was set to -inf in the staged slice by the caller: its
// p, and so its weight, is 0.

// The 8 logits of unit u (fp32 slices: the second half of a tail unit may
// lie past n; the caller ignores it).
template <bool BF16>
__device__ __forceinline__ void race_unit_logits(const unsigned char* lbuf, int u, float l[8]) {
  if (BF16) {
    const uint4 b = reinterpret_cast<const uint4*>(lbuf)[u];
    l[0] = bf16_lo(b.x); l[1] = bf16_hi(b.x); l[2] = bf16_lo(b.y); l[3] = bf16_hi(b.y);
    l[4] = bf16_lo(b.z); l[5] = bf16_hi(b.z); l[6] = bf16_lo(b.w); l[7] = bf16_hi(b.w);
  } else {
    const float4 a = reinterpret_cast<const float4*>(lbuf)[2 * u];
    const float4 b = reinterpret_cast<const float4*>(lbuf)[2 * u + 1];
    l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
    l[4] = b.x; l[5] = b.y; l[6] = b.z; l[7] = b.w;
  }
}

// The 4 logits of group g.
template <bool BF16>
__device__ __forceinline__ void race_group_logits(const unsigned char* lbuf, int g, float l[4]) {
  if (BF16) {
    const uint2 b = reinterpret_cast<const uint2*>(lbuf)[g];
    l[0] = bf16_lo(b.x); l[1] = bf16_hi(b.x); l[2] = bf16_lo(b.y); l[3] = bf16_hi(b.y);
  } else {
    const float4 a = reinterpret_cast<const float4*>(lbuf)[g];
    l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
  }
}

// Weights of one group: p = ex2(l c - m c) / Z (0 below theta when THETA),
// and w = max(p - q, 0) when HAS_Q, else w = p.
template <bool HAS_Q, bool THETA>
__device__ __forceinline__ void race_w4(const float l[4], const float4 q, const RaceView& v,
                                        float w[4]) {
  const unsigned long long c2 = f2_pack(v.c, v.c);
  const unsigned long long nmc2 = f2_pack(-v.mc, -v.mc);
  const unsigned long long iz2 = f2_pack(v.inv_z, v.inv_z);
  const float qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    float z0, z1;
    f2_unpack(f2_fma(f2_pack(l[2 * t], l[2 * t + 1]), c2, nmc2), z0, z1);
    unsigned long long p2 = f2_mul(f2_pack(ex2(z0), ex2(z1)), iz2);
    if (HAS_Q) p2 = f2_sub(p2, f2_pack(qq[2 * t], qq[2 * t + 1]));
    f2_unpack(p2, w[2 * t], w[2 * t + 1]);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (HAS_Q) w[e] = fmaxf(w[e], 0.f);
    if (THETA) w[e] = (l[e] >= v.theta) ? w[e] : 0.f;
  }
}

__device__ __forceinline__ float max4(const float a[4]) {
  return fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
}

// The heaviest entry of the slice in this thread's units (lowest index on
// ties): the race's first bound when nothing better is known.
template <bool BF16, bool HAS_Q, bool THETA>
__device__ void race_slice_heaviest(const RaceView& v, const unsigned char* lbuf,
                                    const float* qbuf, int n, int j0, float& wb, int& jb) {
  const int units = (n + 7) >> 3;
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    float l[8], w[8];
    race_unit_logits<BF16>(lbuf, u, l);
    const float4 q0 = HAS_Q ? reinterpret_cast<const float4*>(qbuf)[2 * u] : make_float4(0, 0, 0, 0);
    const float4 q1 = HAS_Q ? reinterpret_cast<const float4*>(qbuf)[2 * u + 1] : make_float4(0, 0, 0, 0);
    race_w4<HAS_Q, THETA>(l, q0, v, w);
    race_w4<HAS_Q, THETA>(l + 4, q1, v, w + 4);
    const int ne = min(8, n - 8 * u);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < ne && w[e] > wb) {
        wb = w[e];
        jb = j0 + 8 * u + e;
      }
  }
}

template <bool BF16, bool HAS_Q, bool THETA>
__device__ void race_slice_smem(const Params& P, const RaceView& v, const unsigned char* lbuf,
                                const float* qbuf, int n, int j0, float& best, int& best_j,
                                uint16_t* queue) {
  // Units per thread: at most those of the larger slice; the queue holds
  // two groups per unit of this call's slice size.
  constexpr int kUnits = race_units(false);
  const int upt = race_units(P.q != nullptr);
  const int lane = threadIdx.x & 31;
  const int units = (n + 7) >> 3;
  const float cut = best;
  const float lthr = race_logit_floor(v, best);

  // 1. Which of this thread's groups need their draw (bit 2k + h: group h
  // of the thread's k-th unit).
  uint32_t need = 0;
#pragma unroll 2
  for (int k = 0; k < kUnits; ++k) {
    const int u = (int)threadIdx.x + k * (int)blockDim.x;
    if (u >= units) break;
    float l[8];
    race_unit_logits<BF16>(lbuf, u, l);
    const float m0 = max4(l);
    const float m1 = (8 * u + 8 <= n) ? max4(l + 4) : -INFINITY;
    const bool a0 = m0 > lthr, a1 = m1 > lthr;
    if (a0 || a1) {
      const float4 q0 = HAS_Q ? reinterpret_cast<const float4*>(qbuf)[2 * u] : make_float4(0, 0, 0, 0);
      const float4 q1 = HAS_Q ? reinterpret_cast<const float4*>(qbuf)[2 * u + 1] : make_float4(0, 0, 0, 0);
      float w[8];
      race_w4<HAS_Q, THETA>(l, q0, v, w);
      race_w4<HAS_Q, THETA>(l + 4, q1, v, w + 4);
      const float w0 = max4(w), w1 = max4(w + 4);
      if (a0 && w0 > 0.f && w0 * kInvEMin > cut) need |= 1u << (2 * k);
      if (a1 && w1 > 0.f && w1 * kInvEMin > cut) need |= 2u << (2 * k);
    }
  }

  // 2. Pack them into the warp's queue.
  const int cnt = __popc(need);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  uint16_t* qw = queue + (threadIdx.x >> 5) * (32 * 2 * upt);
  int at = incl - cnt;
  while (need) {
    const int b = __ffs(need) - 1;
    need &= need - 1u;
    const int u = (int)threadIdx.x + (b >> 1) * (int)blockDim.x;
    qw[at++] = (uint16_t)(2 * u + (b & 1));
  }
  __syncwarp();

  // 3. Draw and score the queued groups on dense lanes.
  const uint32_t gbase = v.g0 + ((uint32_t)j0 >> 2);
  for (int t = lane; t < total; t += 32) {
    const int g = qw[t];
    float l[4], w[4];
    race_group_logits<BF16>(lbuf, g, l);
    const float4 q = HAS_Q ? reinterpret_cast<const float4*>(qbuf)[g] : make_float4(0, 0, 0, 0);
    race_w4<HAS_Q, THETA>(l, q, v, w);
    const uint4 r = race_words(P.seed, v.greq, v.kstar, gbase + (uint32_t)g);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // -ln U >= 1 - U, so w / (1 - U) bounds the score; 1 - U is exact and
      // the factor (1 + 2e-6) covers the roundings of the score and of this
      // test. Entries that fail cannot reach this lane's best (nor tie it).
      const float v1 = 1.f - race_uniform_from_word(words[e]);
      if (w[e] > 0.f && w[e] * 1.000002f > best * v1) {
        const float sc = race_score(w[e], words[e]);
        const int j = j0 + 4 * g + e;
        if (sc > best || (sc == best && j < best_j)) {
          best = sc;
          best_j = j;
        }
      }
    }
  }
}

// Calls f(bf16, has_q, theta) with the three flags as compile-time
// constants (std::integral_constant-like tags).
template <bool B>
struct RaceFlag {
  static constexpr bool value = B;
};
template <typename F>
__device__ __forceinline__ void race_dispatch(bool bf16, bool has_q, bool theta, F&& f) {
  if (bf16) {
    if (has_q) {
      if (theta) f(RaceFlag<true>{}, RaceFlag<true>{}, RaceFlag<true>{});
      else f(RaceFlag<true>{}, RaceFlag<true>{}, RaceFlag<false>{});
    } else {
      if (theta) f(RaceFlag<true>{}, RaceFlag<false>{}, RaceFlag<true>{});
      else f(RaceFlag<true>{}, RaceFlag<false>{}, RaceFlag<false>{});
    }
  } else {
    if (has_q) {
      if (theta) f(RaceFlag<false>{}, RaceFlag<true>{}, RaceFlag<true>{});
      else f(RaceFlag<false>{}, RaceFlag<true>{}, RaceFlag<false>{});
    } else {
      if (theta) f(RaceFlag<false>{}, RaceFlag<false>{}, RaceFlag<true>{});
      else f(RaceFlag<false>{}, RaceFlag<false>{}, RaceFlag<false>{});
    }
  }
}

__global__ void __launch_bounds__(kRaceThreads, 4)
k_race(Params P) {
  pdl_wait();
  extern __shared__ __align__(128) unsigned char race_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_staged;
  __shared__ unsigned long long s_lb;

  const unsigned n_race = *P.race_count;
  const unsigned t = blockIdx.x;
  if (t >= n_race * (unsigned)P.race_slices) return;
  const int slice = (int)(t / n_race);
  const RaceTask task = P.race_list[t % n_race];
  const int r = task.r;
  const int slot = task.slot;
  // Second race of a sharded call: only where every residual weight was 0,
  // and on p.
  if (P.sh_skip && P.sh_skip[r] != 0ull) return;
  const RaceView v = race_view(P, r, task.row, task.qrow, task.kstar,
                               P.sh_skip ? (int)kRaceP : task.mode, task.x, task.m, task.c,
                               task.inv_z, task.theta, task.z);
  const int V = P.V;
  const uint32_t groups = (uint32_t)((V + 3) / 4);
  const int slice_n = P.race_slice_n;
  const uint32_t g0 = (uint32_t)slice * (uint32_t)(slice_n / 4);
  const uint32_t g1 = min(groups, g0 + (uint32_t)(slice_n / 4));
  const int j0 = (int)(g0 * 4u);
  const int n = min(slice_n, V - j0);
  const int esize = P.bf16 ? 2 : 4;
  const bool resid = (v.mode == kRaceResidual);
  const char* lsrc = (const char*)P.logits + ((long long)v.row * V + j0) * esize;
  const char* qsrc = resid ? (const char*)(P.q + (long long)v.qrow * V + j0) : nullptr;
  unsigned char* lbuf = race_smem;
  float* qbuf = reinterpret_cast<float*>(race_smem + (size_t)slice_n * esize);

  // Stage the slice with bulk copies when every address and size allows it.
  if (threadIdx.x == 0) {
    const uint32_t lbytes = (uint32_t)n * esize, qbytes = resid ? (uint32_t)n * 4u : 0u;
    const bool ok = ((reinterpret_cast<uintptr_t>(lsrc) & 15) == 0) && (lbytes % 16 == 0) &&
                    (!resid || (((reinterpret_cast<uintptr_t>(qsrc) & 15) == 0) &&
                                (qbytes % 16 == 0)));
    s_staged = ok ? 1 : 0;
    if (ok) {
      // Draft probabilities in host memory are staged by the threads below
      // with 16-byte plain loads; the bulk copies take device memory only.
      const bool q_bulk = resid && !P.q_host;
      mbar_init(&bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&bar, lbytes + (q_bulk ? qbytes : 0u));
      bulk_load(lbuf, lsrc, lbytes, &bar);
      if (q_bulk) bulk_load(qbuf, qsrc, qbytes, &bar);
    }
    // The best so far (seeded by the accept scan, raised by other slices
    // as they finish), read once while the copies fly: the whole block must
    // start from the same value, since it decides below whether the block
    // takes the branch with block-wide barriers.
    s_lb = __ldcg(P.race_best + slot);
  }
  __syncthreads();
  const unsigned long long lb = s_lb;
  const bool staged = s_staged != 0;
  if (staged && resid && P.q_host) {
    // n / 4 16-byte vectors (n is a multiple of 4 here); all loads of a
    // thread are issued before its stores.
    constexpr int kVec = kRaceSlice / 4 / kRaceThreads;
    const uint4* src = reinterpret_cast<const uint4*>(qsrc);
    uint4* dst = reinterpret_cast<uint4*>(qbuf);
    const int nv = n / 4;
    uint4 t4[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = (int)threadIdx.x + k * kRaceThreads;
      if (i < nv) t4[k] = ldg_stream(src + i);
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = (int)threadIdx.x + k * kRaceThreads;
      if (i < nv) dst[i] = t4[k];
    }
    __syncthreads();
  }
  if (staged) {
    // Every thread waits for the copies (bounded); all agree on the outcome.
    if (!__syncthreads_and(mbar_wait(&bar, 0) ? 1 : 0)) {
      if (threadIdx.x == 0) atomicOr(P.status, SPEC_STATUS_TIMEOUT);
      // one more bounded wait for the copies in flight, then give up
      __syncthreads_and(mbar_wait(&bar, 0) ? 1 : 0);
      return;
    }
  }

  // Packed with global indices, kept here as local ones.
  float best = lb ? __uint_as_float((uint32_t)(lb >> 32)) : 0.f;
  int best_j = lb ? (int)(0xFFFFFFFFu - (uint32_t)lb) - v.v0 : kNoIndex;
  // Behind the staged slice: the queue of the staged scoring. Unstaged
  // tasks use the slice area for the global path's queue instead.
  uint16_t* queue = reinterpret_cast<uint16_t*>(
      race_smem + (size_t)slice_n * esize + (P.q ? (size_t)slice_n * 4 : 0));
  RaceItem* gqueue = reinterpret_cast<RaceItem*>(race_smem);
  if (v.z > 0.f) {
    if (staged) {
      // A one-hot draft's token is masked by giving it logit -inf here.
      if (v.mode == kRaceMasked && v.x >= j0 && v.x < j0 + n && threadIdx.x == 0) {
        if (P.bf16) reinterpret_cast<unsigned short*>(lbuf)[v.x - j0] = 0xFF80u;
        else reinterpret_cast<float*>(lbuf)[v.x - j0] = -INFINITY;
      }
      __syncthreads();
      const bool theta = v.theta > -INFINITY;
      race_dispatch(P.bf16 != 0, resid, theta, [&](auto bf16, auto hq, auto th) {
        constexpr bool kB = decltype(bf16)::value, kQ = decltype(hq)::value,
                       kT = decltype(th)::value;
        if (best_j == kNoIndex) {
          // No bound yet (the argmax token had weight 0 and no earlier slice
          // has finished): score this slice's heaviest entry first.
          float wb = 0.f;
          int jb = kNoIndex;
          race_slice_heaviest<kB, kQ, kT>(v, lbuf, qbuf, n, j0, wb, jb);
          block_argmax(wb, jb);
          if (jb != kNoIndex && wb > 0.f) {
            const uint4 rw = race_words(P.seed, v.greq, v.kstar, v.g0 + ((uint32_t)jb >> 2));
            const uint32_t words[4] = {rw.x, rw.y, rw.z, rw.w};
            best = race_score(wb, words[jb & 3]);
            best_j = jb;
          }
        }
        race_slice_smem<kB, kQ, kT>(P, v, lbuf, qbuf, n, j0, best, best_j, queue);
      });
    } else {
      race_range_global(P, v, v.mode, g0, g1, best, best_j, gqueue);
    }
  }
  // Each warp raises the race's best itself: no block-wide barrier at the
  // end of the task.
  warp_argmax(best, best_j);
  if ((threadIdx.x & 31) == 0 && best_j != kNoIndex && best > 0.f)
    atomicMax(P.race_best + slot, race_pack(best, best_j + v.v0));
}

// The token of race i (one CTA each), from the best that every slice of
// the race has raised (the kernel runs after k_race); a race whose weights
// were all 0 (rounding only) draws from p over the whole row instead. In a
// sharded call the rank's winner is left for the caller to combine.
__global__ void __launch_bounds__(kRaceThreads)
k_race_token(Params P) {
  pdl_wait();
  __shared__ RaceItem gqueue[kRaceThreads * kRaceGroups];
  const unsigned n_race = *P.race_count;
  const unsigned i = blockIdx.x;
  if (i >= n_race) return;
  const RaceTask task = P.race_list[i];
  const int r = task.r;
  // Second race of a sharded call: only where every residual weight was 0.
  if (P.sh_skip && P.sh_skip[r] != 0ull) return;
  const unsigned long long packed = __ldcg(P.race_best + task.slot);
  if (P.shard) {
    if (threadIdx.x == 0) P.sh_best[r] = packed;
    return;
  }
  if (packed) {
    if (threadIdx.x == 0) P.out_tokens[task.row] = (int)(0xFFFFFFFFu - (uint32_t)packed);
    return;
  }
  const RaceView v = race_view(P, r, task.row, task.qrow, task.kstar, task.mode, task.x, task.m,
                               task.c, task.inv_z, task.theta, task.z);
  float b2 = 0.f;
  int j2 = kNoIndex;
  if (v.z > 0.f)
    race_range_global(P, v, kRaceP, 0u, (uint32_t)((P.V + 3) / 4), b2, j2, gqueue);
  block_argmax(b2, j2);
  if (threadIdx.x == 0) {
    P.out_tokens[v.row] = (j2 == kNoIndex) ? 0 : j2;
    atomicOr(P.status, SPEC_STATUS_EMPTY_RESIDUAL);
  }
}

}  // namespace sv
