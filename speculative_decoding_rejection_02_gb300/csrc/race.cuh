// The recovered / bonus token: exponential race over one target row per
// request (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나": argmax_j w_j / E_j with
// E_j ~ Exp(1) is a draw proportional to w, no normalising sum needed;
// "왜 하필 max(p − q, 0)인가": w = max(p - q, 0) at the first rejection;
// "기본값 greedy 드래프트에서도 분포가 지켜질까": with a one-hot draft, w is p
// with the draft token masked; "드래프트가 제안하고 타깃이 판정한다": the bonus
// token comes from p of the last row).
//
// One CTA per task (request, 8192-entry slice), numbered slice-major so that
// later slices of a request start from the best score its earlier slices
// published (and from the argmax token's score seeded by the accept scan). Four consecutive entries share one Philox4x32-10 draw;
// E = -ln U, score = w / E, the lowest index wins ties. A group whose largest
// weight w satisfies w * kInvEMin <= best (kInvEMin above 1 / the smallest E
// a race uniform can give) cannot produce a winner and skips the draw: exact
// pruning. Since w <= p and p grows with the logit, the same bound (with a
// factor-2 margin for rounding) becomes a logit threshold, so most entries
// cost one compare. Slice winners meet in one 64-bit atomicMax of (score bits,
// ~index); the last task of a request writes the token.
#pragma once
#include "common.cuh"
#include "philox.cuh"
#include "pipe.cuh"

namespace sv {

constexpr int kRaceThreads = 256;
constexpr int kRaceSlice = 8192;  // entries per task (multiple of 4 * kRaceThreads)
constexpr int kRaceGroups = 4;  // groups of 4 entries loaded together per thread
// Above 1 / E_min, E_min = -ln(1 - 2^-24) ~ 5.96e-8 the smallest E a race
// uniform can give: no entry scores more than w * kInvEMin.
constexpr float kInvEMin = 1.7e7f;

// p of one entry of a race row (0 if cut by top-k / top-p).
__device__ __forceinline__ float race_p(float l, const RowStats& s, float mc) {
  return (l >= s.theta) ? ex2(fmaf(l, s.c, -mc)) * s.inv_z : 0.f;
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

// One candidate entry j, scored exactly as the race scores it: the packed
// (score, ~j), or 0 when w_j = 0.
__device__ unsigned long long race_candidate(const Params& P, const RaceDesc& d,
                                             const RowStats& s, long long greq, int j) {
  if (j < 0 || j >= P.V || !(s.z > 0.f)) return 0ull;
  const float l = load_logit(P, d.row, j);
  const float q = (d.mode == kRaceResidual) ? __ldg(P.q + (long long)d.qrow * P.V + j) : 0.f;
  const float w = race_w(race_p(l, s, s.m * s.c), q, j, d.mode, d.x);
  if (!(w > 0.f)) return 0ull;
  const uint4 r = race_words(P.seed, greq, d.kstar, (uint32_t)j >> 2);
  const uint32_t words[4] = {r.x, r.y, r.z, r.w};
  return race_pack(race_score(w, words[j & 3]), j);
}

// A logit at or below the returned value has p * kInvEMin <= best / 2 (p
// is ex2(l c - m c) / Z), so neither its p nor its weight can reach `best`:
//   l <= (log2(best Z / (2 kInvEMin)) + m c) / c.
// The factor 2 absorbs every rounding of this bound and of p itself.
// -inf (nothing skipped) while there is no best yet, the theta cut aside.
__device__ __forceinline__ float race_logit_floor(const RowStats& s, float mc, float best) {
  float t = -INFINITY;
  if (best > 0.f && s.c > 0.f) t = (log2f(best * s.z / (2.f * kInvEMin)) + mc) / s.c;
  // entries below theta have p = 0
  return fmaxf(t, nextafterf(s.theta, -INFINITY));
}

// Groups [g0, g1) of the race row, this thread's share; loads for
// kRaceGroups groups are issued before any of them is scored.
struct RaceItem {
  uint32_t g;  // group (entries 4g .. 4g+3)
  float w[4];  // their weights
};

// `queue`: shared memory for 32 * kRaceGroups items per warp of the block.
__device__ void race_range(const Params& P, const RaceDesc& d, const RowStats& s, int mode,
                           long long greq, uint32_t g0, uint32_t g1, float& best, int& best_j,
                           RaceItem* queue) {
  const int V = P.V;
  const float mc = s.m * s.c;
  const long long lrow = (long long)d.row * V;
  const long long qoff = (long long)d.qrow * V;
  const uintptr_t la = reinterpret_cast<uintptr_t>(P.logits);
  const uintptr_t qa = reinterpret_cast<uintptr_t>(P.q);
  const bool vec = (V % 4 == 0) && ((la & 15) == 0) && (mode != kRaceResidual || (qa & 15) == 0);
  const uint32_t stride = blockDim.x;
  // Groups whose largest logit is <= lthr cannot hold a winner.
  float lthr = race_logit_floor(s, mc, best);
  // Every lane runs the same number of batches (warp-wide ballots inside).
  const uint32_t span = stride * kRaceGroups;
  const uint32_t first = g0 + (threadIdx.x & ~31u);
  for (uint32_t gw = first; gw < g1; gw += span) {
    const uint32_t gb = gw + (threadIdx.x & 31u);
    float l[kRaceGroups][4], q[kRaceGroups][4];
#pragma unroll
    for (int k = 0; k < kRaceGroups; ++k) {
      const uint32_t g = gb + (uint32_t)k * stride;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        l[k][e] = -INFINITY;
        q[k][e] = 0.f;
      }
      if (g < g1) {
        const int j0 = (int)(g * 4u);
        if (vec && j0 + 3 < V) {
          if (P.bf16) {
            const uint2 b = __ldg(reinterpret_cast<const uint2*>(
                reinterpret_cast<const unsigned short*>(P.logits) + lrow + j0));
            l[k][0] = bf16_lo(b.x);
            l[k][1] = bf16_hi(b.x);
            l[k][2] = bf16_lo(b.y);
            l[k][3] = bf16_hi(b.y);
          } else {
            const float4 f = __ldg(reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(P.logits) + lrow + j0));
            l[k][0] = f.x; l[k][1] = f.y; l[k][2] = f.z; l[k][3] = f.w;
          }
          if (mode == kRaceResidual) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(P.q + qoff + j0));
            q[k][0] = f.x; q[k][1] = f.y; q[k][2] = f.z; q[k][3] = f.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (j0 + e < V) {
              l[k][e] = load_logit(P, d.row, j0 + e);
              if (mode == kRaceResidual) q[k][e] = __ldg(P.q + qoff + j0 + e);
            }
          }
        }
      }
    }
    // Decide every group of the batch against one snapshot of the best
    // (the best only grows, so an older snapshot prunes less but never
    // wrongly). Groups that still need their Philox words are packed into
    // a per-warp queue, so that the draws run on dense lanes instead of
    // following each lane's divergent decisions.
    const float cut = best;
    const int lane = threadIdx.x & 31;
    RaceItem* qw = queue + (threadIdx.x >> 5) * (32 * kRaceGroups);
    int n_items = 0;
#pragma unroll
    for (int k = 0; k < kRaceGroups; ++k) {
      const uint32_t g = gb + (uint32_t)k * stride;
      const float lmax = fmaxf(fmaxf(l[k][0], l[k][1]), fmaxf(l[k][2], l[k][3]));
      bool need = false;
      float w[4] = {0.f, 0.f, 0.f, 0.f};
      if (g < g1 && lmax > lthr) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = (int)(g * 4u) + e;
          w[e] = (j < V) ? race_w(race_p(l[k][e], s, mc), q[k][e], j, mode, d.x) : 0.f;
        }
        const float wmax = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
        need = (wmax > 0.f) && (wmax * kInvEMin > cut);
      }
      const unsigned m = __ballot_sync(0xFFFFFFFFu, need);
      if (need) {
        RaceItem& it = qw[n_items + __popc(m & ((1u << lane) - 1u))];
        it.g = g;
        it.w[0] = w[0]; it.w[1] = w[1]; it.w[2] = w[2]; it.w[3] = w[3];
      }
      n_items += __popc(m);
    }
    __syncwarp();
    for (int t = lane; t < n_items; t += 32) {
      const RaceItem it = qw[t];
      const uint4 r = race_words(P.seed, greq, d.kstar, it.g);
      const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (it.w[e] * kInvEMin > cut) {
          const float sc = race_score(it.w[e], words[e]);
          const int j = (int)(it.g * 4u) + e;
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
    if (best != cut) lthr = race_logit_floor(s, mc, best);
  }
}

__global__ void __launch_bounds__(kRaceThreads)
k_race(Params P) {
  const unsigned n_race = *P.race_count;
  const unsigned t = blockIdx.x;
  if (t >= n_race * (unsigned)P.race_slices) return;
  const uint32_t groups = (uint32_t)((P.V + 3) / 4);
  __shared__ int s_last;
  __shared__ unsigned long long s_packed;
  __shared__ RaceItem queue[kRaceThreads * kRaceGroups];
  const int slice = (int)(t / n_race);
  const int r = P.race_list[t % n_race];
  const RaceDesc d = P.race[r];
  const RowStats s = P.rows[d.row];
  const long long greq = P.req_base + r;
  const unsigned long long lb = __ldcg(P.race_best + r);
  float best = lb ? __uint_as_float((uint32_t)(lb >> 32)) : 0.f;
  int best_j = lb ? (int)(0xFFFFFFFFu - (uint32_t)lb) : kNoIndex;
  const uint32_t g0 = (uint32_t)slice * (kRaceSlice / 4);
  const uint32_t g1 = min(groups, g0 + (uint32_t)(kRaceSlice / 4));
  if (s.z > 0.f) race_range(P, d, s, d.mode, greq, g0, g1, best, best_j, queue);
  block_argmax(best, best_j);
  if (threadIdx.x == 0) {
    if (best_j != kNoIndex && best > 0.f) atomicMax(P.race_best + r, race_pack(best, best_j));
    __threadfence();
    const unsigned prev = atomicAdd(P.race_counter + r, 1u);
    s_last = (prev == (unsigned)P.race_slices - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0) {
    __threadfence();
    s_packed = atomicAdd(P.race_best + r, 0ull);
  }
  __syncthreads();
  const unsigned long long packed = s_packed;
  int tok;
  if (packed == 0ull) {
    // Every weight was 0 (rounding only): draw from p over the whole row.
    float b2 = 0.f;
    int j2 = kNoIndex;
    if (s.z > 0.f) race_range(P, d, s, kRaceP, greq, 0u, groups, b2, j2, queue);
    block_argmax(b2, j2);
    tok = (j2 == kNoIndex) ? 0 : j2;
    if (threadIdx.x == 0) atomicOr(P.status, SPEC_STATUS_EMPTY_RESIDUAL);
  } else {
    tok = (int)(0xFFFFFFFFu - (uint32_t)(packed & 0xFFFFFFFFull));
  }
  if (threadIdx.x == 0) P.out_tokens[d.row] = tok;
}

}  // namespace sv
