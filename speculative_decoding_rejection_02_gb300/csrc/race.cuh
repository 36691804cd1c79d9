// The recovered / bonus token: exponential race over one target row per
// request (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나": argmax_j w_j / E_j with
// E_j ~ Exp(1) is a draw proportional to w, no normalising sum needed;
// "왜 하필 max(p − q, 0)인가": w = max(p - q, 0) at the first rejection;
// "기본값 greedy 드래프트에서도 분포가 지켜질까": with a one-hot draft, w is p
// with the draft token masked; "드래프트가 제안하고 타깃이 판정한다": the bonus
// token comes from p of the last row).
//
// The chosen row is cut into slices; one CTA scores one slice: 4 consecutive
// entries share one Philox4x32-10 draw, E = -ln U, score = w / E, the lowest
// index wins ties. Groups whose largest weight cannot beat the thread's best
// even with the smallest possible E skip the draw (exact pruning). Slice
// winners meet in one 64-bit atomicMax of (score bits, ~index); the last CTA
// of the request writes the token.
#pragma once
#include "common.cuh"
#include "philox.cuh"

namespace sv {

constexpr int kRaceThreads = 256;
constexpr int kRaceSlice = 8192;  // entries per CTA (multiple of 4)
// Below the smallest E = -ln(1 - 2^-24) ~ 5.96e-8 that a race uniform can give.
constexpr float kEFloor = 5.0e-8f;

// Weights of entries 4g .. 4g+3 of the race row (0 beyond V).
__device__ __forceinline__ void race_weights(const Params& P, const RaceDesc& d,
                                             const RowStats& s, long long qrow, int mode,
                                             uint32_t g, float w[4]) {
  const int V = P.V;
  const int j0 = (int)(g * 4u);
  float l[4];
  const long long at = (long long)d.row * V + j0;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(P.logits) + (uintptr_t)(at * (P.bf16 ? 2 : 4));
  if (j0 + 3 < V && P.bf16 && (addr & 7) == 0) {
    const uint2 b = __ldg((const uint2*)((const unsigned short*)P.logits + at));
    l[0] = bf16_lo(b.x); l[1] = bf16_hi(b.x); l[2] = bf16_lo(b.y); l[3] = bf16_hi(b.y);
  } else if (j0 + 3 < V && !P.bf16 && (addr & 15) == 0) {
    const float4 f = __ldg((const float4*)((const float*)P.logits + at));
    l[0] = f.x; l[1] = f.y; l[2] = f.z; l[3] = f.w;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) l[e] = (j0 + e < V) ? load_logit(P, d.row, j0 + e) : -INFINITY;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float p = (l[e] >= s.theta) ? exp2f(fmaf(l[e], s.c, -(s.m * s.c))) * s.inv_z : 0.f;
    w[e] = (j0 + e < V) ? p : 0.f;
  }
  if (mode == kRaceResidual) {
    const float* qr = P.q + qrow * V;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (j0 + e < V) w[e] = fmaxf(w[e] - __ldg(qr + j0 + e), 0.f);
  } else if (mode == kRaceMasked) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (j0 + e == d.x) w[e] = 0.f;
  }
}

// Score groups [g_begin, g_end) with this thread's stride; keeps the best.
__device__ __forceinline__ void race_scan(const Params& P, const RaceDesc& d, const RowStats& s,
                                          long long qrow, int mode, long long greq,
                                          uint32_t g_begin, uint32_t g_end, float& best,
                                          int& best_j) {
  for (uint32_t g = g_begin + threadIdx.x; g < g_end; g += blockDim.x) {
    float w[4];
    race_weights(P, d, s, qrow, mode, g, w);
    const float wmax = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
    if (!(wmax > 0.f) || wmax / kEFloor <= best) continue;
    const uint4 r = race_words(P.seed, greq, d.kstar, g);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (w[e] > 0.f) {
        const float E = -logf(race_uniform_from_word(words[e]));
        const float sc = w[e] / E;
        if (sc > best) {
          best = sc;
          best_j = (int)(g * 4u) + e;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kRaceThreads)
k_race(Params P) {
  const int r = blockIdx.x / P.race_slices;
  const int sl = blockIdx.x % P.race_slices;
  const RaceDesc d = P.race[r];
  if (d.mode == kRaceNone) return;
  const RowStats s = P.rows[d.row];
  const long long qrow = (long long)d.row - r;  // draft position index cu[r] + k*
  const long long greq = P.req_base + r;
  const uint32_t groups = (uint32_t)((P.V + 3) / 4);
  const uint32_t g0 = (uint32_t)sl * (kRaceSlice / 4);
  const uint32_t g1 = min(groups, g0 + (uint32_t)(kRaceSlice / 4));

  float best = 0.f;
  int best_j = kNoIndex;
  race_scan(P, d, s, qrow, d.mode, greq, g0, g1, best, best_j);
  block_argmax(best, best_j);

  __shared__ int s_last;
  if (threadIdx.x == 0) {
    if (best_j != kNoIndex && best > 0.f) {
      const unsigned long long packed =
          ((unsigned long long)__float_as_uint(best) << 32) | (0xFFFFFFFFu - (uint32_t)best_j);
      atomicMax(P.race_best + r, packed);
    }
    __threadfence();
    const unsigned prev = atomicAdd(P.race_counter + r, 1u);
    s_last = (prev == (unsigned)P.race_slices - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __shared__ unsigned long long s_packed;
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
    race_scan(P, d, s, qrow, kRaceP, greq, 0u, groups, b2, j2);
    block_argmax(b2, j2);
    tok = (j2 == kNoIndex) ? 0 : j2;
    if (threadIdx.x == 0) atomicOr(P.status, SPEC_STATUS_EMPTY_RESIDUAL);
  } else {
    tok = (int)(0xFFFFFFFFu - (uint32_t)(packed & 0xFFFFFFFFull));
  }
  if (threadIdx.x == 0) P.out_tokens[d.row] = tok;
}

}  // namespace sv
