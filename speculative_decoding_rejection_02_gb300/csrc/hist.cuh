// Exact top-k / top-p on bf16 rows from a count histogram over bf16 values.
//
// A bf16 logit takes one of 65536 values, so the tempered, filtered
// distribution of a row (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나":
// temperature, top-k and top-p applied before the judgement) is fixed by how
// many tokens hold each value. While a row streams through the SM, every
// element adds 1 to the 16-bit counter indexed by its raw bits (one
// shared-memory atomic, two counters per 32-bit word: 128 KB for all values).
// At the row's end the consumers merge -0 into +0, turn counts into masses
// n 2^(v c - m c), scan the values from the largest down and read off the
// top-k and top-p thresholds, Z over the kept set and the kept set itself:
// no sort, no per-element exp, one read of the row, exact for every value.
// A counter can wrap only if more than 65535 tokens of one row share a
// value; the total count then differs from V and the row is left to the
// exact bisection kernel, as are rows with NaN or +inf.
#pragma once
#include "common.cuh"
#include "pipe.cuh"

namespace sv {

constexpr unsigned kPendingSlow = 0x80000000u;  // row left to the exact slow path
constexpr size_t kHist16Bytes = 65536 * 2;      // 16-bit counters for every bf16 value

// Order-preserving 16-bit key of a bf16 value and back.
__device__ __forceinline__ uint32_t bf16_key(uint32_t b) {
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t key_bf16(uint32_t k) {
  return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
}
__device__ __forceinline__ unsigned hist16_count(const uint32_t* h, uint32_t bits) {
  return (h[bits >> 1] >> ((bits & 1u) << 4)) & 0xFFFFu;
}

// Sum of v over consumer threads with a larger index (exclusive suffix sum).
// `scratch` holds one slot per consumer warp.
template <typename T, int kWarps>
__device__ __forceinline__ T suffix_exclusive(T v, T* scratch, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_down_sync(0xFFFFFFFFu, x, o);
    if (lane + o < 32) x += y;
  }
  const T excl = x - v;
  if (lane == 0) scratch[warp] = x;
  named_sync(1, kWarps * 32);
  T above = excl;
  for (int w = warp + 1; w < kWarps; ++w) above += scratch[w];
  named_sync(1, kWarps * 32);
  return above;
}

template <typename T, int kWarps, typename Op>
__device__ __forceinline__ T consumer_reduce(T v, T* scratch, int tid, Op op) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if (lane == 0) scratch[warp] = v;
  named_sync(1, kWarps * 32);
  T r = scratch[0];
  for (int w = 1; w < kWarps; ++w) r = op(r, scratch[w]);
  named_sync(1, kWarps * 32);
  return r;
}

struct HistResult {
  float theta;  // keep iff logit >= theta
  float z;      // sum over kept of 2^(l c - m c)
  int pending;  // 1: leave the row to the exact slow path
};

// Count and mass of one value (mass 0 for -inf and for NaN / +inf, which
// are reported separately).
__device__ __forceinline__ bool bf16_nonfinite(uint32_t bits) {
  return ((bits & 0x7F80u) == 0x7F80u) && bits != 0xFF80u;
}
__device__ __forceinline__ float value_mass(uint32_t bits, unsigned n, float c, float mc) {
  if (!n || bits == 0xFF80u || bf16_nonfinite(bits)) return 0.f;
  return (float)n * ex2(fmaf(__uint_as_float(bits << 16), c, -mc));
}

// Warp-level refinement inside one 128-key block (keys 128 blk + 4 lane ..
// + 3): returns, in every lane of the calling warp,
//   mode 0: the largest key whose weight summed from the top of the block,
//           plus `above`, reaches `target` (top-k: counts);
//   mode 1: the smallest nonempty key >= `from` whose weight strictly above
//           it, plus `above`, is < `target` (top-p: masses).
// `wt(key)` gives the weight of a key (0 below `from`), `nz(key)` whether it
// holds tokens.
// As warp_refine, and *below_sum receives the sum of sw(key) over the
// block's keys >= the returned key.
template <typename Wt, typename Nz, typename Sw>
__device__ __forceinline__ int warp_refine_sum(int blk, float above, float target, int mode,
                                               Wt wt, Nz nz, Sw sw, float* sum_from) {
  const int lane = threadIdx.x & 31;
  float w[4];
  bool nzv[4];
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int key = blk * 128 + 4 * lane + e;
    w[e] = wt(key);
    nzv[e] = nz(key);
    mine += w[e];
  }
  // weight of all lanes above this one (keys of higher lanes are larger)
  float x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_down_sync(0xFFFFFFFFu, x, o);
    if (lane + o < 32) x += y;
  }
  float run = above + (x - mine);  // weight strictly above this lane's keys
  int cand = mode == 0 ? -1 : 0x7FFFFFFF;
#pragma unroll
  for (int e = 3; e >= 0; --e) {
    const int key = blk * 128 + 4 * lane + e;
    if (mode == 0) {
      if (cand < 0 && run < target && run + w[e] >= target) cand = key;
    } else if (nzv[e] && run < target) {
      cand = key;
    }
    run += w[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int c2 = __shfl_xor_sync(0xFFFFFFFFu, cand, o);
    cand = mode == 0 ? max(cand, c2) : min(cand, c2);
  }
  float part = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int key = blk * 128 + 4 * lane + e;
    if (key >= cand) part += sw(key);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
  *sum_from = part;
  return cand;
}

template <typename Wt, typename Nz>
__device__ __forceinline__ int warp_refine(int blk, float above, float target, int mode, Wt wt,
                                           Nz nz) {
  float unused;
  return warp_refine_sum(blk, above, target, mode, wt, nz, wt, &unused);
}


// Row-end processing of the 16-bit value histogram by the kWarps consumer
// warps (all call it). Warp w sums the 128-key blocks w, w + kWarps, ...
// (empty blocks cost one ballot), so dense and sparse key ranges spread
// over all warps; the per-block totals then locate the top-k and top-p
// blocks, which one warp refines to the exact value. Clears the histogram.
template <int kWarps>
__device__ HistResult hist16_finish(uint32_t* h, float m, float c, int tk, float tp, int V,
                                    int tid, float* fscr, int* iscr) {
  constexpr int kBlocks = 512;  // 128 keys each
  static_assert(kWarps * 32 == kBlocks, "one block total per consumer thread");
  __shared__ unsigned blk_cnt[kBlocks];
  __shared__ float blk_mass[kBlocks];
  __shared__ int s_blk, s_key, s_from_blk;
  __shared__ float s_above, s_from;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    // -0 and +0 are one value: move the count of -0 (bits 0x8000) to +0.
    const unsigned neg0 = h[0x4000] & 0xFFFFu;
    h[0x4000] &= 0xFFFF0000u;
    h[0] += neg0;  // a carry out of +0 breaks the total below: detected
  }
  named_sync(1, kWarps * 32);
  const float mc = m * c;
  auto cnt_of = [&](int key) -> unsigned { return hist16_count(h, key_bf16((uint32_t)key)); };
  auto mass_of = [&](int key) -> float {
    const uint32_t bits = key_bf16((uint32_t)key);
    return value_mass(bits, hist16_count(h, bits), c, mc);
  };

  // Pass 1: per-block totals. A block's 128 values are 64 consecutive words;
  // lane l reads words 2l, 2l+1 (keys 4l .. 4l+3 up to the block's order).
  unsigned bad_w = 0;
  for (int blk = warp; blk < kBlocks; blk += kWarps) {
    const uint32_t b0 = key_bf16((uint32_t)blk * 128u), b1 = key_bf16((uint32_t)blk * 128u + 127u);
    const uint32_t bmin = b0 < b1 ? b0 : b1;
    const uint2 q = reinterpret_cast<const uint2*>(h + (bmin >> 1))[lane];
    const bool any = __any_sync(0xFFFFFFFFu, (q.x | q.y) != 0u);
    unsigned cn = 0;
    float ms = 0.f;
    if (any) {
      const uint32_t wd[2] = {q.x, q.y};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {
          const unsigned n = (wd[j] >> (16 * hl)) & 0xFFFFu;
          const uint32_t bits = bmin + (uint32_t)(4 * lane + 2 * j + hl);
          cn += n;
          if (bf16_nonfinite(bits)) bad_w += n;
          else ms += value_mass(bits, n, c, mc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cn += __shfl_xor_sync(0xFFFFFFFFu, cn, o);
        ms += __shfl_xor_sync(0xFFFFFFFFu, ms, o);
      }
    }
    if (lane == 0) {
      blk_cnt[blk] = cn;
      blk_mass[blk] = ms;
    }
  }
  named_sync(1, kWarps * 32);
  // From here thread t holds block t's totals.
  const unsigned cnt_t = blk_cnt[tid];
  const float mass_t = blk_mass[tid];
  const int total = consumer_reduce<int, kWarps>((int)cnt_t, iscr, tid,
                                                 [](int a, int b) { return a + b; });
  const int bad = consumer_reduce<int, kWarps>((int)bad_w, iscr, tid,
                                               [](int a, int b) { return a + b; });
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);

  // top-k: the key holding the k-th largest value (counts from the top).
  int bk = 0;
  if (topk_on) {
    if (tid == 0) s_blk = 0;
    const unsigned run = suffix_exclusive<unsigned, kWarps>(cnt_t, (unsigned*)iscr, tid);
    if (run < (unsigned)tk && run + cnt_t >= (unsigned)tk) {
      s_blk = tid;
      s_above = (float)run;
    }
    named_sync(1, kWarps * 32);
    if (warp == 0) {
      const int blk = s_blk;
      float from = 0.f;
      int key = warp_refine_sum(
          blk, s_above, (float)tk, 0, [&](int k) { return (float)cnt_of(k); },
          [&](int k) { return cnt_of(k) != 0u; }, [&](int k) { return mass_of(k); }, &from);
      if (lane == 0) {
        s_key = key < 0 ? blk * 128 : key;
        s_from = from;
        s_from_blk = blk;
      }
    }
    named_sync(1, kWarps * 32);
    bk = s_key;
  }
  // This block's mass over keys >= key0; the block holding key0 takes the
  // partial sum its refinement produced.
  auto mass_from = [&](int key0, float from) -> float {
    const int k0 = tid * 128;
    if (k0 >= key0) return mass_t;
    if (k0 + 127 < key0) return 0.f;
    return from;
  };
  const float part_k = topk_on ? mass_from(bk, s_from) : mass_t;
  const float zk = consumer_reduce<float, kWarps>(part_k, fscr, tid,
                                                  [](float a, float b) { return a + b; });

  // top-p: keep value v iff the mass strictly above it (within the top-k set)
  // is < top_p * Z_k; the kept values are the top ones down to bp.
  int bp = bk;
  if (topp_on) {
    const float thr = tp * zk;
    const float run = suffix_exclusive<float, kWarps>(part_k, fscr, tid);
    // The lowest block whose mass above is below thr holds the crossing
    // (every lower block has mass above >= thr and is dropped whole).
    if (tid == 0) s_blk = 0x7FFFFFFF;
    named_sync(1, kWarps * 32);
    if (part_k > 0.f && run < thr) atomicMin(&s_blk, tid);
    named_sync(1, kWarps * 32);
    const int blk = s_blk == 0x7FFFFFFF ? 0 : s_blk;
    if (tid == blk) s_above = run;
    named_sync(1, kWarps * 32);
    if (warp == 0) {
      float from = 0.f;
      const int key = warp_refine_sum(
          blk, s_above, thr, 1, [&](int k) { return k >= bk ? mass_of(k) : 0.f; },
          [&](int k) { return k >= bk && cnt_of(k) != 0u; },
          [&](int k) { return k >= bk ? mass_of(k) : 0.f; }, &from);
      if (lane == 0) {
        s_key = (key == 0x7FFFFFFF) ? blk * 128 + 127 : key;
        s_from = from;
      }
    }
    named_sync(1, kWarps * 32);
    bp = s_key;
  }
  float zpart;
  if (topp_on) zpart = mass_from(bp, s_from);
  else zpart = part_k;
  const float z = consumer_reduce<float, kWarps>(zpart, fscr, tid,
                                                 [](float a, float b) { return a + b; });

  // Clear the blocks that held tokens (thread t: block t's 64 words).
  if (cnt_t) {
    const uint32_t b0 = key_bf16((uint32_t)tid * 128u), b1 = key_bf16((uint32_t)tid * 128u + 127u);
    uint4* pz = reinterpret_cast<uint4*>(h + ((b0 < b1 ? b0 : b1) >> 1));
#pragma unroll
    for (int i = 0; i < 16; ++i) pz[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  named_sync(1, kWarps * 32);

  HistResult res;
  res.pending = (total != V) || (bad > 0);
  res.theta = (topk_on || topp_on) ? __uint_as_float(key_bf16((uint32_t)bp) << 16) : -INFINITY;
  res.z = z;
  return res;
}

}  // namespace sv
