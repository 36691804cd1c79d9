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

// Row-end processing of the 16-bit value histogram by the kWarps consumer
// warps (all call it; 128 values per thread, thread t holding the keys
// [128 t, 128 t + 128)). Clears the histogram for the next row.
template <int kWarps>
__device__ HistResult hist16_finish(uint32_t* h, float m, float c, int tk, float tp, int V,
                                    int tid, float* fscr, int* iscr) {
  static_assert(kWarps * 32 * 128 == 65536, "128 keys per consumer thread");
  __shared__ float s_w[128];
  __shared__ unsigned s_n[128];
  __shared__ int s_blk;
  __shared__ float s_above_f;
  __shared__ unsigned s_above_u;
  __shared__ int s_key;
  if (tid == 0) {
    // -0 and +0 are one value: move the count of -0 (bits 0x8000) to +0.
    const unsigned neg0 = h[0x4000] & 0xFFFFu;
    h[0x4000] &= 0xFFFF0000u;
    h[0] += neg0;  // a carry out of +0 breaks the total below: detected
  }
  named_sync(1, kWarps * 32);
  const float mc = m * c;
  const uint32_t k0 = (uint32_t)tid * 128u;
  // This thread's 128 values occupy 64 consecutive words.
  const uint32_t blo = key_bf16(k0), bhi = key_bf16(k0 + 127u);
  const uint32_t bmin = blo < bhi ? blo : bhi;
  const uint4* hw = reinterpret_cast<const uint4*>(h + (bmin >> 1));
  unsigned cnt_t = 0, bad_t = 0;
  float mass_t = 0.f;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const uint4 q = hw[i];
    if ((q.x | q.y | q.z | q.w) == 0u) continue;
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!wd[j]) continue;
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const unsigned n = (wd[j] >> (16 * hl)) & 0xFFFFu;
        const uint32_t bits = bmin + (uint32_t)(8 * i + 2 * j + hl);
        cnt_t += n;
        if (bf16_nonfinite(bits)) bad_t += n;
        else mass_t += value_mass(bits, n, c, mc);
      }
    }
  }
  const int total = consumer_reduce<int, kWarps>((int)cnt_t, iscr, tid,
                                                 [](int a, int b) { return a + b; });
  const int bad = consumer_reduce<int, kWarps>((int)bad_t, iscr, tid,
                                               [](int a, int b) { return a + b; });
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);

  // Weight (count or mass) of key k0 + i for the block being refined.
  auto key_count = [&](int blk, int i) -> unsigned {
    return hist16_count(h, key_bf16((uint32_t)(blk * 128 + i)));
  };

  // top-k: the key holding the k-th largest value (counts from the top).
  int bk = 0;
  if (topk_on) {
    if (tid == 0) s_blk = 0;
    const unsigned run = suffix_exclusive<unsigned, kWarps>(cnt_t, (unsigned*)iscr, tid);
    if (run < (unsigned)tk && run + cnt_t >= (unsigned)tk) {
      s_blk = tid;
      s_above_u = run;
    }
    named_sync(1, kWarps * 32);
    const int blk = s_blk;
    // 128 threads refine the block: suffix counts from the top key down.
    if (tid < 128) s_n[tid] = key_count(blk, tid);
    named_sync(1, kWarps * 32);
    if (tid == 0) {
      unsigned r = s_above_u;
      int key = blk * 128;
      for (int i = 127; i >= 0; --i) {
        const unsigned n = s_n[i];
        if (r < (unsigned)tk && r + n >= (unsigned)tk) { key = blk * 128 + i; break; }
        r += n;
      }
      s_key = key;
    }
    named_sync(1, kWarps * 32);
    bk = s_key;
  }
  // This thread's mass over keys >= key0.
  auto mass_from = [&](int key0) -> float {
    if ((int)k0 >= key0) return mass_t;
    if ((int)k0 + 127 < key0) return 0.f;
    float w = 0.f;
    for (int k = key0; k <= (int)k0 + 127; ++k) {
      const uint32_t bits = key_bf16((uint32_t)k);
      w += value_mass(bits, hist16_count(h, bits), c, mc);
    }
    return w;
  };
  const float part_k = mass_from(bk);
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
    if (tid == blk) s_above_f = run;
    named_sync(1, kWarps * 32);
    if (tid < 128) {
      const int key = blk * 128 + tid;
      const uint32_t bits = key_bf16((uint32_t)key);
      const unsigned n = hist16_count(h, bits);
      s_n[tid] = (key >= bk) ? n : 0u;
      s_w[tid] = (key >= bk) ? value_mass(bits, n, c, mc) : 0.f;
    }
    named_sync(1, kWarps * 32);
    if (tid == 0) {
      float a = s_above_f;
      int key = blk * 128 + 127;
      for (int i = 127; i >= 0; --i) {
        if (s_n[i] && a < thr) key = blk * 128 + i;
        a += s_w[i];
      }
      s_key = key;
    }
    named_sync(1, kWarps * 32);
    bp = s_key;
  }
  const float z = consumer_reduce<float, kWarps>(mass_from(bp), fscr, tid,
                                                 [](float a, float b) { return a + b; });

  // clear for the next row (this thread's 64 words)
  {
    uint4* pz = reinterpret_cast<uint4*>(h + (bmin >> 1));
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
