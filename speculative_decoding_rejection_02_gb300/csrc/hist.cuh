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

// Row-end processing of the 16-bit value histogram by the kWarps consumer
// warps (all call it; 128 values per thread, thread t holding the keys
// [128 t, 128 t + 128)). Clears the histogram for the next row.
template <int kWarps>
__device__ HistResult hist16_finish(uint32_t* h, float m, float c, int tk, float tp, int V,
                                    int tid, float* fscr, int* iscr) {
  static_assert(kWarps * 32 * 128 == 65536, "128 keys per consumer thread");
  if (tid == 0) {
    // -0 and +0 are one value: move the count of -0 (bits 0x8000) to +0.
    const unsigned neg0 = h[0x4000] & 0xFFFFu;
    h[0x4000] &= 0xFFFF0000u;
    h[0] += neg0;  // a carry out of +0 breaks the total below: detected
  }
  named_sync(1, kWarps * 32);
  const float mc = m * c;
  const uint32_t k0 = (uint32_t)tid * 128u;
  // mass of one value (0 for -inf); nonfinite values flagged separately
  auto mass_of = [&](uint32_t bits, unsigned n) -> float {
    if (!n || bits == 0xFF80u) return 0.f;
    return (float)n * ex2(fmaf(__uint_as_float(bits << 16), c, -mc));
  };
  unsigned cnt_t = 0, bad_t = 0;
  float mass_t = 0.f;
  for (uint32_t k = k0; k < k0 + 128u; ++k) {
    const uint32_t bits = key_bf16(k);
    const unsigned n = hist16_count(h, bits);
    cnt_t += n;
    const bool nonfinite = ((bits & 0x7F80u) == 0x7F80u) && bits != 0xFF80u;
    if (nonfinite) bad_t += n;
    else mass_t += mass_of(bits, n);
  }
  const int total = consumer_reduce<int, kWarps>((int)cnt_t, iscr, tid,
                                                 [](int a, int b) { return a + b; });
  const int bad = consumer_reduce<int, kWarps>((int)bad_t, iscr, tid,
                                               [](int a, int b) { return a + b; });
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);

  // top-k: the key holding the k-th largest value (counts from the top).
  int bk = 0;
  if (topk_on) {
    unsigned run = suffix_exclusive<unsigned, kWarps>(cnt_t, (unsigned*)iscr, tid);
    int cand = -1;
    if (run < (unsigned)tk && run + cnt_t >= (unsigned)tk) {
      for (int k = (int)k0 + 127; k >= (int)k0; --k) {
        const unsigned n = hist16_count(h, key_bf16((uint32_t)k));
        if (run < (unsigned)tk && run + n >= (unsigned)tk) cand = k;
        run += n;
      }
    }
    bk = consumer_reduce<int, kWarps>(cand, iscr, tid, [](int a, int b) { return a > b ? a : b; });
    if (bk < 0) bk = 0;
  }
  // mass of this thread's keys >= key0 (walking only when the range is cut)
  auto mass_from = [&](int key0) -> float {
    if ((int)k0 >= key0) return mass_t;
    if ((int)k0 + 127 < key0) return 0.f;
    float w = 0.f;
    for (int k = key0; k <= (int)k0 + 127; ++k) {
      const uint32_t bits = key_bf16((uint32_t)k);
      if ((bits & 0x7F80u) == 0x7F80u && bits != 0xFF80u) continue;
      w += mass_of(bits, hist16_count(h, bits));
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
    float run = suffix_exclusive<float, kWarps>(part_k, fscr, tid);
    int cand = 0x7FFFFFFF;
    if (part_k > 0.f && run < thr) {
      for (int k = (int)k0 + 127; k >= (int)k0 && k >= bk; --k) {
        const uint32_t bits = key_bf16((uint32_t)k);
        const unsigned n = hist16_count(h, bits);
        if (n && run < thr) cand = k;
        if (!((bits & 0x7F80u) == 0x7F80u && bits != 0xFF80u)) run += mass_of(bits, n);
      }
    }
    bp = consumer_reduce<int, kWarps>(cand, iscr, tid, [](int a, int b) { return a < b ? a : b; });
    if (bp == 0x7FFFFFFF) bp = bk;
  }
  const float z = consumer_reduce<float, kWarps>(mass_from(bp), fscr, tid,
                                                 [](float a, float b) { return a + b; });

  // clear for the next row (this thread's 64 words)
  {
    const uint32_t b_lo = key_bf16(k0), b_hi = key_bf16(k0 + 127u);
    const uint32_t w0 = (b_lo < b_hi ? b_lo : b_hi) >> 1;
    uint4* p = reinterpret_cast<uint4*>(h + w0);
#pragma unroll
    for (int i = 0; i < 16; ++i) p[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  named_sync(1, kWarps * 32);

  HistResult res;
  res.pending = (total != V) || (bad > 0);
  res.theta = (topk_on || topp_on) ? __uint_as_float(key_bf16((uint32_t)bp) << 16) : -INFINITY;
  res.z = z;
  return res;
}

}  // namespace sv
