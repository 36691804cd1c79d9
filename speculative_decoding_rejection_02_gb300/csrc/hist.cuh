// Exact top-k / top-p on bf16 rows from a count histogram over bf16 values.
//
// A bf16 logit takes one of at most 65536 values, so the tempered, filtered
// distribution of a row (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나":
// temperature, top-k and top-p applied before the judgement) is fixed by how
// many tokens hold each value. While a row streams through the SM, every
// element adds 1 to its value's bin (a shared-memory atomic); at the row's
// end the consumers turn counts into masses n_b 2^(v_b c - m c), scan the
// bins from the largest value down, and read off the top-k and top-p
// thresholds, Z over the kept set, and the kept set itself: no sort, no
// per-element exp, one read of the row.
//
// Bins, in increasing value: 0 = -inf; 1 .. kFine = negative values with
// 2^-4 <= |v| < 256, one per bf16 value; kNearZero = every |v| < 2^-4 (its
// mass is accumulated per element); kNearZero+1 .. 2 kFine + 1 = positive
// values with 2^-4 <= v < 256; kOutOfRange = |v| >= 256, +inf, NaN. A row
// whose thresholds fall on the near-zero bin, or that has out-of-range
// values, is left to the exact bisection kernel.
#pragma once
#include "common.cuh"
#include "pipe.cuh"

namespace sv {

constexpr int kFineExpLo = 123;                 // 2^-4
constexpr int kFineBinades = 12;                // up to 2^8
constexpr int kFine = kFineBinades * 128;       // 1536 values per sign
constexpr int kFineBase = kFineExpLo << 7;      // bits of 2^-4 without sign
constexpr int kNearZero = kFine + 1;            // 1537
constexpr int kOutOfRange = 2 * kFine + 2;      // 3074
constexpr int kHistBins = 2 * kFine + 3;        // 3075
constexpr unsigned kPendingSlow = 0x80000000u;  // row left to the exact slow path

// Table form of hist_bin, one 32-bit entry per (sign, exponent) = b >> 7:
// bin = base + mul * mantissa with mul in {-1, 0, +1} (low 16 bits: base,
// high 16 bits: mul as a signed value).
__device__ __forceinline__ uint32_t hist_table_entry(uint32_t se) {
  const int e = (int)((se & 0xFFu));
  const bool neg = (se & 0x100u) != 0;
  int base, mul;
  if (e >= kFineExpLo && e < kFineExpLo + kFineBinades) {
    const int f0 = (e - kFineExpLo) << 7;
    if (neg) { base = kFine - f0; mul = -1; }
    else { base = kNearZero + 1 + f0; mul = 1; }
  } else if (e < kFineExpLo) {
    base = kNearZero; mul = 0;
  } else {
    base = kOutOfRange; mul = 0;  // |v| >= 256, inf, NaN; -inf fixed below
  }
  return (uint32_t)(base & 0xFFFF) | ((uint32_t)(mul & 0xFFFF) << 16);
}

// Bin of a bf16 value through the table (exact for every value but -inf,
// which the caller maps to bin 0).
__device__ __forceinline__ int hist_bin_tab(const uint32_t* tab, uint32_t b) {
  const uint32_t t = tab[b >> 7];
  const int base = (int)(t & 0xFFFFu);
  const int mul = (int)(short)(t >> 16);
  return base + mul * (int)(b & 0x7Fu);
}

__device__ __forceinline__ int hist_bin(uint32_t b) {
  const int f = (int)(b & 0x7FFFu) - kFineBase;
  if ((unsigned)f < (unsigned)kFine) return (b & 0x8000u) ? (kFine - f) : (kNearZero + 1 + f);
  if (f < 0) return kNearZero;
  return (b == 0xFF80u) ? 0 : kOutOfRange;
}

// The bf16 value of a fine bin (also -inf for bin 0).
__device__ __forceinline__ float hist_value(int idx) {
  if (idx <= 0) return -INFINITY;
  uint32_t b;
  if (idx <= kFine) b = 0x8000u | (uint32_t)(kFine - idx + kFineBase);
  else b = (uint32_t)(idx - kNearZero - 1 + kFineBase);
  return __uint_as_float(b << 16);
}

constexpr int kHistPer = 7;  // bins per consumer thread (7 * 512 >= kHistBins)

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

// Row-end processing of the histogram by the kWarps consumer warps (all of
// them call it). Clears the histogram for the next row.
template <int kWarps>
__device__ HistResult hist_finish(unsigned* hist, float* nz, float m, float c, int tk, float tp,
                                  int V, int tid, float* fscr, int* iscr) {
  const float mc = m * c;
  const int b0 = tid * kHistPer;
  unsigned cnt[kHistPer];
  float mass[kHistPer];
  const float nz_mass = *nz * ex2(-mc);
#pragma unroll
  for (int i = 0; i < kHistPer; ++i) {
    const int b = b0 + i;
    const unsigned n = (b < kHistBins) ? hist[b] : 0u;
    cnt[i] = n;
    float w = 0.f;
    if (n && b > 0 && b != kOutOfRange)
      w = (b == kNearZero) ? nz_mass : (float)n * ex2(fmaf(hist_value(b), c, -mc));
    mass[i] = w;
  }
  const int oor = consumer_reduce<int, kWarps>(
      (b0 <= kOutOfRange && kOutOfRange < b0 + kHistPer) ? (int)cnt[kOutOfRange - b0] : 0,
      iscr, tid, [](int a, int b) { return a + b; });
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);

  // top-k: the bin holding the k-th largest value (counts from the top).
  int bk = 0;
  if (topk_on) {
    unsigned tc = 0;
#pragma unroll
    for (int i = 0; i < kHistPer; ++i) tc += cnt[i];
    unsigned run = suffix_exclusive<unsigned, kWarps>(tc, (unsigned*)iscr, tid);
    int cand = -1;
#pragma unroll
    for (int i = kHistPer - 1; i >= 0; --i) {
      if (run < (unsigned)tk && run + cnt[i] >= (unsigned)tk) cand = b0 + i;
      run += cnt[i];
    }
    bk = consumer_reduce<int, kWarps>(cand, iscr, tid, [](int a, int b) { return a > b ? a : b; });
    if (bk < 0) bk = 0;
  }
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < kHistPer; ++i)
    if (b0 + i >= bk) part += mass[i];
  const float zk = consumer_reduce<float, kWarps>(part, fscr, tid,
                                                  [](float a, float b) { return a + b; });

  // top-p: keep bin b iff the mass strictly above it (within the top-k set)
  // is < top_p * Z_k; the kept bins are the top ones down to bp.
  int bp = bk;
  if (topp_on) {
    const float thr = tp * zk;
    float tm = 0.f;
#pragma unroll
    for (int i = 0; i < kHistPer; ++i)
      if (b0 + i >= bk) tm += mass[i];
    float run = suffix_exclusive<float, kWarps>(tm, fscr, tid);
    int cand = 0x7FFFFFFF;
#pragma unroll
    for (int i = kHistPer - 1; i >= 0; --i) {
      const int b = b0 + i;
      if (b >= bk && cnt[i] && run < thr) cand = b;
      if (b >= bk) run += mass[i];
    }
    bp = consumer_reduce<int, kWarps>(cand, iscr, tid, [](int a, int b) { return a < b ? a : b; });
    if (bp == 0x7FFFFFFF) bp = bk;
  }
  part = 0.f;
#pragma unroll
  for (int i = 0; i < kHistPer; ++i)
    if (b0 + i >= bp) part += mass[i];
  const float z = consumer_reduce<float, kWarps>(part, fscr, tid,
                                                 [](float a, float b) { return a + b; });

  // clear for the next row
#pragma unroll
  for (int i = 0; i < kHistPer; ++i)
    if (b0 + i < kHistBins) hist[b0 + i] = 0u;
  if (tid == 0) *nz = 0.f;
  named_sync(1, kWarps * 32);

  HistResult res;
  res.pending = (oor > 0) || (topk_on && bk == kNearZero) ||
                ((topk_on || topp_on) && bp == kNearZero);
  res.theta = (topk_on || topp_on) ? hist_value(bp) : -INFINITY;
  res.z = z;
  return res;
}

}  // namespace sv
