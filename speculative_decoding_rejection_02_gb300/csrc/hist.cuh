// Exact top-k / top-p on bf16 rows from a window histogram of values.
//
// A bf16 logit takes one of 65536 values, so the tempered, filtered
// distribution of a row (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나":
// temperature, top-k and top-p applied before the judgement) is fixed by how
// many tokens hold each value. Only values near the row maximum m can decide
// the thresholds. For top-p, the tokens below m - D with
//   D = (log2(V / (1 - top_p)) + 1) / c,   c = log2(e) / T,
// weigh less than (1 - top_p) / 2 in units of the maximum's weight, and
// Z >= 1 in those units, so the mass at or above m - D exceeds top_p Z and
// the top-p boundary lies inside the window [m - D, m]. For top-k the window
// is 30 / c wide (weights down to 2^-30 of the maximum's).
//
// While the row streams, each thread drops an element unless it lies at or
// above (its own running max) - D; every running max is at most m, so every
// element at or above m - D is counted. A counted element adds 1 to the
// counter of its value: one 32-bit counter per bf16 value of magnitude in
// [2^-16, 2^8) (24 binades x 128 values per sign, 24 KB), plus one merged
// counter per sign for the magnitudes below 2^-16, which also sums the
// weights 2^(l c) of its members. A counted value of magnitude 2^8 or more
// (or +inf) sends the row to the exact slow path.
//
// At the row's end the consumers turn counts into masses n 2^(v c - m c),
// scan the values from the largest down and read off the top-k and top-p
// thresholds, Z over the kept set and the kept set itself: exact for every
// value, one read of the row, no sort, no per-element exp beyond the row
// sum. The row goes to the slow path when a threshold falls on a merged
// counter or outside the window (top-k with fewer than k tokens in it), or
// when the row holds NaN or +inf.
#pragma once
#include "common.cuh"
#include "pipe.cuh"

namespace sv {

constexpr unsigned kPendingSlow = 0x80000000u;  // row left to the exact slow path

constexpr int kWinELo = 111;                 // biased exponent of 2^-16
constexpr int kWinBinades = 24;              // magnitudes 2^-16 .. 2^8
constexpr int kWinHalf = kWinBinades * 128;  // single-value counters per sign
constexpr int kWinFine = 2 * kWinHalf;       // 6144
// Items in increasing value order: negative values (most negative first),
// the merged negative and positive counters, positive values.
constexpr int kWinItems = kWinFine + 2;
constexpr int kWinTinyNeg = kWinHalf;
constexpr int kWinTinyPos = kWinHalf + 1;
constexpr float kWinTopKWidth = 30.f;  // top-k window, in units of 1 / c
constexpr float kWinTinyNegLow = -1.52587890625e-05f;  // -2^-16

struct WinHist {
  unsigned cnt[kWinItems];  // counter of fine item i at cnt[i] (the two merged
                            // items keep theirs below)
  unsigned tiny_cnt[2];     // merged counters: [0] negative, [1] positive
  float tiny_w[2];          // their sums of 2^(l c)
  unsigned out_of_range;    // set when a counted value has magnitude >= 2^8
  unsigned pad[1];
};
static_assert(sizeof(WinHist) % 16 == 0, "cleared with 16-byte stores");

// Window half-width D (logit units) of a filtered row; c > 0.
__device__ __forceinline__ float win_delta(float c, int tk, float tp, int V) {
  float d = 0.f;
  if (tp < 1.f) d = (log2f((float)V / (1.f - tp)) + 1.f) / c;
  if (tk > 0 && tk < V) d = fmaxf(d, kWinTopKWidth / c);
  return d;
}

// Item (and counter) index of a bf16 value of magnitude in [2^-16, 2^8);
// `fine` tells whether the magnitude is in that range.
__device__ __forceinline__ int win_slot(uint32_t bits, bool& fine) {
  const int idx = (int)(bits & 0x7FFFu) - kWinELo * 128;
  fine = (unsigned)idx < (unsigned)kWinHalf;
  return (bits & 0x8000u) ? (kWinHalf - 1 - idx) : (kWinHalf + 2 + idx);
}

// Count an element outside the single-value range (merged counter, or the
// out-of-range flag for magnitudes >= 2^8 and +inf).
__device__ __forceinline__ void win_add_rare(WinHist* h, uint32_t bits, float l, float c) {
  const int e = (int)((bits & 0x7FFFu) >> 7);
  const uint32_t pos = ((bits >> 15) & 1u) ^ 1u;
  if (e < kWinELo) {
    atomicAdd(&h->tiny_cnt[pos], 1u);
    atomicAdd(&h->tiny_w[pos], ex2(l * c));
  } else {
    h->out_of_range = 1u;
  }
}

// Shared-memory add of 1 to the counter at byte address `addr`, issued as
// one predicated instruction (no branch around it).
__device__ __forceinline__ void red_add1_if(uint32_t addr, bool on) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "@p red.shared.add.u32 [%0], 1;\n\t}" ::"r"(addr),
      "r"((uint32_t)on)
      : "memory");
}

// Count the elements of 4 words of packed bf16 pairs that lie at or above
// the floor `flo` (-inf never does). The common case is one predicated
// shared-memory add per element; the rare out-of-range ones are redone by
// the warp's lanes that hold any.
__device__ __forceinline__ void win_count(WinHist* h, const uint32_t w[4], float flo, float c) {
  const uint32_t base = smem_addr(h->cnt);
  bool rare = false;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t b0 = w[t] & 0xFFFFu, b1 = w[t] >> 16;
    const float l0 = __uint_as_float(w[t] << 16), l1 = __uint_as_float(w[t] & 0xFFFF0000u);
    bool f0, f1;
    const int k0 = win_slot(b0, f0), k1 = win_slot(b1, f1);
    const bool c0 = l0 >= flo, c1 = l1 >= flo;
    red_add1_if(base + 4u * (uint32_t)k0, c0 && f0);
    red_add1_if(base + 4u * (uint32_t)k1, c1 && f1);
    rare |= (c0 && !f0) || (c1 && !f1);
  }
  if (__any_sync(0xFFFFFFFFu, rare) && rare) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t b0 = w[t] & 0xFFFFu, b1 = w[t] >> 16;
      const float l0 = __uint_as_float(w[t] << 16), l1 = __uint_as_float(w[t] & 0xFFFF0000u);
      bool f0, f1;
      win_slot(b0, f0);
      win_slot(b1, f1);
      if (l0 >= flo && !f0) win_add_rare(h, b0, l0, c);
      if (l1 >= flo && !f1) win_add_rare(h, b1, l1, c);
    }
  }
}

// Value of fine item i (not a merged one).
__device__ __forceinline__ float win_value(int i) {
  if (i < kWinHalf) {
    const uint32_t a = (uint32_t)(kWinHalf - 1 - i) + kWinELo * 128u;
    return __uint_as_float((0x8000u | a) << 16);
  }
  const uint32_t a = (uint32_t)(i - kWinHalf - 2) + kWinELo * 128u;
  return __uint_as_float(a << 16);
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

// Add this CTA's window histogram into a global one and clear it (the
// threads 0 .. nt-1 of the caller's group, tid among them).
__device__ __forceinline__ void win_flush(WinHist* h, WinHist* g, int tid, int nt) {
  for (int i = tid; i < kWinItems; i += nt) {
    const unsigned v = h->cnt[i];
    if (v) {
      atomicAdd(&g->cnt[i], v);
      h->cnt[i] = 0u;
    }
  }
  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      if (h->tiny_cnt[k]) {
        atomicAdd(&g->tiny_cnt[k], h->tiny_cnt[k]);
        atomicAdd(&g->tiny_w[k], h->tiny_w[k]);
      }
      h->tiny_cnt[k] = 0u;
      h->tiny_w[k] = 0.f;
    }
    if (h->out_of_range) atomicOr(&g->out_of_range, 1u);
    h->out_of_range = 0u;
  }
}

// Move a global window histogram into this CTA's (which is clear) and clear
// the global one.
__device__ __forceinline__ void win_take(WinHist* h, WinHist* g, int tid, int nt) {
  for (int i = tid; i < kWinItems; i += nt) {
    const unsigned v = __ldcg(&g->cnt[i]);
    if (v) {
      h->cnt[i] = v;
      g->cnt[i] = 0u;
    }
  }
  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      h->tiny_cnt[k] = __ldcg(&g->tiny_cnt[k]);
      h->tiny_w[k] = __ldcg(&g->tiny_w[k]);
      g->tiny_cnt[k] = 0u;
      g->tiny_w[k] = 0.f;
    }
    h->out_of_range = __ldcg(&g->out_of_range);
    g->out_of_range = 0u;
  }
}

// Row-end processing of the window histogram by the kWarps consumer warps
// (all call it): m the row max, c = log2(e) / T, zfull the sum of
// 2^(l c - m c) over the whole row, lo = m - D the window floor. Thread t
// owns a run of consecutive items (kWinFine / threads fine ones; the merged
// two go to the threads on either side of the sign change), and higher
// threads hold larger values. Each thread reads its items' counts once,
// clears them, and works from registers; items not wholly inside the window
// (values below lo, not all counted) read as empty, so a threshold never
// lands on them. Clears the histogram.
template <int kWarps>
__device__ HistResult win_finish(WinHist* h, float m, float c, float zfull, float lo, int tk,
                                 float tp, int V, int tid, float* fscr, int* iscr) {
  constexpr int kThreads = kWarps * 32;
  constexpr int kPer = kWinFine / kThreads;
  constexpr int kHalfT = kThreads / 2;
  constexpr int kMax = kPer + 1;  // items of the two threads at the sign change
  static_assert(kPer * kThreads == kWinFine, "fine items split evenly over the threads");
  static_assert(kPer * kHalfT == kWinHalf, "the sign change falls between two threads");
  __shared__ int s_item;
  const int i0 = tid < kHalfT ? tid * kPer : tid * kPer + 2 - (tid == kHalfT ? 1 : 0);
  const int ni = (tid == kHalfT - 1 || tid == kHalfT) ? kMax : kPer;
  const float mc = m * c;
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);
  const float emc = ex2(-mc);

  // Counts and masses of this thread's items, in increasing value order.
  unsigned cn[kMax];
  float ms[kMax];
  unsigned my_cnt = 0;
#pragma unroll
  for (int k = 0; k < kMax; ++k) {
    const int i = i0 + k;
    cn[k] = 0u;
    ms[k] = 0.f;
    if (k < ni) {
      unsigned n;
      float w;
      bool whole;
      if (i == kWinTinyNeg || i == kWinTinyPos) {
        const int s = i - kWinTinyNeg;
        n = h->tiny_cnt[s];
        w = h->tiny_w[s] * emc;
        h->tiny_cnt[s] = 0u;
        h->tiny_w[s] = 0.f;
        whole = (s == 0) ? (lo <= kWinTinyNegLow) : (lo <= 0.f);
      } else {
        n = h->cnt[i];
        h->cnt[i] = 0u;
        const float v = win_value(i);
        w = n ? (float)n * ex2(fmaf(v, c, -mc)) : 0.f;
        whole = v >= lo;
      }
      if (whole) {
        cn[k] = n;
        ms[k] = w;
        my_cnt += n;
      }
    }
  }
  auto merged = [](int i) { return i == kWinTinyNeg || i == kWinTinyPos; };
  int pending = (zfull == zfull && m < INFINITY) ? 0 : 1;  // NaN or +inf in the row

  // top-k: the item holding the k-th largest value (counts from the top).
  int ik = -1;  // lowest item kept by top-k (-1: all)
  if (topk_on) {
    if (tid == 0) s_item = -1;
    const unsigned above = suffix_exclusive<unsigned, kWarps>(my_cnt, (unsigned*)iscr, tid);
    if (above < (unsigned)tk && above + my_cnt >= (unsigned)tk) {
      unsigned run = above;
      int found = -1;
#pragma unroll
      for (int k = kMax - 1; k >= 0; --k) {
        if (k < ni && found < 0) {
          run += cn[k];
          if (run >= (unsigned)tk) found = i0 + k;
        }
      }
      s_item = found;
    }
    named_sync(1, kThreads);
    ik = s_item;
    if (ik < 0 || merged(ik)) pending = 1;  // outside the window, or on a merged item
  }

  // Mass of this thread's items in the top-k set.
  float my_mass = 0.f;
#pragma unroll
  for (int k = 0; k < kMax; ++k)
    if (i0 + k >= ik) my_mass += ms[k];
  float zk = zfull;
  if (topk_on)
    zk = consumer_reduce<float, kWarps>(my_mass, fscr, tid, [](float a, float b) { return a + b; });

  // top-p: keep value v iff the mass strictly above it (in the top-k set) is
  // < top_p Z_k: the kept values run from the top down to item ip, the
  // lowest nonempty item whose mass above is below the bar.
  int ikeep = ik;
  float z = zk;
  if (topp_on) {
    const float thr = tp * zk;
    const float above = suffix_exclusive<float, kWarps>(my_mass, fscr, tid);
    int cand = 0x7FFFFFFF;
    float run = above;
#pragma unroll
    for (int k = kMax - 1; k >= 0; --k) {
      const int i = i0 + k;
      if (k < ni && i >= ik) {
        if (cn[k] && run < thr) cand = i;
        run += ms[k];
      }
    }
    if (tid == 0) s_item = 0x7FFFFFFF;
    named_sync(1, kThreads);
    if (cand != 0x7FFFFFFF) atomicMin(&s_item, cand);
    named_sync(1, kThreads);
    const int ip = s_item;
    if (ip == 0x7FFFFFFF || merged(ip)) pending = 1;
    ikeep = ip;
    float zpart = 0.f;
#pragma unroll
    for (int k = 0; k < kMax; ++k)
      if (i0 + k >= ip) zpart += ms[k];
    z = consumer_reduce<float, kWarps>(zpart, fscr, tid, [](float a, float b) { return a + b; });
    // The next value below ip has the kept mass z above it; it is dropped
    // (wherever it lies, inside the window or not) iff z >= thr. Unless
    // top-k ends the set at ip, a kept mass below the bar means the kept set
    // might continue below the window.
    if (!pending && !(topk_on && ip == ik) && !(z >= thr)) pending = 1;
  }

  const unsigned oor = h->out_of_range;
  named_sync(1, kThreads);
  if (tid == 0) h->out_of_range = 0u;

  HistResult res;
  res.pending = (pending || oor != 0u) ? 1 : 0;
  res.theta = (!res.pending && ikeep >= 0) ? win_value(ikeep) : -INFINITY;
  res.z = z;
  return res;
}

}  // namespace sv
