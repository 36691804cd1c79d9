// Exact top-k / top-p on bf16 rows from a histogram of values.
//
// A bf16 logit takes one of 65536 values, so the tempered, filtered
// distribution of a row (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나":
// temperature, top-k and top-p applied before the judgement) is fixed by how
// many tokens hold each value. While the row streams, every element adds 1
// to the counter of its value: per sign, one 32-bit counter per bf16
// magnitude in [2^-16, 2^8) (3072 values), one for all smaller magnitudes
// (whose exact weights 2^(l c), c = log2(e) / T, are summed beside it) and
// one for 2^8 and above (+inf and -inf included). The counters of a bf16
// word's two values come from a few packed 16-bit operations (magnitude
// clamp, sign offset) and one unpredicated shared-memory add each; the -inf
// padding of a stage that the row does not fill is taken out of the
// negative huge counter again.
//
// At the row's end the consumers turn counts into masses n 2^(v c - m c)
// (m the row max): their sum is Z, no per-element exponential is needed.
// Scanning the values from the largest down gives the top-k and top-p
// thresholds, Z over the kept set and the kept set itself: exact for every
// value, one read of the row, no sort. The row goes to the exact slow path
// when a threshold falls on the tiny-value counter, when the row holds NaN,
// +inf or a value of 2^8 and above, or when huge negative values could
// weigh in Z ((m + 2^8) c < 50).
#pragma once
#include "common.cuh"
#include "pipe.cuh"

namespace sv {

constexpr unsigned kPendingSlow = 0x80000000u;  // row left to the exact slow path

// Counter layout: per sign kWinSide slots, slot d of a magnitude in bits
// being clamp(mag, kWinMagLo, kWinMagHi) - kWinMagLo: 0 for |v| < 2^-16, 1 ..
// 3072 for the single values of [2^-16, 2^8), 3073 for |v| >= 2^8. Positive
// values use slots d, negative ones kWinSide + d.
constexpr int kWinSide = 3074;
constexpr int kWinSlots = 2 * kWinSide;      // 6148
constexpr uint32_t kWinMagLo = 0x377Fu;      // the largest bf16 magnitude below 2^-16
constexpr uint32_t kWinMagHi = 0x4380u;      // 2^8
// Items: the slots in increasing value order. Items 0 .. kWinSide-1 are the
// negative side (item 0 the huge negatives, kWinSide-1 the tiny ones), then
// the positive side (tiny first, huge last).
constexpr int kWinItems = kWinSlots;
constexpr int kWinHugeNeg = 0;
constexpr int kWinTinyNeg = kWinSide - 1;
constexpr int kWinTinyPos = kWinSide;
constexpr int kWinHugePos = kWinSlots - 1;

static_assert(kWinSlots == SPEC_SHARD_HIST_INTS, "the sharded histogram rows hold the slots");
static_assert(kWinSlots % 4 == 0, "the counters are cleared with 16-byte stores");

struct WinHist {
  unsigned cnt[kWinSlots];  // by slot
  float tiny_w[2];          // sums of 2^(l c) of the tiny values: [0] negative, [1] positive
  unsigned pad[2];
};
static_assert(sizeof(WinHist) % 16 == 0, "cleared with 16-byte stores");

__device__ __forceinline__ int win_slot_of_item(int i) {
  return i < kWinSide ? kWinSlots - 1 - i : i - kWinSide;
}

// Count every element of 4 words of packed bf16 pairs: per word, the two
// slots from packed 16-bit operations and one shared-memory add per element
// (unpredicated: a packed compare and predicated adds cost about ten more
// instructions per word). mn2 / mx2 keep the smallest / largest magnitudes
// seen (per half), for win_tiny / win_nan.
__device__ __forceinline__ void win_count_all(WinHist* h, const uint32_t w[4], uint32_t& mn2,
                                              uint32_t& mx2) {
  // byte address of slot 0, less the clamp offset folded in
  const uint32_t base = smem_addr(h->cnt) - 4u * kWinMagLo;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t mag2 = w[t] & 0x7FFF7FFFu;
    uint32_t d2;
    asm("min.u16x2 %0, %1, %2;" : "=r"(mn2) : "r"(mn2), "r"(mag2));
    asm("max.u16x2 %0, %1, %2;" : "=r"(mx2) : "r"(mx2), "r"(mag2));
    asm("max.u16x2 %0, %1, %2;" : "=r"(d2) : "r"(mag2), "r"(0x377F377Fu));
    asm("min.u16x2 %0, %1, %2;" : "=r"(d2) : "r"(d2), "r"(0x43804380u));
    // + kWinSide per negative half (no carry: every half stays below 2^16)
    const uint32_t s2 = d2 + ((w[t] >> 15) & 0x00010001u) * (uint32_t)kWinSide;
    asm volatile("red.shared.add.u32 [%0], 1;\n\tred.shared.add.u32 [%1], 1;" ::"r"(
                     base + 4u * (s2 & 0xFFFFu)),
                 "r"(base + 4u * (s2 >> 16))
                 : "memory");
  }
}

// A NaN among a thread's counted elements (largest magnitudes mx2 above
// that of infinity) makes the positive tiny-value weight sum NaN, so the
// row's Z is NaN at its end (also after the histograms of several parts or
// ranks are summed).
__device__ __forceinline__ void win_nan(WinHist* h, uint32_t mx2) {
  if (max(mx2 & 0xFFFFu, mx2 >> 16) > 0x7F80u) atomicAdd(&h->tiny_w[1], __int_as_float(0x7FC00000));
}

// Elements of a stage holding n (bf16) elements, whole 16-byte vectors:
// the padding that win_count_all counted as -inf (negative huge counter).
__device__ __forceinline__ unsigned win_pad(int n, int stage_elems) {
  return (unsigned)(stage_elems - n);
}

// After win_count_all over a thread's words of a stage (smallest magnitudes
// mn2): the rare tiny magnitudes (below 2^-16) also add their weight
// 2^(l c) to their side's sum, on a path the warp takes only when some lane
// holds one. Huge ones need nothing here.
template <int kWords>
__device__ __forceinline__ void win_tiny(WinHist* h, const uint32_t (&w)[kWords], uint32_t mn2,
                                         float c) {
  const bool tiny = min(mn2 & 0xFFFFu, mn2 >> 16) <= kWinMagLo;
  if (__any_sync(0xFFFFFFFFu, tiny) && tiny) {
#pragma unroll
    for (int t = 0; t < 2 * kWords; ++t) {
      const uint32_t b = (t & 1) ? (w[t >> 1] >> 16) : (w[t >> 1] & 0xFFFFu);
      const float l = __uint_as_float(b << 16);
      if ((b & 0x7FFFu) <= kWinMagLo) atomicAdd(&h->tiny_w[(b >> 15) ? 0 : 1], ex2(l * c));
    }
  }
}

// Value of fine item i (not a tiny or huge one).
__device__ __forceinline__ float win_value(int i) {
  if (i < kWinSide) return __uint_as_float((0x8000u | (kWinMagLo + (uint32_t)(kWinSide - 1 - i))) << 16);
  return __uint_as_float((kWinMagLo + (uint32_t)(i - kWinSide)) << 16);
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

// suffix_exclusive, and the sum of v over all the consumer threads.
template <typename T, int kWarps>
__device__ __forceinline__ T suffix_exclusive_total(T v, T* scratch, int tid, T& total) {
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
  T above = excl, all = T(0);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const T sw = scratch[w];
    all += sw;
    if (w > warp) above += sw;
  }
  named_sync(1, kWarps * 32);
  total = all;
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
  float zall;   // sum over the whole row (NaN: a NaN in the row)
  int pending;  // 1: leave the row to the exact slow path
};

// Add this CTA's window histogram into a global one and clear it (the
// threads 0 .. nt-1 of the caller's group, tid among them).
__device__ __forceinline__ void win_flush(WinHist* h, WinHist* g, int tid, int nt) {
  for (int i = tid; i < kWinSlots; i += nt) {
    const unsigned v = h->cnt[i];
    if (v) {
      atomicAdd(&g->cnt[i], v);
      h->cnt[i] = 0u;
    }
  }
  if (tid < 2) {
    if (h->tiny_w[tid] != 0.f) atomicAdd(&g->tiny_w[tid], h->tiny_w[tid]);
    h->tiny_w[tid] = 0.f;
  }
}

// Move a global window histogram into this CTA's (which is clear) and clear
// the global one.
__device__ __forceinline__ void win_take(WinHist* h, WinHist* g, int tid, int nt) {
  for (int i = tid; i < kWinSlots; i += nt) {
    const unsigned v = __ldcg(&g->cnt[i]);
    if (v) {
      h->cnt[i] = v;
      g->cnt[i] = 0u;
    }
  }
  if (tid < 2) {
    h->tiny_w[tid] = __ldcg(&g->tiny_w[tid]);
    g->tiny_w[tid] = 0.f;
  }
}

// Row-end processing of the histogram by the kWarps consumer warps (all
// call it): m the row max, c = log2(e) / T. Thread t owns a run of
// consecutive items (each side's kWinSide items over half the threads, the
// two ends of each side one extra), and higher threads hold larger values.
// Each thread reads its items' counts once, clears them, and works from
// registers: the masses, their sum Z, the top-k item, Z_k, the top-p item and
// Z over the kept set. A huge value that can matter leaves the row to the
// slow path. Clears the histogram (the caller's next barrier orders the
// clearing before later counts).
template <int kWarps>
__device__ HistResult win_finish(WinHist* h, float m, float c, int tk, float tp, int V, int tid,
                                 float* fscr, int* iscr) {
  constexpr int kThreads = kWarps * 32;
  constexpr int kHalfT = kThreads / 2;
  constexpr int kPer = (kWinSide - 2) / kHalfT;
  constexpr int kMax = kPer + 1;  // items of a side's first and last thread
  static_assert(kPer * kHalfT + 2 == kWinSide, "each side splits evenly over half the threads");
  __shared__ int s_item;
  __shared__ float s_z;
  __shared__ int s_huge[2];  // written every row by the huge items' owners
  const int side = tid < kHalfT ? 0 : 1;
  const int u = tid - side * kHalfT;
  const int i0 = side * kWinSide + u * kPer + (u > 0 ? 1 : 0);
  const int ni = (u == 0 || u == kHalfT - 1) ? kMax : kPer;
  const float mc = m * c;
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);
  const float emc = ex2(-mc);

  // Counts and masses of this thread's items, in increasing value order.
  unsigned cn[kMax];
  float ms[kMax];
  unsigned my_cnt = 0;
  bool huge = false;
#pragma unroll
  for (int k = 0; k < kMax; ++k) {
    const int i = i0 + k;
    cn[k] = 0u;
    ms[k] = 0.f;
    if (k < ni) {
      const unsigned n = h->cnt[win_slot_of_item(i)];
      float w;
      bool whole;
      if (i == kWinHugeNeg || i == kWinHugePos) {
        // Values of magnitude 2^8 and above: +inf, NaN or a huge positive
        // value (then the row's max) send the row to the exact path; huge
        // negatives and -inf weigh less than 2^-50 of the max each once
        // (m + 2^8) c >= 50 (out of Z, which then moves by < 2^-32), and
        // need the exact path below that.
        huge |= (n != 0u) && (i == kWinHugePos || !((m + 256.f) * c >= 50.f));
        w = 0.f;
        whole = false;
      } else if (i == kWinTinyNeg || i == kWinTinyPos) {
        // magnitudes below 2^-16: the sum of their weights
        const int sd = (i == kWinTinyNeg) ? 0 : 1;
        w = h->tiny_w[sd] * emc;  // each side's sum has one reader, its owner
        h->tiny_w[sd] = 0.f;
        whole = true;
      } else {
        const float v = win_value(i);
        w = n ? (float)n * ex2(fmaf(v, c, -mc)) : 0.f;
        whole = true;
      }
      if (whole) {
        cn[k] = n;
        ms[k] = w;
        my_cnt += n;
      }
    }
  }
  // Only the first and the last thread own a huge item; the barriers below
  // publish their flags.
  if (tid == 0) s_huge[0] = huge ? 1 : 0;
  if (tid == kThreads - 1) s_huge[1] = huge ? 1 : 0;
  auto merged = [](int i) { return i == kWinTinyNeg || i == kWinTinyPos; };
  int pending = (m < INFINITY) ? 0 : 1;  // +inf in the row (NaN: through Z below)

  // top-k: the item holding the k-th largest value (counts from the top).
  int ik = -1;  // lowest item kept by top-k (-1: all)
  float zfull = 0.f, zk = 0.f;
  if (topk_on) {
    // Z over the whole row from the counts (every value was counted).
    float my_all = 0.f;
#pragma unroll
    for (int k = 0; k < kMax; ++k) my_all += ms[k];
    zfull = consumer_reduce<float, kWarps>(my_all, fscr, tid, [](float a, float b) { return a + b; });
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
    if (ik < 0 || merged(ik)) pending = 1;  // beyond the counted values, or on a merged item
  }

  // Mass of this thread's items in the top-k set (all items without top-k).
  float my_mass = 0.f;
#pragma unroll
  for (int k = 0; k < kMax; ++k)
    if (i0 + k >= ik) my_mass += ms[k];
  if (topk_on)
    zk = consumer_reduce<float, kWarps>(my_mass, fscr, tid, [](float a, float b) { return a + b; });

  // top-p: keep value v iff the mass strictly above it (in the top-k set) is
  // < top_p Z_k: the kept values run from the top down to item ip, the
  // lowest nonempty item whose mass above is below the bar. One suffix scan
  // gives each thread the mass above its items and (without top-k) Z_k;
  // the thread owning ip reads Z over the kept set off its own scan.
  int ikeep = ik;
  float z = zk;
  if (topp_on) {
    if (tid == 0) s_item = 0x7FFFFFFF;  // (ordered before the atomicMin by the scan's barrier)
    float total;
    const float above = suffix_exclusive_total<float, kWarps>(my_mass, fscr, tid, total);
    if (!topk_on) zfull = zk = total;
    const float thr = tp * zk;
    int cand = 0x7FFFFFFF;
    float zc = 0.f;  // the kept mass if cand is the boundary
    float run = above;
#pragma unroll
    for (int k = kMax - 1; k >= 0; --k) {
      const int i = i0 + k;
      if (k < ni && i >= ik) {
        const float next = run + ms[k];
        if (cn[k] && run < thr) {
          cand = i;
          zc = next;
        }
        run = next;
      }
    }
    if (cand != 0x7FFFFFFF) atomicMin(&s_item, cand);
    named_sync(1, kThreads);
    const int ip = s_item;
    if (cand == ip && ip != 0x7FFFFFFF) s_z = zc;  // one owner
    named_sync(1, kThreads);
    if (ip == 0x7FFFFFFF || merged(ip)) pending = 1;
    ikeep = ip;
    z = (ip == 0x7FFFFFFF) ? zk : s_z;
    // The next value below ip has the kept mass z above it; it is dropped
    // iff z >= thr. Unless top-k ends the set at ip, a kept mass below the
    // bar means the set would continue into values that were not counted
    // one by one.
    if (!pending && !(topk_on && ip == ik) && !(z >= thr)) pending = 1;
  }
  if (!(zfull == zfull)) pending = 1;  // NaN in the row

  if (!topk_on && !topp_on) named_sync(1, kThreads);  // (filtered rows have one of them)
  const int any_huge = s_huge[0] | s_huge[1];
  // Every count was read before the barriers above: clear the counters with
  // 16-byte stores (the tiny weights were cleared by their readers).
  {
    uint4* hz = reinterpret_cast<uint4*>(h->cnt);
    for (int i = tid; i < kWinSlots / 4; i += kThreads) hz[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  HistResult res;
  res.pending = (pending || any_huge) ? 1 : 0;
  res.theta = (!res.pending && ikeep >= 0) ? win_value(ikeep) : -INFINITY;
  res.z = z;
  res.zall = zfull;
  return res;
}

}  // namespace sv
