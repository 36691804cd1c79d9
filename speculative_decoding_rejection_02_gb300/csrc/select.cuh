// Top-k / top-p rows the streaming pass does not take — fp32 logits, and bf16
// rows whose length is not a multiple of 16 bytes — (velog "vLLM 커널은 이
// 규칙을 어떻게 옮겼나": temperature, top-k and top-p applied before the
// judgement), settled from a histogram of their bf16-truncated values
// instead of searching the whole key space. For bf16 rows each bin holds one
// value, so its mass bounds meet.
//
// One CTA per row:
//  1. one pass over the row finds the max (lowest argmax), Z (online) and
//     counts every element into the window histogram of hist.cuh by the top
//     16 bits of its value: an exact count per bin, and each bin holds values
//     from a known interval, so its mass lies between count x e(low edge)
//     and count x e(high edge), e(v) = 2^(v c - m c);
//  2. suffix sums of those bounds (and of the counts) leave a short range of
//     bins that can hold the threshold: top-p keeps an element iff the mass
//     above it is below top_p Z, top-k keeps the k largest (ties kept);
//  3. a second look at the row (mostly from L2) sums the exact masses above
//     the range and copies the values inside it to shared memory;
//  4. an 8-ary search over the copied values settles the threshold.
// With top-k and top-p, top-k is settled first, then the whole top-k set is
// copied and top-p is searched over it. Rows it cannot settle this way (NaN,
// +-inf or values of 2^8 and above, more values to copy than the buffer
// holds) are settled by filtered_row_stats in the same CTA.
#pragma once
#include "common.cuh"
#include "hist.cuh"
#include "pipe.cuh"
#include "rows.cuh"

namespace sv {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCand = 16384;  // values copied for the last step, at most
constexpr int kSelItemsPerThread = (kWinItems + kSelThreads - 1) / kSelThreads;  // 13
constexpr int kSelProbes = 7;   // thresholds per search pass
constexpr size_t kSelSmemBytes = sizeof(WinHist) + kSelCand * sizeof(float);

// The fp32 pattern of a value with -0 read as +0 (they are one value: its
// bin must agree with the order of the keys, which do the same).
__device__ __forceinline__ uint32_t sel_bits(float v) {
  const uint32_t b = __float_as_uint(v);
  return b == 0x80000000u ? 0u : b;
}

// Window item of a value, from the top 16 bits of its fp32 pattern (the
// slot mapping of win_count_all, read in increasing value order).
__device__ __forceinline__ int sel_item(float v) {
  const uint32_t b = sel_bits(v);
  const uint32_t mag = (b >> 16) & 0x7FFFu;
  const uint32_t d = min(max(mag, kWinMagLo), kWinMagHi) - kWinMagLo;
  return (b >> 31) ? (kWinSide - 1 - (int)d) : (kWinSide + (int)d);
}

// The value interval [lo, hi] of item i (inclusive bounds are enough for the
// mass bounds). Tiny items span magnitudes below 2^-16, huge ones 2^8 and
// beyond.
__device__ __forceinline__ void sel_item_range(int i, float& lo, float& hi) {
  if (i == kWinHugeNeg) { lo = -INFINITY; hi = -256.f; return; }
  if (i == kWinHugePos) { lo = 256.f; hi = INFINITY; return; }
  if (i == kWinTinyNeg) { lo = -0x1p-16f; hi = 0.f; return; }
  if (i == kWinTinyPos) { lo = 0.f; hi = 0x1p-16f; return; }
  if (i > kWinSide) {
    const uint32_t mag = kWinMagLo + (uint32_t)(i - kWinSide);
    lo = __uint_as_float(mag << 16);
    hi = __uint_as_float((mag + 1u) << 16);
  } else {
    const uint32_t mag = kWinMagLo + (uint32_t)(kWinSide - 1 - i);
    lo = -__uint_as_float((mag + 1u) << 16);
    hi = -__uint_as_float(mag << 16);
  }
}

// Block-wide sums of K values (fixed order: every thread gets the same K
// results); scr holds kSelWarps x K values.
template <int K, typename T>
__device__ __forceinline__ void sel_sum_k(T (&v)[K], T* scr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) scr[warp * K + k] = v[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    T s = T(0);
    for (int w = 0; w < kSelWarps; ++w) s += scr[w * K + k];
    v[k] = s;
  }
  __syncthreads();
}

// Block-wide exclusive suffix sum over threads (threads with a larger index
// first) of K values, and their totals.
template <int K, typename T>
__device__ __forceinline__ void sel_suffix_k(T (&v)[K], T (&total)[K], T* scr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    x[k] = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_down_sync(0xFFFFFFFFu, x[k], o);
      if (lane + o < 32) x[k] += y;
    }
  }
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) scr[warp * K + k] = x[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    T above = x[k] - v[k], all = T(0);
    for (int w = 0; w < kSelWarps; ++w) {
      const T s = scr[w * K + k];
      all += s;
      if (w > warp) above += s;
    }
    v[k] = above;
    total[k] = all;
  }
  __syncthreads();
}

// Visit every element of a row, thread tid taking 16-byte chunks tid,
// tid + 512, ... with four chunks' loads issued before any is used (the
// looks at a row are bound by load latency otherwise); misaligned rows
// element by element.
template <typename F>
__device__ __forceinline__ void sel_row_each(const Params& P, long long row, F&& f) {
  const int V = P.V;
  const int esize = P.bf16 ? 2 : 4;
  const char* rowp = (const char*)P.logits + row * (long long)V * esize;
  const int tid = threadIdx.x;
  int jt = 0;
  if ((reinterpret_cast<uintptr_t>(rowp) & 15) == 0) {
    const int epc = 16 / esize;
    const int nchunk = V / epc;
    jt = nchunk * epc;
    constexpr int kAhead = 4;
    const uint4* src = (const uint4*)rowp;
    int ch = tid;
    for (; ch + (kAhead - 1) * kSelThreads < nchunk; ch += kAhead * kSelThreads) {
      uint4 w[kAhead];
#pragma unroll
      for (int u = 0; u < kAhead; ++u) w[u] = __ldg(src + ch + u * kSelThreads);
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        float e[8];
        unpack_chunk(w[u], P.bf16, e);
        for (int t = 0; t < epc; ++t) f(e[t], (ch + u * kSelThreads) * epc + t);
      }
    }
    for (; ch < nchunk; ch += kSelThreads) {
      float e[8];
      unpack_chunk(__ldg(src + ch), P.bf16, e);
      for (int t = 0; t < epc; ++t) f(e[t], ch * epc + t);
    }
  }
  for (int j = jt + tid; j < V; j += kSelThreads) f(load_logit(P, row, j), j);
}

__device__ __forceinline__ void sel_probes(long long lo, long long hi, long long t[kSelProbes]) {
  const long long span = hi - lo;
#pragma unroll
  for (int i = 0; i < kSelProbes; ++i) {
    const long long step = span * (i + 1) / (kSelProbes + 1);
    t[i] = min(lo + (step > 0 ? step : 1), hi - 1);
  }
}

// The smallest and largest key among the copied values (every thread gets
// them); s_i holds 2 x kSelWarps ints.
__device__ __forceinline__ void sel_key_range(const float* cand, int n, int* s_i, long long& kmin,
                                              long long& kmax) {
  const int tid = threadIdx.x;
  int lo32 = INT_MAX, hi32 = INT_MIN;  // keys with the top bit flipped, as ints
  for (int j = tid; j < n; j += kSelThreads) {
    const int k = (int)(float_key(cand[j]) ^ 0x80000000u);
    lo32 = min(lo32, k);
    hi32 = max(hi32, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo32 = min(lo32, __shfl_xor_sync(0xFFFFFFFFu, lo32, o));
    hi32 = max(hi32, __shfl_xor_sync(0xFFFFFFFFu, hi32, o));
  }
  const int warp = tid >> 5;
  if ((tid & 31) == 0) {
    s_i[warp * 2] = lo32;
    s_i[warp * 2 + 1] = hi32;
  }
  __syncthreads();
  lo32 = INT_MAX;
  hi32 = INT_MIN;
  for (int w = 0; w < kSelWarps; ++w) {
    lo32 = min(lo32, s_i[w * 2]);
    hi32 = max(hi32, s_i[w * 2 + 1]);
  }
  __syncthreads();
  kmin = (long long)((uint32_t)lo32 ^ 0x80000000u);
  kmax = (long long)((uint32_t)hi32 ^ 0x80000000u);
}

// Top-p among the copied values: the smallest key t with A(t) < thr, where
// A(t) = a_hi + the copied mass with key > t; the caller guarantees
// A(kmin - 1) >= thr > A(kmax).
__device__ long long sel_search_topp(const float* cand, int n, float a_hi, float thr, float c,
                                     float mc, float* s_f, int* s_i) {
  long long kmin, kmax;
  sel_key_range(cand, n, s_i, kmin, kmax);
  long long lo = kmin - 1, hi = kmax;
  while (hi - lo > 1) {
    long long t[kSelProbes];
    sel_probes(lo, hi, t);
    float a[kSelProbes];
#pragma unroll
    for (int i = 0; i < kSelProbes; ++i) a[i] = 0.f;
    for (int j = threadIdx.x; j < n; j += kSelThreads) {
      const float v = cand[j];
      const long long k = float_key(v);
      const float e = exp2f(fmaf(v, c, -mc));
#pragma unroll
      for (int i = 0; i < kSelProbes; ++i) a[i] += (k > t[i]) ? e : 0.f;
    }
    sel_sum_k(a, s_f);
    long long nlo = lo, nhi = hi;
#pragma unroll
    for (int i = 0; i < kSelProbes; ++i) {
      if (nhi != hi) continue;
      if (a_hi + a[i] < thr) nhi = t[i]; else nlo = t[i];
    }
    lo = nlo;
    hi = nhi;
  }
  return hi;
}

// Top-k among the copied values: the largest key t with count(key >= t) >=
// krem (1 <= krem <= n).
__device__ long long sel_search_topk(const float* cand, int n, int krem, int* s_i) {
  long long kmin, kmax;
  sel_key_range(cand, n, s_i, kmin, kmax);
  long long lo = kmin, hi = kmax + 1;
  while (hi - lo > 1) {
    long long t[kSelProbes];
    sel_probes(lo, hi, t);
    int cnt[kSelProbes];
#pragma unroll
    for (int i = 0; i < kSelProbes; ++i) cnt[i] = 0;
    for (int j = threadIdx.x; j < n; j += kSelThreads) {
      const long long k = float_key(cand[j]);
#pragma unroll
      for (int i = 0; i < kSelProbes; ++i) cnt[i] += (k >= t[i]);
    }
    sel_sum_k(cnt, s_i);
    long long nlo = lo, nhi = hi;
#pragma unroll
    for (int i = 0; i < kSelProbes; ++i) {
      if (nhi != hi) continue;
      if (cnt[i] >= krem) nlo = t[i]; else nhi = t[i];
    }
    lo = nlo;
    hi = nhi;
  }
  return lo;
}

// The copied mass with key >= keep, and the number of such values.
__device__ void sel_kept(const float* cand, int n, long long keep, float c, float mc, float* s_f,
                         int* s_i, float& mass, int& count) {
  float z = 0.f;
  int k = 0;
  for (int j = threadIdx.x; j < n; j += kSelThreads) {
    const float v = cand[j];
    if ((long long)float_key(v) >= keep) {
      z += exp2f(fmaf(v, c, -mc));
      ++k;
    }
  }
  float fv[1] = {z};
  sel_sum_k<1>(fv, s_f);
  int iv[1] = {k};
  sel_sum_k<1>(iv, s_i);
  mass = fv[0];
  count = iv[0];
}

// Settle filtered row `row` of request r (the whole block calls it). Returns
// false when the row needs filtered_row_stats.
__device__ bool select_row(const Params& P, long long row, int r, WinHist* hist, float* cand) {
  __shared__ float s_f[kSelWarps * kSelProbes];
  __shared__ int s_i[kSelWarps * kSelProbes];
  __shared__ int s_ncand;
  const int tid = threadIdx.x;
  const int V = P.V;
  const float c = kLog2e / __ldg(P.temp + r);
  const int tk = P.top_k ? __ldg(P.top_k + r) : 0;
  const float tp = P.top_p ? __ldg(P.top_p + r) : 1.f;
  const bool topk_on = (tk > 0 && tk < V);
  const bool topp_on = (tp < 1.f);
  if (!topk_on && !topp_on) return false;

  // ---- 1. max, lowest argmax, online Z, NaN, counts ----
  for (int i = tid; i < kWinSlots; i += kSelThreads) hist->cnt[i] = 0u;
  __syncthreads();
  float vmax = -INFINITY, vmc = 0.f, s = 0.f;
  int imax = kNoIndex, nan_seen = 0;
  sel_row_each(P, row, [&](float v, int j) {
    nan_seen |= (v != v);
    if (v > vmax || (imax == kNoIndex && v == v)) {
      const float nmc = __fmul_rn(v, c);
      if (vmax > -INFINITY) s = __fmul_rn(s, ex2(__fsub_rn(vmc, nmc)));
      vmax = v;
      vmc = nmc;
      imax = j;
    }
    if (vmax > -INFINITY) s = __fadd_rn(s, ex2(__fsub_rn(__fmul_rn(v, c), vmc)));
    const uint32_t b = sel_bits(v);
    const uint32_t mag = (b >> 16) & 0x7FFFu;
    const uint32_t d = min(max(mag, kWinMagLo), kWinMagHi) - kWinMagLo;
    atomicAdd(&hist->cnt[d + ((b >> 31) ? (uint32_t)kWinSide : 0u)], 1u);
  });
  float m = vmax;
  int am = imax;
  block_argmax(m, am);
  if (__syncthreads_or(nan_seen) || !(m > -INFINITY) || m == INFINITY) return false;
  const float mc = __fmul_rn(m, c);
  float zpart = (vmax > -INFINITY) ? __fmul_rn(s, ex2(__fsub_rn(vmc, mc))) : 0.f;
  {
    float v1[1] = {zpart};
    sel_sum_k<1>(v1, s_f);
    zpart = v1[0];
  }
  const float z1 = zpart;  // Z from the online sums (fixes the candidate range)
  if (hist->cnt[win_slot_of_item(kWinHugePos)] != 0u) return false;

  // ---- 2. the range of items that can hold the threshold ----
  // Thread t owns items [t K, t K + K), K = kSelItemsPerThread. Mass bounds
  // of item i: count x e(low edge) and count x e(high edge, at most m), with
  // a margin for ex2's rounding.
  const int i0 = tid * kSelItemsPerThread;
  // A fine item of a bf16 row holds a single value: both edges are that value.
  const bool single = P.bf16 != 0;
  auto item_bounds = [&](int i, unsigned& cnt, float& lo_m, float& hi_m) {
    cnt = (i < kWinItems) ? hist->cnt[win_slot_of_item(i)] : 0u;
    lo_m = hi_m = 0.f;
    if (cnt) {
      float lo, hi;
      sel_item_range(i, lo, hi);
      if (single && i != kWinHugeNeg && i != kWinTinyNeg && i != kWinTinyPos &&
          i != kWinHugePos) {
        if (i > kWinSide) hi = lo; else lo = hi;
      }
      const float n = (float)cnt;
      lo_m = n * ex2(fmaf(lo, c, -mc)) * 0.999999f;
      hi_m = n * ex2(fmaf(fminf(hi, m), c, -mc)) * 1.000001f;
    }
  };
  float my_l = 0.f, my_h = 0.f;
  unsigned my_c = 0u;
  for (int k = 0; k < kSelItemsPerThread; ++k) {
    unsigned cn;
    float ml, mh;
    item_bounds(i0 + k, cn, ml, mh);
    my_l += ml;
    my_h += mh;
    my_c += cn;
  }
  int lo_item = kWinItems, hi_item = -1;
  unsigned above_cnt_at = 0u;  // top-k: items above the boundary item
  {
    float fv[2] = {my_l, my_h}, ft[2];
    sel_suffix_k<2>(fv, ft, s_f);
    unsigned uv[1] = {my_c}, ut[1];
    sel_suffix_k<1>(uv, ut, reinterpret_cast<unsigned*>(s_i));
    float above_l = fv[0], above_h = fv[1];
    unsigned above_c = uv[0];
    const float thr = tp * z1;
    const float thr_lo = thr * (1.f - 1e-5f), thr_hi = thr * (1.f + 1e-5f);
    for (int k = kSelItemsPerThread - 1; k >= 0; --k) {
      const int i = i0 + k;
      if (i >= kWinItems) continue;
      unsigned cn;
      float ml, mh;
      item_bounds(i, cn, ml, mh);
      bool cand_item;
      if (topk_on) {
        cand_item = (above_c < (unsigned)tk) && (above_c + cn >= (unsigned)tk);
        if (cand_item) above_cnt_at = above_c;
      } else {
        const bool kept = (above_h + mh < thr_lo);
        const bool dropped = (above_l >= thr_hi);
        cand_item = !kept && !dropped;
      }
      if (cand_item) {
        lo_item = min(lo_item, i);
        hi_item = max(hi_item, i);
      }
      above_l += ml;
      above_h += mh;
      above_c += cn;
    }
  }
  // the range over the block, its element count, and (top-k) the count above it
  int lo_r = lo_item, hi_r = hi_item;
  {
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo_r = min(lo_r, __shfl_xor_sync(0xFFFFFFFFu, lo_r, o));
      hi_r = max(hi_r, __shfl_xor_sync(0xFFFFFFFFu, hi_r, o));
    }
    if (lane == 0) {
      s_i[warp * 2] = lo_r;
      s_i[warp * 2 + 1] = hi_r;
    }
    __syncthreads();
    lo_r = kWinItems;
    hi_r = -1;
    for (int w = 0; w < kSelWarps; ++w) {
      lo_r = min(lo_r, s_i[w * 2]);
      hi_r = max(hi_r, s_i[w * 2 + 1]);
    }
    __syncthreads();
  }
  if (hi_r < 0 || hi_r == kWinHugePos) return false;
  unsigned need = 0u, above_k = 0u;
  for (int k = 0; k < kSelItemsPerThread; ++k) {
    const int i = i0 + k;
    if (i >= lo_r && i <= hi_r && i < kWinItems) need += hist->cnt[win_slot_of_item(i)];
  }
  {
    unsigned uv[2] = {need, (lo_item <= hi_item) ? above_cnt_at : 0u};
    sel_sum_k<2>(uv, reinterpret_cast<unsigned*>(s_i));
    need = uv[0];
    above_k = uv[1];  // top-k: one thread owns the boundary item
  }
  if (need == 0u || need > (unsigned)kSelCand) return false;

  // ---- 3. exact masses above the range and Z; the range's values ----
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  float a_hi = 0.f, a_mid = 0.f;
  sel_row_each(P, row, [&](float v, int) {
    const int it = sel_item(v);
    if (it >= lo_r) {
      const float e = exp2f(fmaf(v, c, -mc));
      if (it > hi_r) {
        a_hi += e;
      } else {
        a_mid += e;
        const int at = atomicAdd(&s_ncand, 1);
        if (at < kSelCand) cand[at] = v;
      }
    }
  });
  {
    float fv[2] = {a_hi, a_mid};
    sel_sum_k<2>(fv, s_f);
    a_hi = fv[0];
    a_mid = fv[1];
  }
  const int n = s_ncand;
  if (n != (int)need) return false;

  // ---- 4. the threshold among the copied values (8-ary search on keys) ----
  long long keep;  // keep the elements whose key is >= keep
  float z_kept = 0.f;
  if (!topk_on) {
    // (Z from the first pass's online sum) the range must hold the
    // boundary: the mass above it below thr, with its own mass added at
    // least thr (else the general routine)
    const float thr = tp * z1;
    if (!(a_hi < thr) || !(a_hi + a_mid >= thr)) return false;
    keep = sel_search_topp(cand, n, a_hi, thr, c, mc, s_f, s_i);
    float mass;
    int cnt;
    sel_kept(cand, n, keep, c, mc, s_f, s_i, mass, cnt);
    z_kept = a_hi + mass;
  } else {
    const int krem = tk - (int)above_k;
    if (krem < 1 || krem > n) return false;
    keep = sel_search_topk(cand, n, krem, s_i);
    float mass;
    int cnt;
    sel_kept(cand, n, keep, c, mc, s_f, s_i, mass, cnt);
    z_kept = a_hi + mass;
    if (topp_on) {
      // Top-p over the top-k set, renormalised (Z_k = z_kept): copy the
      // whole set (the values above the boundary bin and its kept ones)
      // and search it with nothing above.
      const int nk = (int)above_k + cnt;
      if (nk > kSelCand) return false;
      __syncthreads();
      if (tid == 0) s_ncand = 0;
      __syncthreads();
      const long long kk = keep;
      sel_row_each(P, row, [&](float v, int) {
        if ((long long)float_key(v) >= kk) {
          const int at = atomicAdd(&s_ncand, 1);
          if (at < kSelCand) cand[at] = v;
        }
      });
      __syncthreads();
      const int n2 = s_ncand;
      __syncthreads();
      if (n2 != nk) return false;
      // Z_k summed over the copy itself, so that A(kmin - 1) = Z_k >= thr
      // (top_p < 1) and A(kmax) = 0 < thr hold as the search sums them
      sel_kept(cand, n2, 0, c, mc, s_f, s_i, mass, cnt);
      const float thr = tp * mass;
      keep = sel_search_topp(cand, n2, 0.f, thr, c, mc, s_f, s_i);
      sel_kept(cand, n2, keep, c, mc, s_f, s_i, mass, cnt);
      z_kept = mass;
    }
  }
  if (tid == 0) finish_row(P, row, r, kFiltered, m, am, z_kept, key_float((uint32_t)keep), c);
  return true;
}

// One block per row: the filtered rows of batches the streaming pass's
// histogram does not take.
__global__ void __launch_bounds__(kSelThreads, 2)
k_rows_select(Params P) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char sel_smem[];
  WinHist* hist = reinterpret_cast<WinHist*>(sel_smem);
  float* cand = reinterpret_cast<float*>(sel_smem + sizeof(WinHist));
  __shared__ int s_req, s_cls, s_ok;
  const long long row = blockIdx.x;
  if (threadIdx.x == 0) {
    int r = 0;
    s_ok = locate_row(P, row, r);
    s_req = r;
    s_cls = s_ok ? row_class(P, r) : kArgmaxOnly;
  }
  __syncthreads();
  if (!s_ok || s_cls != kFiltered) return;
  if (!select_row(P, row, s_req, hist, cand)) {
    __syncthreads();
    filtered_row_stats(P, BlockGroup(), row, s_req);
  }
}

}  // namespace sv
