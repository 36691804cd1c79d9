// Target-row pass: the sampling constraints and row statistics of every
// target row (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나": temperature, top-k
// and top-p turn the target logits into p before the judgement; "기본값 greedy
// 드래프트에서도 분포가 지켜질까": temperature-0 rows need only the argmax).
//
// Two kernels share the work by row class:
//  * k_rows_stream — argmax-only and plain-softmax rows. Each row is cut into
//    slices; one CTA streams one slice once from HBM with 16-byte loads and
//    reduces (max, lowest argmax, sum of exp2((l - m) log2e / T)) in
//    registers and warp shuffles. The last CTA of a row (atomic counter)
//    merges the slice partials and evaluates p at the row's draft token.
//  * k_rows_filtered — rows with top-k and/or top-p. One CTA per row finds
//    the thresholds exactly by an 8-ary search over order-preserving keys
//    (counts for top-k, probability mass for top-p; seven thresholds per
//    pass), re-reading the row each pass.
#pragma once
#include "common.cuh"
#include "pipe.cuh"

namespace sv {

constexpr int kStreamThreads = 256;
constexpr int kStreamChunks = 8;  // 16-byte loads per thread per slice
constexpr int kSliceBf16 = kStreamThreads * kStreamChunks * 8;  // 16384
constexpr int kSliceF32 = kStreamThreads * kStreamChunks * 4;   // 8192

__device__ __forceinline__ int unpack_chunk(uint4 v, int bf16, float* f) {
  if (bf16) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    return 8;
  }
  f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  return 4;
}

// Partials written by other CTAs of the row: read through L2, not L1.
__device__ __forceinline__ SlicePartial load_partial(const SlicePartial* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  SlicePartial q;
  q.m = __int_as_float(v.x);
  q.s = __int_as_float(v.y);
  q.argmax = v.z;
  q.pad = v.w;
  return q;
}

// Write the statistics of one finished row and p at its draft token x
// (x < 0: the row has no draft token; lx is the logit at x when 0 <= x < V).
__device__ void finish_row_x(const Params& P, long long row, int cls, float m, int argmax,
                             float z, float theta, float c, int x, float lx) {
  unsigned st = 0;
  if (cls != kArgmaxOnly) {
    if (m == INFINITY || !(z == z)) st |= SPEC_STATUS_NONFINITE;
    else if (m == -INFINITY) st |= SPEC_STATUS_NO_FINITE;
  }
  float p_x = 0.f;
  if (x >= 0 && x < P.Vg) {
    if (cls == kArgmaxOnly) {
      p_x = (x == argmax) ? 1.f : 0.f;
    } else if (st == 0) {
      p_x = (lx >= theta) ? exp2f(fmaf(lx, c, -__fmul_rn(m, c))) / z : 0.f;
    }
  }
  RowStats s;
  s.m = m;
  s.c = c;
  s.inv_z = 1.f / z;
  s.theta = theta;
  s.argmax = argmax;
  s.p_x = p_x;
  s.status = st;
  s.z = z;
  P.rows[row] = s;
  // Under early exit a row's problems count only if the row is at or before
  // its request's stop: the accept step reports them then.
  if (st && !(P.flags & SPEC_FLAG_EARLY_EXIT)) atomicOr(P.status, st);
}

// The draft token of target row `row` of request r (-1 for the last row).
__device__ __forceinline__ int draft_of_row(const Params& P, long long row, int r) {
  const int c0 = __ldg(P.cu + r);
  const int gamma = __ldg(P.cu + r + 1) - c0;
  const long long i = row - ((long long)c0 + r);
  return (i >= 0 && i < gamma && c0 + i < P.N) ? __ldg(P.ids + c0 + i) : -1;
}

__device__ void finish_row(const Params& P, long long row, int r, int cls, float m, int argmax,
                           float z, float theta, float c) {
  const int x = draft_of_row(P, row, r);
  const float lx = (x >= 0 && x < P.V) ? load_logit(P, row, x) : 0.f;
  finish_row_x(P, row, cls, m, argmax, z, theta, c, x, lx);
}

// Row lookup shared by both kernels; returns false (and flags the status
// word) when the offsets do not place `row` inside its request.
__device__ __forceinline__ bool locate_row(const Params& P, long long row, int& r) {
  r = request_of_row(P.cu, P.B, row);
  const int c0 = __ldg(P.cu + r), c1 = __ldg(P.cu + r + 1);
  const long long i = row - ((long long)c0 + r);
  if (c0 < 0 || c1 < c0 || c1 > P.N || i < 0 || i > c1 - c0) {
    atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
    return false;
  }
  return true;
}

__global__ void __launch_bounds__(kStreamThreads)
k_rows_stream(Params P) {
  pdl_wait();
  pdl_trigger();
  const int spr = P.slices_per_row;
  const long long row = (long long)blockIdx.x / spr;
  const int slice = (int)(blockIdx.x % spr);
  __shared__ int s_req, s_cls, s_ok, s_last;
  if (threadIdx.x == 0) {
    int r = 0;
    s_ok = locate_row(P, row, r);
    s_req = r;
    s_cls = s_ok ? row_class(P, r) : kArgmaxOnly;
  }
  __syncthreads();
  if (!s_ok || s_cls == kFiltered) return;
  const int r = s_req, cls = s_cls;
  const int V = P.V;
  const int esize = P.bf16 ? 2 : 4;
  const int slice_elems = P.bf16 ? kSliceBf16 : kSliceF32;
  const int j0 = slice * slice_elems;
  const int j1 = min(V, j0 + slice_elems);
  const float c = (cls == kSoftmax) ? kLog2e / __ldg(P.temp + r) : 0.f;
  const char* rowp = (const char*)P.logits + row * (long long)V * esize;

  float vmax = -INFINITY;
  int imax = kNoIndex;
  uint4 v[kStreamChunks];
  int nchunk = 0, jt = j0;
  const bool aligned = ((reinterpret_cast<uintptr_t>(rowp) & 15) == 0);
  if (aligned) {
    const int epc = 16 / esize;
    nchunk = (j1 - j0) / epc;
    jt = j0 + nchunk * epc;
    const char* base = rowp + (long long)j0 * esize;
#pragma unroll
    for (int k = 0; k < kStreamChunks; ++k) {
      const int ch = threadIdx.x + k * kStreamThreads;
      v[k] = ch < nchunk ? ldg_stream(base + (long long)ch * 16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kStreamChunks; ++k) {
      const int ch = threadIdx.x + k * kStreamThreads;
      if (ch < nchunk) {
        float f[8];
        const int n = unpack_chunk(v[k], P.bf16, f);
        float m8 = f[0];
#pragma unroll
        for (int e = 1; e < 8; ++e)
          if (e < n) m8 = fmaxf(m8, f[e]);
        if (m8 > vmax || (imax == kNoIndex && m8 == m8)) {
          int e = 0;
          while (e < n - 1 && !(f[e] == m8)) ++e;
          vmax = m8;
          imax = j0 + ch * epc + e;
        }
      }
    }
  }
  // Scalar part: a misaligned row, or the tail after the last full chunk.
  for (int j = jt + threadIdx.x; j < j1; j += kStreamThreads) {
    const float f = load_logit(P, row, j);
    if (f > vmax || (imax == kNoIndex && f == f)) {
      vmax = f;
      imax = j;
    }
  }
  float m = vmax;
  int am = imax;
  block_argmax(m, am);

  float s = 0.f;
  const float mc = m * c;
  if (cls == kSoftmax && m > -INFINITY) {
    if (aligned) {
#pragma unroll
      for (int k = 0; k < kStreamChunks; ++k) {
        const int ch = threadIdx.x + k * kStreamThreads;
        if (ch < nchunk) {
          float f[8];
          const int n = unpack_chunk(v[k], P.bf16, f);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < n) s += exp2f(fmaf(f[e], c, -mc));
        }
      }
    }
    for (int j = jt + threadIdx.x; j < j1; j += kStreamThreads)
      s += exp2f(fmaf(load_logit(P, row, j), c, -mc));
    s = block_sum(s);
  }

  if (threadIdx.x == 0) {
    SlicePartial part;
    part.m = m;
    part.s = s;
    part.argmax = am;
    part.pad = 0;
    P.partials[row * spr + slice] = part;
    __threadfence();
    const unsigned prev = atomicAdd(P.row_counter + row, 1u);
    s_last = (prev == (unsigned)spr - 1u);
  }
  __syncthreads();
  if (!s_last || threadIdx.x >= 32) return;

  // Last slice of the row: merge the partials (warp 0).
  __threadfence();
  const int lane = threadIdx.x;
  float mm = -INFINITY;
  int aa = kNoIndex;
  for (int t = lane; t < spr; t += 32) {
    const SlicePartial q = load_partial(P.partials + row * spr + t);
    argmax_combine(mm, aa, q.m, q.argmax);
  }
  warp_argmax(mm, aa);
  float z = 0.f;
  if (cls == kSoftmax) {
    for (int t = lane; t < spr; t += 32) {
      const SlicePartial q = load_partial(P.partials + row * spr + t);
      if (q.m > -INFINITY) z += q.s * exp2f(q.m * c - mm * c);
    }
    z = warp_sum(z);
  }
  if (lane == 0) {
    if (aa == kNoIndex) aa = 0;
    P.row_counter[row] = 0u;
    finish_row(P, row, r, cls, mm, aa, z, -INFINITY, c);
  }
}

// ---------------------------------------------------------------------------
// Filtered rows: exact thresholds by an 8-ary search on order-preserving keys.
// ---------------------------------------------------------------------------
constexpr int kFilterThreads = 512;

// Visit every element (value, index) of a row, in increasing index per
// thread, thread `tid` of `nt`.
template <typename F>
__device__ __forceinline__ void row_for_each(const Params& P, long long row, int tid, int nt,
                                             F&& f) {
  const int V = P.V;
  const int esize = P.bf16 ? 2 : 4;
  const char* rowp = (const char*)P.logits + row * (long long)V * esize;
  int jt = 0;
  if ((reinterpret_cast<uintptr_t>(rowp) & 15) == 0) {
    const int epc = 16 / esize;
    const int nchunk = V / epc;
    jt = nchunk * epc;
    for (int ch = tid; ch < nchunk; ch += nt) {
      float e[8];
      const int n = unpack_chunk(__ldg((const uint4*)rowp + ch), P.bf16, e);
      for (int t = 0; t < n; ++t) f(e[t], ch * epc + t);
    }
  }
  for (int j = jt + tid; j < V; j += nt) f(load_logit(P, row, j), j);
}

// The whole block as a thread group (for filtered_row_stats).
struct BlockGroup {
  __device__ int tid() const { return threadIdx.x; }
  __device__ int size() const { return blockDim.x; }
  __device__ void sync() const { __syncthreads(); }
  template <typename T>
  __device__ T sum(T x) const { return block_sum(x); }
  __device__ void argmax(float& v, int& i) const { block_argmax(v, i); }
};

__device__ __forceinline__ uint32_t elem_key(float v, int bf16) {
  const uint32_t k = float_key(v);
  return bf16 ? (k >> 16) : k;
}

// Smallest float whose key is `k` (key width 16 for bf16, 32 for fp32).
__device__ __forceinline__ float key_threshold(uint32_t k, int bf16) {
  if (bf16) {
    const uint32_t k32 = (k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu);
    return key_float(k32);
  }
  return key_float(k);
}

// The searches below test kSearchProbes thresholds per pass (an 8-ary
// search over the keys): a pass reads the row once and reduces
// kSearchProbes sums, so a 32-bit key space takes at most 11 passes.
constexpr int kSearchProbes = 7;

// The thresholds of one pass over the open interval (lo, hi), hi - lo >= 2:
// non-decreasing, each strictly inside it.
__device__ __forceinline__ void search_probes(long long lo, long long hi,
                                              long long t[kSearchProbes]) {
  const long long span = hi - lo;
#pragma unroll
  for (int i = 0; i < kSearchProbes; ++i) {
    const long long step = span * (i + 1) / (kSearchProbes + 1);
    t[i] = min(lo + (step > 0 ? step : 1), hi - 1);
  }
}

// Sum of v[0..K-1] over the group, in a fixed order (every thread gets the
// same K results); scr holds 32 x K values.
template <int K, typename T, typename G>
__device__ __forceinline__ void group_sum_k(const G& g, T (&v)[K], T* scr) {
  const int lane = g.tid() & 31, warp = g.tid() >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) scr[warp * K + k] = v[k];
  g.sync();
  const int nw = g.size() >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    T s = T(0);
    for (int w = 0; w < nw; ++w) s += scr[w * K + k];
    v[k] = s;
  }
  g.sync();
}

// One filtered row of request r, exactly, by a thread group G (all of its
// threads call it; thread 0 writes the row's statistics).
template <typename G>
__device__ __noinline__ void filtered_row_stats(const Params& P, const G& g, long long row, int r) {
  __shared__ float s_fsum[32 * kSearchProbes];
  __shared__ int s_isum[32 * kSearchProbes];
  const int bf16 = P.bf16;
  const float c = kLog2e / __ldg(P.temp + r);
  const int tk = P.top_k ? __ldg(P.top_k + r) : 0;
  const float tp = P.top_p ? __ldg(P.top_p + r) : 1.f;
  const bool topk_on = (tk > 0 && tk < P.V);
  const bool topp_on = (tp < 1.f);

  float vmax = -INFINITY;
  int imax = kNoIndex;
  int nan_seen = 0;
  row_for_each(P, row, g.tid(), g.size(), [&](float v, int j) {
    if (v > vmax || (imax == kNoIndex && v == v)) { vmax = v; imax = j; }
    nan_seen |= (v != v);
  });
  float m = vmax;
  int am = imax;
  g.argmax(m, am);
  nan_seen = g.sum(nan_seen);
  if (am == kNoIndex) am = 0;
  if (nan_seen || m == INFINITY || m == -INFINITY) {
    if (g.tid() == 0)
      finish_row(P, row, r, kFiltered, nan_seen ? NAN : m, am,
                 (nan_seen || m == INFINITY) ? NAN : 0.f, -INFINITY, c);
    return;
  }

  const float mc = m * c;
  const long long key_space = bf16 ? (1ll << 16) : (1ll << 32);
  long long kk = 0;  // top-k key threshold (keep key >= kk)
  if (topk_on) {
    long long lo = 0, hi = key_space;  // count(key >= lo) >= k > count(key >= hi)
    while (hi - lo > 1) {
      long long t[kSearchProbes];
      search_probes(lo, hi, t);
      int cnt[kSearchProbes];
#pragma unroll
      for (int i = 0; i < kSearchProbes; ++i) cnt[i] = 0;
      row_for_each(P, row, g.tid(), g.size(), [&](float v, int) {
        const long long k = elem_key(v, bf16);
#pragma unroll
        for (int i = 0; i < kSearchProbes; ++i) cnt[i] += (k >= t[i]);
      });
      group_sum_k(g, cnt, s_isum);
      long long nlo = lo, nhi = hi;
#pragma unroll
      for (int i = 0; i < kSearchProbes; ++i) {
        if (nhi != hi) continue;
        if (cnt[i] >= tk) nlo = t[i]; else nhi = t[i];
      }
      lo = nlo;
      hi = nhi;
    }
    kk = lo;
  }
  float zk = 0.f;
  row_for_each(P, row, g.tid(), g.size(), [&](float v, int) {
    if ((long long)elem_key(v, bf16) >= kk) zk += exp2f(fmaf(v, c, -mc));
  });
  zk = g.sum(zk);

  long long kp = kk;  // final key threshold
  if (topp_on) {
    const float thr = tp * zk;
    long long lo = kk - 1, hi = (long long)elem_key(m, bf16);  // A(lo) >= thr > A(hi)
    while (hi - lo > 1) {
      long long t[kSearchProbes];
      search_probes(lo, hi, t);
      float a[kSearchProbes];
#pragma unroll
      for (int i = 0; i < kSearchProbes; ++i) a[i] = 0.f;
      row_for_each(P, row, g.tid(), g.size(), [&](float v, int) {
        const long long k = elem_key(v, bf16);
        if (k >= kk) {
          const float e = exp2f(fmaf(v, c, -mc));
#pragma unroll
          for (int i = 0; i < kSearchProbes; ++i) a[i] += (k > t[i]) ? e : 0.f;
        }
      });
      group_sum_k(g, a, s_fsum);
      long long nlo = lo, nhi = hi;
#pragma unroll
      for (int i = 0; i < kSearchProbes; ++i) {
        if (nhi != hi) continue;
        if (a[i] < thr) nhi = t[i]; else nlo = t[i];
      }
      lo = nlo;
      hi = nhi;
    }
    kp = hi;
  }
  float z = 0.f;
  row_for_each(P, row, g.tid(), g.size(), [&](float v, int) {
    if ((long long)elem_key(v, bf16) >= kp) z += exp2f(fmaf(v, c, -mc));
  });
  z = g.sum(z);
  if (g.tid() == 0) {
    const float theta = (kp <= 0) ? -INFINITY : key_threshold((uint32_t)kp, bf16);
    finish_row(P, row, r, kFiltered, m, am, z, theta, c);
  }
}

// One filtered row, exactly, by the whole block (all threads call it).
__device__ void filtered_row(const Params& P, long long row) {
  __shared__ int s_req, s_cls, s_ok;
  if (threadIdx.x == 0) {
    int r = 0;
    s_ok = locate_row(P, row, r);
    s_req = r;
    s_cls = s_ok ? row_class(P, r) : kArgmaxOnly;
  }
  __syncthreads();
  if (!s_ok || s_cls != kFiltered) return;
  filtered_row_stats(P, BlockGroup(), row, s_req);
}

// Without the streaming pass's histogram: block b settles row b. With it:
// the blocks share out the rows that pass listed as unsettled.
__global__ void __launch_bounds__(kFilterThreads, 2)
k_rows_filtered(Params P) {
  pdl_wait();
  pdl_trigger();
  if (!P.fast_filtered) {
    filtered_row(P, blockIdx.x);
    return;
  }
  const unsigned n = *P.pending_count;
  for (unsigned i = blockIdx.x; i < n; i += gridDim.x) {
    filtered_row(P, P.pending_rows[i]);
    __syncthreads();
  }
}

}  // namespace sv
