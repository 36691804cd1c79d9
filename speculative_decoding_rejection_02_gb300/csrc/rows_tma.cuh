// Persistent, bulk-copy pipelined target-row pass (the same statistics as
// k_rows_stream, for rows whose byte length is a multiple of 16).
//
// Each CTA owns rows blockIdx.x, blockIdx.x + gridDim.x, ... and streams
// every row exactly once from HBM through a ring of shared-memory stages:
//  * warp 16 (producer) looks up the next row's request and settings with
//    warp-parallel loads while the current row streams, and lane 0 issues
//    one 1-D bulk copy (TMA) per stage, signalling an mbarrier;
//  * warps 0..15 (consumers) wait on the stage, fold it into per-thread
//    (max, lowest argmax, online sum of exp2((l - m) log2e / T)) in
//    registers, capture the logit at the row's draft token, release the
//    stage, and at the row's end reduce over the 512 consumers and write the
//    row statistics and p(x).
// Variants (template flags below): rows with top-k / top-p also counted
// into the window histogram (FILT); rows taken from the early-exit work
// queue and judged at their end, possibly in parts (EARLY); one rank's
// columns of a vocab-sharded call, exporting local statistics (SHARD).
// Without parts a row never leaves its CTA.
#pragma once
#include "common.cuh"
#include "pipe.cuh"
#include "rows.cuh"
#include "hist.cuh"
#include "early.cuh"

namespace sv {

constexpr int kTmaConsumerWarps = 16;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaThreads = kTmaConsumers + 32;
constexpr int kTmaStages = 3;
// Stage size: 32 KB for the softmax / argmax rows; 24 KB next to the 24 KB
// window histogram of the top-k / top-p variant (two CTAs per SM either way).
__host__ __device__ constexpr int tma_stage_bytes(bool filt) { return filt ? 24576 : 32768; }
__host__ __device__ constexpr int tma_vec_per_thread(bool filt) {
  return tma_stage_bytes(filt) / 16 / kTmaConsumers;
}

struct StageMeta {
  long long row;  // -1: end of work
  int cls;
  float c;
  int x;     // draft token of the row (-1: none)
  int j0;    // first element of the stage within the row
  int n;     // elements in the stage
  int last;  // 1 on the row's last stage
  int tk;    // top-k of the row's request (filtered rows)
  float tp;  // top-p of the row's request (filtered rows)
  int r;        // request of the row
  int pos;      // position of the row within its request (0 .. gamma)
  int gamma;    // draft tokens of the request
  int c0;       // cu_num_draft[r]
  int part;     // part of the row (early exit; 0 otherwise)
};

__host__ __device__ constexpr size_t tma_ring_bytes(bool filt) {
  return (size_t)kTmaStages * tma_stage_bytes(filt) + 2 * kTmaStages * sizeof(uint64_t) +
         kTmaStages * sizeof(StageMeta);
}
constexpr size_t kTmaSmemBytes = tma_ring_bytes(false);
// The top-k / top-p variant adds the window histogram (16-byte aligned).
constexpr size_t kTmaHistOffset = (tma_ring_bytes(true) + 255) & ~size_t(255);
constexpr size_t kTmaFiltSmemBytes = kTmaHistOffset + sizeof(WinHist);

struct RowInfo {
  long long row;
  int cls;  // -1: skip this row
  float c;
  int x;
  int tk;
  float tp;
  int r, pos, gamma, c0;  // request, position in it, its draft count, cu[r]
};

// Warp-parallel lookup of the request owning `row` and its settings (all 32
// lanes call it; every lane gets the result). Two or three dependent rounds
// of loads instead of a serial binary search.
// take_filtered: take every row (true) or skip the rows with top-k / top-p.
__device__ RowInfo warp_row_info(const Params& P, long long row, bool take_filtered) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = P.B;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const bool le = probe < hi && ((long long)__ldg(P.cu + probe) + probe <= row);
    const unsigned m = __ballot_sync(0xFFFFFFFFu, le);
    const int last = m ? 31 - __clz(m) : 0;
    lo = lo + last * step;
    hi = min(hi, lo + step);
  }
  const int r = lo;
  RowInfo info;
  info.row = row;
  int c0 = 0, c1 = 0, cls = kArgmaxOnly;
  float T = 0.f;
  if (lane == 0) {
    c0 = __ldg(P.cu + r);
    c1 = __ldg(P.cu + r + 1);
    if (!P.greedy_call) T = __ldg(P.temp + r);
  }
  c0 = __shfl_sync(0xFFFFFFFFu, c0, 0);
  c1 = __shfl_sync(0xFFFFFFFFu, c1, 0);
  const long long i = row - ((long long)c0 + r);
  if (c0 < 0 || c1 < c0 || c1 > P.N || i < 0 || i > c1 - c0) {
    if (lane == 0) atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
    info.cls = -1;
    info.c = 0.f;
    info.x = -1;
    info.tk = 0;
    info.tp = 1.f;
    info.r = r;
    info.pos = 0;
    info.gamma = 0;
    info.c0 = 0;
    return info;
  }
  int x = -1, tk = 0;
  float tp = 1.f;
  if (lane == 0) {
    cls = row_class(P, r);
    if (i < c1 - c0) x = __ldg(P.ids + c0 + i);
    if (cls == kFiltered) {
      tk = P.top_k ? __ldg(P.top_k + r) : 0;
      tp = P.top_p ? __ldg(P.top_p + r) : 1.f;
    }
  }
  cls = __shfl_sync(0xFFFFFFFFu, cls, 0);
  T = __shfl_sync(0xFFFFFFFFu, T, 0);
  info.x = __shfl_sync(0xFFFFFFFFu, x, 0);
  info.r = r;
  info.pos = (int)i;
  info.gamma = c1 - c0;
  info.c0 = c0;
  info.tk = __shfl_sync(0xFFFFFFFFu, tk, 0);
  info.tp = __shfl_sync(0xFFFFFFFFu, tp, 0);
  info.cls = (!take_filtered && cls == kFiltered) ? -1 : cls;
  info.c = (cls != kArgmaxOnly) ? kLog2e / T : 0.f;
  return info;
}

// A part's statistics written by another CTA (read through L2).
__device__ __forceinline__ PartStat load_part(const PartStat* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  PartStat q;
  q.m = __int_as_float(a.x);
  q.z = __int_as_float(a.y);
  q.argmax = a.z;
  q.lx = __int_as_float(a.w);
  q.has_lx = b.x;
  q.pad[0] = b.y;
  q.pad[1] = b.z;
  q.pad[2] = b.w;
  return q;
}

// The kTmaConsumers consumer threads as a thread group (for the exact
// filtered-row search inside the row pass); fs / is: one slot per warp.
struct ConsumerGroup {
  float* fs;
  int* is;
  __device__ int tid() const { return threadIdx.x; }
  __device__ int size() const { return kTmaConsumers; }
  __device__ void sync() const { named_sync(1, kTmaConsumers); }
  __device__ float sum(float x) const {
    return consumer_reduce<float, kTmaConsumerWarps>(x, fs, threadIdx.x,
                                                     [](float a, float b) { return a + b; });
  }
  __device__ int sum(int x) const {
    return consumer_reduce<int, kTmaConsumerWarps>(x, is, threadIdx.x,
                                                   [](int a, int b) { return a + b; });
  }
  __device__ void argmax(float& v, int& i) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_argmax(v, i);
    if (lane == 0) {
      fs[warp] = v;
      is[warp] = i;
    }
    sync();
    v = fs[0];
    i = is[0];
    for (int w = 1; w < kTmaConsumerWarps; ++w) argmax_combine(v, i, fs[w], is[w]);
    sync();
  }
};

// FILT = false: argmax-only and plain-softmax rows (batches without top-k /
// top-p, or whose filtered rows all go to the exact slow kernel).
// FILT = true (bf16 only): every row; on rows with top-k / top-p the
// elements near the row max are also counted into the window histogram of
// hist.cuh, and rows it cannot settle are listed for the slow kernel.
// EARLY: rows come from the early-exit work queue (early.cuh) and each row's
// position is judged at its end.
// SHARD: the rows hold one rank's columns of a vocab-sharded call; the row
// end exports the local statistics (and window histogram) instead of
// finishing the row (shard.cuh combines them).
template <bool BF16, bool FILT, bool EARLY = false, bool SHARD = false>
__global__ void __launch_bounds__(kTmaThreads, 2)
k_rows_tma(Params P, long long R) {
  pdl_wait();
  pdl_trigger();
  static_assert(!FILT || BF16, "the histogram path is for bf16 rows");
  constexpr int kTmaStageBytes = tma_stage_bytes(FILT);
  constexpr int kTmaVecPerThread = tma_vec_per_thread(FILT);
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTmaStages * kTmaStageBytes);
  uint64_t* empty = full + kTmaStages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(empty + kTmaStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTmaConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  constexpr int esize = BF16 ? 2 : 4;
  const long long row_bytes = (long long)P.V * esize;

  if (warp == kTmaConsumerWarps) {
    // ---------------- producer warp ----------------
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    const int nchunks = (int)((row_bytes + kTmaStageBytes - 1) / kTmaStageBytes);
    if constexpr (EARLY) {
      // Rows come from the work queue; the next one is taken only after the
      // current row is issued (it may not be queued yet).
      for (;;) {
        long long item = -1;
        if (lane == 0) item = queue_pop(P);
        item = __shfl_sync(0xFFFFFFFFu, item, 0);
        if (item < 0) break;
        const long long row = item >> 3;
        const int part = (int)(item & 7);
        const RowInfo cur = warp_row_info(P, row, true);
        const char* src = (const char*)P.logits + row * row_bytes;
        const long long off0 = (long long)part * P.part_bytes;
        const long long off1 = min(off0 + P.part_bytes, row_bytes);
        const int nch = (int)((off1 - off0 + kTmaStageBytes - 1) / kTmaStageBytes);
        for (int ch = 0; ch < nch && ok; ++ch) {
          int waited = 1;
          if (lane == 0) waited = mbar_wait(&empty[stage], phase ^ 1u) ? 1 : 0;
          waited = __shfl_sync(0xFFFFFFFFu, waited, 0);
          if (!waited) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const long long off = off0 + (long long)ch * kTmaStageBytes;
            const uint32_t bytes = (uint32_t)min((long long)kTmaStageBytes, off1 - off);
            StageMeta& M = meta[stage];
            M.row = row;
            M.cls = cur.cls;
            M.c = cur.c;
            M.x = cur.x;
            M.j0 = (int)(off / esize);
            M.n = (int)(bytes / esize);
            M.last = (ch == nch - 1) ? 1 : 0;
            M.tk = cur.tk;
            M.tp = cur.tp;
            M.r = cur.r;
            M.pos = cur.pos;
            M.gamma = cur.gamma;
            M.c0 = cur.c0;
            M.part = part;
            mbar_arrive_expect_tx(&full[stage], bytes);
            bulk_load(ring + (size_t)stage * kTmaStageBytes, src + off, bytes, &full[stage]);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kTmaStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    } else {
      // Rows blockIdx.x, then either blockIdx.x + gridDim.x, + 2 gridDim.x,
      // ... or, with a ticket counter, gridDim.x + the tickets this CTA
      // takes in turn (CTAs whose rows were cheap take more of them).
      auto next_row = [&](long long r0) -> long long {
        if (!P.row_ticket) return r0 + gridDim.x;
        unsigned t = 0;
        if (lane == 0) t = atomicAdd(P.row_ticket, 1u);
        return (long long)gridDim.x + __shfl_sync(0xFFFFFFFFu, t, 0);
      };
      long long row = blockIdx.x;
      RowInfo cur;
      cur.cls = -1;
      while (row < R) {  // first row with work
        cur = warp_row_info(P, row, FILT);  // FILT: every row
        if (cur.cls >= 0) break;
        row = next_row(row);
      }
      // The next row is looked up while this one streams: at its first
      // stage by stride, at its last with tickets (so that a ticket goes to
      // the CTA about to be free).
      const int look_at = P.row_ticket ? nchunks - 1 : 0;
      while (row < R && ok) {
        RowInfo next;
        next.cls = -1;
        long long nrow = R;
        bool next_done = false;
        const char* src = (const char*)P.logits + row * row_bytes;
        // the draft token as a local column (-1: another rank's)
        const int xl = SHARD ? ((cur.x >= P.v0 && cur.x - P.v0 < P.V) ? cur.x - P.v0 : -1)
                             : cur.x;
        for (int ch = 0; ch < nchunks; ++ch) {
          int waited = 1;
          if (lane == 0) waited = mbar_wait(&empty[stage], phase ^ 1u) ? 1 : 0;
          waited = __shfl_sync(0xFFFFFFFFu, waited, 0);
          if (!waited) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const long long off = (long long)ch * kTmaStageBytes;
            const uint32_t bytes = (uint32_t)min((long long)kTmaStageBytes, row_bytes - off);
            StageMeta& M = meta[stage];
            M.row = row;
            M.cls = cur.cls;
            M.c = cur.c;
            M.x = xl;
            M.j0 = (int)(off / esize);
            M.n = (int)(bytes / esize);
            M.last = (ch == nchunks - 1) ? 1 : 0;
            M.tk = cur.tk;
            M.tp = cur.tp;
            mbar_arrive_expect_tx(&full[stage], bytes);
            bulk_load(ring + (size_t)stage * kTmaStageBytes, src + off, bytes, &full[stage]);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kTmaStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (ch == look_at) {
            nrow = next_row(row);
            while (nrow < R) {
              next = warp_row_info(P, nrow, FILT);
              if (next.cls >= 0) break;
              nrow = next_row(nrow);
            }
            next_done = true;
          }
        }
        if (!next_done) break;
        row = nrow;
        cur = next;
      }
    }
    if (lane == 0) {
      // Every issued copy has landed before the block may exit. This runs
      // before the end marker: the marker advances a full barrier once more,
      // after which the parity of that stage's last copy would name the
      // (incomplete) current phase.
      for (int s = 0; s < kTmaStages; ++s)
        if (((issued >> s) & 1u) && !mbar_wait(&full[s], (issued_parity >> s) & 1u)) {
          atomicOr(P.status, SPEC_STATUS_TIMEOUT);
          ok = false;
        }
      if (ok && mbar_wait(&empty[stage], phase ^ 1u)) {
        meta[stage].row = -1;
        mbar_arrive(&full[stage]);
      } else {
        atomicOr(P.status, SPEC_STATUS_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  __shared__ float red_m[kTmaConsumerWarps], red_s[kTmaConsumerWarps];
  __shared__ int red_i[kTmaConsumerWarps];
  __shared__ float bc_m, s_lx;
  __shared__ int s_has_lx, s_last_part;
  __shared__ float s_zfull;
  __shared__ int bc_i;
  __shared__ float fscr[kTmaConsumerWarps];
  __shared__ int iscr[kTmaConsumerWarps];
  const int tid = threadIdx.x;
  constexpr int epc = 16 / esize;
  if (tid == 0) s_has_lx = 0;
  // Window histogram of the current filtered row (FILT only).
  WinHist* hist = reinterpret_cast<WinHist*>(smem + kTmaHistOffset);
  if (FILT) {
    uint4* hz = reinterpret_cast<uint4*>(hist);
    for (int i = tid; i < (int)(sizeof(WinHist) / 16); i += kTmaConsumers)
      hz[i] = make_uint4(0u, 0u, 0u, 0u);
    named_sync(1, kTmaConsumers);
  }
  int stage = 0;
  uint32_t phase = 0;
  // Running state of the current row: max, its lowest index, fl(max * c),
  // and the sum of 2^(l c - fl(max c)) over this thread's elements.
  float vmax = -INFINITY, vmc = 0.f, s = 0.f;
  int imax = kNoIndex;  // first element of the vector holding vmax (kNoIndex: none)
  uint4 mvec = make_uint4(0u, 0u, 0u, 0u);  // that vector
  for (;;) {
    int landed = 1;
    if (lane == 0) landed = mbar_wait(&full[stage], phase) ? 1 : 0;
    if (!__shfl_sync(0xFFFFFFFFu, landed, 0)) {
      if (lane == 0) atomicOr(P.status, SPEC_STATUS_TIMEOUT);
      break;
    }
    const StageMeta M = meta[stage];
    if (M.row < 0) break;
    const uint4* buf = reinterpret_cast<const uint4*>(ring + (size_t)stage * kTmaStageBytes);
    const int nvec = M.n / epc;
    // The row sum Z runs on softmax rows (top-k / top-p rows take theirs
    // from the window histogram, which counts every element).
    const bool soft = (M.cls == kSoftmax);
    // This thread's vectors of the stage, in increasing element order; the
    // missing ones read as -inf (no max, no mass).
    constexpr uint32_t pad = BF16 ? 0xFF80FF80u : 0xFF800000u;
    uint4 v[kTmaVecPerThread];
    if (nvec == kTmaVecPerThread * kTmaConsumers) {
      // a full stage (every stage but a row's or part's last)
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k) v[k] = buf[tid + k * kTmaConsumers];
    } else {
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k) {
        const int idx = tid + k * kTmaConsumers;
        v[k] = idx < nvec ? buf[idx] : make_uint4(pad, pad, pad, pad);
      }
    }
    float m32;
    // per-vector maxima (bf16: packed pairs), then the stage max
    uint32_t vm[kTmaVecPerThread];
    if (BF16) {
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k) {
        const __nv_bfloat162 h = __hmax2(__hmax2(u32_as_bf162(v[k].x), u32_as_bf162(v[k].y)),
                                         __hmax2(u32_as_bf162(v[k].z), u32_as_bf162(v[k].w)));
        memcpy(&vm[k], &h, sizeof h);
      }
      __nv_bfloat162 h = u32_as_bf162(vm[0]);
#pragma unroll
      for (int k = 1; k < kTmaVecPerThread; ++k) h = __hmax2(h, u32_as_bf162(vm[k]));
      m32 = fmaxf(__low2float(h), __high2float(h));
    } else {
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k)
        vm[k] = __float_as_uint(
            fmaxf(fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                  fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
      m32 = __uint_as_float(vm[0]);
#pragma unroll
      for (int k = 1; k < kTmaVecPerThread; ++k) m32 = fmaxf(m32, __uint_as_float(vm[k]));
    }
    if (m32 > vmax || (imax == kNoIndex && m32 > -INFINITY)) {
      // New running max: rescale, and remember the vector that holds it.
      // (every product and sum of Z with its own rounding: no instantiation
      // of this kernel may fuse them, so all give the same statistics)
      const float nmc = __fmul_rn(m32, M.c);
      if (soft && vmax > -INFINITY) s = __fmul_rn(s, ex2(__fsub_rn(vmc, nmc)));
      // The lowest index holding it: the first vector whose max it is, then
      // the first element of that vector.
      int kk = kTmaVecPerThread - 1;
#pragma unroll
      for (int k = kTmaVecPerThread - 2; k >= 0; --k) {
        const float mk = BF16 ? fmaxf(bf16_lo(vm[k]), bf16_hi(vm[k])) : __uint_as_float(vm[k]);
        if (mk == m32) kk = k;
      }
      uint4 vk = v[kTmaVecPerThread - 1];
#pragma unroll
      for (int k = kTmaVecPerThread - 2; k >= 0; --k)
        if (k == kk) vk = v[k];
      // Keep that vector; its element is found once, at the row's end.
      vmax = m32;
      vmc = nmc;
      imax = M.j0 + (tid + kk * kTmaConsumers) * epc;
      mvec = vk;
    }
    if (soft && vmax > -INFINITY) {
      const unsigned long long c2 = f2_pack(M.c, M.c);
      const unsigned long long nmc2 = f2_pack(-vmc, -vmc);
      unsigned long long acc0 = 0ull, acc1 = 0ull;  // (+0, +0) pairs
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k) {
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        if (BF16) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const unsigned long long x2 = f2_pack(bf16_lo(w[t]), bf16_hi(w[t]));
            float z0, z1;
            f2_unpack(f2_fma(x2, c2, nmc2), z0, z1);
            const unsigned long long e2 = f2_pack(ex2(z0), ex2(z1));
            if (t & 1) acc1 = f2_add(acc1, e2); else acc0 = f2_add(acc0, e2);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 4; t += 2) {
            const unsigned long long x2 =
                f2_pack(__uint_as_float(w[t]), __uint_as_float(w[t + 1]));
            float z0, z1;
            f2_unpack(f2_fma(x2, c2, nmc2), z0, z1);
            const unsigned long long e2 = f2_pack(ex2(z0), ex2(z1));
            if (t & 2) acc1 = f2_add(acc1, e2); else acc0 = f2_add(acc0, e2);
          }
        }
      }
      float a0, a1, a2, a3;
      f2_unpack(acc0, a0, a1);
      f2_unpack(acc1, a2, a3);
      s = __fadd_rn(s, __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3)));
    }
    if (FILT && M.cls == kFiltered) {
      // Count every element into the window histogram. The padding of a
      // row's (or part's) last stage is -inf and lands in the negative huge
      // counter; thread 0 takes it out again.
      uint32_t words[4 * kTmaVecPerThread];
      uint32_t mn2 = 0xFFFFFFFFu, mx2 = 0u;
#pragma unroll
      for (int k = 0; k < kTmaVecPerThread; ++k) {
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        words[4 * k] = v[k].x;
        words[4 * k + 1] = v[k].y;
        words[4 * k + 2] = v[k].z;
        words[4 * k + 3] = v[k].w;
        win_count_all(hist, w, mn2, mx2);
      }
      win_tiny(hist, words, mn2, M.c);
      win_nan(hist, mx2);
      if (tid == 0 && nvec < kTmaVecPerThread * kTmaConsumers)
        atomicSub(&hist->cnt[win_slot_of_item(kWinHugeNeg)],
                  win_pad(M.n, kTmaVecPerThread * kTmaConsumers * epc));
    }
    {
      // The draft token's logit, captured by the thread that holds it.
      const int dx = M.x - M.j0;
      if (dx >= 0 && dx < M.n) {
        const int vx = dx / epc;
        if ((vx % kTmaConsumers) == tid) {
          const int k = vx / kTmaConsumers;
          uint4 vk = v[0];
#pragma unroll
          for (int t = 1; t < kTmaVecPerThread; ++t)
            if (t == k) vk = v[t];
          float f[8];
          unpack_chunk(vk, BF16, f);
          float lx = f[0];
#pragma unroll
          for (int e = 1; e < epc; ++e)
            if (e == dx - vx * epc) lx = f[e];
          s_lx = lx;
          s_has_lx = 1;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == kTmaStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (M.last) {
      float m = vmax;
      int a = kNoIndex;
      if (imax != kNoIndex) {
        float f[8];
        unpack_chunk(mvec, BF16, f);
#pragma unroll
        for (int e = epc - 1; e >= 0; --e)
          if (f[e] == vmax) a = imax + e;
      }
      warp_argmax(m, a);
      if (lane == 0) {
        red_m[warp] = m;
        red_i[warp] = a;
      }
      named_sync(1, kTmaConsumers);
      if (warp == 0) {
        m = lane < kTmaConsumerWarps ? red_m[lane] : -INFINITY;
        a = lane < kTmaConsumerWarps ? red_i[lane] : kNoIndex;
        warp_argmax(m, a);
        if (lane == 0) {
          bc_m = m;
          bc_i = a;
        }
      }
      named_sync(1, kTmaConsumers);
      m = bc_m;
      a = bc_i;
      if constexpr (SHARD) {
        // Local statistics of this rank's columns (global indices).
        const float mc = __fmul_rn(m, M.c);
        float part = 0.f;
        if (soft && vmax > -INFINITY && m > -INFINITY) part = __fmul_rn(s, ex2(__fsub_rn(vmc, mc)));
        part = warp_sum(part);
        if (lane == 0) red_s[warp] = part;
        if (FILT && M.cls == kFiltered) {
          int* hout = P.sh_hist + M.row * (long long)SPEC_SHARD_HIST_INTS;
          for (int i = tid; i < kWinSlots; i += kTmaConsumers) {
            hout[i] = (int)hist->cnt[i];
            hist->cnt[i] = 0u;
          }
          if (tid < 2) {
            P.sh_hist_w[2 * M.row + tid] = hist->tiny_w[tid];
            hist->tiny_w[tid] = 0.f;
          }
        }
        named_sync(1, kTmaConsumers);
        if (tid == 0) {
          float z = 0.f;
          if (soft)
            for (int w = 0; w < kTmaConsumerWarps; ++w) z += red_s[w];
          P.sh_m[M.row] = m;
          P.sh_z[M.row] = z;
          P.sh_arg[M.row] = (a == kNoIndex) ? 0x7FFFFFFF : a + P.v0;
          P.sh_lx[M.row] = s_has_lx ? s_lx : -INFINITY;
          P.rows[M.row].m = m;  // the local max, for the rescale
          s_has_lx = 0;
        }
        named_sync(1, kTmaConsumers);
        vmax = -INFINITY;
        vmc = 0.f;
        s = 0.f;
        imax = kNoIndex;
        continue;
      }
      float zmerged = 0.f;
      if (EARLY && P.parts > 1) {
        // End of one part of the row: publish the part's statistics (and add
        // its window histogram to the request's global one). The CTA that
        // ends the row's last part merges them and judges the position.
        const float mc = __fmul_rn(m, M.c);
        float part = 0.f;
        if (soft && vmax > -INFINITY && m > -INFINITY) part = __fmul_rn(s, ex2(__fsub_rn(vmc, mc)));
        part = warp_sum(part);
        if (lane == 0) red_s[warp] = part;
        WinHist* ghist = reinterpret_cast<WinHist*>(P.part_hist) + M.r;
        if (FILT && M.cls == kFiltered) {
          win_flush(hist, ghist, tid, kTmaConsumers);
          __threadfence();
        }
        named_sync(1, kTmaConsumers);
        if (tid == 0) {
          PartStat ps;
          ps.m = m;
          ps.z = 0.f;
          if (soft)
            for (int w = 0; w < kTmaConsumerWarps; ++w) ps.z += red_s[w];
          ps.argmax = a;
          ps.lx = s_has_lx ? s_lx : 0.f;
          ps.has_lx = s_has_lx;
          ps.pad[0] = ps.pad[1] = ps.pad[2] = 0;
          s_has_lx = 0;
          PartStat* mine = P.part_stats + (size_t)M.r * kMaxParts;
          mine[M.part] = ps;
          __threadfence();
          const unsigned prev = atomicAdd(P.part_done + M.r, 1u);
          s_last_part = (prev == (unsigned)P.parts - 1u) ? 1 : 0;
          if (s_last_part) {
            __threadfence();
            P.part_done[M.r] = 0u;
            float mm = -INFINITY, zz = 0.f, lxx = 0.f;
            int aa = kNoIndex;
            for (int k = 0; k < P.parts; ++k) {
              const PartStat q = load_part(mine + k);
              argmax_combine(mm, aa, q.m, q.argmax);
              if (q.has_lx) lxx = q.lx;
            }
            const float mmc = mm * M.c;
            for (int k = 0; k < P.parts; ++k) {
              const PartStat q = load_part(mine + k);
              if (q.argmax != kNoIndex && q.m > -INFINITY) zz += q.z * ex2(q.m * M.c - mmc);
            }
            bc_m = mm;
            bc_i = aa;
            s_zfull = zz;
            s_lx = lxx;
          }
        }
        named_sync(1, kTmaConsumers);
        if (!s_last_part) {
          vmax = -INFINITY;
          vmc = 0.f;
          s = 0.f;
          imax = kNoIndex;
          continue;
        }
        m = bc_m;
        a = bc_i;
        zmerged = s_zfull;
        if (FILT && M.cls == kFiltered) {
          win_take(hist, ghist, tid, kTmaConsumers);
          named_sync(1, kTmaConsumers);
        }
      }
      if (FILT && M.cls == kFiltered) {
        const HistResult hr =
            win_finish<kTmaConsumerWarps>(hist, m, M.c, M.tk, M.tp, P.V, tid, fscr, iscr);
        const bool unsettled = hr.pending || !(m > -INFINITY);
        if (unsettled && EARLY) {
          // The judgement needs this row now: settle it exactly here.
          filtered_row_stats(P, ConsumerGroup{fscr, iscr}, M.row, M.r);
        } else if (tid == 0) {
          if (unsettled) {
            RowStats ps;
            ps.m = m;
            ps.c = M.c;
            ps.inv_z = 0.f;
            ps.theta = -INFINITY;
            ps.argmax = 0;
            ps.p_x = 0.f;
            ps.status = kPendingSlow;
            ps.z = 0.f;
            P.rows[M.row] = ps;
            P.pending_rows[atomicAdd(P.pending_count, 1u)] = M.row;
          } else {
            finish_row_x(P, M.row, M.cls, m, a == kNoIndex ? 0 : a, hr.z, hr.theta, M.c, M.x,
                         s_lx);
          }
        }
        if (EARLY && tid == 0) early_decide(P, M.r, M.pos, M.gamma, M.c0);
        named_sync(1, kTmaConsumers);
        vmax = -INFINITY;
        vmc = 0.f;
        s = 0.f;
        imax = kNoIndex;
        continue;
      }
      const float mc = __fmul_rn(m, M.c);
      const bool merged_row = EARLY && P.parts > 1;
      float part = 0.f;
      if (!merged_row) {
        if (soft && vmax > -INFINITY && m > -INFINITY) part = __fmul_rn(s, ex2(__fsub_rn(vmc, mc)));
        part = warp_sum(part);
        if (lane == 0) red_s[warp] = part;
        named_sync(1, kTmaConsumers);
      }
      if (tid == 0) {
        float z = merged_row ? zmerged : 0.f;
        if (soft && !merged_row)
          for (int w = 0; w < kTmaConsumerWarps; ++w) z += red_s[w];
        finish_row_x(P, M.row, M.cls, m, a == kNoIndex ? 0 : a, z, -INFINITY, M.c, M.x, s_lx);
        if (EARLY) early_decide(P, M.r, M.pos, M.gamma, M.c0);
      }
      named_sync(1, kTmaConsumers);
      vmax = -INFINITY;
      vmc = 0.f;
      s = 0.f;
      imax = kNoIndex;
    }
  }
}

}  // namespace sv
