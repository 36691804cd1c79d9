// Early-exit verification with each judged row resident in a thread-block
// cluster (velog "드래프트가 제안하고 타깃이 판정한다": the first rejection
// ends the round and the later positions are discarded, so their rows need
// never be read; the token at the stop is drawn from the row just judged).
//
// One cluster of C CTAs (C = 1, 2, 4 or 8) verifies one request at a time.
// CTA k of the cluster holds elements [k S, (k + 1) S) of the request's
// current target row in its shared memory (S elements of at most 64 KB, so a
// 512 KB bf16 row at V = 256000 spans 8 CTAs). Position by position:
//  1. each CTA pulls its part of the row with bulk copies (TMA, untiled) and
//     folds it into (max, lowest argmax, sum of 2^(l c - m c)) and, when the
//     part holds it, the draft token's logit;
//  2. the CTAs swap these partials through distributed shared memory; each
//     combines the C of them in rank order, so every CTA holds the same row
//     statistics and takes the same accept decision (the test of k_accept);
//  3. on acceptance the next row replaces this one; at the first rejection,
//     or after the last draft token, the exponential race for the output
//     token runs on the parts still in shared memory (only that position's
//     draft probabilities are read, streamed through a two-stage ring), and
//     the CTAs swap their best (score, index) to pick the winner.
// A request's rows after its stop are never read and the row at the stop is
// read once. Requests are taken by atomic ticket, one per cluster at a time.
//
// Exchanges: every CTA writes its 32-byte record into slot [rank] of every
// CTA's exchange array and arrives (release, cluster scope) on every CTA's
// exchange mbarrier, which expects C arrivals; all threads then wait
// (acquire, cluster scope, bounded). Two barriers and two slot arrays
// alternate: a CTA can publish exchange e + 2 only after exchange e + 1 has
// completed, which needs every CTA's arrival for e + 1, which each CTA makes
// only after it has read exchange e. The CTAs of a cluster leave together
// through one cluster barrier, so none exits while another may still write
// into its shared memory.
#pragma once
#include "common.cuh"
#include "philox.cuh"
#include "pipe.cuh"
#include "race.cuh"
#include "rows.cuh"

namespace sv {

constexpr int kResWarps = 16;
constexpr int kResThreads = kResWarps * 32;
constexpr int kResMaxCluster = 8;
constexpr int kResPartBytes = 65536;   // a CTA's part of a row, at most
constexpr int kResChunkBytes = 16384;  // one bulk copy (the part takes up to 4)
constexpr int kResChunks = kResPartBytes / kResChunkBytes;
constexpr int kResVecPerThread = kResChunkBytes / 16 / kResThreads;  // 2
constexpr int kResQEntries = 4096;     // draft probabilities per ring stage (16 KB)
constexpr int kResQStages = 2;
constexpr int kResSubEntries = 8192;   // entries per scoring call without q
static_assert(kResVecPerThread * 16 * kResThreads == kResChunkBytes, "chunk / thread split");
// Scoring calls take at most 2 units (8 entries) per thread: within the
// per-warp queue that race_slice_smem sizes for either kind of call.
static_assert(kResSubEntries / 8 <= 2 * kResThreads && kResQEntries / 8 <= 2 * kResThreads &&
                  race_units(true) >= 2,
              "race queue too small for the scoring calls");

// Shared memory (dynamic): the part, the draft-probability ring (which holds
// the scoring queue in calls without draft probabilities), the queue of calls
// with them, the mbarriers and the exchange slots.
constexpr size_t kResOffQ = kResPartBytes;
constexpr size_t kResQRingBytes = (size_t)kResQStages * kResQEntries * sizeof(float);
constexpr size_t kResQueueBytesQ = (size_t)kResWarps * 32 * 2 * race_units(true) * sizeof(uint16_t);
constexpr size_t kResQueueBytesNoQ =
    (size_t)kResWarps * 32 * 2 * race_units(false) * sizeof(uint16_t);
static_assert(kResQueueBytesNoQ <= kResQRingBytes, "no-q queue lives in the ring");
constexpr size_t kResOffQueue = kResOffQ + kResQRingBytes;
constexpr size_t kResOffBar = kResOffQueue + kResQueueBytesQ;
constexpr int kResBars = kResChunks + kResQStages + 2;
constexpr size_t kResOffSlots = kResOffBar + kResBars * sizeof(uint64_t);
struct __align__(16) ResSlot {
  float m;        // max over the part
  float z;        // sum of 2^(l c - fl(m c)) over the part
  int argmax;     // lowest index of the part max (kNoIndex: none)
  float lx;       // the draft token's logit (when has_lx)
  int has_lx;
  int req;        // request ticket (rank 0's record)
  unsigned long long best;  // the part's race winner, packed (score, ~index)
};
static_assert(sizeof(ResSlot) == 32, "two 16-byte stores per record");
static_assert(kResOffSlots % 16 == 0, "slots are written as 16-byte vectors");
constexpr size_t kResSmemBytes = kResOffSlots + 2 * kResMaxCluster * sizeof(ResSlot);

// --------------------------------------------------------------------------
// Cluster primitives (inline PTX, sm_90 and later)
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `p` (a shared variable of this CTA) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}
// Exchange waits: probes that may suspend the thread for up to
// kClusterHintNs (the phase is completed by other CTAs' arrivals), at most
// kClusterTries of them: about a second in all.
constexpr uint32_t kClusterHintNs = 2000;
constexpr uint32_t kClusterTries = 1u << 19;
__device__ __forceinline__ bool mbar_try_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kClusterHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kClusterTries; ++i)
    if (mbar_try_acq_cluster(bar, parity)) return true;
  return false;
}
// All threads of every CTA of the cluster (used once at the start and once
// at the end of the kernel).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Order this CTA's earlier generic-proxy accesses of shared memory before
// later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Publish `mine` (thread 0's) as exchange e and wait for the other CTAs'
// records. Returns the same outcome in every thread; false on timeout.
__device__ __forceinline__ bool res_exchange(ResSlot* slots, uint64_t* xbar, uint32_t e,
                                             uint32_t rank, uint32_t C, const ResSlot& mine) {
  const uint32_t b = e & 1u;
  if (threadIdx.x == 0) {
    const uint4 lo = make_uint4(__float_as_uint(mine.m), __float_as_uint(mine.z),
                                (uint32_t)mine.argmax, __float_as_uint(mine.lx));
    const uint4 hi = make_uint4((uint32_t)mine.has_lx, (uint32_t)mine.req,
                                (uint32_t)(mine.best & 0xFFFFFFFFull), (uint32_t)(mine.best >> 32));
    const ResSlot* dst = slots + b * kResMaxCluster + rank;
    for (uint32_t k = 0; k < C; ++k) {
      const uint32_t a = cluster_map(dst, k);
      st_cluster_v4(a, lo);
      st_cluster_v4(a + 16u, hi);
    }
    for (uint32_t k = 0; k < C; ++k) mbar_arrive_cluster(cluster_map(&xbar[b], k));
  }
  const bool ok = mbar_wait_cluster(&xbar[b], (e >> 1) & 1u);
  return __syncthreads_and(ok ? 1 : 0) != 0;
}

// The records of exchange e (valid after res_exchange returned true).
__device__ __forceinline__ const ResSlot* res_records(const ResSlot* slots, uint32_t e) {
  return slots + (e & 1u) * kResMaxCluster;
}

// Race over this CTA's part (elements j0 .. j0 + n - 1, logits resident at
// lbuf) in the given mode; returns the part's winner packed (0: none). Every
// thread returns the same value. The running best starts from the score of
// token seed_j (a valid candidate, so a lower bound of the winner's score;
// -1: none), computed by thread 0 from global memory while the first copies
// fly; s_seed is a shared word for it. For residual weights the part's draft
// probabilities are streamed through the ring; on a timeout `ok` turns false
// (after the copies in flight have landed or given up).
template <bool BF16>
__device__ unsigned long long res_race(const Params& P, const RaceView& v, int mode,
                                       unsigned char* lbuf, float* qring, uint64_t* qbar,
                                       uint32_t& q_phase, uint16_t* queue, int j0, int n,
                                       int seed_j, unsigned long long* s_seed, bool& ok) {
  constexpr int esize = BF16 ? 2 : 4;
  const bool resid = (mode == kRaceResidual) && n > 0 && v.z > 0.f;
  const int nst = resid ? (n + kResQEntries - 1) / kResQEntries : 0;
  const float* qsrc = resid ? P.q + (long long)v.qrow * P.V + j0 : nullptr;
  uint32_t issued = 0;  // stages issued and not yet waited (bit per ring slot)
  if (threadIdx.x == 0) {
    for (int s = 0; s < kResQStages && s < nst; ++s) {
      const uint32_t bytes = (uint32_t)min(kResQEntries, n - s * kResQEntries) * 4u;
      mbar_arrive_expect_tx(&qbar[s], bytes);
      bulk_load(qring + s * kResQEntries, qsrc + s * kResQEntries, bytes, &qbar[s]);
    }
    *s_seed = (seed_j >= 0) ? race_candidate(P, v, seed_j) : 0ull;
  }
  for (int s = 0; s < kResQStages && s < nst; ++s) issued |= 1u << s;
  __syncthreads();
  const unsigned long long seed_best = *s_seed;
  float best = seed_best ? __uint_as_float((uint32_t)(seed_best >> 32)) : 0.f;
  int best_j = seed_best ? (int)(0xFFFFFFFFu - (uint32_t)seed_best) : kNoIndex;
  if (n > 0 && v.z > 0.f) {
    if (resid) {
      for (int s = 0; s < nst; ++s) {
        const int slot = s % kResQStages;
        const uint32_t par = (q_phase >> slot) & 1u;
        const bool landed = mbar_wait(&qbar[slot], par);
        if (!__syncthreads_and(landed ? 1 : 0)) {
          ok = false;  // this stage's copy is still counted as in flight
          break;
        }
        q_phase ^= 1u << slot;
        issued &= ~(1u << slot);
        const int js = s * kResQEntries;
        const int ns = min(kResQEntries, n - js);
        const unsigned char* lb = lbuf + (size_t)js * esize;
        const float* qb = qring + slot * kResQEntries;
        if (best_j == kNoIndex) {
          // No bound yet: score the stage's heaviest entry first.
          float wb = 0.f;
          int jb = kNoIndex;
          race_slice_heaviest<BF16, true, false>(v, lb, qb, ns, j0 + js, wb, jb);
          block_argmax(wb, jb);
          if (jb != kNoIndex && wb > 0.f) {
            const uint4 rw = race_words(P.seed, v.greq, v.kstar, v.g0 + ((uint32_t)jb >> 2));
            const uint32_t words[4] = {rw.x, rw.y, rw.z, rw.w};
            best = race_score(wb, words[jb & 3]);
            best_j = jb;
          }
        }
        race_slice_smem<BF16, true, false>(P, v, lb, qb, ns, j0 + js, best, best_j, queue);
        __syncthreads();  // the stage is free again
        if (s + kResQStages < nst) {
          if (threadIdx.x == 0) {
            const int jn = (s + kResQStages) * kResQEntries;
            const uint32_t bytes = (uint32_t)min(kResQEntries, n - jn) * 4u;
            mbar_arrive_expect_tx(&qbar[slot], bytes);
            bulk_load(qring + slot * kResQEntries, qsrc + jn, bytes, &qbar[slot]);
          }
          issued |= 1u << slot;
        }
      }
      if (!ok) {
        // Let the copies still in flight land (bounded) before the ring is
        // given up.
        for (int slot = 0; slot < kResQStages; ++slot)
          if ((issued >> slot) & 1u) {
            mbar_wait(&qbar[slot], (q_phase >> slot) & 1u);
            q_phase ^= 1u << slot;
          }
        __syncthreads();
        return 0ull;
      }
    } else {
      for (int js = 0; js < n; js += kResSubEntries) {
        const int ns = min(kResSubEntries, n - js);
        const unsigned char* lb = lbuf + (size_t)js * esize;
        if (best_j == kNoIndex) {
          float wb = 0.f;
          int jb = kNoIndex;
          race_slice_heaviest<BF16, false, false>(v, lb, nullptr, ns, j0 + js, wb, jb);
          block_argmax(wb, jb);
          if (jb != kNoIndex && wb > 0.f) {
            const uint4 rw = race_words(P.seed, v.greq, v.kstar, v.g0 + ((uint32_t)jb >> 2));
            const uint32_t words[4] = {rw.x, rw.y, rw.z, rw.w};
            best = race_score(wb, words[jb & 3]);
            best_j = jb;
          }
        }
        race_slice_smem<BF16, false, false>(P, v, lb, nullptr, ns, j0 + js, best, best_j, queue);
      }
    }
  }
  block_argmax(best, best_j);
  return (best_j != kNoIndex && best > 0.f) ? race_pack(best, best_j) : 0ull;
}

template <bool BF16>
__global__ void __launch_bounds__(kResThreads, 2)
k_resident(Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* lbuf = smem;
  float* qring = reinterpret_cast<float*>(smem + kResOffQ);
  uint16_t* queue = reinterpret_cast<uint16_t*>(smem + (P.q ? kResOffQueue : kResOffQ));
  uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + kResOffBar);
  uint64_t* qbar = cbar + kResChunks;
  uint64_t* xbar = qbar + kResQStages;
  ResSlot* slots = reinterpret_cast<ResSlot*>(smem + kResOffSlots);
  __shared__ float red_m[kResWarps], red_s[kResWarps];
  __shared__ int red_i[kResWarps];
  __shared__ float s_lx;
  __shared__ int s_has_lx;
  __shared__ unsigned long long s_seed;
  __shared__ int s_acc;

  constexpr int esize = BF16 ? 2 : 4;
  constexpr int epc = 16 / esize;
  const uint32_t rank = cluster_rank(), C = cluster_ctas();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V;
  const int S = P.res_part;  // elements per part (a multiple of 8)
  const int j0 = (int)rank * S;
  const int n = max(0, min(S, V - j0));  // this CTA's elements
  const uint32_t pbytes = (uint32_t)n * esize;  // a multiple of 16
  const int nch = (int)((pbytes + kResChunkBytes - 1) / kResChunkBytes);

  if (tid == 0) {
    for (int i = 0; i < kResChunks + kResQStages; ++i) mbar_init(&cbar[i], 1);
    mbar_init(&xbar[0], C);
    mbar_init(&xbar[1], C);
    fence_mbar_init();
    s_has_lx = 0;
  }
  __syncthreads();
  cluster_sync_all();  // every barrier of the cluster is set up before any remote arrival

  uint32_t rows_done = 0;  // rows loaded into the part: the chunk barriers' phase
  uint32_t q_phase = 0;    // bit per ring slot
  uint32_t xe = 0;         // exchanges so far
  bool ok = true;
  ResSlot mine;
  mine.m = -INFINITY;
  mine.z = 0.f;
  mine.argmax = kNoIndex;
  mine.lx = 0.f;
  mine.has_lx = 0;
  mine.req = -1;
  mine.best = 0ull;

  // Requests by ticket: rank 0 takes them, every CTA learns them through an
  // exchange (the next request's ticket rides on the first row's exchange
  // of the current one).
  int r = -1;
  bool need_ticket = true;
  while (ok) {
    if (need_ticket) {
      ResSlot t = mine;
      if (rank == 0 && tid == 0) t.req = (int)atomicAdd(P.queue_ctl, 1u);
      if (!res_exchange(slots, xbar, xe, rank, C, t)) {
        ok = false;
        break;
      }
      r = res_records(slots, xe)[0].req;
      ++xe;
    }
    if (r < 0 || r >= P.B) break;
    need_ticket = true;
    const bool lead = (rank == 0 && tid == 0);  // writes the request's outputs
    const int c0 = __ldg(P.cu + r), c1 = __ldg(P.cu + r + 1);
    bool bad = (c0 < 0 || c1 < c0 || c1 > P.N);
    if (r == 0 && c0 != 0) bad = true;
    if (r == P.B - 1 && c1 != P.N) bad = true;
    if (bad) {
      if (lead) {
        atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
        P.num_accepted[r] = 0;
      }
      continue;
    }
    const int cur = r;
    const int gamma = c1 - c0;
    const long long row0 = (long long)c0 + r;
    const long long greq = P.req_base + r;
    const int cls = row_class(P, r);
    const bool greedy = (cls == kArgmaxOnly);
    const float c = greedy ? 0.f : kLog2e / __ldg(P.temp + r);
    const bool soft = (cls == kSoftmax);

    for (int pos = 0; pos <= gamma && ok; ++pos) {
      const long long row = row0 + pos;
      const int x = (pos < gamma) ? __ldg(P.ids + c0 + pos) : -1;
      const bool valid = (x >= 0 && x < V);
      // ---- 1. this CTA's part of the row ----
      if (tid == 0 && nch > 0) {
        fence_proxy_async_smem();
        const char* src = (const char*)P.logits + (row * V + j0) * esize;
        for (int ch = 0; ch < nch; ++ch) {
          const uint32_t off = (uint32_t)ch * kResChunkBytes;
          const uint32_t bytes = min((uint32_t)kResChunkBytes, pbytes - off);
          mbar_arrive_expect_tx(&cbar[ch], bytes);
          bulk_load(lbuf + off, src + off, bytes, &cbar[ch]);
        }
      }
      // q(x) for the judgement, fetched while the part lands, and with the
      // first row the next request's ticket.
      float qx = 1.f;
      if (tid == 0 && !greedy && pos < gamma && P.q)
        qx = valid ? __ldg(P.q + (long long)(c0 + pos) * V + x) : 0.f;
      int ticket = -1;
      if (pos == 0 && rank == 0 && tid == 0) ticket = (int)atomicAdd(P.queue_ctl, 1u);
      float vmax = -INFINITY, vmc = 0.f, s = 0.f;
      int imax = kNoIndex;
      uint4 mvec = make_uint4(0u, 0u, 0u, 0u);
      bool landed_all = true;
      for (int ch = 0; ch < nch; ++ch) {
        const bool landed = mbar_wait(&cbar[ch], rows_done & 1u);
        if (!__syncthreads_and(landed ? 1 : 0)) {
          landed_all = false;
          // this chunk and the later ones: wait (bounded) once more for them
          for (int k = ch; k < nch; ++k) mbar_wait(&cbar[k], rows_done & 1u);
          break;
        }
        const uint4* buf = reinterpret_cast<const uint4*>(lbuf + (size_t)ch * kResChunkBytes);
        const int cj0 = j0 + ch * (kResChunkBytes / esize);
        const int cbytes = (int)min((uint32_t)kResChunkBytes, pbytes - (uint32_t)ch * kResChunkBytes);
        const int nvec = cbytes / 16;
        constexpr uint32_t pad = BF16 ? 0xFF80FF80u : 0xFF800000u;
        uint4 v[kResVecPerThread];
#pragma unroll
        for (int k = 0; k < kResVecPerThread; ++k) {
          const int idx = tid + k * kResThreads;
          v[k] = idx < nvec ? buf[idx] : make_uint4(pad, pad, pad, pad);
        }
        float m32;
        uint32_t vm[kResVecPerThread];
        if (BF16) {
#pragma unroll
          for (int k = 0; k < kResVecPerThread; ++k) {
            const __nv_bfloat162 h =
                __hmax2(__hmax2(u32_as_bf162(v[k].x), u32_as_bf162(v[k].y)),
                        __hmax2(u32_as_bf162(v[k].z), u32_as_bf162(v[k].w)));
            memcpy(&vm[k], &h, sizeof h);
          }
          __nv_bfloat162 h = u32_as_bf162(vm[0]);
#pragma unroll
          for (int k = 1; k < kResVecPerThread; ++k) h = __hmax2(h, u32_as_bf162(vm[k]));
          m32 = fmaxf(__low2float(h), __high2float(h));
        } else {
#pragma unroll
          for (int k = 0; k < kResVecPerThread; ++k)
            vm[k] = __float_as_uint(
                fmaxf(fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                      fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
          m32 = __uint_as_float(vm[0]);
#pragma unroll
          for (int k = 1; k < kResVecPerThread; ++k) m32 = fmaxf(m32, __uint_as_float(vm[k]));
        }
        if (m32 > vmax || (imax == kNoIndex && m32 > -INFINITY)) {
          // New running max: rescale the sum, remember the vector holding it.
          const float nmc = __fmul_rn(m32, c);
          if (soft && vmax > -INFINITY) s = __fmul_rn(s, ex2(__fsub_rn(vmc, nmc)));
          int kk = kResVecPerThread - 1;
#pragma unroll
          for (int k = kResVecPerThread - 2; k >= 0; --k) {
            const float mk = BF16 ? fmaxf(bf16_lo(vm[k]), bf16_hi(vm[k])) : __uint_as_float(vm[k]);
            if (mk == m32) kk = k;
          }
          uint4 vk = v[kResVecPerThread - 1];
#pragma unroll
          for (int k = kResVecPerThread - 2; k >= 0; --k)
            if (k == kk) vk = v[k];
          vmax = m32;
          vmc = nmc;
          imax = cj0 + (tid + kk * kResThreads) * epc;
          mvec = vk;
        }
        if (soft && vmax > -INFINITY) {
          const unsigned long long c2 = f2_pack(c, c);
          const unsigned long long nmc2 = f2_pack(-vmc, -vmc);
          unsigned long long acc0 = 0ull, acc1 = 0ull;
#pragma unroll
          for (int k = 0; k < kResVecPerThread; ++k) {
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            if (BF16) {
#pragma unroll
              for (int t4 = 0; t4 < 4; ++t4) {
                const unsigned long long x2 = f2_pack(bf16_lo(w[t4]), bf16_hi(w[t4]));
                float z0, z1;
                f2_unpack(f2_fma(x2, c2, nmc2), z0, z1);
                const unsigned long long e2 = f2_pack(ex2(z0), ex2(z1));
                if (t4 & 1) acc1 = f2_add(acc1, e2); else acc0 = f2_add(acc0, e2);
              }
            } else {
#pragma unroll
              for (int t4 = 0; t4 < 4; t4 += 2) {
                const unsigned long long x2 =
                    f2_pack(__uint_as_float(w[t4]), __uint_as_float(w[t4 + 1]));
                float z0, z1;
                f2_unpack(f2_fma(x2, c2, nmc2), z0, z1);
                const unsigned long long e2 = f2_pack(ex2(z0), ex2(z1));
                if (t4 & 2) acc1 = f2_add(acc1, e2); else acc0 = f2_add(acc0, e2);
              }
            }
          }
          float a0, a1, a2, a3;
          f2_unpack(acc0, a0, a1);
          f2_unpack(acc1, a2, a3);
          s = __fadd_rn(s, __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3)));
        }
        // The draft token's logit, captured by the thread that holds it.
        const int dx = x - cj0;
        if (dx >= 0 && dx < cbytes / esize) {
          const int vx = dx / epc;
          if ((vx % kResThreads) == tid) {
            const int k = vx / kResThreads;
            uint4 vk = v[0];
#pragma unroll
            for (int t4 = 1; t4 < kResVecPerThread; ++t4)
              if (t4 == k) vk = v[t4];
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
      ++rows_done;
      if (!landed_all) {
        if (tid == 0) atomicOr(P.status, SPEC_STATUS_TIMEOUT);
        ok = false;
        break;
      }
      // ---- 2. the part's statistics, then the whole row's ----
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
      __syncthreads();
      m = red_m[0];
      a = red_i[0];
      for (int w = 1; w < kResWarps; ++w) argmax_combine(m, a, red_m[w], red_i[w]);
      const float mc = __fmul_rn(m, c);
      float part = 0.f;
      if (soft && vmax > -INFINITY && m > -INFINITY) part = __fmul_rn(s, ex2(__fsub_rn(vmc, mc)));
      part = warp_sum(part);
      if (lane == 0) red_s[warp] = part;
      __syncthreads();
      ResSlot rec = mine;
      if (tid == 0) {
        float z = 0.f;
        if (soft)
          for (int w = 0; w < kResWarps; ++w) z += red_s[w];
        rec.m = m;
        rec.z = z;
        rec.argmax = a;
        rec.lx = s_has_lx ? s_lx : 0.f;
        rec.has_lx = s_has_lx;
        rec.req = ticket;
        s_has_lx = 0;
      }
      if (!res_exchange(slots, xbar, xe, rank, C, rec)) {
        ok = false;
        break;
      }
      const ResSlot* rs = res_records(slots, xe);
      ++xe;
      if (pos == 0) {
        r = rs[0].req;
        need_ticket = false;
      }
      float mm = -INFINITY, lxx = 0.f;
      int aa = kNoIndex;
      for (uint32_t k = 0; k < C; ++k) {
        argmax_combine(mm, aa, rs[k].m, rs[k].argmax);
        if (rs[k].has_lx) lxx = rs[k].lx;
      }
      float zz = 0.f;
      if (soft) {
        const float mmc = __fmul_rn(mm, c);
        for (uint32_t k = 0; k < C; ++k)
          if (rs[k].argmax != kNoIndex && rs[k].m > -INFINITY)
            zz = __fadd_rn(zz, __fmul_rn(rs[k].z, ex2(__fsub_rn(__fmul_rn(rs[k].m, c), mmc))));
      }
      const int amax = (aa == kNoIndex) ? 0 : aa;
      unsigned st = 0;
      if (!greedy) {
        if (mm == INFINITY || !(zz == zz)) st |= SPEC_STATUS_NONFINITE;
        else if (mm == -INFINITY) st |= SPEC_STATUS_NO_FINITE;
      }
      // ---- 3. the judgement (as k_accept and early exit take it) ----
      if (!greedy && st) {
        // Unusable target row: nothing is emitted for this request.
        if (lead) {
          atomicOr(P.status, st);
          for (int i = 0; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
          if (P.p_at_draft)
            for (int i = 0; i < gamma; ++i) P.p_at_draft[c0 + i] = 0.f;
          P.num_accepted[cur] = 0;
        }
        break;
      }
      int k = gamma;
      if (pos < gamma) {
        // One thread judges (the test runs in float64, which is slow here)
        // and tells the others.
        if (tid == 0) {
          bool acc;
          float pa;
          if (greedy) {
            acc = (x == amax);
            pa = acc ? 1.f : 0.f;
          } else {
            pa = valid ? exp2f(fmaf(lxx, c, -__fmul_rn(mm, c))) / zz : 0.f;
            const double u = accept_uniform(P.seed, greq, pos);
            acc = (qx > 0.f) && ((double)pa / (double)qx >= u);
          }
          s_acc = acc ? 1 : 0;
          if (lead) {
            if (!valid) atomicOr(P.status, SPEC_STATUS_BAD_TOKEN);
            if (P.p_at_draft) P.p_at_draft[c0 + pos] = pa;
            if (acc) P.out_tokens[row] = x;
          }
        }
        __syncthreads();
        if (s_acc) continue;
        k = pos;
      }
      // ---- the round ends at k = pos: the argmax, or the race ----
      int tok = amax;
      if (!greedy) {
        int mode;
        if (k < gamma) {
          if (P.flags & SPEC_FLAG_NAIVE) mode = kRaceP;
          else if (P.q) mode = kRaceResidual;
          else mode = valid ? kRaceMasked : kRaceP;
        } else {
          mode = kRaceP;
        }
        const RaceView v = race_view(P, cur, (int)row, c0 + k, k, mode, (k < gamma) ? x : -1, mm,
                                     c, 1.f / zz, -INFINITY, zz);
        // A one-hot draft's token is masked by giving it logit -inf here.
        const bool mask_here = (mode == kRaceMasked && x >= j0 && x < j0 + n);
        uint32_t saved = 0u;
        if (mask_here && tid == 0) {
          if (BF16) {
            saved = reinterpret_cast<unsigned short*>(lbuf)[x - j0];
            reinterpret_cast<unsigned short*>(lbuf)[x - j0] = 0xFF80u;
          } else {
            saved = reinterpret_cast<uint32_t*>(lbuf)[x - j0];
            reinterpret_cast<float*>(lbuf)[x - j0] = -INFINITY;
          }
        }
        bool rok = true;
        // The argmax token's score bounds the winner's from below.
        unsigned long long packed = res_race<BF16>(P, v, mode, lbuf, qring, qbar, q_phase, queue,
                                                   j0, n, amax, &s_seed, rok);
        if (mask_here && tid == 0) {
          if (BF16) reinterpret_cast<unsigned short*>(lbuf)[x - j0] = (unsigned short)saved;
          else reinterpret_cast<uint32_t*>(lbuf)[x - j0] = saved;
        }
        __syncthreads();
        if (!rok) {
          if (tid == 0) atomicOr(P.status, SPEC_STATUS_TIMEOUT);
          ok = false;
          break;
        }
        ResSlot br = mine;
        br.best = packed;
        if (!res_exchange(slots, xbar, xe, rank, C, br)) {
          ok = false;
          break;
        }
        const ResSlot* bs = res_records(slots, xe);
        ++xe;
        unsigned long long win = 0ull;
        for (uint32_t q = 0; q < C; ++q) win = bs[q].best > win ? bs[q].best : win;
        if (win == 0ull) {
          // Every weight was 0 (rounding only): draw from p over the row.
          const RaceView vp = race_view(P, cur, (int)row, c0 + k, k, kRaceP, -1, mm, c,
                                        1.f / zz, -INFINITY, zz);
          br.best = res_race<BF16>(P, vp, kRaceP, lbuf, qring, qbar, q_phase, queue, j0, n, -1,
                                   &s_seed, rok);
          if (!res_exchange(slots, xbar, xe, rank, C, br)) {
            ok = false;
            break;
          }
          const ResSlot* ps = res_records(slots, xe);
          ++xe;
          for (uint32_t q = 0; q < C; ++q) win = ps[q].best > win ? ps[q].best : win;
          if (lead) atomicOr(P.status, SPEC_STATUS_EMPTY_RESIDUAL);
        }
        tok = win ? (int)(0xFFFFFFFFu - (uint32_t)(win & 0xFFFFFFFFull)) : 0;
      }
      if (lead) {
        P.out_tokens[row] = tok;
        for (int i = k + 1; i <= gamma; ++i) P.out_tokens[row0 + i] = -1;
        if (P.p_at_draft)
          for (int i = k + 1; i < gamma; ++i) P.p_at_draft[c0 + i] = __int_as_float(0x7FC00000);
        P.num_accepted[cur] = k;
      }
      break;
    }
  }
  // Leave together: no CTA exits while another may still write into it.
  __syncthreads();
  cluster_sync_all();
}

}  // namespace sv
