// Shared device-side definitions of the verifier library: kernel parameters,
// workspace records, element decoding and block reductions.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/spec_verify.h"

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxParts = 8;  // queue items carry (row << 3) | part
constexpr int kNoIndex = 0x7FFFFFFF;

// Row classes decided on the device from the request's sampling settings.
enum RowClass : int {
  kArgmaxOnly = 0,  // temperature 0 (or the greedy entry point)
  kSoftmax = 1,     // temperature > 0, no top-k / top-p
  kFiltered = 2,    // temperature > 0 with top-k and/or top-p
};

// Race modes written by the accept scan for the kernel that draws the token.
enum RaceMode : int {
  kRaceNone = 0,      // nothing to draw (temperature 0 or unusable request)
  kRaceResidual = 1,  // w = max(p - q, 0) with q the draft_probs row
  kRaceMasked = 2,    // one-hot draft: w = p with the draft token masked
  kRaceP = 3,         // bonus token or naive control: w = p
  kRaceMatch = 4,     // sampler-match request: a race on every row, then k_match
};

// Per target row: what the accept scan and the race need.
struct RowStats {
  float m;          // max logit of the row
  float c;          // log2(e) / T (0 on argmax-only rows)
  float inv_z;      // 1 / Z, Z = sum over kept tokens of exp((l - m) / T)
  float theta;      // a token is kept iff its logit >= theta (-inf: all kept)
  int argmax;       // lowest index of the max logit
  float p_x;        // p of the row's draft token (rows before the last)
  unsigned status;  // SPEC_STATUS_* bits found on this row
  float z;          // Z
};

// One slice of a row in the streaming pass.
struct SlicePartial {
  float m;     // max over the slice
  float s;     // sum of exp2((l - m) c) over the slice
  int argmax;  // lowest index of the slice max
  int pad;
};

// Per request: the token to draw after the accept scan.
struct RaceDesc {
  int mode;    // RaceMode
  int kstar;   // position of the drawn token (0 .. gamma)
  int x;       // draft token at kstar (masked in kRaceMasked)
  int row;     // target row of kstar (= output slot)
  int qrow;    // draft_probs row of kstar (= cu[r] + kstar)
};

// Everything one race task needs, written by the accept scan so that a race
// CTA starts its copies after a single dependent load.
struct RaceTask {
  int r;        // request
  int row;      // target row of k* (= output slot)
  int qrow;     // draft_probs row of k*
  int kstar;    // position k* (the race's Philox position)
  int mode;     // RaceMode
  int x;        // draft token at k*
  float m, c, inv_z, theta, z;  // RowStats of the row
  int slot;     // index into race_best (request, or row for sampler-match)
};

// One part of a row streamed by one CTA under early exit (rows are split
// into parts so that a request's rows, which are judged one after another,
// each spread over several SMs).
struct __align__(16) PartStat {
  float m;      // max over the part
  float z;      // sum of 2^(l c - fl(m c)) over the part (softmax / filtered rows)
  int argmax;   // lowest index of the part max (kNoIndex: none)
  float lx;     // logit at the row's draft token, if the part holds it
  int has_lx;   // 1 when lx is set
  int pad[3];
};

// Device view of one call.
struct Params {
  int B, V, N;
  const int* cu;
  const int* ids;
  const void* logits;
  int bf16;  // 1: bf16 logits, 0: fp32
  const float* q;
  int q_host;  // 1: q is page-locked host memory (read with plain loads)
  const float* temp;
  const int* top_k;
  const float* top_p;
  unsigned long long seed;
  long long req_base;
  unsigned flags;
  int greedy_call;  // 1 when called through spec_verify_greedy
  int fast_filtered;  // 1 when the streaming pass handled top-k / top-p rows
  int* out_tokens;
  int* num_accepted;
  float* p_at_draft;
  // workspace
  RowStats* rows;
  SlicePartial* partials;
  unsigned* row_counter;
  RaceDesc* race;
  unsigned long long* race_best;  // per race slot: packed (score, ~index)
  RaceTask* race_list;   // races to draw (order not fixed)
  unsigned* race_count;  // entries in race_list
  unsigned* status;
  long long* pending_rows;  // filtered rows left to the exact slow kernel
  unsigned* pending_count;  // entries in pending_rows (race_count + 1)
  unsigned* row_ticket;     // full row pass: rows after the first wave by ticket
                            // (race_count + 2; null: by stride)
  // Early exit (SPEC_FLAG_EARLY_EXIT): the row pass's work queue.
  int early;
  int test_stall;           // 1: leave the early-exit queue empty, short waits (tests)
  long long* queue;         // [q_cap] items (row << 3) | part
  unsigned* queue_ready;    // [q_cap] 1 once the slot holds its item
  unsigned* queue_ctl;      // control words, see early.cuh
  int q_cap;
  int parts;                // parts per row (1: a row stays in one CTA)
  long long part_bytes;     // bytes per part (the last one may be shorter)
  PartStat* part_stats;     // [max_batch x kMaxParts]: one row in flight per request
  unsigned* part_done;      // [max_batch] parts of the request's current row done
  void* part_hist;          // [max_batch] WinHist: merged window histograms
  int slices_per_row;
  int race_slices;
  int race_slice_n;          // entries per race task (a power of two, at most race_slice())
  int res_part;              // early exit in clusters: elements of a row per CTA
  // Vocab-sharded calls: the local columns are global v0 .. v0 + V - 1.
  int v0;                    // 0 otherwise
  int Vg;                    // the full vocabulary (V otherwise)
  int shard;                 // 1 in a sharded call
  float* sh_m;
  float* sh_z;
  int* sh_arg;
  float* sh_lx;
  float* sh_qx;
  int* sh_hist;              // [R x SPEC_SHARD_HIST_INTS]
  float* sh_hist_w;          // [R x 2]
  unsigned long long* sh_best;    // race output of a sharded call
  const unsigned long long* sh_skip;  // race on p only where this combined best is 0
};

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ __nv_bfloat162 u32_as_bf162(uint32_t w) {
  __nv_bfloat162 h;
  memcpy(&h, &w, sizeof h);
  return h;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float load_logit(const Params& P, long long row, int j) {
  const long long at = row * (long long)P.V + j;
  if (P.bf16) {
    const unsigned short b = __ldg((const unsigned short*)P.logits + at);
    return __uint_as_float((uint32_t)b << 16);
  }
  return __ldg((const float*)P.logits + at);
}

// Read-only 16-byte load that does not allocate in L1 (the rows are streamed).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Order-preserving 32-bit key of a float (-0 and +0 share the key of +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// ---------------------------------------------------------------------------
// Request lookup: the largest r with cu[r] + r <= row (rows of request r are
// cu[r] + r .. cu[r+1] + r). Valid offsets are checked by the caller.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int request_of_row(const int* cu, int B, long long row) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)__ldg(cu + mid) + mid <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int row_class(const Params& P, int r) {
  if (P.greedy_call) return kArgmaxOnly;
  const float T = __ldg(P.temp + r);
  if (!(T > 0.f)) return kArgmaxOnly;
  const int k = P.top_k ? __ldg(P.top_k + r) : 0;
  const float tp = P.top_p ? __ldg(P.top_p + r) : 1.f;
  const bool topk_on = (k > 0 && k < P.V);
  const bool topp_on = (tp < 1.f);
  return (topk_on || topp_on) ? kFiltered : kSoftmax;
}

// ---------------------------------------------------------------------------
// Block reductions (blockDim.x a multiple of 32, at most 1024)
// ---------------------------------------------------------------------------
// (max value, lowest index among equal maxima); kNoIndex marks "no element".
__device__ __forceinline__ void argmax_combine(float& v, int& i, float v2, int i2) {
  if (i2 == kNoIndex) return;
  if (i == kNoIndex || v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    argmax_combine(v, i, v2, i2);
  }
}

template <typename T>
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// Block-wide (max, argmax); result valid in every thread.
__device__ __forceinline__ void block_argmax(float& v, int& i) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_argmax(v, i);
  __syncthreads();
  if (lane == 0) { sv[warp] = v; si[warp] = i; }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  v = lane < nw ? sv[lane] : -INFINITY;
  i = lane < nw ? si[lane] : kNoIndex;
  warp_argmax(v, i);
}

template <typename T>
__device__ __forceinline__ T block_sum(T x) {
  __shared__ T s[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_sum(x);
  __syncthreads();
  if (lane == 0) s[warp] = x;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  x = lane < nw ? s[lane] : T(0);
  return warp_sum(x);
}

}  // namespace sv
