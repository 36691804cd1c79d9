// C ABI of the verifier library (declared in include/spec_verify.h): handle
// and workspace management, host-side argument checks, and the launch
// sequence of one verification call.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/spec_verify.h"
#include "accept.cuh"
#include "common.cuh"
#include "philox.cuh"
#include "race.cuh"
#include "resident.cuh"
#include "rows.cuh"
#include "rows_tma.cuh"
#include "select.cuh"
#include "shard.cuh"

struct spec_verify_handle {
  spec_verify_config cfg;
  int sm_count;
  void* ws;  // one allocation for everything below
  sv::RowStats* rows;
  sv::SlicePartial* partials;
  unsigned* row_counter;
  sv::RaceDesc* race;
  unsigned long long* race_best;
  sv::RaceTask* race_list;
  unsigned* race_count;  // [3]: races listed, rows left to the slow kernel, row tickets
  long long* pending_rows;
  long long* queue;      // early exit: [q_cap] items
  unsigned* queue_ready;  // [q_cap]
  unsigned* queue_ctl;    // [kQueueCtl]
  int q_cap;
  sv::PartStat* part_stats;  // [max_batch x kMaxParts] (NULL: rows are not split)
  unsigned* part_done;       // [max_batch]
  void* part_hist;           // [max_batch] WinHist
  unsigned* status;
  int max_slices;
  cudaEvent_t phase[4];
  int n_phase;
  int tma_blocks;   // resident CTAs of k_rows_tma<.., false> on the device
  int filt_blocks;  // resident CTAs of k_rows_tma<true, true>
  int res_clusters[4];  // co-resident clusters of k_resident with 1, 2, 4, 8 CTAs
};

namespace {

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// Shared-memory sizes of every row-pass instantiation (current device).
bool set_row_pass_smem() {
  const int plain = (int)sv::kTmaSmemBytes, filt = (int)sv::kTmaFiltSmemBytes;
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  return cudaFuncSetAttribute(sv::k_rows_select, a, (int)sv::kSelSmemBytes) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, false>, a, plain) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<false, false>, a, plain) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, true>, a, filt) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, false, true>, a, plain) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<false, false, true>, a, plain) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, true, true>, a, filt) == cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, false, false, true>, a, plain) ==
             cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<false, false, false, true>, a, plain) ==
             cudaSuccess &&
         cudaFuncSetAttribute(sv::k_rows_tma<true, true, false, true>, a, filt) == cudaSuccess;
}

// Early exit in clusters: the shared memory of k_resident and how many
// clusters of 1, 2, 4 and 8 CTAs fit on the device at once (0: none).
void resident_setup(int out[4]) {
  for (int i = 0; i < 4; ++i) out[i] = 0;
  const int smem = (int)sv::kResSmemBytes;
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if (cudaFuncSetAttribute(sv::k_resident<true>, a, smem) != cudaSuccess ||
      cudaFuncSetAttribute(sv::k_resident<false>, a, smem) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  for (int i = 0; i < 4; ++i) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(1u << i);
    cfg.blockDim = dim3(sv::kResThreads);
    cfg.dynamicSmemBytes = sv::kResSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1u << i;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sv::k_resident<true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    out[i] = n;
  }
}

// Cluster size (1, 2, 4 or 8; 0: the batch cannot take the resident path)
// for rows of V elements of esize bytes: the fewest CTAs whose parts fit,
// doubled while the batch's requests all still run at once, so that small
// batches spread each row over more SMs.
int resident_cluster(const spec_verify_handle* h, int V, int esize, int B, int& part) {
  int i = 0;
  for (; i < 4; ++i) {
    const int C = 1 << i;
    const long long S = (((long long)V + C - 1) / C + 7) / 8 * 8;
    if (S * esize <= sv::kResPartBytes && h->res_clusters[i] > 0) break;
  }
  if (i == 4) return 0;
  while (i < 3 && h->res_clusters[i + 1] > 0 && (long long)B <= h->res_clusters[i + 1]) ++i;
  const int C = 1 << i;
  part = (int)((((long long)V + C - 1) / C + 7) / 8 * 8);
  return C;
}

// Control words of the early-exit queue, and its slots beyond one per row
// part: each persistent CTA takes one more ticket than it gets items.
constexpr size_t kQueueCtl = 4;
constexpr size_t kQueueSpare = 1024;
// Early exit splits a row into parts of about this many bytes (at most
// sv::kMaxParts) so that each judged row spreads over several SMs: rows with
// top-k / top-p (slow per element) in parts of ~128 KB, the others in parts
// of ~512 KB (measured: smaller parts only add per-part overhead there).
constexpr long long kPartTarget = 512 * 1024;
constexpr long long kPartTargetFiltered = 128 * 1024;

// Launch a kernel that depends on the previous one in the stream with
// programmatic dependent launch: it may be launched while that kernel runs
// (after its pdl_trigger) and waits in pdl_wait for its completion, so the
// launch latency between the kernels of one call overlaps the previous
// kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int check_batch(const spec_verify_config* cfg, const spec_verify_batch* b, bool greedy) {
  if (!cfg || !b) return SPEC_ERR_INVALID_ARG;
  if (b->B < 0 || b->N < 0 || b->V < 1) return SPEC_ERR_INVALID_ARG;
  if (b->logits_dtype != SPEC_F32 && b->logits_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (b->B == 0) return SPEC_OK;
  if (!b->cu_num_draft || !b->target_logits || !b->out_tokens || !b->num_accepted)
    return SPEC_ERR_INVALID_ARG;
  if (b->N > 0 && !b->draft_token_ids) return SPEC_ERR_INVALID_ARG;
  if (!greedy && !b->temperature) return SPEC_ERR_INVALID_ARG;
  if (!greedy) {
    const unsigned known = SPEC_FLAG_NAIVE | SPEC_FLAG_SAMPLER_MATCH | SPEC_FLAG_EARLY_EXIT;
    if ((b->flags & ~known) ||
        ((b->flags & SPEC_FLAG_SAMPLER_MATCH) &&
         (b->flags & (SPEC_FLAG_NAIVE | SPEC_FLAG_EARLY_EXIT))))
      return SPEC_ERR_INVALID_ARG;
  }
  if (b->B > cfg->max_batch || b->V > cfg->max_vocab ||
      (long long)b->N + b->B > cfg->max_rows)
    return SPEC_ERR_CAPACITY;
  return SPEC_OK;
}

// Where draft_probs lives: device (or managed) memory, or page-locked host
// memory that the device reads in place (its device alias is used; the race
// then reads those rows with plain loads). Pageable host memory is rejected.
int resolve_q(sv::Params& P) {
  P.q_host = 0;
  if (!P.q) return SPEC_OK;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, P.q) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeHost) {
    if (!a.devicePointer) return SPEC_ERR_INVALID_ARG;
    P.q = static_cast<const float*>(a.devicePointer);
    P.q_host = 1;
  } else if (a.type == cudaMemoryTypeUnregistered) {
    return SPEC_ERR_INVALID_ARG;
  }
  return SPEC_OK;
}

// The kernel parameters of a call: the batch and the handle's workspace.
sv::Params make_params(spec_verify_handle* h, const spec_verify_batch* b, bool greedy) {
  sv::Params P;
  std::memset(&P, 0, sizeof P);
  P.B = b->B;
  P.V = b->V;
  P.N = b->N;
  P.cu = b->cu_num_draft;
  P.ids = b->draft_token_ids;
  P.logits = b->target_logits;
  P.bf16 = (b->logits_dtype == SPEC_BF16) ? 1 : 0;
  P.q = greedy ? nullptr : b->draft_probs;
  P.q_host = 0;
  P.temp = b->temperature;
  P.top_k = greedy ? nullptr : b->top_k;
  P.top_p = greedy ? nullptr : b->top_p;
  P.seed = b->seed;
  P.req_base = b->request_base;
  P.flags = greedy ? 0u : b->flags;
  P.greedy_call = greedy ? 1 : 0;
  P.fast_filtered = 0;
  P.out_tokens = b->out_tokens;
  P.num_accepted = b->num_accepted;
  P.p_at_draft = b->p_at_draft;
  P.rows = h->rows;
  P.partials = h->partials;
  P.row_counter = h->row_counter;
  P.race = h->race;
  P.race_best = h->race_best;
  P.race_list = h->race_list;
  P.race_count = h->race_count;
  P.pending_rows = h->pending_rows;
  P.pending_count = h->race_count + 1;
  P.early = (!greedy && (b->flags & SPEC_FLAG_EARLY_EXIT)) ? 1 : 0;
  P.test_stall = (h->cfg.flags & SPEC_CONFIG_TEST_WAIT_TIMEOUT) ? 1 : 0;
  P.queue = h->queue;
  P.queue_ready = h->queue_ready;
  P.queue_ctl = h->queue_ctl;
  P.q_cap = h->q_cap;
  P.parts = 1;
  P.part_bytes = 0;
  P.part_stats = h->part_stats;
  P.part_done = h->part_done;
  P.part_hist = h->part_hist;
  P.status = h->status;
  const int slice = P.bf16 ? sv::kSliceBf16 : sv::kSliceF32;
  P.slices_per_row = (b->V + slice - 1) / slice;
  const int rslice = sv::race_slice(P.q != nullptr);
  P.race_slice_n = rslice;
  P.race_slices = (b->V + rslice - 1) / rslice;
  P.v0 = 0;
  P.Vg = b->V;
  return P;
}

int launch(spec_verify_handle* h, const spec_verify_batch* b, cudaStream_t stream, bool greedy) {
  if (!h) return SPEC_ERR_NOT_INIT;
  int rc = check_batch(&h->cfg, b, greedy);
  if (rc != SPEC_OK) return rc;
  if (b->B == 0) return SPEC_OK;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return SPEC_ERR_CUDA;

  sv::Params P = make_params(h, b, greedy);
  rc = resolve_q(P);
  if (rc != SPEC_OK) return rc;
  const long long R = (long long)b->N + b->B;
  const bool match = !greedy && (P.flags & SPEC_FLAG_SAMPLER_MATCH);
  // Races: one per request (its k* row), or one per row under sampler-match.
  const long long races = match ? R : (long long)b->B;
  // Too few race tasks to give every SM two: smaller slices (the race of a
  // small batch is latency-bound, so more CTAs finish it sooner).
  while (P.race_slice_n > sv::kRaceSliceMin && races * P.race_slices < 2ll * h->sm_count) {
    P.race_slice_n /= 2;
    P.race_slices = (b->V + P.race_slice_n - 1) / P.race_slice_n;
  }
  if (R * P.slices_per_row > 0x7FFFFFFFll || races * P.race_slices > 0x7FFFFFFFll)
    return SPEC_ERR_CAPACITY;
  const bool timed = h->n_phase >= 4;
  if (timed) cudaEventRecord(h->phase[0], stream);
  if (!greedy && cudaMemsetAsync(h->race_count, 0, 3 * sizeof(unsigned), stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const int esize = P.bf16 ? 2 : 4;
  const bool rows_aligned = (((long long)b->V * esize) % 16 == 0) &&
                            ((reinterpret_cast<uintptr_t>(b->target_logits) & 15) == 0);
  const bool filters = !greedy && (P.top_k || P.top_p);
  P.fast_filtered = (rows_aligned && h->tma_blocks > 0 && h->filt_blocks > 0 && P.bf16 &&
                     filters) ? 1 : 0;
  if (P.early) {
    // Handles created with SPEC_CONFIG_EARLY_RESIDENT, rows without top-k /
    // top-p: each request in a cluster that keeps the judged row in shared
    // memory (rows 16-byte aligned and at most 8 parts of 64 KB, draft
    // probabilities in device memory and 16-byte aligned).
    int part = 0;
    const int C = ((h->cfg.flags & SPEC_CONFIG_EARLY_RESIDENT) && !filters && rows_aligned &&
                   !P.q_host && !P.test_stall &&
                   (!P.q || (reinterpret_cast<uintptr_t>(P.q) & 15) == 0))
                      ? resident_cluster(h, b->V, esize, b->B, part)
                      : 0;
    if (C > 0) {
      P.res_part = part;
      const int fit = h->res_clusters[C == 1 ? 0 : C == 2 ? 1 : C == 4 ? 2 : 3];
      const int ncl = b->B < fit ? b->B : fit;
      if (cudaMemsetAsync(h->queue_ctl, 0, kQueueCtl * sizeof(unsigned), stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof cfg);
      cfg.gridDim = dim3((unsigned)(ncl * C));
      cfg.blockDim = dim3(sv::kResThreads);
      cfg.dynamicSmemBytes = sv::kResSmemBytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const cudaError_t e = P.bf16 ? cudaLaunchKernelEx(&cfg, sv::k_resident<true>, P)
                                   : cudaLaunchKernelEx(&cfg, sv::k_resident<false>, P);
      if (timed) {
        // one kernel: its time is the rows phase
        cudaEventRecord(h->phase[1], stream);
        cudaEventRecord(h->phase[2], stream);
        cudaEventRecord(h->phase[3], stream);
      }
      if (e != cudaSuccess || cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
      }
      return SPEC_OK;
    }
    // The work queue pays off when the batch's requests can keep every SM
    // busy; otherwise (and for rows the bulk copies cannot take) the full
    // pass runs and the accept scan applies the same early-exit semantics.
    const int qblocks = P.fast_filtered ? h->filt_blocks : h->tma_blocks;
    const bool queue_ok = rows_aligned && h->tma_blocks > 0 && (!filters || P.fast_filtered);
    const bool big = (long long)b->B >= 2ll * qblocks;
    if (!queue_ok || !(big || (h->cfg.flags & SPEC_CONFIG_EARLY_QUEUE)) ||
        (h->cfg.flags & SPEC_CONFIG_EARLY_FULL_PASS))
      P.early = 0;
  }
  // Early exit: split each row into parts of about the target size (whole
  // stages) when the workspace has room for it. The queue takes every row
  // part plus one closing ticket per CTA; whole rows that still do not fit
  // take the full pass instead.
  int parts = 1;
  long long part_bytes = (long long)b->V * esize;
  if (P.early) {
    const long long row_bytes = (long long)b->V * esize;
    const long long stage = P.fast_filtered ? sv::tma_stage_bytes(true) : sv::tma_stage_bytes(false);
    const long long target = P.fast_filtered ? kPartTargetFiltered : kPartTarget;
    parts = (int)((row_bytes + target - 1) / target);
    parts = parts < 1 ? 1 : (parts > sv::kMaxParts ? sv::kMaxParts : parts);
    part_bytes = ((row_bytes + parts - 1) / parts + stage - 1) / stage * stage;
    parts = (int)((row_bytes + part_bytes - 1) / part_bytes);
    const long long tickets = (long long)(P.fast_filtered ? h->filt_blocks : h->tma_blocks);
    if (!h->part_stats || R * parts + tickets > h->q_cap) parts = 1;
    if (R + tickets > h->q_cap) P.early = 0;
  }
  if (P.early) {
    // Rows from the work queue, judged as they finish; no accept kernel.
    P.parts = parts;
    P.part_bytes = parts > 1 ? part_bytes : (long long)b->V * esize;
    if (cudaMemsetAsync(h->queue_ctl, 0, kQueueCtl * sizeof(unsigned), stream) != cudaSuccess ||
        cudaMemsetAsync(h->queue_ready, 0, (size_t)h->q_cap * sizeof(unsigned), stream) !=
            cudaSuccess)
      return SPEC_ERR_CUDA;
    if (parts > 1 &&
        (cudaMemsetAsync(h->part_done, 0, (size_t)b->B * sizeof(unsigned), stream) != cudaSuccess ||
         (filters && cudaMemsetAsync(h->part_hist, 0, (size_t)b->B * sizeof(sv::WinHist),
                                     stream) != cudaSuccess)))
      return SPEC_ERR_CUDA;
    sv::k_early_init<<<(b->B + 255) / 256, 256, 0, stream>>>(P);
    const int blocks = P.fast_filtered ? h->filt_blocks : h->tma_blocks;
    const long long items = (long long)b->B * parts;  // in flight at most
    const int grid = items < blocks ? (int)items : blocks;
    if (P.fast_filtered)
      launch_after(sv::k_rows_tma<true, true, true>, grid, sv::kTmaThreads, sv::kTmaFiltSmemBytes,
                   stream, P, R);
    else if (P.bf16)
      launch_after(sv::k_rows_tma<true, false, true>, grid, sv::kTmaThreads, sv::kTmaSmemBytes,
                   stream, P, R);
    else
      launch_after(sv::k_rows_tma<false, false, true>, grid, sv::kTmaThreads, sv::kTmaSmemBytes,
                   stream, P, R);
    if (timed) {
      cudaEventRecord(h->phase[1], stream);
      cudaEventRecord(h->phase[2], stream);
    }
    launch_after(sv::k_race, (unsigned)(races * P.race_slices), sv::kRaceThreads,
                 sv::race_smem_bytes(P.bf16 ? 2 : 4, P.q != nullptr), stream, P);
    launch_after(sv::k_race_token, (unsigned)races, sv::kRaceThreads, 0, stream, P);
    if (timed) cudaEventRecord(h->phase[3], stream);
    if (cudaPeekAtLastError() != cudaSuccess) {
      cudaGetLastError();
      return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
  }
  // Rows after the row pass's first wave go by ticket when there are any
  // (the counter was cleared with the race counters; greedy calls keep the
  // stride order).
  if (P.fast_filtered) {
    // One pass over every row; the filtered rows it cannot settle are listed.
    const long long fgrid = R < h->filt_blocks ? R : h->filt_blocks;
    if (!greedy && R > fgrid) P.row_ticket = h->race_count + 2;
    sv::k_rows_tma<true, true><<<(unsigned)fgrid, sv::kTmaThreads, sv::kTmaFiltSmemBytes,
                                 stream>>>(P, R);
  } else if (rows_aligned && h->tma_blocks > 0) {
    const long long grid = R < h->tma_blocks ? R : h->tma_blocks;
    if (!greedy && R > grid) P.row_ticket = h->race_count + 2;
    if (P.bf16)
      sv::k_rows_tma<true, false><<<(unsigned)grid, sv::kTmaThreads, sv::kTmaSmemBytes, stream>>>(
          P, R);
    else
      sv::k_rows_tma<false, false><<<(unsigned)grid, sv::kTmaThreads, sv::kTmaSmemBytes,
                                     stream>>>(P, R);
  } else {
    sv::k_rows_stream<<<(unsigned)(R * P.slices_per_row), sv::kStreamThreads, 0, stream>>>(P);
  }
  if (filters) {
    // Every filtered row (one block each), settled from a histogram of its
    // truncated values; or only the rows the streaming pass listed.
    const long long cap = 2ll * h->sm_count;
    const long long sgrid = P.fast_filtered ? (R < cap ? R : cap) : R;
    if (!P.fast_filtered)
      launch_after(sv::k_rows_select, (unsigned)R, sv::kSelThreads, sv::kSelSmemBytes, stream, P);
    else
      launch_after(sv::k_rows_filtered, (unsigned)sgrid, sv::kFilterThreads, 0, stream, P);
  }
  if (timed) cudaEventRecord(h->phase[1], stream);
  launch_after(sv::k_accept, (unsigned)((b->B + sv::kAcceptWarps - 1) / sv::kAcceptWarps),
               sv::kAcceptWarps * 32, 0, stream, P);
  if (timed) cudaEventRecord(h->phase[2], stream);
  if (!greedy) {
    launch_after(sv::k_race, (unsigned)(races * P.race_slices), sv::kRaceThreads,
                 sv::race_smem_bytes(P.bf16 ? 2 : 4, P.q != nullptr), stream, P);
    launch_after(sv::k_race_token, (unsigned)races, sv::kRaceThreads, 0, stream, P);
    if (match)
      launch_after(sv::k_match, (unsigned)((b->B + sv::kAcceptWarps - 1) / sv::kAcceptWarps),
                   sv::kAcceptWarps * 32, 0, stream, P);
  }
  if (timed) cudaEventRecord(h->phase[3], stream);
  if (cudaPeekAtLastError() != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_verify_check_batch(const spec_verify_config* cfg, const spec_verify_batch* b) {
  return check_batch(cfg, b, false);
}

int spec_verify_init(spec_verify_handle** out, const spec_verify_config* cfg) {
  if (!out) return SPEC_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || cfg->max_batch < 1 || cfg->max_rows < 1 || cfg->max_vocab < 1)
    return SPEC_ERR_INVALID_ARG;
  if (cfg->max_rows < cfg->max_batch) return SPEC_ERR_INVALID_ARG;
  if (cfg->flags & ~(SPEC_CONFIG_TEST_WAIT_TIMEOUT | SPEC_CONFIG_EARLY_QUEUE |
                     SPEC_CONFIG_EARLY_FULL_PASS | SPEC_CONFIG_EARLY_RESIDENT))
    return SPEC_ERR_INVALID_ARG;
  if ((cfg->flags & SPEC_CONFIG_EARLY_RESIDENT) &&
      (cfg->flags & (SPEC_CONFIG_EARLY_QUEUE | SPEC_CONFIG_EARLY_FULL_PASS)))
    return SPEC_ERR_INVALID_ARG;
  if (cudaSetDevice(cfg->device) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return SPEC_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return SPEC_ERR_UNSUPPORTED;

  spec_verify_handle* h = new (std::nothrow) spec_verify_handle();
  if (!h) return SPEC_ERR_CUDA;
  h->cfg = *cfg;
  h->sm_count = prop.multiProcessorCount;
  int per_sm = 0;
  int filt_per_sm = 0;
  if (!set_row_pass_smem() ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv::k_rows_tma<true, false>,
                                                    sv::kTmaThreads,
                                                    sv::kTmaSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    per_sm = 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&filt_per_sm, sv::k_rows_tma<true, true>,
                                                    sv::kTmaThreads,
                                                    sv::kTmaFiltSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    filt_per_sm = 0;
  }
  h->tma_blocks = per_sm * prop.multiProcessorCount;
  h->filt_blocks = filt_per_sm * prop.multiProcessorCount;
  resident_setup(h->res_clusters);
  if (cudaFuncSetAttribute(sv::k_race, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sv::kRaceSmemMax) != cudaSuccess) {
    delete h;
    return SPEC_ERR_CUDA;
  }
  h->max_slices = (cfg->max_vocab + sv::kSliceF32 - 1) / sv::kSliceF32;

  const size_t n_rows = (size_t)cfg->max_rows, n_b = (size_t)cfg->max_batch;
  const size_t sz_rows = align_up(n_rows * sizeof(sv::RowStats));
  const size_t sz_part = align_up(n_rows * h->max_slices * sizeof(sv::SlicePartial));
  const size_t sz_rcnt = align_up(n_rows * sizeof(unsigned));
  // Race slots and tasks: one per row covers sampler-match batches.
  const size_t sz_race = align_up(n_b * sizeof(sv::RaceDesc));
  const size_t sz_best = align_up(n_rows * sizeof(unsigned long long));
  const size_t sz_list = align_up(n_rows * sizeof(sv::RaceTask));
  const size_t sz_lcnt = align_up(3 * sizeof(unsigned));
  const size_t sz_pend = align_up(n_rows * sizeof(long long));
  const size_t qcap = n_rows * sv::kMaxParts + kQueueSpare;
  const size_t sz_queue = align_up(qcap * sizeof(long long));
  const size_t sz_qready = align_up(qcap * sizeof(unsigned));
  const size_t sz_qctl = align_up(kQueueCtl * sizeof(unsigned));
  const size_t sz_pstat = align_up(n_b * sv::kMaxParts * sizeof(sv::PartStat));
  const size_t sz_pdone = align_up(n_b * sizeof(unsigned));
  const size_t sz_phist = align_up(n_b * sizeof(sv::WinHist));
  const size_t sz_stat = align_up(sizeof(unsigned));
  const size_t total = sz_rows + sz_part + sz_rcnt + sz_race + sz_best + sz_list +
                       sz_lcnt + sz_pend + sz_queue + sz_qready + sz_qctl + sz_pstat + sz_pdone +
                       sz_phist + sz_stat;
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    delete h;
    return SPEC_ERR_CUDA;
  }
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return SPEC_ERR_CUDA;
  }
  char* p = (char*)h->ws;
  h->rows = (sv::RowStats*)p; p += sz_rows;
  h->partials = (sv::SlicePartial*)p; p += sz_part;
  h->row_counter = (unsigned*)p; p += sz_rcnt;
  h->race = (sv::RaceDesc*)p; p += sz_race;
  h->race_best = (unsigned long long*)p; p += sz_best;
  h->race_list = (sv::RaceTask*)p; p += sz_list;
  h->race_count = (unsigned*)p; p += sz_lcnt;
  h->pending_rows = (long long*)p; p += sz_pend;
  h->queue = (long long*)p; p += sz_queue;
  h->queue_ready = (unsigned*)p; p += sz_qready;
  h->queue_ctl = (unsigned*)p; p += sz_qctl;
  h->q_cap = (int)qcap;
  h->part_stats = (sv::PartStat*)p; p += sz_pstat;
  h->part_done = (unsigned*)p; p += sz_pdone;
  h->part_hist = p; p += sz_phist;
  h->status = (unsigned*)p;
  *out = h;
  return SPEC_OK;
}

int spec_verify_run(spec_verify_handle* h, const spec_verify_batch* b, void* stream) {
  return launch(h, b, (cudaStream_t)stream, false);
}

int spec_verify_greedy(spec_verify_handle* h, const spec_verify_batch* b, void* stream) {
  return launch(h, b, (cudaStream_t)stream, true);
}

int spec_verify_status(spec_verify_handle* h, unsigned* bits) {
  if (!h) return SPEC_ERR_NOT_INIT;
  if (!bits) return SPEC_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPEC_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaMemset(h->status, 0, sizeof v) != cudaSuccess) return SPEC_ERR_CUDA;
  *bits = v;
  return v ? SPEC_ERR_DEVICE_STATUS : SPEC_OK;
}

int spec_verify_set_phase_events(spec_verify_handle* h, void* const* events, int n) {
  if (!h) return SPEC_ERR_NOT_INIT;
  if (n == 0) {
    h->n_phase = 0;
    return SPEC_OK;
  }
  if (n < 4 || !events) return SPEC_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return SPEC_ERR_INVALID_ARG;
    h->phase[i] = (cudaEvent_t)events[i];
  }
  h->n_phase = 4;
  return SPEC_OK;
}

void spec_verify_destroy(spec_verify_handle* h) {
  if (!h) return;
  cudaSetDevice(h->cfg.device);
  cudaDeviceSynchronize();
  cudaFree(h->ws);
  delete h;
}

// ---------------------------------------------------------------------------
// Vocab-sharded verification (the protocol is in include/spec_verify.h).
// ---------------------------------------------------------------------------
static int shard_setup(spec_verify_handle* h, const spec_verify_batch* b, const spec_shard* sh,
                       sv::Params& P, bool& filters) {
  if (!h) return SPEC_ERR_NOT_INIT;
  if (!sh) return SPEC_ERR_INVALID_ARG;
  int rc = check_batch(&h->cfg, b, false);
  if (rc != SPEC_OK) return rc;
  if (b->flags) return SPEC_ERR_UNSUPPORTED;
  if (sh->v0 < 0 || (sh->v0 & 3) || sh->V_global < 1 || sh->v0 + b->V > sh->V_global ||
      sh->V_global > 0x7FFFFFFF - 8)
    return SPEC_ERR_INVALID_ARG;
  if (b->B == 0) return SPEC_OK;
  const long long esize = (b->logits_dtype == SPEC_BF16) ? 2 : 4;
  filters = b->top_k || b->top_p;
  const bool aligned = ((long long)b->V * esize) % 16 == 0 &&
                       (reinterpret_cast<uintptr_t>(b->target_logits) & 15) == 0;
  if (!aligned || h->tma_blocks <= 0 || (filters && (esize != 2 || h->filt_blocks <= 0)))
    return SPEC_ERR_UNSUPPORTED;
  if (!sh->m || !sh->z || !sh->argmax || !sh->lx || !sh->best || !sh->best_p ||
      (b->draft_probs && !sh->qx) || (filters && (!sh->hist || !sh->hist_w)))
    return SPEC_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return SPEC_ERR_CUDA;
  P = make_params(h, b, false);
  rc = resolve_q(P);
  if (rc != SPEC_OK) return rc;
  P.shard = 1;
  P.v0 = (int)sh->v0;
  P.Vg = sh->V_global;
  P.sh_m = sh->m;
  P.sh_z = sh->z;
  P.sh_arg = sh->argmax;
  P.sh_lx = sh->lx;
  P.sh_qx = b->draft_probs ? sh->qx : nullptr;
  P.sh_hist = sh->hist;
  P.sh_hist_w = sh->hist_w;
  P.sh_best = sh->best;
  P.sh_skip = nullptr;
  return SPEC_OK;
}

static int launched() {
  if (cudaPeekAtLastError() != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

int spec_verify_shard_rows(spec_verify_handle* h, const spec_verify_batch* b,
                           const spec_shard* sh, void* stream) {
  sv::Params P;
  bool filters = false;
  int rc = shard_setup(h, b, sh, P, filters);
  if (rc != SPEC_OK || b->B == 0) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const long long R = (long long)b->N + b->B;
  if (filters) {
    const long long grid = R < h->filt_blocks ? R : h->filt_blocks;
    sv::k_rows_tma<true, true, false, true><<<(unsigned)grid, sv::kTmaThreads,
                                               sv::kTmaFiltSmemBytes, s>>>(P, R);
  } else {
    const long long grid = R < h->tma_blocks ? R : h->tma_blocks;
    if (P.bf16)
      sv::k_rows_tma<true, false, false, true><<<(unsigned)grid, sv::kTmaThreads,
                                                  sv::kTmaSmemBytes, s>>>(P, R);
    else
      sv::k_rows_tma<false, false, false, true><<<(unsigned)grid, sv::kTmaThreads,
                                                   sv::kTmaSmemBytes, s>>>(P, R);
  }
  return launched();
}

int spec_verify_shard_rescale(spec_verify_handle* h, const spec_verify_batch* b,
                              const spec_shard* sh, void* stream) {
  sv::Params P;
  bool filters = false;
  int rc = shard_setup(h, b, sh, P, filters);
  if (rc != SPEC_OK || b->B == 0) return rc;
  const long long R = (long long)b->N + b->B;
  const long long n = R > b->N ? R : b->N;
  sv::k_shard_rescale<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(P);
  return launched();
}

int spec_verify_shard_judge(spec_verify_handle* h, const spec_verify_batch* b,
                            const spec_shard* sh, void* stream) {
  sv::Params P;
  bool filters = false;
  int rc = shard_setup(h, b, sh, P, filters);
  if (rc != SPEC_OK || b->B == 0) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const long long R = (long long)b->N + b->B;
  if ((long long)b->B * P.race_slices > 0x7FFFFFFFll) return SPEC_ERR_CAPACITY;
  sv::k_shard_finish<<<(unsigned)R, sv::kShardFinishThreads, filters ? sizeof(sv::WinHist) : 0,
                       s>>>(P);
  if (cudaMemsetAsync(h->race_count, 0, 2 * sizeof(unsigned), s) != cudaSuccess ||
      cudaMemsetAsync(sh->best, 0, (size_t)b->B * sizeof(unsigned long long), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  sv::k_accept<<<(b->B + sv::kAcceptWarps - 1) / sv::kAcceptWarps, sv::kAcceptWarps * 32, 0, s>>>(
      P);
  sv::k_race<<<(unsigned)((long long)b->B * P.race_slices), sv::kRaceThreads,
               sv::race_smem_bytes(P.bf16 ? 2 : 4, P.q != nullptr), s>>>(P);
  sv::k_race_token<<<(unsigned)b->B, sv::kRaceThreads, 0, s>>>(P);
  return launched();
}

int spec_verify_shard_race_p(spec_verify_handle* h, const spec_verify_batch* b,
                             const spec_shard* sh, void* stream) {
  sv::Params P;
  bool filters = false;
  int rc = shard_setup(h, b, sh, P, filters);
  if (rc != SPEC_OK || b->B == 0) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  P.sh_skip = sh->best;
  P.sh_best = sh->best_p;
  if (cudaMemsetAsync(sh->best_p, 0, (size_t)b->B * sizeof(unsigned long long), s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  sv::k_shard_race_reset<<<(b->B + 255) / 256, 256, 0, s>>>(P);
  sv::k_race<<<(unsigned)((long long)b->B * P.race_slices), sv::kRaceThreads,
               sv::race_smem_bytes(P.bf16 ? 2 : 4, P.q != nullptr), s>>>(P);
  sv::k_race_token<<<(unsigned)b->B, sv::kRaceThreads, 0, s>>>(P);
  return launched();
}

int spec_verify_shard_emit(spec_verify_handle* h, const spec_verify_batch* b,
                           const spec_shard* sh, void* stream) {
  sv::Params P;
  bool filters = false;
  int rc = shard_setup(h, b, sh, P, filters);
  if (rc != SPEC_OK || b->B == 0) return rc;
  sv::k_shard_emit<<<(b->B + 255) / 256, 256, 0, (cudaStream_t)stream>>>(P, sh->best,
                                                                          sh->best_p);
  return launched();
}

const char* spec_verify_strerror(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_NOT_INIT: return "null handle";
    case SPEC_ERR_CAPACITY: return "batch exceeds the handle's maxima";
    case SPEC_ERR_DEVICE_STATUS: return "device status bits set";
    default: return "unknown error code";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// spec_verify_run_noalloc: the same launch sequence on a workspace carved out
// of one file-scope device array instead of cudaMalloc'ed memory.
// ---------------------------------------------------------------------------
namespace {

// Sizes of the workspace pieces at the no-allocation limits.
constexpr size_t kNaRows = SPEC_NOALLOC_MAX_ROWS;
constexpr size_t kNaBatch = SPEC_NOALLOC_MAX_BATCH;
constexpr size_t kNaSlices = (SPEC_NOALLOC_MAX_VOCAB + sv::kSliceF32 - 1) / sv::kSliceF32;
constexpr size_t na_align(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kNaOffRows = 0;
constexpr size_t kNaOffPart = kNaOffRows + na_align(kNaRows * sizeof(sv::RowStats));
constexpr size_t kNaOffRcnt = kNaOffPart + na_align(kNaRows * kNaSlices * sizeof(sv::SlicePartial));
constexpr size_t kNaOffRace = kNaOffRcnt + na_align(kNaRows * sizeof(unsigned));
constexpr size_t kNaOffBest = kNaOffRace + na_align(kNaBatch * sizeof(sv::RaceDesc));
constexpr size_t kNaOffList = kNaOffBest + na_align(kNaRows * sizeof(unsigned long long));
constexpr size_t kNaOffLcnt = kNaOffList + na_align(kNaRows * sizeof(sv::RaceTask));
constexpr size_t kNaOffPend = kNaOffLcnt + na_align(3 * sizeof(unsigned));
// Early exit without row parts: one queue slot per row, plus the spare.
constexpr size_t kNaQueueCap = kNaRows + kQueueSpare;
constexpr size_t kNaOffQueue = kNaOffPend + na_align(kNaRows * sizeof(long long));
constexpr size_t kNaOffQready = kNaOffQueue + na_align(kNaQueueCap * sizeof(long long));
constexpr size_t kNaOffQctl = kNaOffQready + na_align(kNaQueueCap * sizeof(unsigned));
constexpr size_t kNaOffStat = kNaOffQctl + na_align(kQueueCtl * sizeof(unsigned));
constexpr size_t kNaBytes = kNaOffStat + na_align(sizeof(unsigned));
static_assert(kNaBytes <= SPEC_NOALLOC_SCRATCH_BYTES, "no-allocation scratch too small");

constexpr int kNaMaxDevices = 64;
struct NoallocDevice {
  bool ready;
  char* base;  // device address of g_noalloc_scratch on this device
  int sm_count;
  int tma_blocks;
  int filt_blocks;
  int res_clusters[4];
};
NoallocDevice g_na_dev[kNaMaxDevices];
std::mutex g_na_mutex;

}  // namespace

// The scratch of spec_verify_run_noalloc (one copy per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

extern "C" int spec_verify_run_noalloc(const spec_verify_batch* b, void* stream,
                                       unsigned* device_status) {
  if (!b) return SPEC_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kNaMaxDevices) return SPEC_ERR_UNSUPPORTED;
  spec_verify_config cfg;
  cfg.device = dev;
  cfg.max_batch = SPEC_NOALLOC_MAX_BATCH;
  cfg.max_rows = SPEC_NOALLOC_MAX_ROWS;
  cfg.max_vocab = SPEC_NOALLOC_MAX_VOCAB;
  cfg.flags = 0;
  int rc = check_batch(&cfg, b, false);
  if (rc != SPEC_OK) return rc;

  NoallocDevice nd;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    NoallocDevice& slot = g_na_dev[dev];
    if (!slot.ready) {
      // Once per device, with that device current: resolve the array's
      // device address and set the kernels' shared-memory attributes.
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SPEC_ERR_CUDA;
      if (!(prop.major == 10 && prop.minor == 3)) return SPEC_ERR_UNSUPPORTED;
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
      }
      int per_sm = 0, filt_per_sm = 0;
      if (!set_row_pass_smem() ||
          cudaFuncSetAttribute(sv::k_race, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sv::kRaceSmemMax) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv::k_rows_tma<true, false>,
                                                        sv::kTmaThreads,
                                                        sv::kTmaSmemBytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&filt_per_sm, sv::k_rows_tma<true, true>,
                                                        sv::kTmaThreads,
                                                        sv::kTmaFiltSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
      }
      resident_setup(slot.res_clusters);
      slot.base = (char*)ptr;
      slot.sm_count = prop.multiProcessorCount;
      slot.tma_blocks = per_sm * prop.multiProcessorCount;
      slot.filt_blocks = filt_per_sm * prop.multiProcessorCount;
      slot.ready = true;
    }
    nd = slot;
  }
  if (b->B == 0) return SPEC_OK;

  // A handle on the stack whose workspace points into the array.
  spec_verify_handle h;
  std::memset(&h, 0, sizeof h);
  h.cfg = cfg;
  h.sm_count = nd.sm_count;
  h.ws = nd.base;
  h.rows = (sv::RowStats*)(nd.base + kNaOffRows);
  h.partials = (sv::SlicePartial*)(nd.base + kNaOffPart);
  h.row_counter = (unsigned*)(nd.base + kNaOffRcnt);
  h.race = (sv::RaceDesc*)(nd.base + kNaOffRace);
  h.race_best = (unsigned long long*)(nd.base + kNaOffBest);
  h.race_list = (sv::RaceTask*)(nd.base + kNaOffList);
  h.race_count = (unsigned*)(nd.base + kNaOffLcnt);
  h.pending_rows = (long long*)(nd.base + kNaOffPend);
  h.queue = (long long*)(nd.base + kNaOffQueue);
  h.queue_ready = (unsigned*)(nd.base + kNaOffQready);
  h.queue_ctl = (unsigned*)(nd.base + kNaOffQctl);
  h.q_cap = (int)kNaQueueCap;
  h.status = device_status ? device_status : (unsigned*)(nd.base + kNaOffStat);
  h.max_slices = (int)kNaSlices;
  h.n_phase = 0;
  h.tma_blocks = nd.tma_blocks;
  h.filt_blocks = nd.filt_blocks;
  for (int i = 0; i < 4; ++i) h.res_clusters[i] = nd.res_clusters[i];
  // The slice counters must start at zero: clear them (the array keeps the
  // previous call's contents).
  cudaStream_t s = (cudaStream_t)stream;
  const size_t rows = (size_t)b->N + (size_t)b->B;
  if (cudaMemsetAsync(h.row_counter, 0, rows * sizeof(unsigned), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return launch(&h, b, s, false);
}
