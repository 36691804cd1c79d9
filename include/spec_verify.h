/*
 * spec_verify.h — C ABI of the GB300 speculative-sampling verifier.
 *
 * One call verifies a ragged batch of draft-then-verify rounds: for request r
 * with gamma_r = cu_num_draft[r+1] - cu_num_draft[r] draft tokens it reads the
 * target's logits at gamma_r + 1 positions, applies the request's temperature,
 * top-k and top-p to get p, accepts draft token x_i while u_i <= p_i(x_i) /
 * q_i(x_i), resamples the first rejected position from norm(max(0, p - q)) by
 * the exponential race argmax_j w_j / E_j, and emits a bonus token from
 * p_{gamma+1} when every draft token is accepted. Temperature-0 requests accept
 * while the draft equals the target argmax and emit the argmax.
 *
 * Sources of the operation (web pages; titles and sections):
 *  - velog, "vLLM speculative decoding이 기각 토큰을 다시 뽑는 이유":
 *      "드래프트가 제안하고 타깃이 판정한다" (accept rule, bonus token),
 *      "왜 하필 max(p − q, 0)인가" (residual distribution, App. A.1),
 *      "vLLM 커널은 이 규칙을 어떻게 옮겼나" (output = accepted + recovered +
 *        bonus tokens; float64 uniforms; exponential race; temperature / top-k /
 *        top-p applied before the judgement),
 *      "기본값 greedy 드래프트에서도 분포가 지켜질까" (draft_probs absent = one-hot
 *        draft; temperature-0 requests judged by argmax agreement).
 *  - cortexys.team, "초안 모델로 생성 속도를 높이는 추측 디코딩", section 방법
 *      (Algorithm 1: gamma drafts, one parallel target pass over gamma + 1
 *      positions, left-to-right verification).
 *  - mlxcel, "투기적 디코딩", section 기본 라운드 (a round emits 1 .. K + 1
 *      tokens).
 *
 * Randomness. Every random number is a Philox4x32-10 draw (Salmon et al.,
 * SC'11) with key = seed and counter = (c0, position, global request, tag):
 *   accept uniform of position i:  c0 = 0, tag 0; the top 52 bits m of words
 *     0..1 give u = (2m + 1) 2^-53 in (0, 1) as a double (never 0, so a
 *     p = 0 token is never accepted);
 *   race uniform of vocabulary entry j at position k: c0 = j / 4, tag 1,
 *     word j mod 4; U = (2 (w >> 9) + 1) 2^-24 in (0, 1), E = -ln U.
 * "global request" = request_base + r, so a batch split across calls (or
 * GPUs) draws exactly what the whole batch would.
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers unless stated; the caller owns
 *    them. The library owns only the workspace it allocates in
 *    spec_verify_init (row statistics, per-request scratch, status word).
 *  - Calls are asynchronous on the given stream and never synchronise the
 *    host. Errors found on the device (bad offsets, bad token ids, non-finite
 *    logits) set bits in a device status word; nothing traps. Read the word
 *    with spec_verify_status after synchronising the stream.
 *  - Return value: SPEC_OK (0) or a negative SPEC_ERR_* code. Argument errors
 *    are detected on the host before anything is enqueued; nothing is
 *    enqueued when a call fails.
 *  - A handle is not thread-safe and its workspace serves one call at a time:
 *    use one handle per stream (calls on one stream are ordered).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)   /* null pointer, negative size, bad enum */
#define SPEC_ERR_UNSUPPORTED (-2)   /* device is not sm_103 */
#define SPEC_ERR_CUDA (-3)          /* a CUDA runtime call failed */
#define SPEC_ERR_NOT_INIT (-4)      /* null handle */
#define SPEC_ERR_CAPACITY (-5)      /* batch exceeds the handle's maxima */
#define SPEC_ERR_DEVICE_STATUS (-6) /* spec_verify_status: device bits set */

/* Device status bits (spec_verify_status). */
#define SPEC_STATUS_NONFINITE 0x1u      /* NaN or +inf logit in a T > 0 row */
#define SPEC_STATUS_NO_FINITE 0x2u      /* T > 0 row whose logits are all -inf */
#define SPEC_STATUS_BAD_TOKEN 0x4u      /* draft token id outside [0, V) */
#define SPEC_STATUS_EMPTY_RESIDUAL 0x8u /* all residual weights 0: raced on p */
#define SPEC_STATUS_BAD_OFFSETS 0x10u   /* cu_num_draft not 0 .. N, non-decreasing */
#define SPEC_STATUS_TIMEOUT 0x20u       /* an on-chip pipeline wait gave up: the
                                           outputs of the call are not valid, and
                                           the handle's workspace may be left
                                           dirty (destroy it and create another) */
#define SPEC_STATUS_UNSETTLED 0x40u     /* vocab-sharded call: a top-k / top-p row
                                           the window histogram could not settle;
                                           its request emits nothing */

/* Batch flags. */
#define SPEC_FLAG_NAIVE 0x1u /* negative control: resample rejected positions
                                from p instead of the residual (biased; for
                                tests of the statistics only) */
/* Sampler-match acceptance (mlxcel, "투기적 디코딩", section "mlxcel의 프롬프트
 * 조회"): for every temperature > 0 request the target's sampler draws a
 * fresh token y_i from p_i at each position i = 0 .. gamma (the exponential
 * race over w = p_i, keyed by position i); x_i is accepted iff x_i == y_i and
 * the first mismatch, or the end of the block, emits y_i. draft_probs is not
 * read. Lossless for any draft; for one-hot drafts it accepts x with
 * probability p(x), as the rejection rule does. Temperature-0 requests keep
 * the argmax match. Cannot be combined with SPEC_FLAG_NAIVE. */
#define SPEC_FLAG_SAMPLER_MATCH 0x2u
/* Early-exit verification (velog, "드래프트가 제안하고 타깃이 판정한다": the
 * first rejection ends the round and the later positions are discarded):
 * only the rows up to each request's first rejection count. Every emitted
 * token and count is the one the full pass gives; the differences are that
 * an unusable row (NaN, +inf, all -inf) or an invalid draft token after the
 * stop does not void the request or set a status bit, and p_at_draft is NaN
 * at the positions after the stop. Schedules, all with the same results:
 *  - when the batch has enough requests to keep every SM busy (B at least
 *    twice the row pass's resident CTAs) and its rows are 16-byte aligned
 *    (bf16 if top_k / top_p are given), the rows are read position by
 *    position from a work queue and the rows after the stop are never read;
 *    the token at the stop is drawn afterwards, reading that row again;
 *  - otherwise every row is read (faster for small batches);
 *  - on handles created with SPEC_CONFIG_EARLY_RESIDENT, batches without
 *    top_k / top_p whose rows are 16-byte aligned and at most 8 x 64 KB,
 *    with draft_probs (if given) in device memory and 16-byte aligned, are
 *    verified one request per thread-block cluster that holds the judged
 *    row in its shared memory: the rows up to the stop are read once each
 *    and the token at the stop is drawn from the row held (the fewest HBM
 *    bytes; slower than the work queue on a GPU the call has to itself).
 * Cannot be combined with SPEC_FLAG_SAMPLER_MATCH. */
#define SPEC_FLAG_EARLY_EXIT 0x4u

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef struct spec_verify_handle spec_verify_handle; /* opaque */

typedef struct {
  int device;          /* CUDA device ordinal */
  int max_batch;       /* largest B of any call */
  long long max_rows;  /* largest N + B (target rows) of any call */
  int max_vocab;       /* largest V of any call */
  unsigned flags;      /* SPEC_CONFIG_* (0 in normal use) */
} spec_verify_config;

/* Handle flags (spec_verify_config.flags). */
#define SPEC_CONFIG_EARLY_QUEUE 0x2u       /* test only: early-exit calls take the work
                                              queue whenever the rows allow it, whatever
                                              the batch size */
#define SPEC_CONFIG_EARLY_FULL_PASS 0x4u   /* test only: early-exit calls read every row
                                              and apply the early-exit semantics in the
                                              accept scan, whatever the batch */
#define SPEC_CONFIG_EARLY_RESIDENT 0x8u    /* early-exit calls whose batch allows it
                                              keep each judged row resident in a
                                              thread-block cluster (see
                                              SPEC_FLAG_EARLY_EXIT); not with the two
                                              flags above */
#define SPEC_CONFIG_TEST_WAIT_TIMEOUT 0x1u /* test only (no counterpart on the pages):
                                              early-exit calls leave their work queue
                                              empty and its waits give up after a few
                                              polls, so the call ends with
                                              SPEC_STATUS_TIMEOUT and garbage outputs;
                                              no asynchronous copy is issued */

typedef struct {
  int B;                       /* requests in the batch, >= 0 */
  int V;                       /* vocabulary size, >= 1 */
  int N;                       /* total draft tokens = cu_num_draft[B] (host copy) */
  const int* cu_num_draft;     /* [B+1] device; cu[0] = 0, non-decreasing,
                                  cu[B] = N; gamma_r = cu[r+1] - cu[r] */
  const int* draft_token_ids;  /* [N] device; x of request r, position i at
                                  cu[r] + i */
  const void* target_logits;   /* [(N+B) x V] device, row-major, dtype below;
                                  the gamma_r + 1 rows of request r are rows
                                  cu[r] + r .. cu[r+1] + r */
  spec_dtype logits_dtype;     /* SPEC_F32 or SPEC_BF16 */
  const float* draft_probs;    /* [N x V] fp32 (row cu[r] + i is q_i of
                                  request r), or NULL: one-hot greedy draft,
                                  q_i(x_i) = 1. Device memory, or page-locked
                                  host memory (cudaHostAlloc / registered),
                                  which the kernels read in place: only the
                                  gathered q_i(x_i) and the rows of rejected
                                  requests cross the host link. Pageable host
                                  memory: SPEC_ERR_INVALID_ARG. The memory
                                  must not change until the call completes. */
  const float* temperature;    /* [B] device; 0 => argmax-match path; > 0 */
  const int* top_k;            /* [B] device or NULL; <= 0 or >= V => off */
  const float* top_p;          /* [B] device or NULL; >= 1 => off; in (0, 1] */
  unsigned long long seed;     /* Philox key */
  long long request_base;      /* global index of request 0 (RNG counter) */
  unsigned flags;              /* SPEC_FLAG_* */
  int* out_tokens;             /* [N+B] device out; slots cu[r]+r .. cu[r+1]+r:
                                  the accepted drafts, then the recovered or
                                  bonus token, then -1 */
  int* num_accepted;           /* [B] device out; accepted drafts per request */
  float* p_at_draft;           /* [N] device out or NULL: p_i(x_i) for every
                                  draft position (at T = 0: 1 if x_i is the
                                  argmax else 0) */
} spec_verify_batch;

/*
 * spec_verify_init — create a handle on cfg->device and allocate its
 * workspace for batches up to the configured maxima.
 *   h   [out] receives the handle (NULL on failure).
 *   cfg [in]  host pointer; maxima must be >= 1.
 * Returns SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED (not an sm_103
 * device) or SPEC_ERR_CUDA. Synchronous.
 */
int spec_verify_init(spec_verify_handle** h, const spec_verify_config* cfg);

/*
 * spec_verify_run — verify one batch (velog sections above; cortexys 방법).
 * Every request uses its own temperature / top-k / top-p; temperature-0
 * requests take the argmax-match path, the others the probabilistic one.
 *   h [in] handle; b [in] host pointer to the batch description (device
 *   arrays inside); stream [in] a cudaStream_t (NULL = legacy default stream).
 * b->flags may hold SPEC_FLAG_NAIVE, SPEC_FLAG_SAMPLER_MATCH and
 * SPEC_FLAG_EARLY_EXIT, but SPEC_FLAG_SAMPLER_MATCH with neither of the
 * others; anything else is SPEC_ERR_INVALID_ARG.
 * Returns SPEC_OK, SPEC_ERR_NOT_INIT, SPEC_ERR_INVALID_ARG, SPEC_ERR_CAPACITY
 * or SPEC_ERR_CUDA (launch failure). Asynchronous.
 */
int spec_verify_run(spec_verify_handle* h, const spec_verify_batch* b,
                    void* stream);

/*
 * spec_verify_greedy — the temperature-0 verification for the whole batch
 * (velog, "기본값 greedy 드래프트에서도 분포가 지켜질까": accept while the draft
 * equals the target argmax; emit the argmax of the first mismatching row, or
 * of the last row). Ignores temperature, top_k, top_p, draft_probs, seed and
 * flags (those pointers may be NULL). Same returns as spec_verify_run.
 */
int spec_verify_greedy(spec_verify_handle* h, const spec_verify_batch* b,
                       void* stream);

/*
 * spec_verify_status — read and clear the device status word (a bitwise OR of
 * SPEC_STATUS_* over every call since the last read). Synchronises the
 * handle's device. *device_error_bits receives the bits (host pointer).
 * Returns SPEC_OK when no bit is set, SPEC_ERR_DEVICE_STATUS when some are,
 * SPEC_ERR_NOT_INIT or SPEC_ERR_CUDA.
 */
int spec_verify_status(spec_verify_handle* h, unsigned* device_error_bits);

/*
 * spec_verify_check_batch — the host-side argument checks of spec_verify_run,
 * without a handle or a device: null pointers, sizes, dtype, and the maxima of
 * cfg. Returns SPEC_OK, SPEC_ERR_INVALID_ARG or SPEC_ERR_CAPACITY.
 */
int spec_verify_check_batch(const spec_verify_config* cfg,
                            const spec_verify_batch* b);

/*
 * spec_verify_set_phase_events — timing hook for profiling. With n >= 4
 * events set (cudaEvent_t values cast to void*, created by the caller on the
 * handle's device), every later run / greedy call records, on its stream,
 * events[0] before its first kernel, events[1] after the target-row pass,
 * events[2] after the accept scan and events[3] after the race (equal to
 * events[2] for spec_verify_greedy). n = 0 (events may be NULL) turns the
 * hook off. The caller keeps ownership of the events.
 * Returns SPEC_OK, SPEC_ERR_NOT_INIT or SPEC_ERR_INVALID_ARG.
 */
int spec_verify_set_phase_events(spec_verify_handle* h, void* const* events, int n);

/*
 * spec_verify_run_noalloc — spec_verify_run for callers that cannot allocate
 * device memory: code running inside an allocator or memory-pool callback
 * (allocating there would re-enter the allocator), a process whose device
 * memory is all owned by another framework's caching allocator (a private
 * cudaMalloc would sit outside its budget and its pool), and latency-bound
 * loops that must not pay for cudaMalloc, which can synchronise the device.
 * It needs no handle and calls no cudaMalloc, cudaFree or allocating library
 * routine: its
 * scratch (row statistics, slice partials, race state) lives in one
 * file-scope device array of the library, SPEC_NOALLOC_SCRATCH_BYTES bytes
 * on every GPU that loads the library, held until the process exits.
 * The sources of the method have no counterpart of this entry point; it
 * computes exactly what spec_verify_run computes.
 *   b      [in]  host pointer to the batch (device arrays inside), on the
 *                current CUDA device;
 *   stream [in]  a cudaStream_t (NULL = legacy default stream);
 *   device_status [in/out] device pointer to one unsigned that receives the
 *                SPEC_STATUS_* bits of the call (OR-ed in: clear it first),
 *                or NULL to drop them.
 * Limits: B <= SPEC_NOALLOC_MAX_BATCH, N + B <= SPEC_NOALLOC_MAX_ROWS,
 * V <= SPEC_NOALLOC_MAX_VOCAB; larger batches return SPEC_ERR_CAPACITY and
 * enqueue nothing. The first call on a device resolves the array's device
 * address (cudaGetSymbolAddress) and sets kernel attributes; make that first
 * call outside any stream capture. Every call shares the one array, so calls
 * whose kernels overlap on the GPU (other streams, other threads) race and
 * give wrong results: serialise them. The counters it relies on are cleared
 * by every call. Returns SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_CAPACITY,
 * SPEC_ERR_UNSUPPORTED or SPEC_ERR_CUDA. Asynchronous.
 */
#define SPEC_NOALLOC_MAX_BATCH 2048
#define SPEC_NOALLOC_MAX_ROWS 8192
#define SPEC_NOALLOC_MAX_VOCAB 262144
#define SPEC_NOALLOC_SCRATCH_BYTES (5u << 20)
int spec_verify_run_noalloc(const spec_verify_batch* b, void* stream,
                            unsigned* device_status);

/* spec_verify_destroy — free the workspace and the handle (NULL is a no-op).
 * Synchronises the handle's device first. */
void spec_verify_destroy(spec_verify_handle* h);

/* spec_verify_strerror — static description of a return code. */
const char* spec_verify_strerror(int code);

/*
 * ---------------------------------------------------------------------------
 * Vocab-sharded (tensor-parallel) verification.
 *
 * The verification of one batch when each of n ranks holds the target
 * logits (and draft probabilities) of a contiguous slice of the vocabulary
 * only. It computes what spec_verify_run computes (velog sections above):
 * the row statistics are sums, maxima and a value histogram, so they
 * combine across slices; the exponential race is a maximum of w_j / E_j with
 * E_j keyed by the global index j, so each rank races its own columns and
 * the winners combine by a maximum. Between the calls below the caller
 * all-reduces the named spec_shard arrays over the n ranks (NCCL, gloo),
 * in this order:
 *   spec_verify_shard_rows      then all-reduce MAX: m
 *   spec_verify_shard_rescale   then all-reduce SUM: z, qx, hist, hist_w;
 *                                    MIN: argmax; MAX: lx
 *   spec_verify_shard_judge     then all-reduce MAX: best
 *   spec_verify_shard_race_p    then all-reduce MAX: best_p
 *   spec_verify_shard_emit      (out_tokens, num_accepted as spec_verify_run)
 * Every rank passes the same cu_num_draft, draft_token_ids (global ids),
 * temperature, top_k, top_p, seed and request_base; b->V is the local
 * slice width and target_logits / draft_probs hold the local columns
 * ([(N+B) x V] and [N x V]). Requirements: 16-byte aligned local rows
 * (b->V * element size a multiple of 16, aligned base), v0 a multiple of 4,
 * bf16 logits when top_k / top_p are given, no flags; otherwise
 * SPEC_ERR_UNSUPPORTED. A top-k / top-p row whose thresholds the window
 * histogram cannot settle (a threshold on a value of magnitude below 2^-16
 * or at least 2^8, or a top-k set reaching more than 30 / c below the max)
 * sets SPEC_STATUS_UNSETTLED and its request emits nothing. The caller owns
 * every array; all are device memory. The handle keeps state between the
 * five calls of one batch: one batch at a time per handle, same stream.
 * ---------------------------------------------------------------------------
 */
#define SPEC_SHARD_HIST_INTS 6148 /* ints per row of spec_shard.hist */

typedef struct {
  long long v0;        /* global index of the first local column */
  int V_global;        /* the full vocabulary size */
  float* m;            /* [N+B] local row max; the caller makes it the global max */
  float* z;            /* [N+B] sum of 2^((l - m) log2(e) / T) over the local columns
                          (T > 0 rows), rescaled to the global max by
                          spec_verify_shard_rescale */
  int* argmax;         /* [N+B] lowest global index of the local max; after the
                          rescale INT_MAX unless the local max is the global one */
  float* lx;           /* [N+B] logit at the row's draft token when it is a local
                          column, else -inf */
  float* qx;           /* [N] q(x) when x is a local column, else 0; NULL when
                          draft_probs is NULL */
  int* hist;           /* [(N+B) x SPEC_SHARD_HIST_INTS] window histogram counts of
                          top-k / top-p rows (NULL when the batch has no top_k and
                          no top_p) */
  float* hist_w;       /* [(N+B) x 2] sums of 2^(l c) of the counted values below 2^-16
                          in magnitude, negative then positive (NULL as hist) */
  unsigned long long* best;    /* [B] race winner of the local columns, (score bits
                                  << 32) | (0xFFFFFFFF - global index); 0: none */
  unsigned long long* best_p;  /* [B] the race on p for requests whose combined best
                                  is 0 (every residual weight 0); 0 otherwise */
} spec_shard;

/* spec_verify_shard_rows — local row statistics and window histograms of
 * the local columns. Same returns as spec_verify_run. */
int spec_verify_shard_rows(spec_verify_handle* h, const spec_verify_batch* b,
                           const spec_shard* sh, void* stream);
/* spec_verify_shard_rescale — with sh->m holding the global maxima: rescale
 * z to them, keep argmax only where the local max is the global one, gather
 * q(x) of local draft tokens into qx. */
int spec_verify_shard_rescale(spec_verify_handle* h, const spec_verify_batch* b,
                              const spec_shard* sh, void* stream);
/* spec_verify_shard_judge — from the combined statistics: the rows'
 * thresholds and Z, the accept scan (num_accepted and the accepted tokens
 * are final here), and the race over the local columns into best. */
int spec_verify_shard_judge(spec_verify_handle* h, const spec_verify_batch* b,
                            const spec_shard* sh, void* stream);
/* spec_verify_shard_race_p — for requests whose combined best is 0, the
 * race over p of the local columns into best_p (0 for the others). */
int spec_verify_shard_race_p(spec_verify_handle* h, const spec_verify_batch* b,
                             const spec_shard* sh, void* stream);
/* spec_verify_shard_emit — write each request's recovered / bonus token
 * from the combined best (best_p where best is 0). */
int spec_verify_shard_emit(spec_verify_handle* h, const spec_verify_batch* b,
                           const spec_shard* sh, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
