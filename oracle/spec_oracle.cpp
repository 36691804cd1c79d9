// Speculative-sampling verifier: plain, slow, single-threaded CPU ORACLE.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
// execute this file; only the test-suite, the smoke check and the CPU
// baseline leg of the benchmark use it. It shares no source, header, table
// or helper with the CUDA library: the Philox generator below is written
// here a second time, from its published definition.
//
// Everything is computed in IEEE double from exactly decoded inputs
// (bf16 -> float -> double, float -> double). Each step follows, in order,
// the method as the source pages state it:
//
//  [cortexys]  "초안 모델로 생성 속도를 높이는 추측 디코딩", section 방법
//              (Algorithm 1: draft, parallel target pass, left-to-right verify)
//  [velog]     "vLLM speculative decoding이 기각 토큰을 다시 뽑는 이유",
//              sections "드래프트가 제안하고 타깃이 판정한다" (accept rule),
//              "왜 하필 max(p − q, 0)인가" (residual law, App. A.1),
//              "vLLM 커널은 이 규칙을 어떻게 옮겼나" (float64 uniforms,
//              exponential race, sampling constraints before the judgement),
//              "기본값 greedy 드래프트에서도 분포가 지켜질까" (one-hot draft,
//              temperature 0 argmax match)
//  [mlxcel]    "투기적 디코딩", section 기본 라운드 (1..K+1 tokens per round),
//              section "mlxcel의 프롬프트 조회" (sampler-match acceptance)
//
// Readings where the pages leave a step open are stated at the function
// that takes them.
//
// Parity pins (what ties this oracle to something other than itself):
//  - Philox4x32-10: the Random123 known-answer vectors (tests/golden).
//  - accept rule + residual law: exhaustive exact enumeration, V<=4, gamma<=2.
//  - exponential race: chi-square against w/sum(w); zero weights never win.
//  - top-k / top-p sets: brute force sort + cumulative sum on small V.
//  - the 5-token worked example of [velog] "Java로 규칙을 재현해 본 결과".
//  - E[tokens per round] = (1 - a^(g+1)) / (1 - a) of [cortexys] 식 1.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <limits>

extern "C" {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11). Ten rounds; each round multiplies counter words
// 0 and 2 by the published constants, crosses the halves, and mixes the key;
// the key is advanced by the published Weyl increments between rounds.
// ---------------------------------------------------------------------------
void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                      uint32_t out[4]) {
  const uint64_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = mul0 * (uint64_t)c0;
    uint64_t prod1 = mul1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// Counter layout used by the verifier: (c0, position, request, tag); the key
// is the 64-bit seed. Tag 0 = accept uniforms, tag 1 = race uniforms.
static const uint32_t OR_TAG_ACCEPT = 0u;
static const uint32_t OR_TAG_RACE = 1u;

static void or_draw(uint64_t seed, uint32_t c0, uint32_t position,
                    uint32_t request, uint32_t tag, uint32_t out[4]) {
  uint32_t ctr[4] = {c0, position, request, tag};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  or_philox4x32_10(ctr, key, out);
}

// Accept uniform u in (0,1) as a double ([velog] "vLLM 커널은 이 규칙을 어떻게
// 옮겼나": the uniforms are float64 so that u = 0 cannot let a p = 0 token
// through). Reading: the top 52 bits of the first two words give m, and
// u = (2m + 1) * 2^-53, which is exact in double and never 0 or 1.
double or_accept_uniform(uint64_t seed, int64_t request, int32_t position) {
  uint32_t w[4];
  or_draw(seed, 0u, (uint32_t)position, (uint32_t)request, OR_TAG_ACCEPT, w);
  uint64_t bits = ((uint64_t)w[0] << 32) | (uint64_t)w[1];
  uint64_t m52 = bits >> 12;
  return (2.0 * (double)m52 + 1.0) * std::ldexp(1.0, -53);
}

// Race uniform U_j in (0,1) for vocabulary entry j of the row at `position`:
// word (j mod 4) of the draw with c0 = j / 4. U = (2 (w >> 9) + 1) 2^-24 is
// exact in float, so E = -ln U is never 0 and never infinite.
float or_race_uniform(uint64_t seed, int64_t request, int32_t position,
                      int64_t j) {
  uint32_t w[4];
  or_draw(seed, (uint32_t)(j >> 2), (uint32_t)position, (uint32_t)request,
          OR_TAG_RACE, w);
  uint32_t word = w[j & 3];
  double u = (2.0 * (double)(word >> 9) + 1.0) * std::ldexp(1.0, -24);
  return (float)u;  // exact: 24 significant bits
}

// ---------------------------------------------------------------------------
// Input decoding: bf16 is the high half of an IEEE float.
// ---------------------------------------------------------------------------
double or_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double or_logit(const void* logits, int dtype, int64_t row, int V,
                       int j) {
  int64_t at = row * (int64_t)V + j;
  if (dtype == 1) return or_bf16_to_double(((const uint16_t*)logits)[at]);
  return (double)((const float*)logits)[at];
}

// ---------------------------------------------------------------------------
// Temperature 0: the argmax, lowest index among equal maxima ([velog]
// "기본값 greedy 드래프트에서도 분포가 지켜질까": temperature-0 requests are
// judged by argmax agreement only).
// ---------------------------------------------------------------------------
int or_argmax(const double* l, int V) {
  int best = 0;
  for (int j = 1; j < V; ++j)
    if (l[j] > l[best]) best = j;
  return best;
}

typedef struct {
  double m;            // max logit of the row
  int argmax;          // lowest index attaining m
  int n_kept;          // tokens with p > 0 after top-k and top-p
  double theta;        // smallest kept logit value (-inf when nothing cut)
  double z_kept;       // sum over kept tokens of exp((l - m) / T)
  double topp_margin;  // relative margin of the top-p boundary decision
  int status;          // 0 ok; 1 non-finite input; 2 no finite logit
} or_row_info;

// ---------------------------------------------------------------------------
// Sampling constraints -> p  ([velog] "vLLM 커널은 이 규칙을 어떻게 옮겼나":
// temperature, top-k and top-p are applied to the target logits before the
// judgement; p is the distribution after the sampling settings).
//
// Readings (the page defers the order to an article that is not given):
//  * temperature first; top-k compares raw logits (the same order as the
//    tempered ones for T > 0); top-p acts on the tempered distribution after
//    it has been renormalised over the top-k set.
//  * top-k keeps every token whose logit is >= the k-th largest logit
//    (ties at the boundary are all kept); k <= 0 or k >= V disables it.
//  * top-p keeps token j iff the probability mass of kept tokens with a
//    strictly larger logit is < top_p; top_p >= 1 disables it. Equal logits
//    are therefore kept or dropped together.
//  * p is renormalised over the finally kept set.
// Returns status (0 ok).
// ---------------------------------------------------------------------------
int or_target_probs(const double* l, int V, double T, int top_k, double top_p,
                    double* p, or_row_info* info) {
  info->status = 0;
  info->topp_margin = std::numeric_limits<double>::infinity();
  for (int j = 0; j < V; ++j) {
    if (std::isnan(l[j]) || l[j] == std::numeric_limits<double>::infinity()) {
      info->status = 1;
      return 1;
    }
  }
  int am = or_argmax(l, V);
  double m = l[am];
  info->m = m;
  info->argmax = am;
  if (!(m > -std::numeric_limits<double>::infinity())) {
    info->status = 2;
    return 2;
  }

  // top-k on raw logits.
  std::vector<char> keep(V, 1);
  if (top_k > 0 && top_k < V) {
    std::vector<double> sorted(l, l + V);
    std::sort(sorted.begin(), sorted.end(), std::greater<double>());
    double kth = sorted[top_k - 1];
    for (int j = 0; j < V; ++j) keep[j] = (l[j] >= kth) ? 1 : 0;
  }

  // Tempered, top-k renormalised distribution.
  std::vector<double> e(V, 0.0);
  double zk = 0.0;
  for (int j = 0; j < V; ++j) {
    if (keep[j]) {
      e[j] = std::exp((l[j] - m) / T);
      zk += e[j];
    }
  }

  // top-p over distinct logit values, largest first.
  if (top_p < 1.0) {
    std::vector<int> order;
    for (int j = 0; j < V; ++j)
      if (keep[j]) order.push_back(j);
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return l[a] > l[b]; });
    double above = 0.0;  // mass of kept tokens with a strictly larger logit
    double last_kept_above = -1.0;
    double first_dropped_above = -1.0;
    size_t g = 0;
    bool cutting = false;
    while (g < order.size()) {
      size_t h = g;
      double group_mass = 0.0;
      while (h < order.size() && l[order[h]] == l[order[g]]) {
        group_mass += e[order[h]] / zk;
        ++h;
      }
      if (!cutting && above < top_p) {
        last_kept_above = above;
      } else {
        if (!cutting) first_dropped_above = above;
        cutting = true;
        for (size_t t = g; t < h; ++t) keep[order[t]] = 0;
      }
      above += group_mass;
      g = h;
    }
    double margin = (top_p - last_kept_above) / top_p;
    if (first_dropped_above >= 0.0)
      margin = std::min(margin, (first_dropped_above - top_p) / top_p);
    info->topp_margin = margin;
  }

  double z = 0.0;
  int n_kept = 0;
  double theta = std::numeric_limits<double>::infinity();
  for (int j = 0; j < V; ++j) {
    if (keep[j]) {
      z += e[j];
      ++n_kept;
      theta = std::min(theta, l[j]);
    }
  }
  bool all_kept = (n_kept == V);
  for (int j = 0; j < V; ++j) p[j] = keep[j] ? e[j] / z : 0.0;
  info->n_kept = n_kept;
  info->theta = all_kept ? -std::numeric_limits<double>::infinity() : theta;
  info->z_kept = z;
  return 0;
}

// ---------------------------------------------------------------------------
// Accept test ([velog] "드래프트가 제안하고 타깃이 판정한다" and "vLLM 커널은 이
// 규칙을 어떻게 옮겼나"): accept x iff q(x) > 0 and p(x) / q(x) >= u, the
// ratio taken as an IEEE double division.
// ---------------------------------------------------------------------------
int or_accept(double p_x, double q_x, double u) {
  return (q_x > 0.0 && p_x / q_x >= u) ? 1 : 0;
}

// Residual weights at a rejected position ([velog] "왜 하필 max(p − q, 0)인가"):
// w = max(p - q, 0). With a one-hot (greedy) draft ([velog] "기본값 greedy
// 드래프트에서도 분포가 지켜질까") q is the indicator of x, so w is p with the
// draft token masked out. mode: 0 = probabilistic (q given), 1 = one-hot at x,
// 2 = naive control (w = p; biased, used only as a negative control, [velog]
// "Java로 규칙을 재현해 본 결과").
void or_residual_weights(const double* p, const double* q, int x, int mode,
                         int V, double* w) {
  for (int j = 0; j < V; ++j) {
    if (mode == 0) {
      w[j] = std::max(p[j] - q[j], 0.0);
    } else if (mode == 1) {
      w[j] = (j == x) ? 0.0 : p[j];
    } else {
      w[j] = p[j];
    }
  }
}

// Exponential race ([velog] "vLLM 커널은 이 규칙을 어떻게 옮겼나"): the index of
// the largest w_j / E_j with E_j ~ Exp(1) is a draw proportional to w, with
// no normalising sum. E_j = -ln U_j from the race stream of this row; the
// lowest index wins ties (strict comparison). Entries with w_j = 0 cannot win.
// Returns the winner, or -1 when every weight is 0. *margin receives
// (s1 - s2) / s1 for the two best scores (inf when only one is positive).
int or_race(const double* w, int V, uint64_t seed, int64_t request,
            int32_t position, double* margin) {
  int best = -1;
  double s1 = 0.0, s2 = 0.0;
  for (int j = 0; j < V; ++j) {
    if (!(w[j] > 0.0)) continue;
    double U = (double)or_race_uniform(seed, request, position, j);
    double E = -std::log(U);
    double s = w[j] / E;
    if (best < 0 || s > s1) {
      s2 = s1;
      s1 = s;
      best = j;
    } else if (s > s2) {
      s2 = s;
    }
  }
  if (margin) {
    *margin = (best >= 0 && s2 > 0.0) ? (s1 - s2) / s1
                                      : std::numeric_limits<double>::infinity();
  }
  return best;
}

// ---------------------------------------------------------------------------
// One verification call over a ragged batch.
// ---------------------------------------------------------------------------
typedef struct {
  int B;
  int V;
  const int* cu_num_draft;      // [B+1], gamma_r = cu[r+1] - cu[r]
  const int* draft_token_ids;   // [N]
  const void* target_logits;    // [(N+B) x V]; rows of r at cu[r]+r .. cu[r+1]+r
  int logits_dtype;             // 0 = float32, 1 = bf16 bits (uint16)
  const float* draft_probs;     // [N x V] or NULL (one-hot draft at x)
  const float* temperature;     // [B]
  const int* top_k;             // [B] or NULL
  const float* top_p;           // [B] or NULL
  uint64_t seed;
  int64_t request_base;         // global index of request 0 (RNG key)
  unsigned flags;               // bit 0: naive resample-from-p control
                                // bit 1: sampler-match acceptance
                                // bit 2: early exit (rows after the first
                                //        rejection are never examined)
} or_batch;

// Per-call outputs and the decision log used to excuse near-tie decisions.
typedef struct {
  int* out_tokens;          // [N+B], -1 beyond the emitted tokens
  int* num_accepted;        // [B]
  double* p_at_draft;       // [N] p_i(x_i) (indicator of the argmax at T = 0)
  double* accept_margin;    // [N] |p/q - u| / u of each judged position
  double* topp_margin;      // [N+B] per target row
  double* race_margin;      // [B]
  unsigned* req_status;     // [B] bit 0 non-finite, bit 1 no finite logit,
                            //     bit 2 bad token id, bit 3 empty residual
  double* row_race_margin;  // [N+B] margin of the race drawn on each target
                            //       row (+inf where no race was drawn)
} or_outputs;

static void or_verify_one(const or_batch* b, int r, const or_outputs* o) {
  const int V = b->V;
  const int c0 = b->cu_num_draft[r];
  const int gamma = b->cu_num_draft[r + 1] - c0;
  const int64_t row0 = (int64_t)c0 + r;  // first target row of request r
  const int64_t greq = b->request_base + r;
  // Reading: a temperature that is not > 0 (0, negative, NaN) takes the
  // temperature-0 path.
  const double T = (double)b->temperature[r];
  const int tk = b->top_k ? b->top_k[r] : 0;
  const double tp = b->top_p ? (double)b->top_p[r] : 1.0;
  const double inf = std::numeric_limits<double>::infinity();
  unsigned status = 0;

  for (int s = 0; s <= gamma; ++s) {
    o->out_tokens[row0 + s] = -1;
    o->topp_margin[row0 + s] = inf;
    o->row_race_margin[row0 + s] = inf;
  }
  for (int i = 0; i < gamma; ++i) o->accept_margin[c0 + i] = inf;
  o->race_margin[r] = inf;
  o->num_accepted[r] = 0;

  std::vector<double> l(V), p(V), q(V), w(V);
  std::vector<int> argmax_row(gamma + 1, 0);
  auto load_row = [&](int s) {
    for (int j = 0; j < V; ++j)
      l[j] = or_logit(b->target_logits, b->logits_dtype, row0 + s, V, j);
  };
  auto draft = [&](int i) { return b->draft_token_ids[c0 + i]; };
  auto valid = [&](int x) { return x >= 0 && x < V; };
  for (int i = 0; i < gamma; ++i)
    if (!valid(draft(i))) status |= 4u;

  // Early exit ([velog] "드래프트가 제안하고 타깃이 판정한다": the first
  // rejection ends the round, the later positions are discarded): the rows
  // are examined in position order and the scan stops at the first
  // rejection, so no row after it is read. Reading: an unusable row after
  // the stop therefore does not void the request, and p_i(x_i) is left
  // unset (NaN) for the positions after the stop. Every decision taken is
  // the one below.
  const bool early = (b->flags & 4u) != 0 && !(b->flags & 2u);
  int k_star = gamma;
  bool stopped = false;  // early exit: the scan already found k_star

  // The accept test of position i (step 2), once its row has been examined.
  auto judge = [&](int i) -> bool {
    const int x = draft(i);
    if (!(T > 0.0)) return x == argmax_row[i];
    const double p_x = o->p_at_draft[c0 + i];
    const double q_x = b->draft_probs
                           ? (valid(x) ? (double)b->draft_probs[(int64_t)(c0 + i) * V + x] : 0.0)
                           : 1.0;
    const double u = or_accept_uniform(b->seed, greq, i);
    if (q_x > 0.0) o->accept_margin[c0 + i] = std::fabs(p_x / q_x - u) / u;
    return or_accept(p_x, q_x, u) != 0;
  };

  // Step 1: the target pass over all gamma+1 rows ([cortexys] 방법: the
  // target evaluates every candidate position in one parallel pass). Every
  // draft position gets p_i(x_i), whether or not the scan reaches it.
  for (int i = 0; i <= gamma && !stopped; ++i) {
    load_row(i);
    if (!(T > 0.0)) {
      argmax_row[i] = or_argmax(l.data(), V);
      if (i < gamma) o->p_at_draft[c0 + i] = (draft(i) == argmax_row[i]) ? 1.0 : 0.0;
      if (early && i < gamma && !judge(i)) {
        k_star = i;
        stopped = true;
      }
      continue;
    }
    or_row_info info;
    int st = or_target_probs(l.data(), V, T, tk, tp, p.data(), &info);
    if (st != 0) {
      // Unusable row (NaN / +inf / no finite logit): nothing is emitted.
      o->req_status[r] = status | ((st == 1) ? 1u : 2u);
      return;
    }
    o->topp_margin[row0 + i] = info.topp_margin;
    if (i < gamma) o->p_at_draft[c0 + i] = valid(draft(i)) ? p[draft(i)] : 0.0;
    if (early && i < gamma && !judge(i)) {
      k_star = i;
      stopped = true;
    }
  }

  // Sampler-match acceptance ([mlxcel] "투기적 디코딩", section "mlxcel의
  // 프롬프트 조회"): at every position the target's own sampler draws a fresh
  // token y_i from p_i; the draft is accepted iff it equals y_i, and the first
  // mismatch (or the end of the block) emits y_i. Readings: the draw is the
  // same exponential race over w = p_i, keyed by position i (so y_gamma is
  // exactly the bonus draw of the rejection rule); draft_probs is not read
  // (the rule never looks at q); temperature-0 requests keep the argmax
  // match, which is the same rule with the argmax as the sampler.
  if ((b->flags & 2u) && T > 0.0) {
    int k_match = gamma;
    for (int i = 0; i <= gamma; ++i) {
      load_row(i);
      or_row_info info;
      or_target_probs(l.data(), V, T, tk, tp, p.data(), &info);
      double margin;
      const int y = or_race(p.data(), V, b->seed, greq, i, &margin);
      o->row_race_margin[row0 + i] = margin;
      o->out_tokens[row0 + i] = y;
      if (i == gamma || draft(i) != y) {
        k_match = i;
        o->race_margin[r] = margin;
        break;
      }
    }
    o->num_accepted[r] = k_match;
    o->req_status[r] = status;
    return;
  }

  // Step 2: left-to-right accept scan; stop at the first rejection (already
  // done above under early exit).
  if (!early) {
    for (int i = 0; i < gamma; ++i) {
      if (!judge(i)) {
        k_star = i;
        break;
      }
    }
  }

  // Step 3: the token at k*: the argmax at temperature 0; otherwise a race
  // over the residual (first rejection) or over p (bonus, all accepted).
  int out_token;
  if (!(T > 0.0)) {
    out_token = argmax_row[k_star];
  } else {
    load_row(k_star);
    or_row_info info;
    or_target_probs(l.data(), V, T, tk, tp, p.data(), &info);
    if (k_star < gamma) {
      int x = draft(k_star);
      int mode;
      if (b->flags & 1u) {
        mode = 2;
      } else if (b->draft_probs) {
        mode = 0;
        for (int j = 0; j < V; ++j)
          q[j] = (double)b->draft_probs[(int64_t)(c0 + k_star) * V + j];
      } else {
        mode = valid(x) ? 1 : 2;
      }
      or_residual_weights(p.data(), q.data(), x, mode, V, w.data());
    } else {
      // Reading: the bonus token is drawn with the same race, w = p.
      for (int j = 0; j < V; ++j) w[j] = p[j];
    }
    double margin;
    out_token = or_race(w.data(), V, b->seed, greq, k_star, &margin);
    if (out_token < 0) {
      // Every residual weight is 0 (reachable only through rounding).
      // Reading: fall back to w = p and record it.
      status |= 8u;
      out_token = or_race(p.data(), V, b->seed, greq, k_star, &margin);
    }
    o->race_margin[r] = margin;
    o->row_race_margin[row0 + k_star] = margin;
  }

  for (int i = 0; i < k_star; ++i) o->out_tokens[row0 + i] = draft(i);
  o->out_tokens[row0 + k_star] = out_token;
  o->num_accepted[r] = k_star;
  o->req_status[r] = status;
}

// Verify every request of the batch. Returns 0.
int or_verify(const or_batch* b, const or_outputs* o) {
  for (int r = 0; r < b->B; ++r) or_verify_one(b, r, o);
  return 0;
}

// Verify only the listed requests (outputs of the others are left as they
// are). Used to check sampled requests of batches too large to run whole.
int or_verify_requests(const or_batch* b, const int* reqs, int n_reqs,
                       const or_outputs* o) {
  for (int t = 0; t < n_reqs; ++t) {
    int r = reqs[t];
    if (r < 0 || r >= b->B) return -1;
    or_verify_one(b, r, o);
  }
  return 0;
}

}  // extern "C"
