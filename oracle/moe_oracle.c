/*
 * CPU fp64 oracle for the forward pass of one sparse Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check of __graft_entry__ and
 * the CPU-baseline leg of bench.py load this library. The product (the CUDA
 * library in sparse_mixture_experts_66_b300/) never calls it, and the two share
 * no code, headers or tables.
 *
 * Inputs arrive as float32 arrays: both fp32 and bf16 stored values convert to
 * float32 and then to double exactly, so the oracle sees the same numbers as
 * the GPU. Every intermediate is double. Loops are plain: no blocking, fusion
 * or reordering beyond what the formulas state. OpenMP only splits
 * independent tokens or experts across threads; it never changes the order of
 * any sum.
 *
 * Sources, by page title and section:
 *   [WIKI]  "Mixture-of-Experts" (beta.fermi.ai wiki): the step-by-step
 *           mechanism (steps 1-7) with its pseudocode, "Communication cost in
 *           distributed settings" (C = gamma*k*T/N), the load-balancing
 *           auxiliary loss, and the worked N=4, k=2, T=5, C=2 example.
 *   [SYN]   "Mixture of Experts (MoE): Architecture, Routing, and Scaling"
 *           (syntave.com): "Core Architecture" (FFN(x) = W2*GELU(W1*x+b1)+b2,
 *           y = sum over top-k of G(x)_i * E_i(x)), "Importance Loss and Z-Loss",
 *           "Expert Choice Routing".
 *   [TGS]   "Mixture of Experts: Scaling Language Models with Sparse
 *           Activation" (tempatgunting.com): "Routing Mechanisms" (softmax,
 *           top-k, renormalise), "The Load Balancing Crisis", "Training
 *           Dynamics and Stability" (z-loss), "Expert Choice Routing".
 *   [CORE]  "Mixture of Experts: How Sparse Routing Scales Transformers"
 *           (corecocept.com): "Inside the Router" (renormalised combine).
 *
 * Pins (tests/test_oracle_pins.py): the worked capacity example, brute force
 * on tiny inputs, gates summing to 1 and equal to the softmax of the top-k
 * logits, counts_kept = min(counts_raw, C), dropped pairs contributing exactly
 * zero, N=1/k=1 against a dense FFN, k=N/no-cap against the full soft mixture,
 * GELU identities, token and expert relabelling, uniform-routing statistics.
 * Parity unpinned: none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FLAG_RENORM_SURVIVORS 1u
#define ORACLE_FLAG_IDENTITY_FALLBACK 2u
#define ORACLE_FLAG_SHARED_EXPERT 4u

/* GELU with the exact Gaussian CDF: GELU(u) = u * Phi(u) = u/2 * (1 + erf(u/sqrt 2)).
 * [SYN] "Core Architecture": the FFN's nonlinearity is GELU (nn.GELU's default,
 * which is the erf form). */
double moe_oracle_gelu(double u) { return 0.5 * u * (1.0 + erf(u / sqrt(2.0))); }

/* Step 1 of [WIKI]: router logits l[t,e] = x_t . W_g[e] (+ optional per-expert
 * logit bias, an input of the skewed workload). */
void moe_oracle_router_logits(int64_t T, int64_t d, int32_t N, const float *x, const float *w_g,
                              const float *router_bias, double *logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t e = 0; e < N; ++e) {
      double acc = 0.0;
      for (int64_t i = 0; i < d; ++i) acc += (double)x[t * d + i] * (double)w_g[(int64_t)e * d + i];
      if (router_bias) acc += (double)router_bias[e];
      logits[t * N + e] = acc;
    }
  }
}

/* Step 1 of [WIKI]: softmax over the N experts, p[t,e] = exp(l[t,e]) / sum_e' exp(l[t,e']),
 * evaluated with the row maximum subtracted (the same value, without overflow). */
void moe_oracle_softmax(int64_t T, int32_t N, const double *logits, double *probs) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + t * N;
    double m = l[0];
    for (int32_t e = 1; e < N; ++e)
      if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int32_t e = 0; e < N; ++e) s += exp(l[e] - m);
    for (int32_t e = 0; e < N; ++e) probs[t * N + e] = exp(l[e] - m) / s;
  }
}

/* Step 2 of [WIKI]: the k experts with the largest softmax score. Softmax is
 * strictly increasing in the logit, so ranking by logit selects the same
 * experts (this is also the form of the [TGS] router code, which takes top-k of
 * the logits). Ties go to the lower expert index; the k picks are listed in
 * rank order (largest first). */
void moe_oracle_topk(int64_t T, int32_t N, int32_t k, const double *logits, int32_t *idx) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + t * N;
    for (int32_t j = 0; j < k; ++j) {
      int32_t best = -1;
      for (int32_t e = 0; e < N; ++e) {
        int taken = 0;
        for (int32_t jj = 0; jj < j; ++jj)
          if (idx[t * k + jj] == e) taken = 1;
        if (taken) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower index on ties */
      }
      idx[t * k + j] = best;
    }
  }
}

/* Steps 2-3 of [WIKI]: score[t,j] = p[t, idx_j] (the softmax score of the pick)
 * and the combine weight gate[t,j] = score[t,j] / sum_j' score[t,j'], i.e. the
 * top-k scores renormalised to sum to 1 ([TGS] "Routing Mechanisms", [CORE]
 * "Inside the Router"). */
void moe_oracle_gates(int64_t T, int32_t N, int32_t k, const double *probs, const int32_t *idx,
                      double *score, double *gate) {
  for (int64_t t = 0; t < T; ++t) {
    double s = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      score[t * k + j] = probs[t * N + idx[t * k + j]];
      s += score[t * k + j];
    }
    for (int32_t j = 0; j < k; ++j) gate[t * k + j] = score[t * k + j] / s;
  }
}

/* Expert capacity, [WIKI] "Communication cost in distributed settings":
 * C = gamma * k*T/N, rounded up to a whole token. A capacity factor <= 0 or
 * infinite means no limit, i.e. C = T (no expert can receive more than T). */
int64_t moe_oracle_capacity(int64_t T, int32_t N, int32_t k, double cf) {
  if (!(cf > 0.0) || isinf(cf)) return T;
  double c = ceil(cf * (double)(T * (int64_t)k) / (double)N);
  if (c > (double)T) return T;
  return (int64_t)c;
}

typedef struct {
  double score;
  int64_t t;
  int32_t j;
} oracle_request;

/* Higher score first; equal scores: lower token first. */
static int request_order(const void *pa, const void *pb) {
  const oracle_request *a = (const oracle_request *)pa, *b = (const oracle_request *)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  if (a->t < b->t) return -1;
  if (a->t > b->t) return 1;
  return 0;
}

static int request_token_order(const void *pa, const void *pb) {
  const oracle_request *a = (const oracle_request *)pa, *b = (const oracle_request *)pb;
  return (a->t > b->t) - (a->t < b->t);
}

/* Step 4 of [WIKI] and its worked example: an expert accepts at most C of the
 * requests routed to it; when more arrive, the lowest-scoring ones are dropped
 * for that expert. Equal scores: the lower token index is kept.
 * Outputs per expert: counts_raw (requests), counts_kept (accepted), and per
 * request slot[t,j] = the rank of the pair among the expert's accepted
 * requests in ascending token order (the order of the pseudocode's
 * expert_buffer), or -1 when dropped. */
void moe_oracle_capacity_assign(int64_t T, int32_t N, int32_t k, int64_t C, const int32_t *idx,
                                const double *score, int32_t *counts_raw, int32_t *counts_kept,
                                int32_t *slot) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t e = 0; e < N; ++e) {
    int64_t n = 0;
    for (int64_t i = 0; i < T * k; ++i)
      if (idx[i] == e) ++n;
    oracle_request *req = (oracle_request *)malloc(sizeof(oracle_request) * (size_t)(n > 0 ? n : 1));
    int64_t m = 0;
    for (int64_t t = 0; t < T; ++t)
      for (int32_t j = 0; j < k; ++j)
        if (idx[t * k + j] == e) {
          req[m].score = score[t * k + j];
          req[m].t = t;
          req[m].j = j;
          ++m;
        }
    qsort(req, (size_t)n, sizeof(oracle_request), request_order);
    int64_t keep = n < C ? n : C;
    for (int64_t r = keep; r < n; ++r) slot[req[r].t * k + req[r].j] = -1;
    qsort(req, (size_t)keep, sizeof(oracle_request), request_token_order);
    for (int64_t r = 0; r < keep; ++r) slot[req[r].t * k + req[r].j] = (int32_t)r;
    counts_raw[e] = (int32_t)n;
    counts_kept[e] = (int32_t)keep;
    free(req);
  }
}

/* One expert on one token, [SYN] "Core Architecture":
 * E(x) = W2 * GELU(W1 * x + b1) + b2, with W1 [d_ff, d], W2 [d, d_ff]. */
void moe_oracle_expert_ffn(int64_t d, int64_t d_ff, const float *xrow, const float *w1e,
                           const float *b1e, const float *w2e, const float *b2e, double *h,
                           double *out) {
  for (int64_t f = 0; f < d_ff; ++f) {
    double acc = 0.0;
    for (int64_t i = 0; i < d; ++i) acc += (double)w1e[f * d + i] * (double)xrow[i];
    h[f] = moe_oracle_gelu(acc + (double)b1e[f]);
  }
  for (int64_t o = 0; o < d; ++o) {
    double acc = 0.0;
    for (int64_t f = 0; f < d_ff; ++f) acc += (double)w2e[o * d_ff + f] * h[f];
    out[o] = acc + (double)b2e[o];
  }
}

/* Steps 5-7 of [WIKI] for one token: y_t = sum over the accepted picks j (in
 * rank order) of w_j * E_{idx_j}(x_t); a dropped pair adds nothing.
 * w_j is the renormalised gate of step 3. Variants the pages also describe:
 *  - RENORM_SURVIVORS: w_j = gate_j / sum of the accepted gates ([WIKI] worked
 *    example: "renormalize over the surviving expert alone");
 *  - IDENTITY_FALLBACK: a token whose picks were all dropped outputs x_t (the
 *    pseudocode's residual fallback); without it such a token outputs 0;
 *  - SHARED_EXPERT: an always-active expert (weights given separately) is added
 *    to every token ([TGS] "Comparing MoE Architectures"). */
static void combine_token(int64_t t, int64_t d, int32_t k, int64_t d_ff, uint32_t flags,
                          const float *x, const float *w1, const float *b1, const float *w2,
                          const float *b2, const float *sw1, const float *sb1, const float *sw2,
                          const float *sb2, const int32_t *idx, const double *gate,
                          const int32_t *slot, double *h, double *o, double *yrow) {
  for (int64_t i = 0; i < d; ++i) yrow[i] = 0.0;
  double kept_sum = 0.0;
  int kept = 0;
  for (int32_t j = 0; j < k; ++j)
    if (slot[t * k + j] >= 0) {
      kept_sum += gate[t * k + j];
      ++kept;
    }
  for (int32_t j = 0; j < k; ++j) {
    if (slot[t * k + j] < 0) continue;
    int64_t e = idx[t * k + j];
    double w = gate[t * k + j];
    if (flags & ORACLE_FLAG_RENORM_SURVIVORS) w = w / kept_sum;
    moe_oracle_expert_ffn(d, d_ff, x + t * d, w1 + e * d_ff * d, b1 + e * d_ff, w2 + e * d * d_ff,
                          b2 + e * d, h, o);
    for (int64_t i = 0; i < d; ++i) yrow[i] += w * o[i];
  }
  if (kept == 0 && (flags & ORACLE_FLAG_IDENTITY_FALLBACK))
    for (int64_t i = 0; i < d; ++i) yrow[i] = (double)x[t * d + i];
  if (flags & ORACLE_FLAG_SHARED_EXPERT) {
    moe_oracle_expert_ffn(d, d_ff, x + t * d, sw1, sb1, sw2, sb2, h, o);
    for (int64_t i = 0; i < d; ++i) yrow[i] += o[i];
  }
}

/* The whole layer forward, steps 1-7 of [WIKI] in order. Routing and capacity
 * always cover all T tokens (capacity couples the batch). The expert FFNs and
 * the combine run for the n_sel tokens listed in sel (all T tokens, in order,
 * when sel is NULL); y has one row of d doubles per listed token.
 * Optional outputs (NULL to skip): logits and probs [T,N]. Required: idx,
 * score, gate, slot [T,k]; counts_raw, counts_kept [N]; y.
 * Returns 0, or -1 for invalid sizes. */
int moe_oracle_forward(int64_t T, int64_t d, int32_t N, int32_t k, int64_t d_ff, double cf,
                       uint32_t flags, const float *x, const float *w_g, const float *router_bias,
                       const float *w1, const float *b1, const float *w2, const float *b2,
                       const float *sw1, const float *sb1, const float *sw2, const float *sb2,
                       int64_t n_sel, const int64_t *sel, double *logits_out, double *probs_out,
                       int32_t *idx, double *score, double *gate, int32_t *counts_raw,
                       int32_t *counts_kept, int32_t *slot, double *y) {
  if (T < 1 || d < 1 || N < 1 || k < 1 || k > N || d_ff < 1) return -1;
  double *logits = logits_out ? logits_out : (double *)malloc(sizeof(double) * (size_t)(T * N));
  double *probs = probs_out ? probs_out : (double *)malloc(sizeof(double) * (size_t)(T * N));
  moe_oracle_router_logits(T, d, N, x, w_g, router_bias, logits);
  moe_oracle_softmax(T, N, logits, probs);
  moe_oracle_topk(T, N, k, logits, idx);
  moe_oracle_gates(T, N, k, probs, idx, score, gate);
  int64_t C = moe_oracle_capacity(T, N, k, cf);
  moe_oracle_capacity_assign(T, N, k, C, idx, score, counts_raw, counts_kept, slot);
  int64_t n = sel ? n_sel : T;
#pragma omp parallel
  {
    double *h = (double *)malloc(sizeof(double) * (size_t)d_ff);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int64_t s = 0; s < n; ++s) {
      int64_t t = sel ? sel[s] : s;
      combine_token(t, d, k, d_ff, flags, x, w1, b1, w2, b2, sw1, sb1, sw2, sb2, idx, gate, slot, h,
                    o, y + s * d);
    }
    free(h);
    free(o);
  }
  if (!logits_out) free(logits);
  if (!probs_out) free(probs);
  return 0;
}

/* Router statistics of one batch.
 *  f_e: the fraction of the T*k router picks that chose expert e, so that
 *       sum_e f_e = 1 (the normalisation under which [WIKI] "The load-balancing
 *       auxiliary loss" states the minimum N*N*(1/N)^2 = 1);
 *  P_e: the mean router probability of expert e over the batch;
 *  aux = N * sum_e f_e * P_e ([TGS] "The Load Balancing Crisis", without the
 *        training coefficient alpha);
 *  zloss = (1/T) * sum_t (log sum_e exp l[t,e])^2 ([TGS] "Training Dynamics and
 *        Stability"), without the coefficient beta. */
void moe_oracle_router_stats(int64_t T, int32_t N, int32_t k, const double *logits,
                             const double *probs, const int32_t *idx, double *f, double *P,
                             double *aux, double *zloss) {
  for (int32_t e = 0; e < N; ++e) {
    f[e] = 0.0;
    P[e] = 0.0;
  }
  for (int64_t i = 0; i < T * k; ++i) f[idx[i]] += 1.0;
  for (int32_t e = 0; e < N; ++e) f[e] /= (double)(T * k);
  for (int32_t e = 0; e < N; ++e) {
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += probs[t * N + e];
    P[e] = s / (double)T;
  }
  double a = 0.0;
  for (int32_t e = 0; e < N; ++e) a += f[e] * P[e];
  *aux = (double)N * a;
  double z = 0.0;
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + t * N;
    double m = l[0];
    for (int32_t e = 1; e < N; ++e)
      if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int32_t e = 0; e < N; ++e) s += exp(l[e] - m);
    double lse = m + log(s);
    z += lse * lse;
  }
  *zloss = z / (double)T;
}

/* Expert-choice routing ([TGS] and [SYN] "Expert Choice Routing"): each expert
 * takes the C tokens with the highest router probability p[t,e] (equal
 * probabilities: lower token first). A token's output is the sum, over the
 * experts that took it (in expert order), of p[t,e] * E_e(x_t); a token no
 * expert took outputs 0. taken[t*N+e] = 1 when expert e took token t.
 * counts[e] = tokens taken by e. y is [T, d]. */
void moe_oracle_expert_choice(int64_t T, int64_t d, int32_t N, int64_t d_ff, int64_t C,
                              const float *x, const double *probs, const float *w1,
                              const float *b1, const float *w2, const float *b2, int32_t *taken,
                              int32_t *counts, double *y) {
  memset(taken, 0, sizeof(int32_t) * (size_t)(T * N));
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t e = 0; e < N; ++e) {
    oracle_request *req = (oracle_request *)malloc(sizeof(oracle_request) * (size_t)T);
    for (int64_t t = 0; t < T; ++t) {
      req[t].score = probs[t * N + e];
      req[t].t = t;
      req[t].j = 0;
    }
    qsort(req, (size_t)T, sizeof(oracle_request), request_order);
    int64_t keep = C < T ? C : T;
    for (int64_t r = 0; r < keep; ++r) taken[req[r].t * N + e] = 1;
    counts[e] = (int32_t)keep;
    free(req);
  }
#pragma omp parallel
  {
    double *h = (double *)malloc(sizeof(double) * (size_t)d_ff);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      for (int64_t i = 0; i < d; ++i) y[t * d + i] = 0.0;
      for (int32_t e = 0; e < N; ++e) {
        if (!taken[t * N + e]) continue;
        moe_oracle_expert_ffn(d, d_ff, x + t * d, w1 + (int64_t)e * d_ff * d, b1 + (int64_t)e * d_ff,
                              w2 + (int64_t)e * d * d_ff, b2 + (int64_t)e * d, h, o);
        for (int64_t i = 0; i < d; ++i) y[t * d + i] += probs[t * N + e] * o[i];
      }
    }
    free(h);
    free(o);
  }
}
