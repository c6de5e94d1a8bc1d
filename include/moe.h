/*
 * moe.h - C ABI of the B300 (sm_103a) sparse Mixture-of-Experts layer forward.
 *
 * One call of moe_forward computes, for a batch of T tokens x [T, d]:
 *   1. router   l = x W_g^T (+ optional per-expert logit bias), p = softmax(l),
 *               the top-k experts by score, and their scores renormalised to
 *               sum to 1 (the combine weights, "gates");
 *   2. capacity C = ceil(cf * T * k / N): an expert keeps at most C of the
 *               (token, expert) requests routed to it, the highest-scoring
 *               ones (equal scores: lower token index first); the rest are
 *               dropped for that expert;
 *   3. dispatch the kept requests are gathered into per-expert row segments;
 *   4. experts  E_e(x) = W2[e] GELU(W1[e] x + b1[e]) + b2[e], GELU with erf;
 *   5. combine  y_t = sum over the kept picks j of gate_j * E_{idx_j}(x_t).
 * Sources, by page and section: "Mixture-of-Experts" (beta.fermi.ai wiki),
 * the step-by-step mechanism, steps 1-7, and "Communication cost in
 * distributed settings" for C; "Mixture of Experts (MoE): Architecture,
 * Routing, and Scaling" (syntave.com), "Core Architecture", for the FFN.
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers owned by the caller, contiguous row-major,
 *     16-byte aligned. The library never allocates or frees device memory.
 *   - Weights use the [out, in] layout of a linear layer: W_g [N, d],
 *     W1 [N, d_ff, d], b1 [N, d_ff], W2 [N, d, d_ff], b2 [N, d].
 *   - x, W_g, W1, b1, W2, b2, x_perm, h, y_perm and y are in the configured
 *     dtype (fp32 or bf16); router outputs, gates and the logit bias are fp32;
 *     indices are int32.
 *   - Calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return without synchronising. Argument errors are detected
 *     on the host and returned before anything is enqueued. Errors found by
 *     kernels (a wait that timed out, an index out of bounds) are recorded in
 *     the workspace's status word and read with moe_get_device_status.
 *   - Kernels are launched with programmatic stream serialisation: a kernel
 *     may be scheduled while the previous kernel on the stream finishes, but
 *     waits for that kernel's completion before it touches global memory, so
 *     stream order holds as usual.
 *   - Every entry point returns a moe_status; moe_last_error() gives the text
 *     of the last failure on the calling thread. Nothing throws across the ABI.
 *   - Limits: T >= 1, T*k < 2^31; 1 <= N <= 256; 1 <= k <= min(N, 8);
 *     d and d_ff >= 8 and multiples of 8 (bf16) or 4 (fp32).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
#if defined(__GNUC__)
#pragma GCC visibility push(default) /* the library builds with hidden visibility */
#endif

typedef void *moe_stream_t; /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, a misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2, /* valid shape outside what the kernels support */
  MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,     /* device: a pipeline wait exceeded its limit */
  MOE_ERR_BOUNDS = 6       /* device: an index was out of range */
} moe_status;

typedef enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

/* Flag bits of moe_config.flags. 0 selects the default contract:
 * dropped pairs add nothing and keep the other picks' original gates, and a
 * token whose picks were all dropped outputs 0 (the caller's residual path
 * then carries x). */
enum {
  /* After drops, divide a token's surviving gates by their sum ("Mixture-of-
   * Experts" wiki, worked example: renormalise over the surviving expert). */
  MOE_FLAG_RENORM_SURVIVORS = 1u,
  /* A token whose picks were all dropped outputs x_t (the wiki pseudocode's
   * identity fallback). */
  MOE_FLAG_IDENTITY_FALLBACK = 2u,
  /* An always-active shared expert (its own W1, b1, W2, b2 with the same
   * d_ff) is added to every token's output after the routed sum ("Mixture of
   * Experts: Scaling Language Models with Sparse Activation", "Comparing MoE
   * Architectures": shared experts). Run moe_shared_expert before
   * moe_combine, or moe_forward_shared. */
  MOE_FLAG_SHARED_EXPERT = 4u,
  /* The router also stores every token's full probability row and the
   * logsumexp of its logits in the workspace (probs, lse), for
   * moe_router_stats. Routing results are unchanged. */
  MOE_FLAG_ROUTER_STATS = 8u,
  /* Expert-choice routing ("Mixture of Experts (MoE): Architecture, Routing,
   * and Scaling" and "Mixture of Experts: Scaling Language Models with Sparse
   * Activation", "Expert Choice Routing"): instead of each token picking k
   * experts, each expert takes the C tokens with the highest probability
   * p[t, e] (equal probabilities: lower token first; C from cfg's k and
   * capacity_factor as usual), and a token's output is the sum, in expert
   * order, of p[t, e] * E_e(x_t) over the experts that took it (0 if none).
   * Only moe_forward runs it (with MOE_FLAG_ROUTER_STATS at most); the
   * workspace's row_of is then [T, N] (the row of token t at expert e, or
   * -1) and probs holds p. */
  MOE_FLAG_EXPERT_CHOICE = 16u
};

typedef struct {
  int64_t T;              /* tokens in the batch */
  int64_t d;              /* model width */
  int64_t d_ff;           /* expert hidden width */
  int32_t N;              /* experts */
  int32_t k;              /* experts per token */
  double capacity_factor; /* <= 0 or +inf: no limit (C = T) */
  moe_dtype dtype;        /* storage type of x, weights, x_perm, h and y */
  uint32_t flags;         /* MOE_FLAG_* bits; 0 = default contract */
} moe_config;

/* Byte offsets of the buffers inside a workspace (all 256-byte aligned).
 * rows = R_max, the row capacity of the permuted buffers: every expert segment
 * starts on a multiple of 128 rows (for decode-shaped configs, bf16 with
 * T*k <= 64*N: 64 rows, or 32 rows when T*k <= 16*N), so
 * R_max = floor((min(T*k, N*C) + 127*N) / 128) * 128
 * bounds the rows in use. */
typedef struct {
  size_t status;      /* int32[16]; [0] first device error code, [1] kernel id, [2] detail */
  size_t topk_idx;    /* int32 [T, k]  picks in rank order */
  size_t gate;        /* fp32  [T, k]  renormalised top-k scores (combine weights) */
  size_t score;       /* fp32  [T, k]  softmax probability of each pick (capacity ranking) */
  size_t counts_raw;  /* int32 [N]     requests per expert */
  size_t counts_kept; /* int32 [N]     accepted requests per expert (<= C) */
  size_t offsets;     /* int32 [N+1]   first row of each expert segment; [N] = rows in use */
  size_t sel_thr;     /* uint32 [N]    capacity selection scratch */
  size_t sel_eq;      /* int32 [N]     capacity selection scratch */
  size_t row_of;      /* int32 [T, k]  row of each pick in the permuted buffers, -1 dropped */
  size_t row_token;   /* int32 [rows]  token of each permuted row, -1 for padding */
  size_t row_gate;    /* fp32  [rows]  combine weight of each permuted row, 0 for padding */
  size_t x_perm;      /* dtype [rows, d]    tokens gathered per expert */
  size_t h;           /* dtype [rows, d_ff] expert hidden activations */
  size_t y_perm;      /* dtype [rows, d]    gate-scaled expert outputs */
  size_t y_split;     /* fp32  [S-1, rows, d] decode-shaped configs only: the second GEMM's extra K slices */
  size_t ffn_sync;    /* int32 bf16 configs: completion counters of h tiles (per expert in decode-shaped
                       * configs, else per 256-row block) and an exit count, read by the fused expert
                       * FFN; zero between calls (moe_workspace_init, moe_dispatch and every
                       * completed moe_expert_ffn leave them zero) */
  size_t probs;       /* fp32  [T, N]  MOE_FLAG_ROUTER_STATS only: p[t, e] for every expert */
  size_t lse;         /* fp32  [T]     MOE_FLAG_ROUTER_STATS only: logsumexp of token t's logits */
  size_t shared_offsets; /* int32 [2]  MOE_FLAG_SHARED_EXPERT only: the shared expert's one segment */
  size_t h_shared;    /* dtype [Tp, d_ff] MOE_FLAG_SHARED_EXPERT only: its hidden activations, Tp = T
                       * rounded up to 128 */
  size_t y_shared;    /* dtype [Tp, d]    MOE_FLAG_SHARED_EXPERT only: its output */
  size_t shared_sync; /* int32        MOE_FLAG_SHARED_EXPERT only: completion counters of its FFN */
  size_t total;       /* bytes of the whole workspace */
  int64_t rows;       /* R_max */
  int64_t capacity;   /* C */
} moe_workspace_layout;

/* Version string of the library. */
const char *moe_version(void);

/* Text of the last error returned on the calling thread ("" if none). */
const char *moe_last_error(void);

/* Expert capacity C = ceil(cf * T * k / N), or T when cf <= 0, cf = inf or
 * the formula exceeds T ("Mixture-of-Experts" wiki, "Communication cost in
 * distributed settings": C = gamma * k * T / N). Returns -1 for an invalid
 * config. */
int64_t moe_capacity(const moe_config *cfg);

/* Fill *out with the workspace layout of cfg. */
moe_status moe_get_workspace_layout(const moe_config *cfg, moe_workspace_layout *out);

/* Bytes of workspace moe_forward needs for cfg (0 for an invalid config). */
size_t moe_workspace_bytes(const moe_config *cfg);

/* Clear the status word and the expert FFN's completion counters of a
 * workspace. Call once after allocating it (the status word is sticky: later
 * calls never clear it). Enqueued on stream. */
moe_status moe_workspace_init(const moe_config *cfg, void *ws, moe_stream_t stream);

/* Wait for stream, then return the workspace's device status: MOE_OK, or the
 * first MOE_ERR_TIMEOUT / MOE_ERR_BOUNDS a kernel recorded since the last
 * moe_workspace_init (its kernel id and detail go to moe_last_error). */
moe_status moe_get_device_status(void *ws, moe_stream_t stream);

/* Step 1-3 of the wiki mechanism: router logits in fp32 (never rounded to
 * bf16), softmax over N, top-k by logit (ties: lower expert first; picks in
 * rank order), renormalised gates.
 *   x [T, d] dtype, w_g [N, d] dtype, router_bias [N] fp32 or NULL;
 *   out: topk_idx int32 [T, k], gate fp32 [T, k], score fp32 [T, k].
 *   ws: a workspace of cfg (its status word is used). */
moe_status moe_route(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                     int32_t *topk_idx, float *gate, float *score, void *ws, moe_stream_t stream);

/* Router statistics of the last routed batch ("Mixture-of-Experts" wiki, the
 * load-balancing auxiliary loss; "Mixture of Experts (MoE): Architecture,
 * Routing, and Scaling", "Importance Loss and Z-Loss"). Needs a workspace of
 * a cfg with MOE_FLAG_ROUTER_STATS on which moe_route (or moe_forward) ran.
 *   counts_raw [N] int32: requests per expert from moe_dispatch (router picks,
 *   before capacity). Out (device, fp32): f [N] = counts_raw[e] / (T*k);
 *   P [N] = mean over tokens of p[t, e]; losses [2] = {N * sum_e f[e] P[e]
 *   (the auxiliary balance loss, 1 at a perfectly uniform split), mean over
 *   tokens of logsumexp(logits)^2 (the z-loss)}. Sums run in a fixed order:
 *   deterministic. MOE_ERR_INVALID_ARG without the flag. */
moe_status moe_router_stats(const moe_config *cfg, void *ws, const int32_t *counts_raw, float *f, float *P,
                            float *losses, moe_stream_t stream);

/* Steps 4-5: capacity enforcement and dispatch. Per expert, keep the top C
 * requests by (score desc, token asc); number the kept rows of each expert in
 * ascending token order inside a segment that starts at offsets[e] (a
 * multiple of 128 rows, or of the decode chunk size for decode-shaped configs:
 * see moe_workspace_layout); gather x into those rows (padding rows are zero).
 *   in:  x [T, d], topk_idx, gate, score [T, k] (as written by moe_route);
 *   out: counts_raw [N], counts_kept [N], offsets [N+1], row_of [T, k],
 *        row_token [rows], row_gate [rows] (the gate of each kept pick; 0
 *        on padding rows), x_perm [rows, d] in dtype.
 *   rows = moe_workspace_layout.rows. ws: a workspace of cfg (selection
 *   scratch and status word). Deterministic: no atomics decide any output. */
moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *topk_idx, const float *gate,
                        const float *score, int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets,
                        int32_t *row_of, int32_t *row_token, float *row_gate, void *x_perm, void *ws,
                        moe_stream_t stream);

/* Step 6: the expert FFNs over the permuted rows, two grouped GEMMs.
 *   h[r]      = GELU(x_perm[r] W1[e]^T + b1[e])                (dtype)
 *   y_perm[r] = row_gate[r] * (h[r] W2[e]^T + b2[e])           (dtype)
 * for every row r of expert e's segment [offsets[e], offsets[e+1]).
 *   row_gate may be NULL (no scaling). h [rows, d_ff] may be NULL to use the
 *   workspace's h buffer. Accumulation is fp32 (bf16 inputs: tensor cores,
 *   tcgen05, accumulating in tensor memory). For decode-shaped configs (bf16,
 *   T*k <= 64*N) the second GEMM is split along d_ff: y_perm receives the
 *   first slice and the workspace's y_split (fp32) the others, which moe_combine
 *   (given the same workspace) adds in slice order. For bf16 configs both
 *   GEMMs run in one launch, whose second-GEMM tiles wait (bounded,
 *   MOE_ERR_TIMEOUT) on completion counters in the workspace's ffn_sync
 *   (zero on entry; the launch's last CTA leaves them zero). */
moe_status moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const void *w1,
                          const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                          void *y_perm, void *ws, moe_stream_t stream);

/* The shared expert over every token: y_shared[t] = W2s GELU(W1s x_t + b1s)
 * + b2s into the workspace of a cfg with MOE_FLAG_SHARED_EXPERT (x [T, d],
 * sw1 [d_ff, d], sb1 [d_ff], sw2 [d, d_ff], sb2 [d], all in dtype). Same
 * arithmetic as moe_expert_ffn (one expert whose segment is the whole batch,
 * unscaled); moe_combine then adds it. */
moe_status moe_shared_expert(const moe_config *cfg, const void *x, const void *sw1, const void *sb1,
                             const void *sw2, const void *sb2, void *ws, moe_stream_t stream);

/* Step 7: y[t] = sum over j < k with row_of[t,j] >= 0, in j order, of
 * y_perm[row_of[t,j]], added in fp32 and rounded once to dtype. No atomics. For
 * decode-shaped configs each pick's term is first completed with the same row
 * of the workspace's y_split slices, added in slice order.
 *   gate [T, k] is read only under MOE_FLAG_RENORM_SURVIVORS (the sum is then
 *   divided by the token's kept-gate sum); x [T, d] only under
 *   MOE_FLAG_IDENTITY_FALLBACK (a token with no kept pick outputs x_t). Either
 *   may be NULL otherwise. Under MOE_FLAG_SHARED_EXPERT the workspace's
 *   y_shared row is added last. ws: a workspace of cfg (status word). */
moe_status moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *row_of, const float *gate,
                       const void *x, void *y, void *ws, moe_stream_t stream);

/* moe_forward plus the shared expert (cfg must carry MOE_FLAG_SHARED_EXPERT):
 * route, dispatch, the routed expert FFNs, moe_shared_expert, combine. */
moe_status moe_forward_shared(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                              const void *w1, const void *b1, const void *w2, const void *b2, const void *sw1,
                              const void *sb1, const void *sw2, const void *sb2, void *y, void *ws,
                              moe_stream_t stream);

/* The whole layer forward: moe_route, moe_dispatch, moe_expert_ffn and
 * moe_combine on the workspace's buffers, y [T, d] in dtype. After the
 * stream reaches the end of the call, every intermediate (picks, gates,
 * counts, offsets, row maps, x_perm, h, y_perm) can be read from the
 * workspace at the offsets of moe_get_workspace_layout. No host
 * synchronisation happens inside the call. */
moe_status moe_forward(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                       const void *w1, const void *b1, const void *w2, const void *b2, void *y, void *ws,
                       moe_stream_t stream);

/* The layer forward for callers that cannot allocate device memory (plugin
 * or custom-op hosts that provide inputs and outputs but no workspace, code
 * whose memory belongs to an allocator that forbids direct cudaMalloc, or
 * paths that must avoid cudaMalloc's device synchronisation). The pages have
 * no counterpart: this is a property of the library, not of the method.
 * Same arguments and result as moe_forward, minus the workspace: the scratch
 * is a file-scope device array of 32 MiB that every GPU loading the library
 * keeps until the process exits. Configs whose moe_workspace_bytes exceeds
 * 32 MiB return MOE_ERR_WORKSPACE before anything is enqueued. The first call
 * on a device looks up the array's address (once per device): make it before
 * any stream capture. All calls share the array and it keeps the last call's
 * contents; each call clears its status word first. Calls whose GPU work
 * overlaps race. Device-side errors are not readable afterwards (the status
 * word is not the caller's): only host-side errors are returned. Never
 * allocates. */
moe_status moe_forward_noalloc(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                               const void *w1, const void *b1, const void *w2, const void *b2, void *y,
                               moe_stream_t stream);

/* Self-test of the library's failure handling (the pages have no counterpart:
 * this checks a property of the library, not of the method). Every wait inside
 * the pipelined kernels, on an mbarrier phase or on a completion counter that
 * another CTA raises, is bounded: when its limit passes, the kernel records
 * MOE_ERR_TIMEOUT in the workspace's status word and leaves cleanly. This call
 * launches one CTA that runs those same two wait routines on a barrier that
 * nothing arms and on a counter that nothing raises, each for limit_ns
 * nanoseconds (1000 .. 10^9), so that a test can watch both give up.
 *   ws: any workspace (only its 64-byte status word, at offset 0, is used;
 *   moe_get_device_status then returns MOE_ERR_TIMEOUT until moe_workspace_init
 *   clears it). result: device int32[8], 16-byte aligned: [0] and [1] are 1 if
 *   the barrier / counter wait succeeded (0 is expected), [2] and [3] the
 *   microseconds each wait lasted, [4] the counter (cleared here before the
 *   launch). MOE_ERR_INVALID_ARG for a limit outside the range or a bad
 *   pointer. */
moe_status moe_selftest_wait_timeout(void *ws, int64_t limit_ns, int32_t *result, moe_stream_t stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
