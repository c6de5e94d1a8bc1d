// The C ABI declared in include/moe.h: argument checks, workspace layout and
// the stream-ordered sequence of kernel launches. No allocation, no host
// synchronisation (except moe_get_device_status, which exists to wait).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "moe_internal.cuh"

using namespace moe;

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

int64_t capacity_of(int64_t T, int32_t N, int32_t k, double cf) {
  if (!(cf > 0.0) || isinf(cf)) return T;
  const double c = ceil(cf * (double)(T * (int64_t)k) / (double)N);
  if (!(c < (double)T)) return T;
  return (int64_t)c;
}

moe_status check_config(const moe_config *cfg, Dims *D) {
  if (!cfg) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
  if (cfg->T < 1) return fail(MOE_ERR_INVALID_ARG, "T must be >= 1 (got %lld)", (long long)cfg->T);
  if (cfg->N < 1 || cfg->N > 256) return fail(MOE_ERR_INVALID_ARG, "N must be in [1, 256] (got %d)", cfg->N);
  if (cfg->k < 1 || cfg->k > cfg->N || cfg->k > 8)
    return fail(MOE_ERR_INVALID_ARG, "k must be in [1, min(N, 8)] (got %d)", cfg->k);
  if (cfg->T * (int64_t)cfg->k >= ((int64_t)1 << 31)) return fail(MOE_ERR_INVALID_ARG, "T*k must be < 2^31");
  if (cfg->dtype != MOE_DT_F32 && cfg->dtype != MOE_DT_BF16)
    return fail(MOE_ERR_INVALID_ARG, "dtype must be MOE_DT_F32 or MOE_DT_BF16");
  const int64_t mult = cfg->dtype == MOE_DT_BF16 ? 8 : 4;
  if (cfg->d < 8 || cfg->d % mult || cfg->d_ff < 8 || cfg->d_ff % mult)
    return fail(MOE_ERR_INVALID_ARG, "d and d_ff must be >= 8 and multiples of %lld (got d=%lld d_ff=%lld)",
                (long long)mult, (long long)cfg->d, (long long)cfg->d_ff);
  if (cfg->flags & ~(uint32_t)(MOE_FLAG_RENORM_SURVIVORS | MOE_FLAG_IDENTITY_FALLBACK | MOE_FLAG_ROUTER_STATS |
                               MOE_FLAG_SHARED_EXPERT | MOE_FLAG_EXPERT_CHOICE))
    return fail(MOE_ERR_INVALID_ARG, "unknown flag bits 0x%x", cfg->flags);
  const bool ec = (cfg->flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  if (ec && (cfg->flags & ~(uint32_t)(MOE_FLAG_EXPERT_CHOICE | MOE_FLAG_ROUTER_STATS)))
    return fail(MOE_ERR_INVALID_ARG, "MOE_FLAG_EXPERT_CHOICE combines only with MOE_FLAG_ROUTER_STATS");
  if (ec && cfg->T * (int64_t)cfg->N >= ((int64_t)1 << 31)) return fail(MOE_ERR_INVALID_ARG, "T*N must be < 2^31");
  if (isnan(cfg->capacity_factor)) return fail(MOE_ERR_INVALID_ARG, "capacity_factor is NaN");
  D->T = cfg->T;
  D->d = cfg->d;
  D->d_ff = cfg->d_ff;
  D->N = cfg->N;
  D->C = capacity_of(cfg->T, cfg->N, cfg->k, cfg->capacity_factor);
  // expert choice: every token offers itself to every expert, so the
  // selection, dispatch and combine run with k = N requests per token
  D->k = ec ? cfg->N : cfg->k;
  int64_t S = cfg->T * (int64_t)D->k;
  if ((int64_t)cfg->N * D->C < S) S = (int64_t)cfg->N * D->C;
  D->R_max = (S + (int64_t)(kRowAlign - 1) * cfg->N) / kRowAlign * kRowAlign;
  if (D->R_max >= ((int64_t)1 << 31)) return fail(MOE_ERR_INVALID_ARG, "too many permuted rows");
  D->dt = cfg->dtype;
  D->flags = cfg->flags;
  return MOE_OK;
}

// The shared expert as a one-expert FFN whose segment is the whole batch,
// rounded up to 128 rows.
Dims shared_dims(const Dims &D) {
  Dims S1 = D;
  S1.N = 1;
  S1.k = 1;
  S1.C = D.T;  // the one expert takes every token
  S1.R_max = (D.T + kRowAlign - 1) / kRowAlign * kRowAlign;
  return S1;
}
int64_t shared_sync_ints(const Dims &D) { return ffn_blocks_max(shared_dims(D)) + 1; }

void make_layout(const Dims &D, moe_workspace_layout *L) {
  const size_t es = D.dt == MOE_DT_BF16 ? 2 : 4;
  const size_t Tk = (size_t)(D.T * D.k), R = (size_t)D.R_max, N = (size_t)D.N;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L->status = take(64);
  L->topk_idx = take(Tk * 4);
  L->gate = take(Tk * 4);
  L->score = take(Tk * 4);
  L->counts_raw = take(N * 4);
  L->counts_kept = take(N * 4);
  L->offsets = take((N + 1) * 4);
  L->sel_thr = take(N * 4);
  L->sel_eq = take(N * 4);
  L->row_of = take(Tk * 4);
  L->row_token = take(R * 4);
  L->row_gate = take(R * 4);
  L->x_perm = take(R * (size_t)D.d * es);
  L->h = take(R * (size_t)D.d_ff * es);
  L->y_perm = take(R * (size_t)D.d * es);
  const int S = decode_splits(D);
  L->y_split = take(S > 1 ? (size_t)(S - 1) * R * (size_t)D.d * 4 : 0);
  L->ffn_sync = take((size_t)ffn_sync_ints(D) * 4);
  const bool stats = (D.flags & (MOE_FLAG_ROUTER_STATS | MOE_FLAG_EXPERT_CHOICE)) != 0;
  L->probs = take(stats ? (size_t)D.T * N * 4 : 0);
  L->lse = take(stats ? (size_t)D.T * 4 : 0);
  const bool shared = (D.flags & MOE_FLAG_SHARED_EXPERT) != 0;
  const Dims S1 = shared_dims(D);
  L->shared_offsets = take(shared ? 8 : 0);
  L->h_shared = take(shared ? (size_t)S1.R_max * (size_t)D.d_ff * es : 0);
  L->y_shared = take(shared ? (size_t)S1.R_max * (size_t)D.d * es : 0);
  L->shared_sync = take(shared ? (size_t)shared_sync_ints(D) * 4 : 0);
  L->total = off;
  L->rows = D.R_max;
  L->capacity = D.C;
}

#define AT(ws, off, T) reinterpret_cast<T>(static_cast<char *>(ws) + (off))

moe_status check_ptrs(std::initializer_list<const void *> ps, const char *what) {
  for (const void *p : ps) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "%s: a required pointer is NULL", what);
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s: pointer %p is not 16-byte aligned", what, p);
  }
  return MOE_OK;
}

moe_status check_opt(const void *p, const char *what) {
  if (p && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s: pointer %p is not 16-byte aligned", what, p);
  return MOE_OK;
}

#define TRY(expr)                          \
  do {                                     \
    moe_status _st = (expr);               \
    if (_st != MOE_OK) return _st;         \
  } while (0)

moe_status do_route(const Dims &D, const moe_workspace_layout &L, const void *x, const void *w_g,
                    const float *router_bias, int32_t *topk_idx, float *gate, float *score, void *ws,
                    cudaStream_t s) {
  // with MOE_FLAG_ROUTER_STATS (or expert choice) the router also stores full
  // probability rows and logsumexps
  const bool ec = (D.flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  const bool stats = ec || (D.flags & MOE_FLAG_ROUTER_STATS) != 0;
  float *probs = stats ? AT(ws, L.probs, float *) : nullptr;
  float *lse = stats ? AT(ws, L.lse, float *) : nullptr;
  Dims Dr = D;
  if (ec) Dr.k = 1;  // expert choice uses the probabilities; the top-1 pick is not read
  cudaError_t e = D.dt == MOE_DT_BF16 && !router_split(Dr)
                      ? launch_router_tc(Dr, x, w_g, router_bias, topk_idx, gate, score, probs, lse,
                                         AT(ws, L.status, int32_t *), s)
                      : launch_router(Dr, x, w_g, router_bias, topk_idx, gate, score, probs, lse,
                                      AT(ws, L.status, int32_t *), s);
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  return MOE_OK;
}

moe_status do_dispatch(const Dims &D, const moe_workspace_layout &L, const void *x, const int32_t *topk_idx,
                       const float *gate, const float *score, int32_t *counts_raw, int32_t *counts_kept,
                       int32_t *offsets, int32_t *row_of, int32_t *row_token, float *row_gate, void *x_perm,
                       void *ws, cudaStream_t s) {
  int32_t *status = AT(ws, L.status, int32_t *);
  cudaError_t e = launch_capacity(D, topk_idx, gate, score, counts_raw, counts_kept, offsets,
                                  AT(ws, L.sel_thr, uint32_t *), AT(ws, L.sel_eq, int32_t *), row_of, row_token,
                                  row_gate, AT(ws, L.ffn_sync, int32_t *), status, s);
  if (e != cudaSuccess) return cuda_fail(e, "capacity launch");
  e = launch_permute(D, x, offsets, row_token, x_perm, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "permute launch");
  return MOE_OK;
}

moe_status do_ffn(const Dims &D, const moe_workspace_layout &L, const void *x_perm, const int32_t *offsets,
                  const void *w1, const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                  void *y_perm, void *ws, cudaStream_t s) {
  int32_t *status = AT(ws, L.status, int32_t *);
  if (decode_splits(D) > 0) {
    cudaError_t e = launch_ffn_decode(D, x_perm, offsets, w1, b1, w2, b2, row_gate, h, y_perm,
                                      AT(ws, L.y_split, float *), AT(ws, L.ffn_sync, int32_t *), status, s);
    if (e == cudaErrorNotSupported)
      return fail(MOE_ERR_UNSUPPORTED, "expert FFN: decode shape not supported by the tensor-core kernels");
    if (e != cudaSuccess) return cuda_fail(e, "expert FFN (decode, tensor cores)");
    return MOE_OK;
  }
  if (D.dt == MOE_DT_BF16) {
    cudaError_t e = launch_ffn_tc(D, x_perm, D.R_max, offsets, w1, b1, w2, b2, row_gate, h, y_perm,
                                  AT(ws, L.ffn_sync, int32_t *), status, s);
    if (e == cudaErrorNotSupported)
      return fail(MOE_ERR_UNSUPPORTED, "expert FFN: shape not supported by the tensor-core kernels");
    if (e != cudaSuccess) return cuda_fail(e, "expert FFN (tensor cores)");
    return MOE_OK;
  }
  cudaError_t e = launch_ffn_simt(D, 1, x_perm, D.R_max, D.d, w1, b1, D.d_ff, nullptr, offsets, h, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "expert GEMM1 launch");
  e = launch_ffn_simt(D, 2, h, D.R_max, D.d_ff, w2, b2, D.d, row_gate, offsets, y_perm, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "expert GEMM2 launch");
  return MOE_OK;
}

moe_status do_combine(const Dims &D, const moe_workspace_layout &L, const void *y_perm, const int32_t *row_of,
                      const float *gate, const void *x, void *y, void *ws, cudaStream_t s) {
  const int S = decode_splits(D);
  const void *y_shared = (D.flags & MOE_FLAG_SHARED_EXPERT) ? AT(ws, L.y_shared, const void *) : nullptr;
  cudaError_t e = launch_combine(D, y_perm, S > 1 ? AT(ws, L.y_split, const float *) : nullptr, S > 1 ? S - 1 : 0,
                                 row_of, gate, x, y_shared, y, AT(ws, L.status, int32_t *), s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return MOE_OK;
}

// The shared expert's FFN over x (T rows; TMA or the SIMT loads zero-fill the
// rows up to the 128-row multiple) into the workspace's y_shared.
moe_status do_shared(const Dims &D, const moe_workspace_layout &L, const void *x, const void *sw1, const void *sb1,
                     const void *sw2, const void *sb2, void *ws, cudaStream_t s) {
  const Dims S1 = shared_dims(D);
  int32_t *status = AT(ws, L.status, int32_t *);
  int32_t *offs = AT(ws, L.shared_offsets, int32_t *);
  void *h = AT(ws, L.h_shared, void *);
  void *y_sh = AT(ws, L.y_shared, void *);
  cudaError_t e = launch_shared_setup(offs, S1.R_max, AT(ws, L.shared_sync, int32_t *), shared_sync_ints(D), s);
  if (e != cudaSuccess) return cuda_fail(e, "shared expert setup");
  if (D.dt == MOE_DT_BF16) {
    e = launch_ffn_tc(S1, x, D.T, offs, sw1, sb1, sw2, sb2, nullptr, h, y_sh, AT(ws, L.shared_sync, int32_t *),
                      status, s);
    if (e != cudaSuccess) return cuda_fail(e, "shared expert FFN (tensor cores)");
    return MOE_OK;
  }
  e = launch_ffn_simt(S1, 1, x, D.T, D.d, sw1, sb1, D.d_ff, nullptr, offs, h, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "shared expert GEMM1 launch");
  e = launch_ffn_simt(S1, 2, h, S1.R_max, D.d_ff, sw2, sb2, D.d, nullptr, offs, y_sh, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "shared expert GEMM2 launch");
  return MOE_OK;
}

}  // namespace

void moe::set_last_error(const char *text) { snprintf(g_err, sizeof(g_err), "%s", text); }

int moe::num_sms() {
  static PerDevice<int> cache;
  int n = 0;
  const cudaError_t e = cache.get(
      [](int *v) {
        int dev = 0;
        cudaError_t r = cudaGetDevice(&dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
        if (r != cudaSuccess || *v <= 0) {
          cudaGetLastError();
          *v = 148;
        }
        return cudaSuccess;
      },
      &n);
  return e == cudaSuccess && n > 0 ? n : 148;
}

extern "C" {

const char *moe_version(void) { return "sparse-moe-b300 0.1 (sm_103a)"; }

const char *moe_last_error(void) { return g_err; }

int64_t moe_capacity(const moe_config *cfg) {
  Dims D{};
  if (check_config(cfg, &D) != MOE_OK) return -1;
  return D.C;
}

moe_status moe_get_workspace_layout(const moe_config *cfg, moe_workspace_layout *out) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (!out) return fail(MOE_ERR_INVALID_ARG, "layout output is NULL");
  make_layout(D, out);
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_config *cfg) {
  Dims D;
  if (check_config(cfg, &D) != MOE_OK) return 0;
  moe_workspace_layout L;
  make_layout(D, &L);
  return L.total;
}

moe_status moe_workspace_init(const moe_config *cfg, void *ws, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  TRY(check_ptrs({ws}, "moe_workspace_init"));
  moe_workspace_layout L;
  make_layout(D, &L);
  cudaError_t e = cudaMemsetAsync(ws, 0, 64, (cudaStream_t)stream);
  if (e == cudaSuccess && ffn_sync_ints(D) > 0)
    e = cudaMemsetAsync(AT(ws, L.ffn_sync, void *), 0, (size_t)ffn_sync_ints(D) * 4, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return MOE_OK;
}

moe_status moe_get_device_status(void *ws, moe_stream_t stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  int32_t h[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  if (h[0] == 0) return MOE_OK;
  if (h[0] == MOE_ERR_TIMEOUT || h[0] == MOE_ERR_BOUNDS)
    return fail((moe_status)h[0], "device error %d recorded by kernel %d (detail %d)", h[0], h[1], h[2]);
  return fail(MOE_ERR_CUDA, "unknown device status %d (kernel %d, detail %d)", h[0], h[1], h[2]);
}

moe_status moe_route(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                     int32_t *topk_idx, float *gate, float *score, void *ws, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (D.flags & MOE_FLAG_EXPERT_CHOICE)
    return fail(MOE_ERR_INVALID_ARG, "moe_route: expert-choice routing runs only through moe_forward");
  TRY(check_ptrs({x, w_g, topk_idx, gate, score, ws}, "moe_route"));
  TRY(check_opt(router_bias, "moe_route router_bias"));
  moe_workspace_layout L;
  make_layout(D, &L);
  return do_route(D, L, x, w_g, router_bias, topk_idx, gate, score, ws, (cudaStream_t)stream);
}

moe_status moe_router_stats(const moe_config *cfg, void *ws, const int32_t *counts_raw, float *f, float *P,
                            float *losses, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (!(D.flags & MOE_FLAG_ROUTER_STATS))
    return fail(MOE_ERR_INVALID_ARG, "moe_router_stats: the config lacks MOE_FLAG_ROUTER_STATS");
  TRY(check_ptrs({ws, counts_raw, f, P, losses}, "moe_router_stats"));
  moe_workspace_layout L;
  make_layout(D, &L);
  cudaError_t e = launch_router_stats(D, AT(ws, L.probs, const float *), AT(ws, L.lse, const float *), counts_raw,
                                      f, P, losses, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "router statistics launch");
  return MOE_OK;
}

moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *topk_idx, const float *gate,
                        const float *score, int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets,
                        int32_t *row_of, int32_t *row_token, float *row_gate, void *x_perm, void *ws,
                        moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (D.flags & MOE_FLAG_EXPERT_CHOICE)
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: expert-choice routing runs only through moe_forward");
  TRY(check_ptrs({x, topk_idx, gate, score, counts_raw, counts_kept, offsets, row_of, row_token, row_gate, x_perm,
                  ws},
                 "moe_dispatch"));
  moe_workspace_layout L;
  make_layout(D, &L);
  return do_dispatch(D, L, x, topk_idx, gate, score, counts_raw, counts_kept, offsets, row_of, row_token, row_gate,
                     x_perm, ws, (cudaStream_t)stream);
}

moe_status moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const void *w1,
                          const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                          void *y_perm, void *ws, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (D.flags & MOE_FLAG_EXPERT_CHOICE)
    return fail(MOE_ERR_INVALID_ARG, "moe_expert_ffn: expert-choice routing runs only through moe_forward");
  TRY(check_ptrs({x_perm, offsets, w1, b1, w2, b2, y_perm, ws}, "moe_expert_ffn"));
  TRY(check_opt(row_gate, "moe_expert_ffn row_gate"));
  TRY(check_opt(h, "moe_expert_ffn h"));
  moe_workspace_layout L;
  make_layout(D, &L);
  if (!h) h = AT(ws, L.h, void *);
  return do_ffn(D, L, x_perm, offsets, w1, b1, w2, b2, row_gate, h, y_perm, ws, (cudaStream_t)stream);
}

moe_status moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *row_of, const float *gate,
                       const void *x, void *y, void *ws, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (D.flags & MOE_FLAG_EXPERT_CHOICE)
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: expert-choice routing runs only through moe_forward");
  TRY(check_ptrs({y_perm, row_of, y, ws}, "moe_combine"));
  if ((D.flags & MOE_FLAG_RENORM_SURVIVORS)) TRY(check_ptrs({gate}, "moe_combine gate (renormalise flag)"));
  if ((D.flags & MOE_FLAG_IDENTITY_FALLBACK)) TRY(check_ptrs({x}, "moe_combine x (identity fallback flag)"));
  moe_workspace_layout L;
  make_layout(D, &L);
  return do_combine(D, L, y_perm, row_of, gate, x, y, ws, (cudaStream_t)stream);
}

moe_status moe_shared_expert(const moe_config *cfg, const void *x, const void *sw1, const void *sb1,
                             const void *sw2, const void *sb2, void *ws, moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (!(D.flags & MOE_FLAG_SHARED_EXPERT))
    return fail(MOE_ERR_INVALID_ARG, "moe_shared_expert: the config lacks MOE_FLAG_SHARED_EXPERT");
  TRY(check_ptrs({x, sw1, sb1, sw2, sb2, ws}, "moe_shared_expert"));
  moe_workspace_layout L;
  make_layout(D, &L);
  return do_shared(D, L, x, sw1, sb1, sw2, sb2, ws, (cudaStream_t)stream);
}

moe_status moe_forward(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                       const void *w1, const void *b1, const void *w2, const void *b2, void *y, void *ws,
                       moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (D.flags & MOE_FLAG_SHARED_EXPERT)
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: MOE_FLAG_SHARED_EXPERT needs the shared weights "
                                     "(use moe_forward_shared)");
  TRY(check_ptrs({x, w_g, w1, b1, w2, b2, y, ws}, "moe_forward"));
  TRY(check_opt(router_bias, "moe_forward router_bias"));
  moe_workspace_layout L;
  make_layout(D, &L);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *topk_idx = AT(ws, L.topk_idx, int32_t *);
  float *gate = AT(ws, L.gate, float *);
  float *score = AT(ws, L.score, float *);
  int32_t *offsets = AT(ws, L.offsets, int32_t *);
  int32_t *row_of = AT(ws, L.row_of, int32_t *);
  float *row_gate = AT(ws, L.row_gate, float *);
  void *x_perm = AT(ws, L.x_perm, void *);
  void *y_perm = AT(ws, L.y_perm, void *);
  TRY(do_route(D, L, x, w_g, router_bias, topk_idx, gate, score, ws, s));
  if (D.flags & MOE_FLAG_EXPERT_CHOICE) {
    // every token offers itself to every expert (request j of token t goes to
    // expert j), ranked and weighted by p[t, j]: the capacity step then keeps
    // each expert's C most probable tokens
    cudaError_t e = launch_ec_pattern(topk_idx, D.T, D.N, s);
    if (e != cudaSuccess) return cuda_fail(e, "expert-choice request pattern");
    gate = score = AT(ws, L.probs, float *);
  }
  TRY(do_dispatch(D, L, x, topk_idx, gate, score, AT(ws, L.counts_raw, int32_t *), AT(ws, L.counts_kept, int32_t *),
                  offsets, row_of, AT(ws, L.row_token, int32_t *), row_gate, x_perm, ws, s));
  TRY(do_ffn(D, L, x_perm, offsets, w1, b1, w2, b2, row_gate, AT(ws, L.h, void *), y_perm, ws, s));
  TRY(do_combine(D, L, y_perm, row_of, gate, x, y, ws, s));
  return MOE_OK;
}

moe_status moe_forward_shared(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                              const void *w1, const void *b1, const void *w2, const void *b2, const void *sw1,
                              const void *sb1, const void *sw2, const void *sb2, void *y, void *ws,
                              moe_stream_t stream) {
  Dims D;
  TRY(check_config(cfg, &D));
  if (!(D.flags & MOE_FLAG_SHARED_EXPERT))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward_shared: the config lacks MOE_FLAG_SHARED_EXPERT");
  TRY(check_ptrs({x, w_g, w1, b1, w2, b2, sw1, sb1, sw2, sb2, y, ws}, "moe_forward_shared"));
  TRY(check_opt(router_bias, "moe_forward_shared router_bias"));
  moe_workspace_layout L;
  make_layout(D, &L);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *topk_idx = AT(ws, L.topk_idx, int32_t *);
  float *gate = AT(ws, L.gate, float *);
  float *score = AT(ws, L.score, float *);
  int32_t *offsets = AT(ws, L.offsets, int32_t *);
  int32_t *row_of = AT(ws, L.row_of, int32_t *);
  float *row_gate = AT(ws, L.row_gate, float *);
  void *x_perm = AT(ws, L.x_perm, void *);
  void *y_perm = AT(ws, L.y_perm, void *);
  TRY(do_route(D, L, x, w_g, router_bias, topk_idx, gate, score, ws, s));
  TRY(do_dispatch(D, L, x, topk_idx, gate, score, AT(ws, L.counts_raw, int32_t *), AT(ws, L.counts_kept, int32_t *),
                  offsets, row_of, AT(ws, L.row_token, int32_t *), row_gate, x_perm, ws, s));
  TRY(do_ffn(D, L, x_perm, offsets, w1, b1, w2, b2, row_gate, AT(ws, L.h, void *), y_perm, ws, s));
  TRY(do_shared(D, L, x, sw1, sb1, sw2, sb2, ws, s));
  TRY(do_combine(D, L, y_perm, row_of, gate, x, y, ws, s));
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(void *ws, int64_t limit_ns, int32_t *result, moe_stream_t stream) {
  TRY(check_ptrs({ws, result}, "moe_selftest_wait_timeout"));
  if (limit_ns < 1000 || limit_ns > 1000000000)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in [1000, 1e9] (got %lld)", (long long)limit_ns);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(result, 0, 8 * sizeof(int32_t), s);
  if (e == cudaSuccess)
    e = launch_wait_expiry(static_cast<int32_t *>(ws), result + 4, (unsigned long long)limit_ns, result, s);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test");
  return MOE_OK;
}

}  // extern "C"
