// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "moe.h"

namespace moe {

// Every expert segment of the permuted buffers starts on a multiple of this
// many rows, so that a 128-row GEMM tile never spans two experts.
constexpr int kRowAlign = 128;
// Decode-shaped batches (at most this many expected rows per expert,
// T*k <= 64*N) run the swap-AB expert GEMMs, whose token chunks are 64 rows,
// or 32 rows when an expert averages at most 16 (T*k <= 16*N): their segments
// start on multiples of the chunk size instead.
constexpr int kDecodeRowsPerExpert = 64;
constexpr int kDecodeSmallRowsPerExpert = 16;

// Kernel ids recorded next to a device error code in the status word.
enum KernelId : int32_t {
  kKRouter = 1,
  kKCapSelect = 2,
  kKCapAssign = 3,
  kKPermute = 4,
  kKGemmSimt = 5,
  kKCombine = 6,
  kKGemmTc = 7,
  kKGemmTcDecode = 8,
  kKSelfTest = 9,
};

// ---- per-device host state ---------------------------------------------
// One-time facts and settings that belong to a device (its SM count, a
// kernel's opt-in shared-memory size, how many clusters fit at once) are kept
// per device: one process may drive several GPUs, and cudaFuncSetAttribute
// applies only to the device that is current when it is called. A value is
// made once per device, with that device current, under a lock, so first
// calls from several host threads are safe.
constexpr int kMaxDevices = 64;

template <typename T> class PerDevice {
 public:
  // *out = the current device's value; make(T *) fills it on first use and
  // returns a cudaError_t (the value is kept only when make succeeds).
  template <typename Make> cudaError_t get(Make &&make, T *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[dev]) {
      T v{};
      e = make(&v);
      if (e != cudaSuccess) return e;
      val_[dev] = v;
      ready_[dev] = true;
    }
    *out = val_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool ready_[kMaxDevices] = {};
  T val_[kMaxDevices] = {};
};

// Streaming multiprocessors of the current device (148 if it cannot be read).
int num_sms();

struct Dims {
  int64_t T, d, d_ff;
  int32_t N, k;
  int64_t C;      // capacity
  int64_t R_max;  // row capacity of the permuted buffers
  moe_dtype dt;
  uint32_t flags;
};

// Record the first device-side error: status[0] = code, status[1] = kernel,
// status[2] = detail. Later errors leave the first one in place.
__device__ __forceinline__ void report_error(int32_t *status, int32_t code, int32_t kernel, int32_t detail) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = kernel;
    status[2] = detail;
  }
}

// Programmatic dependent launch. Every kernel is launched with programmatic
// stream serialisation: it may start while the previous kernel of the stream
// finishes, and waits for that kernel's completion and memory (pdl_wait)
// before it touches global memory. The persistent tensor-core kernels let
// their successor launch as soon as a CTA has no work left (pdl_trigger); the
// other kernels let it launch as their CTAs exit. What overlaps is the launch
// latency and the prologue (barrier set-up, tensor-memory allocation) that
// needs no global memory.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialisation (and clusters of `cluster`
// CTAs along x when cluster > 1).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            unsigned cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Exact GELU, u * Phi(u), with CUDA's erff (fp32 path).
__device__ __forceinline__ float gelu_erf(float u) { return 0.5f * u * (1.0f + erff(u * 0.70710678118654752440f)); }

// GELU for the bf16 tensor-core epilogue: u * Phi(u) with erf from the
// rational-exponential approximation of Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (Hastings):
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),
//   t = 1 / (1 + p z), z >= 0, |error| <= 1.5e-7,
// evaluated without branches (one reciprocal, one exp2). The result is stored
// in bf16 (relative step 2^-8), so the approximation is invisible in h. For
// u < 0 the complement is used directly, so tiny outputs lose no precision:
//   GELU(u) = u (1 - q/2) for u >= 0,  u q/2 for u < 0,  q = erfc(|u|/sqrt 2).
__device__ __forceinline__ float gelu_as(float u) {
  const float z = fabsf(u) * 0.70710678118654752440f;
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, z, 1.0f)));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
  const float q = poly * exp2f(-z * z * 1.44269504088896341f);
  return u >= 0.f ? u * fmaf(-0.5f, q, 1.0f) : 0.5f * u * q;
}

// gelu_as on two values at once, with the multiply-adds on the packed
// two-lane fp32 units (one instruction per pair) and the reciprocal and exp2
// per value. Same erf (A&S 7.1.26, x = |u|/sqrt 2), arranged to need no sign
// select and no cancellation: GELU(u) = max(u, 0) - |u| erfc(x)/2, with
// erfc(x)/2 = (sum of a_i t^i)/2 * exp(-x^2); the factor -1/2 is folded into
// the coefficients, 1/sqrt 2 into p and into the exponent (-u^2/2, base 2).
__device__ __forceinline__ float2 gelu_as2(float2 u) {
  const float2 au = make_float2(fabsf(u.x), fabsf(u.y));
  const float2 den = __ffma2_rn(make_float2(0.23164188826636f, 0.23164188826636f), au, make_float2(1.0f, 1.0f));
  float2 t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t.x) : "f"(den.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t.y) : "f"(den.y));
  float2 p = __ffma2_rn(t, make_float2(-0.5307027145f, -0.5307027145f), make_float2(0.7265760135f, 0.7265760135f));
  p = __ffma2_rn(t, p, make_float2(-0.7107068705f, -0.7107068705f));
  p = __ffma2_rn(t, p, make_float2(0.142248368f, 0.142248368f));
  p = __ffma2_rn(t, p, make_float2(-0.127414796f, -0.127414796f));
  p = __fmul2_rn(t, p);  // -(sum of a_i t^i)/2
  const float2 arg = __fmul2_rn(__fmul2_rn(u, u), make_float2(-0.72134752044448170f, -0.72134752044448170f));
  float2 e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(arg.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(arg.y));
  return __ffma2_rn(au, __fmul2_rn(p, e), make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)));  // relu(u) - |u| erfc/2
}

// The expert whose segment holds row r: offsets is non-decreasing, N+1 long.
__device__ __forceinline__ int segment_of(const int32_t *offsets, int N, int64_t r) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {  // largest e with offsets[e] <= r
    int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Replace the calling thread's moe_last_error() text.
void set_last_error(const char *text);

// ---- launchers (each returns the launch's cudaError_t) ----
// Batches small enough that the router splits each token's columns over a
// CTA's warps (few tokens would leave most SMs idle otherwise).
constexpr int64_t kSplitRouterMaxT = 1024;
inline bool router_split(const Dims &D) { return D.T <= kSplitRouterMaxT; }

// probs [T, N] and lse [T] (both NULL unless router statistics are on): every
// token's full probability row and the logsumexp of its logits.
cudaError_t launch_router(const Dims &D, const void *x, const void *w_g, const float *router_bias,
                          int32_t *topk_idx, float *gate, float *score, float *probs, float *lse, int32_t *status,
                          cudaStream_t s);

// Router on the tensor cores (bf16 inputs, N <= 256); cudaErrorNotSupported otherwise.
cudaError_t launch_router_tc(const Dims &D, const void *x, const void *w_g, const float *router_bias,
                             int32_t *topk_idx, float *gate, float *score, float *probs, float *lse, int32_t *status,
                             cudaStream_t s);

// Router statistics from the stored probabilities (fixed-order reductions):
// P [N] column means, losses[1] = mean lse^2, then f [N] and losses[0] = aux.
cudaError_t launch_router_stats(const Dims &D, const float *probs, const float *lse, const int32_t *counts_raw,
                                float *f, float *P, float *losses, cudaStream_t s);

cudaError_t launch_capacity(const Dims &D, const int32_t *topk_idx, const float *gate, const float *score,
                            int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets, uint32_t *sel_thr,
                            int32_t *sel_eq, int32_t *row_of, int32_t *row_token, float *row_gate,
                            int32_t *ffn_sync, int32_t *status, cudaStream_t s);

// Number of K slices of the decode-mode second GEMM (>= 1), or 0 when the
// config is not decode-shaped (bf16 and T*k <= 64*N).
int decode_splits(const Dims &D);
// Token rows per chunk of the decode-mode expert FFN (32 or 64).
int decode_chunk_rows(const Dims &D);
// Segment alignment of the permuted buffers for this config.
inline int row_align(const Dims &D) { return decode_splits(D) > 0 ? decode_chunk_rows(D) : kRowAlign; }

// Swap-AB expert FFNs for decode-shaped batches, both GEMMs in one launch.
// y_split holds the second GEMM's K slices 1..S-1 (S = decode_splits), each
// [R_max, d] fp32; h_done [N + 1] int32 counts stored h tiles per expert
// (zero on entry, left zero on exit).
cudaError_t launch_ffn_decode(const Dims &D, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                              void *y_perm, float *y_split, int32_t *h_done, int32_t *status, cudaStream_t s);

cudaError_t launch_permute(const Dims &D, const void *x, const int32_t *offsets, const int32_t *row_token,
                           void *x_perm, int32_t *status, cudaStream_t s);

// y_split / nsplit: the extra K slices of a decode-mode second GEMM (nsplit
// buffers of [R_max, d] after y_perm's own), added in slice order.
// y_perm and y_shared ([Tp, d] or NULL: the shared expert's output, added
// last) are in x's dtype; y_split is fp32.
cudaError_t launch_combine(const Dims &D, const void *y_perm, const float *y_split, int nsplit,
                           const int32_t *row_of, const float *gate, const void *x, const void *y_shared, void *y,
                           int32_t *status, cudaStream_t s);

// Grouped GEMM over expert segments with the two fused epilogues.
//   epi 1: out[r, n] = GELU(A[r] . B[e, n] + bias[e, n])            (dtype)
//   epi 2: out[r, n] = row_gate[r] * (A[r] . B[e, n] + bias[e, n])  (fp32)
// a_rows: rows of A that exist (rows past it read as zeros).
cudaError_t launch_ffn_simt(const Dims &D, int epi, const void *A, int64_t a_rows, int64_t K, const void *B,
                            const void *bias, int64_t N_out, const float *row_gate, const int32_t *offsets, void *out,
                            int32_t *status, cudaStream_t s);

// tcgen05 path (bf16). Returns cudaErrorNotSupported when the shape is not
// handled, so the caller can report MOE_ERR_UNSUPPORTED.
// Upper bound on the 256-row blocks of the permuted rows (one completion
// counter each in the fused tensor-core FFN): sum over experts of
// ceil(segment / 256) <= R_max / 256 + N.
inline int64_t ffn_blocks_max(const Dims &D) { return D.R_max / 256 + D.N; }

// Completion counters of the fused expert FFNs (bf16 configs): one per
// expert (decode-shaped) or per 256-row block, plus an exit count. They are
// zero between launches: set to zero by the workspace init and by every
// dispatch, and reset by the last CTA of every FFN launch.
inline int64_t ffn_sync_ints(const Dims &D) {
  if (D.dt != MOE_DT_BF16) return 0;
  return (decode_splits(D) > 0 ? (int64_t)D.N : ffn_blocks_max(D)) + 1;
}

// Both expert GEMMs of a bf16 config in one launch on CTA pairs; blk_done
// [ffn_blocks_max + 1] int32 counts stored h tiles per block (zero on entry,
// left zero on exit).
// a_rows: rows of x_perm that exist (TMA zero-fills the rest up to R_max).
cudaError_t launch_ffn_tc(const Dims &D, const void *x_perm, int64_t a_rows, const int32_t *offsets, const void *w1,
                          const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                          void *y_perm, int32_t *blk_done, int32_t *status, cudaStream_t s);

// Self-test of the bounded waits: one CTA waits on an mbarrier nothing arms
// and on a counter (*counter stays 0) nothing raises, each for limit_ns.
cudaError_t launch_wait_expiry(int32_t *status, const int32_t *counter, unsigned long long limit_ns,
                               int32_t *result, cudaStream_t s);

// Expert-choice requests: idx[t * N + j] = j for every token.
cudaError_t launch_ec_pattern(int32_t *idx, int64_t T, int N, cudaStream_t s);

// The shared expert's single segment {0, Tp} and zeroed FFN counters.
cudaError_t launch_shared_setup(int32_t *offsets, int64_t rows, int32_t *sync, int64_t n_sync, cudaStream_t s);

}  // namespace moe
