// K1, the fused router: gate projection, softmax over N experts, top-k and
// renormalisation of the top-k scores.
//
// "Mixture-of-Experts" (beta.fermi.ai wiki), step-by-step mechanism, steps
// 1-3: logits x W_g, softmax over the N experts, the k largest by score,
// renormalised to sum to 1. Softmax is strictly increasing in the logit, so
// ranking the fp32 logits picks the same experts as ranking the scores. The
// logits are accumulated and kept in fp32 (never rounded to bf16), following
// "Inside the Router" of "Mixture of Experts: How Sparse Routing Scales
// Transformers" (router logits at higher precision).
//
// Layout of the work: one warp owns two tokens. Lanes stream the two token
// rows with 16-byte loads (lane l takes every 32nd vector) against the rows of
// W_g for a chunk of 8 experts (L1-resident), so each lane holds 2 x 8 partial
// dot products. A shuffle reduce-scatter (offsets 16, 8, 4, 2, then a final
// exchange at offset 1: 16 shuffles) leaves lane L with the full logit of
// token L/16, expert (L/2)%8 of the chunk. With N <= 8 the whole softmax and
// top-k then run in registers: the 16 lanes of a token reduce with shuffles
// at offsets 8, 4, 2 (lanes L and L^1 hold the same value). With more experts
// the chunk logits go to shared memory and each token is finished by the warp
// with lane L holding experts L, L+32, ...
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kTokPerWarp = 2;
constexpr int kTokPerBlock = kWarps * kTokPerWarp;
constexpr int kEC = 8;  // experts per chunk
constexpr size_t kMaxStagedW = 96 * 1024;  // W_g bytes staged in shared memory per CTA
constexpr unsigned kFull = 0xffffffffu;

template <typename T> struct VecN;
template <> struct VecN<float> { static constexpr int n = 4; };
template <> struct VecN<__nv_bfloat16> { static constexpr int n = 8; };

__device__ __forceinline__ void load16(const float *p, float (&v)[4]) {
  float4 q = __ldg(reinterpret_cast<const float4 *>(p));
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// W_g rows may live in shared memory (staged) or global memory: generic loads.
__device__ __forceinline__ void load16w(const float *p, float (&v)[4]) {
  float4 q = *reinterpret_cast<const float4 *>(p);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load16w(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 q = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// 16 values per lane -> lane L returns the warp-wide sum of value (L >> 1) & 15.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int n = 16, off = 16; n >= 2; n >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
    const int h = n >> 1;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  return v[0] + __shfl_xor_sync(kFull, v[0], 1);
}

// Partial logits of 2 tokens x 8 experts (e0 .. e0+7) for this lane's slice.
// Each pass first issues the loads of kBatch vectors of both token rows (so
// that many bytes are in flight per lane), then walks the expert rows (L1).
constexpr int kBatch = 4;
// x0, x1 and w_g point at the first column of a slice of len columns; d is
// the row stride of W_g.
template <typename T>
__device__ __forceinline__ void chunk_logits(const T *__restrict__ x0, const T *__restrict__ x1, bool has1,
                                             const T *__restrict__ w_g, int d, int len, int N, int e0, int lane,
                                             float (&acc)[16]) {
  constexpr int V = VecN<T>::n;
  const int nvec = len / V;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int vb = lane; vb < nvec; vb += 32 * kBatch) {
    float xa[kBatch][V], xb[kBatch][V];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int v = vb + 32 * j;
      if (v < nvec) {
        load16(x0 + (int64_t)v * V, xa[j]);
        if (has1) {
          load16(x1 + (int64_t)v * V, xb[j]);
        } else {
#pragma unroll
          for (int q = 0; q < V; ++q) xb[j][q] = 0.f;
        }
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) xa[j][q] = xb[j][q] = 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < kEC; ++e) {
      if (e0 + e < N) {
        const T *wr = w_g + (int64_t)(e0 + e) * d;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int v = vb + 32 * j;
          if (v < nvec) {
            float wv[V];
            load16w(wr + (int64_t)v * V, wv);
#pragma unroll
            for (int q = 0; q < V; ++q) {
              acc[e] = fmaf(xa[j][q], wv[q], acc[e]);
              acc[8 + e] = fmaf(xb[j][q], wv[q], acc[8 + e]);
            }
          }
        }
      }
    }
  }
}

// N <= 8: everything in registers. W_g is staged in shared memory by one
// cooperative load per CTA (when it fits), so the projection reads it at
// shared-memory latency instead of a chain of cache misses.
template <typename T, bool kStageW>
__global__ void __launch_bounds__(kWarps * 32) router_small_kernel(const T *__restrict__ x, const T *__restrict__ w_g,
                                                                   const float *__restrict__ router_bias, int64_t T_,
                                                                   int d, int N, int k, int32_t *__restrict__ topk_idx,
                                                                   float *__restrict__ gate,
                                                                   float *__restrict__ score,
                                                                   float *__restrict__ probs,
                                                                   float *__restrict__ lse) {
  pdl_wait();
  extern __shared__ uint4 s_w[];  // [N * d * sizeof(T) / 16]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T *w = w_g;
  if (kStageW) {
    const int nv = N * d * (int)sizeof(T) / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(w_g);
    for (int i = threadIdx.x; i < nv; i += kWarps * 32) s_w[i] = __ldg(src + i);
    __syncthreads();
    w = reinterpret_cast<const T *>(s_w);
  }
  const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * kTokPerWarp;
  if (t0 >= T_) return;
  const bool has1 = t0 + 1 < T_;
  float acc[16];
  chunk_logits(x + t0 * d, x + (t0 + 1) * d, has1, w, d, d, N, 0, lane, acc);
  float l = reduce_scatter16(acc, lane);
  const int e = (lane >> 1) & 7;
  const int64_t t = t0 + (lane >> 4);
  const bool valid = e < N;
  if (valid && router_bias) l += router_bias[e];
  if (!valid) l = -INFINITY;
  float m = l;
#pragma unroll
  for (int off = 8; off >= 2; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  const float ex = valid ? expf(l - m) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 8; off >= 2; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  if (probs && t < T_) {  // router statistics (lanes L and L^1 hold the same expert)
    if (valid && (lane & 1) == 0) probs[t * N + e] = ex / s;
    if ((lane & 15) == 0) lse[t] = m + logf(s);
  }
  bool taken = !valid;
  float sel_ex[8];
  int sel_e[8];
  float sel_sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      float bv = taken ? -INFINITY : l;
      int be = taken ? 0x7fffffff : e;
#pragma unroll
      for (int off = 8; off >= 2; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (be == e) taken = true;
      sel_e[j] = be;
      sel_ex[j] = expf(bv - m);
      sel_sum += sel_ex[j];
    }
  }
  if ((lane & 15) == 0 && t < T_) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        topk_idx[t * k + j] = sel_e[j];
        score[t * k + j] = sel_ex[j] / s;
        gate[t * k + j] = sel_ex[j] / sel_sum;
      }
    }
  }
}

// Softmax, top-k and renormalisation of one token by one warp: lane L holds
// the logits of experts L, L+32, ... (no bias yet) in lv. Ties go to the lower
// expert; the picks are written in rank order.
__device__ __forceinline__ void finish_token(float (&lv)[8], const float *__restrict__ router_bias, int N, int k,
                                             int lane, int64_t t, int32_t *__restrict__ topk_idx,
                                             float *__restrict__ gate, float *__restrict__ score,
                                             float *__restrict__ probs, float *__restrict__ lse) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < N) {
      if (router_bias) lv[i] += router_bias[e];
      m = fmaxf(m, lv[i]);
    } else {
      lv[i] = -INFINITY;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i < N) s += expf(lv[i] - m);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  if (probs) {  // router statistics: the full probability row and the logsumexp
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < N) probs[t * N + lane + 32 * i] = expf(lv[i] - m) / s;
    if (lane == 0) lse[t] = m + logf(s);
  }
  uint32_t taken = 0;
  float sel_ex[8];
  int sel_e[8];
  float sel_sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < N && !(taken & (1u << i)) && (lv[i] > bv || (lv[i] == bv && e < be))) {
          bv = lv[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_e[j] = be;
      sel_ex[j] = expf(bv - m);
      sel_sum += sel_ex[j];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        topk_idx[t * k + j] = sel_e[j];
        score[t * k + j] = sel_ex[j] / s;
        gate[t * k + j] = sel_ex[j] / sel_sum;
      }
    }
  }
}

// Any N <= 256: chunk logits through shared memory.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) router_kernel(const T *__restrict__ x, const T *__restrict__ w_g,
                                                             const float *__restrict__ router_bias, int64_t T_,
                                                             int d, int N, int k, int32_t *__restrict__ topk_idx,
                                                             float *__restrict__ gate, float *__restrict__ score,
                                                             float *__restrict__ probs, float *__restrict__ lse) {
  pdl_wait();
  extern __shared__ float s_logits[];  // [kTokPerBlock][N]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * kTokPerWarp;
  if (t0 >= T_) return;
  const bool has1 = t0 + 1 < T_;
  float *my = s_logits + warp * kTokPerWarp * N;
  for (int e0 = 0; e0 < N; e0 += kEC) {
    float acc[16];
    chunk_logits(x + t0 * d, x + (t0 + 1) * d, has1, w_g, d, d, N, e0, lane, acc);
    const float r = reduce_scatter16(acc, lane);
    const int e = e0 + ((lane >> 1) & 7);
    if ((lane & 1) == 0 && e < N) my[(lane >> 4) * N + e] = r;
  }
  __syncwarp();
  for (int tk = 0; tk < kTokPerWarp; ++tk) {
    const int64_t t = t0 + tk;
    if (t >= T_) break;
    const float *L = my + tk * N;
    float lv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) lv[i] = lane + 32 * i < N ? L[lane + 32 * i] : -INFINITY;
    finish_token(lv, router_bias, N, k, lane, t, topk_idx, gate, score, probs, lse);
  }
}

// Small batches: one CTA per pair of tokens, the 8 warps splitting d. Each
// warp forms the partial logits of both tokens over its slice of columns
// (8 experts at a time), the partials meet in shared memory and are summed in
// warp order (deterministic), and warps 0 and 1 finish one token each. The
// many CTAs keep enough bytes of x in flight even when T is a few dozen.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) router_split_kernel(const T *__restrict__ x,
                                                                   const T *__restrict__ w_g,
                                                                   const float *__restrict__ router_bias,
                                                                   int64_t T_, int d, int N, int k,
                                                                   int32_t *__restrict__ topk_idx,
                                                                   float *__restrict__ gate,
                                                                   float *__restrict__ score,
                                                                   float *__restrict__ probs,
                                                                   float *__restrict__ lse) {
  pdl_wait();
  extern __shared__ float s_part[];  // [kWarps][kTokPerWarp][N]
  constexpr int V = VecN<T>::n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = (int64_t)blockIdx.x * kTokPerWarp;
  const bool has1 = t0 + 1 < T_;
  const int nv = d / V;
  const int v0 = warp * nv / kWarps, v1 = (warp + 1) * nv / kWarps;
  const int c0 = v0 * V, len = (v1 - v0) * V;
  float *my = s_part + warp * kTokPerWarp * N;
  for (int e0 = 0; e0 < N; e0 += kEC) {
    float acc[16];
    chunk_logits(x + t0 * d + c0, x + (t0 + 1) * d + c0, has1, w_g + c0, d, len, N, e0, lane, acc);
    const float r = reduce_scatter16(acc, lane);
    const int e = e0 + ((lane >> 1) & 7);
    if ((lane & 1) == 0 && e < N) my[(lane >> 4) * N + e] = r;
  }
  __syncthreads();
  if (warp < kTokPerWarp) {
    const int64_t t = t0 + warp;
    if (t < T_) {
      float lv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        float v = 0.f;
        if (e < N)
          for (int w = 0; w < kWarps; ++w) v += s_part[(w * kTokPerWarp + warp) * N + e];
        lv[i] = v;
      }
      finish_token(lv, router_bias, N, k, lane, t, topk_idx, gate, score, probs, lse);
    }
  }
}

}  // namespace

// The three SIMT router kernels share one argument list.
template <typename T>
static cudaError_t launch_router_t(const Dims &D, const T *x, const T *w_g, const float *router_bias,
                                   int32_t *topk_idx, float *gate, float *score, float *probs, float *lse,
                                   cudaStream_t s) {
  if (router_split(D)) {
    const unsigned g = (unsigned)((D.T + kTokPerWarp - 1) / kTokPerWarp);
    const size_t smem = sizeof(float) * kWarps * kTokPerWarp * D.N;
    return launch_k(router_split_kernel<T>, dim3(g), dim3(kWarps * 32), smem, s, 1u, x, w_g, router_bias, D.T,
                    (int)D.d, D.N, D.k, topk_idx, gate, score, probs, lse);
  }
  const unsigned grid = (unsigned)((D.T + kTokPerBlock - 1) / kTokPerBlock);
  if (D.N <= kEC) {
    const size_t wbytes = (size_t)D.N * D.d * sizeof(T);
    const bool stage = wbytes <= kMaxStagedW;
    const size_t smem = stage ? wbytes : 0;
    auto kern = stage ? router_small_kernel<T, true> : router_small_kernel<T, false>;
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    return launch_k(kern, dim3(grid), dim3(kWarps * 32), smem, s, 1u, x, w_g, router_bias, D.T, (int)D.d, D.N, D.k,
                    topk_idx, gate, score, probs, lse);
  }
  const size_t smem = sizeof(float) * kTokPerBlock * D.N;
  return launch_k(router_kernel<T>, dim3(grid), dim3(kWarps * 32), smem, s, 1u, x, w_g, router_bias, D.T, (int)D.d,
                  D.N, D.k, topk_idx, gate, score, probs, lse);
}

cudaError_t launch_router(const Dims &D, const void *x, const void *w_g, const float *router_bias,
                          int32_t *topk_idx, float *gate, float *score, float *probs, float *lse, int32_t *status,
                          cudaStream_t s) {
  (void)status;
  if (D.dt == MOE_DT_BF16)
    return launch_router_t(D, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w_g, router_bias, topk_idx, gate,
                           score, probs, lse, s);
  return launch_router_t(D, (const float *)x, (const float *)w_g, router_bias, topk_idx, gate, score, probs, lse, s);
}

}  // namespace moe
