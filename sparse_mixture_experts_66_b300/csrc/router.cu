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
// Layout of the work: a CTA of 8 warps owns 32 consecutive tokens, 4 per
// warp. A warp streams its 4 token rows with 16-byte loads (each lane takes
// every 32nd vector) against the rows of W_g for a chunk of 8 experts, so
// each lane holds 4 x 8 = 32 partial dot products. One shuffle
// reduce-scatter (31 shuffles) leaves lane L with the full logit of token
// L/8, expert L%8 of the chunk. Logits go to shared memory; then each warp
// reduces its tokens' softmax and top-k across lanes with shuffles (lane L
// holds experts L, L+32, ...).
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kTokPerWarp = 4;
constexpr int kTokPerBlock = kWarps * kTokPerWarp;
constexpr int kEC = 8;  // experts per chunk: kTokPerWarp * kEC = 32 partial sums per lane
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

// 32 values per lane -> lane L returns the warp-wide sum of value L.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      float send = up ? v[i] : v[i + half];
      float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, half);
    }
  }
  return v[0];
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) router_kernel(const T *__restrict__ x, const T *__restrict__ w_g,
                                                             const float *__restrict__ router_bias, int64_t T_,
                                                             int d, int N, int k, int32_t *__restrict__ topk_idx,
                                                             float *__restrict__ gate, float *__restrict__ score) {
  extern __shared__ float s_logits[];  // [kTokPerBlock][N]
  constexpr int V = VecN<T>::n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok0 = (int64_t)blockIdx.x * kTokPerBlock + warp * kTokPerWarp;
  const int nvec = d / V;

  for (int e0 = 0; e0 < N; e0 += kEC) {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float xv[kTokPerWarp][V];
#pragma unroll
      for (int tk = 0; tk < kTokPerWarp; ++tk) {
        if (tok0 + tk < T_) {
          load16(x + (tok0 + tk) * (int64_t)d + (int64_t)v * V, xv[tk]);
        } else {
#pragma unroll
          for (int q = 0; q < V; ++q) xv[tk][q] = 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < kEC; ++e) {
        if (e0 + e < N) {
          float wv[V];
          load16(w_g + (int64_t)(e0 + e) * d + (int64_t)v * V, wv);
#pragma unroll
          for (int tk = 0; tk < kTokPerWarp; ++tk)
#pragma unroll
            for (int q = 0; q < V; ++q) acc[tk * kEC + e] = fmaf(xv[tk][q], wv[q], acc[tk * kEC + e]);
        }
      }
    }
    const float r = reduce_scatter32(acc, lane);
    const int tk = lane >> 3, e = e0 + (lane & 7);
    if (e < N) s_logits[(warp * kTokPerWarp + tk) * N + e] = r;
  }
  __syncwarp();

  for (int tk = 0; tk < kTokPerWarp; ++tk) {
    const int64_t t = tok0 + tk;
    if (t >= T_) break;
    const float *L = s_logits + (warp * kTokPerWarp + tk) * N;
    float lv[8];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      lv[i] = -INFINITY;
      if (e < N) {
        lv[i] = L[e];
        if (router_bias) lv[i] += router_bias[e];
        m = fmaxf(m, lv[i]);
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
}

}  // namespace

cudaError_t launch_router(const Dims &D, const void *x, const void *w_g, const float *router_bias,
                          int32_t *topk_idx, float *gate, float *score, int32_t *status, cudaStream_t s) {
  (void)status;
  const unsigned grid = (unsigned)((D.T + kTokPerBlock - 1) / kTokPerBlock);
  const size_t smem = sizeof(float) * kTokPerBlock * D.N;
  if (D.dt == MOE_DT_BF16) {
    router_kernel<__nv_bfloat16><<<grid, kWarps * 32, smem, s>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w_g, router_bias, D.T, (int)D.d, D.N, D.k, topk_idx,
        gate, score);
  } else {
    router_kernel<float><<<grid, kWarps * 32, smem, s>>>((const float *)x, (const float *)w_g, router_bias, D.T,
                                                         (int)D.d, D.N, D.k, topk_idx, gate, score);
  }
  return cudaGetLastError();
}

}  // namespace moe
