// Router statistics of a routed batch, from the probability rows and
// logsumexps the router stores under MOE_FLAG_ROUTER_STATS.
//
// "Mixture-of-Experts" (beta.fermi.ai wiki), the load-balancing auxiliary
// loss: f_e = the fraction of the router's picks that went to expert e,
// P_e = the mean router probability of e over the batch, aux = N * sum_e
// f_e P_e, which is 1 at a perfectly uniform split. "Mixture of Experts (MoE):
// Architecture, Routing, and Scaling", "Importance Loss and Z-Loss": z-loss =
// the mean over tokens of logsumexp(logits)^2.
//
// Two launches, both with sums in a fixed order, so the results are
// deterministic: one CTA per expert sums its probability column (thread i
// takes tokens i, i + 256, ...; then a fixed tree across the CTA), and one
// more CTA sums lse^2; then one warp forms f from the pick counts and the
// auxiliary loss in expert order.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 256;

// Fixed-order sum over the CTA: per-warp shuffle trees, then warp 0 adds the
// 8 warp sums in warp order.
__device__ __forceinline__ float block_sum(float v, float *s_warp) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  float total = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kStatThreads / 32; ++w) total += s_warp[w];
  return total;
}

// CTA e < N: P[e] = mean_t probs[t, e]; CTA N: losses[1] = mean_t lse[t]^2.
__global__ void __launch_bounds__(kStatThreads) stats_column_kernel(const float *__restrict__ probs,
                                                                    const float *__restrict__ lse, int64_t T_, int N,
                                                                    float *__restrict__ P, float *__restrict__ losses) {
  pdl_wait();
  __shared__ float s_warp[kStatThreads / 32];
  const int e = blockIdx.x;
  float acc = 0.f;
  if (e < N) {
    for (int64_t t = threadIdx.x; t < T_; t += kStatThreads) acc += probs[t * N + e];
  } else {
    for (int64_t t = threadIdx.x; t < T_; t += kStatThreads) acc += lse[t] * lse[t];
  }
  const float total = block_sum(acc, s_warp);
  if (threadIdx.x == 0) {
    if (e < N) P[e] = total / (float)T_;
    else losses[1] = total / (float)T_;
  }
}

// f[e] = counts_raw[e] / (T*k); losses[0] = N * sum_e f[e] P[e], in expert order.
__global__ void __launch_bounds__(32) stats_aux_kernel(const int32_t *__restrict__ counts_raw, const float *P,
                                                       int64_t T_, int k, int N, float *__restrict__ f,
                                                       float *__restrict__ losses) {
  pdl_wait();
  const float picks = (float)((double)T_ * k);
  for (int e = threadIdx.x; e < N; e += 32) f[e] = (float)counts_raw[e] / picks;
  __syncwarp();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int e = 0; e < N; ++e) a += ((float)counts_raw[e] / picks) * P[e];
    losses[0] = (float)N * a;
  }
}

}  // namespace

cudaError_t launch_router_stats(const Dims &D, const float *probs, const float *lse, const int32_t *counts_raw,
                                float *f, float *P, float *losses, cudaStream_t s) {
  cudaError_t e = launch_k(stats_column_kernel, dim3((unsigned)D.N + 1), dim3(kStatThreads), 0, s, 1u, probs, lse,
                           D.T, (int)D.N, P, losses);
  if (e != cudaSuccess) return e;
  return launch_k(stats_aux_kernel, dim3(1), dim3(32), 0, s, 1u, counts_raw, (const float *)P, D.T, (int)D.k,
                  (int)D.N, f, losses);
}

}  // namespace moe
