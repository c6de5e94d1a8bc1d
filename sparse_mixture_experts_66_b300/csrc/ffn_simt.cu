// K8, the expert FFNs on CUDA cores (fp32 FMA): the path of fp32 workloads.
//
// "Mixture of Experts (MoE): Architecture, Routing, and Scaling" (syntave.com),
// "Core Architecture": FFN(x) = W2 GELU(W1 x + b1) + b2, one FFN per expert.
// Rows of the permuted buffer are grouped by expert in segments that start on
// multiples of 128 rows, so a 64-row tile belongs to exactly one expert.
//   epilogue 1: out = GELU(acc + b1[e])                   (first GEMM)
//   epilogue 2: out = row_gate[r] * (acc + b2[e])         (second GEMM, in x's dtype)
// fp32 is kept on CUDA cores on purpose: tf32 tensor cores round the inputs
// to a 10-bit mantissa, which cannot meet a 1e-4 relative bound.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

// kRowBound: A has fewer rows than the segments cover (the shared expert reads
// x in place); rows past a_rows read as zeros.
template <typename Tin, typename Tout, int EPI, bool kRowBound>
__global__ void __launch_bounds__(256) ffn_simt_kernel(const Tin *__restrict__ A, int64_t a_rows, int64_t K,
                                                       const Tin *__restrict__ B, const Tin *__restrict__ bias,
                                                       int64_t N_out, const float *__restrict__ row_gate,
                                                       const int32_t *__restrict__ offsets, int N_exp,
                                                       Tout *__restrict__ out) {
  pdl_wait();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int64_t m0 = (int64_t)blockIdx.y * BM;
  if (m0 >= offsets[N_exp]) return;
  const int e = segment_of(offsets, N_exp, m0);
  const int64_t n0 = (int64_t)blockIdx.x * BN;
  const Tin *Be = B + (int64_t)e * N_out * K;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int64_t k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int l = tid + q * 256;
      const int r = l / BK, c = l % BK;
      const int64_t kk = k0 + c;
      As[c][r] = (kk < K && (!kRowBound || m0 + r < a_rows)) ? to_f32(A[(m0 + r) * K + kk]) : 0.f;
      const int64_t n = n0 + r;
      Bs[c][r] = (kk < K && n < N_out) ? to_f32(Be[n * K + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = m0 + ty * 4 + i;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= N_out) continue;
      const float v = acc[i][j] + to_f32(bias[(int64_t)e * N_out + n]);
      if (EPI == 1) {
        out[r * N_out + n] = from_f32<Tout>(gelu_erf(v));
      } else {
        out[r * N_out + n] = from_f32<Tout>(row_gate ? row_gate[r] * v : v);
      }
    }
  }
}

}  // namespace

cudaError_t launch_ffn_simt(const Dims &D, int epi, const void *A, int64_t a_rows, int64_t K, const void *B,
                            const void *bias, int64_t N_out, const float *row_gate, const int32_t *offsets, void *out,
                            int32_t *status, cudaStream_t s) {
  (void)status;
  const dim3 grid((unsigned)((N_out + BN - 1) / BN), (unsigned)(D.R_max / BM));
  const bool bound = a_rows < D.R_max;
  if (D.dt == MOE_DT_F32) {
    auto kern = epi == 1 ? (bound ? ffn_simt_kernel<float, float, 1, true> : ffn_simt_kernel<float, float, 1, false>)
                         : (bound ? ffn_simt_kernel<float, float, 2, true> : ffn_simt_kernel<float, float, 2, false>);
    return launch_k(kern, grid, dim3(256), 0, s, 1u, (const float *)A, a_rows, K, (const float *)B,
                    (const float *)bias, N_out, row_gate, offsets, D.N, (float *)out);
  }
  if (epi == 1)
    return launch_k(bound ? ffn_simt_kernel<__nv_bfloat16, __nv_bfloat16, 1, true>
                          : ffn_simt_kernel<__nv_bfloat16, __nv_bfloat16, 1, false>,
                    grid, dim3(256), 0, s, 1u, (const __nv_bfloat16 *)A, a_rows, K, (const __nv_bfloat16 *)B,
                    (const __nv_bfloat16 *)bias, N_out, row_gate, offsets, D.N, (__nv_bfloat16 *)out);
  return launch_k(bound ? ffn_simt_kernel<__nv_bfloat16, __nv_bfloat16, 2, true>
                        : ffn_simt_kernel<__nv_bfloat16, __nv_bfloat16, 2, false>,
                  grid, dim3(256), 0, s, 1u, (const __nv_bfloat16 *)A, a_rows, K, (const __nv_bfloat16 *)B,
                  (const __nv_bfloat16 *)bias, N_out, row_gate, offsets, D.N, (__nv_bfloat16 *)out);
}

}  // namespace moe
