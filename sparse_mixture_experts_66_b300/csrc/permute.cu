// K3, dispatch gather, and K6, combine.
//
// Dispatch, "Mixture-of-Experts" (beta.fermi.ai wiki) step 5: gather each
// expert's kept tokens into a per-expert batch. x_perm[r] = x[row_token[r]]
// for every row in use; padding rows are written as zeros so that every row
// a GEMM tile reads is finite. One warp per row, 16-byte vectors, so each
// warp reads and writes whole contiguous rows (coalesced).
//
// Combine, step 7: y_t = sum over the token's kept picks, in pick order, of
// the gate-scaled expert output (the scaling is fused into the second expert
// GEMM). Each token's rows are found through row_of, so the sum is a gather,
// with no atomics and a fixed order: the result is deterministic. Variants:
// renormalise over the surviving picks (wiki worked example), and the
// pseudocode's identity fallback for a token whose picks were all dropped.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) permute_kernel(const uint4 *__restrict__ x, int64_t vec_per_row,
                                                              const int32_t *__restrict__ offsets, int N,
                                                              const int32_t *__restrict__ row_token, int64_t T,
                                                              int64_t R_max, uint4 *__restrict__ x_perm,
                                                              int32_t *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t rows = offsets[N];
  if (rows > R_max) rows = R_max;  // a failed assign leaves offsets unchecked; never write past the buffer
  for (int64_t r = (int64_t)blockIdx.x * kWarps + warp; r < rows; r += (int64_t)gridDim.x * kWarps) {
    const int32_t t = row_token[r];
    uint4 *dst = x_perm + r * vec_per_row;
    if (t >= 0 && t < T) {
      const uint4 *src = x + (int64_t)t * vec_per_row;
      for (int64_t v0 = lane; v0 < vec_per_row; v0 += 32 * 4) {  // 4 loads in flight before the stores
        uint4 tmp[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (v0 + 32 * j < vec_per_row) tmp[j] = __ldg(src + v0 + 32 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (v0 + 32 * j < vec_per_row) dst[v0 + 32 * j] = tmp[j];
      }
    } else {
      if (t >= T && lane == 0) report_error(status, MOE_ERR_BOUNDS, kKPermute, (int32_t)r);
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int64_t v = lane; v < vec_per_row; v += 32) dst[v] = z;
    }
  }
}

template <typename T> struct Store4;
template <> struct Store4<float> {
  static __device__ __forceinline__ void st(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
  static __device__ __forceinline__ float4 ld(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
};
template <> struct Store4<__nv_bfloat16> {
  static __device__ __forceinline__ void st(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
  }
  static __device__ __forceinline__ float4 ld(const __nv_bfloat16 *p) {
    uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
  }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const float *__restrict__ y_perm,
                                                              const float *__restrict__ y_split, int nsplit,
                                                              int64_t d,
                                                              const int32_t *__restrict__ row_of,
                                                              const float *__restrict__ gate,
                                                              const T *__restrict__ x, int64_t T_, int k,
                                                              int64_t R_max, uint32_t flags, T *__restrict__ y,
                                                              int32_t *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < T_; t += (int64_t)gridDim.x * kWarps) {
    int32_t rows[8];
    int nkept = 0;
    float kept_gate = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      rows[j] = -1;
      if (j < k) {
        int32_t r = row_of[t * k + j];
        if (r >= R_max) {
          if (lane == 0) report_error(status, MOE_ERR_BOUNDS, kKCombine, (int32_t)t);
          r = -1;
        }
        rows[j] = r;
        if (r >= 0) {
          ++nkept;
          if (flags & MOE_FLAG_RENORM_SURVIVORS) kept_gate += gate[t * k + j];
        }
      }
    }
    const bool renorm = (flags & MOE_FLAG_RENORM_SURVIVORS) && nkept > 0;
    const bool identity = (flags & MOE_FLAG_IDENTITY_FALLBACK) && nkept == 0;
    constexpr int B = 4;  // column groups per pass: B loads per kept pick in flight
    for (int64_t c0 = (int64_t)lane * 4; c0 < d; c0 += 128 * B) {
      float4 acc[B];
#pragma unroll
      for (int b = 0; b < B; ++b) acc[b] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (rows[j] >= 0) {
          // the pick's row: y_perm, then the K slices of a decode-mode GEMM in order
          for (int sl = 0; sl <= nsplit; ++sl) {
            float4 v[B];
            const float *src = (sl == 0 ? y_perm : y_split + (int64_t)(sl - 1) * R_max * d) + (int64_t)rows[j] * d;
#pragma unroll
            for (int b = 0; b < B; ++b)
              if (c0 + 128 * b < d) v[b] = __ldg(reinterpret_cast<const float4 *>(src + c0 + 128 * b));
#pragma unroll
            for (int b = 0; b < B; ++b) {
              if (c0 + 128 * b < d) {
                acc[b].x += v[b].x;
                acc[b].y += v[b].y;
                acc[b].z += v[b].z;
                acc[b].w += v[b].w;
              }
            }
          }
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int64_t c = c0 + 128 * b;
        if (c >= d) continue;
        float4 a = acc[b];
        if (renorm) {
          a.x /= kept_gate;
          a.y /= kept_gate;
          a.z /= kept_gate;
          a.w /= kept_gate;
        }
        if (identity) a = Store4<T>::ld(x + t * d + c);
        Store4<T>::st(y + t * d + c, a);
      }
    }
  }
}

unsigned grid_for(int64_t items, int per_block) {
  int64_t g = (items + per_block - 1) / per_block;
  const int64_t cap = 148 * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace

cudaError_t launch_permute(const Dims &D, const void *x, const int32_t *offsets, const int32_t *row_token,
                           void *x_perm, int32_t *status, cudaStream_t s) {
  const size_t es = D.dt == MOE_DT_BF16 ? 2 : 4;
  const int64_t vpr = D.d * (int64_t)es / 16;
  permute_kernel<<<grid_for(D.R_max, kWarps), kWarps * 32, 0, s>>>((const uint4 *)x, vpr, offsets, D.N, row_token,
                                                                   D.T, D.R_max, (uint4 *)x_perm, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Dims &D, const float *y_perm, const float *y_split, int nsplit,
                           const int32_t *row_of, const float *gate, const void *x, void *y, int32_t *status,
                           cudaStream_t s) {
  const unsigned g = grid_for(D.T, kWarps);
  if (!y_split) nsplit = 0;
  if (D.dt == MOE_DT_BF16)
    combine_kernel<__nv_bfloat16><<<g, kWarps * 32, 0, s>>>(y_perm, y_split, nsplit, D.d, row_of, gate,
                                                            (const __nv_bfloat16 *)x, D.T, D.k, D.R_max, D.flags,
                                                            (__nv_bfloat16 *)y, status);
  else
    combine_kernel<float><<<g, kWarps * 32, 0, s>>>(y_perm, y_split, nsplit, D.d, row_of, gate, (const float *)x,
                                                    D.T, D.k, D.R_max, D.flags, (float *)y, status);
  return cudaGetLastError();
}

}  // namespace moe
