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
constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kWarps * 32) permute_kernel(const uint4 *__restrict__ x, int64_t vec_per_row,
                                                              const int32_t *__restrict__ offsets, int N,
                                                              const int32_t *__restrict__ row_token, int64_t T,
                                                              int64_t R_max, uint4 *__restrict__ x_perm,
                                                              int32_t *status) {
  pdl_wait();
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

// W (4 or 8) consecutive values of a row as floats, loaded through the
// read-only path, and stored back in the row's type.
template <int W>
__device__ __forceinline__ void ldv(const float *p, float (&v)[W]) {
#pragma unroll
  for (int i = 0; i < W; i += 4) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p + i));
    v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
  }
}
template <int W>
__device__ __forceinline__ void ldv(const __nv_bfloat16 *p, float (&v)[W]) {
  uint32_t w[W / 2];
  if (W == 8) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    w[0] = u.x; w[1] = u.y; w[W / 2 - 2] = u.z; w[W / 2 - 1] = u.w;
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    w[0] = u.x; w[W / 2 - 1] = u.y;
  }
#pragma unroll
  for (int i = 0; i < W / 2; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <int W>
__device__ __forceinline__ void stv(float *p, const float (&v)[W]) {
#pragma unroll
  for (int i = 0; i < W; i += 4) *reinterpret_cast<float4 *>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <int W>
__device__ __forceinline__ void stv(__nv_bfloat16 *p, const float (&v)[W]) {
  uint32_t w[W / 2];
#pragma unroll
  for (int i = 0; i < W / 2; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  if (W == 8) *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[W / 2 - 2], w[W / 2 - 1]);
  else *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[W / 2 - 1]);
}

// A 16-byte vector as W values of T, widened exactly to fp32.
template <typename T, int W> __device__ __forceinline__ void widen(uint4 q, float (&v)[W]);
template <> __device__ __forceinline__ void widen<float, 4>(uint4 q, float (&v)[4]) {
  v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y); v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
}
template <> __device__ __forceinline__ void widen<__nv_bfloat16, 8>(uint4 q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Combine, without K slices: a CTA owns U = 8 / KM tokens (KM >= k); its
// threads take W columns at a time (8 for bf16, 4 for fp32). The
// CTA reads the U x KM row indices once and turns them into source-row
// pointers (null for a dropped pick), so the column loop holds no index
// arithmetic, and every condition in it is uniform across the CTA. A thread
// keeps one 16-byte load per source row in flight (y_perm is in x's dtype: 8
// bf16 or 4 fp32 columns). The picks of a token are added, as fp32, in pick
// order, and the sum is rounded once to x's dtype.
constexpr int kC8Threads = 128;
template <typename T, int KM, int W>
__global__ void __launch_bounds__(kC8Threads) combine_kernel(const T *__restrict__ y_perm, int64_t d,
                                                             const int32_t *__restrict__ row_of,
                                                             const float *__restrict__ gate,
                                                             const T *__restrict__ x,
                                                             const T *__restrict__ y_shared, int64_t T_, int k,
                                                             int64_t R_max, uint32_t flags, T *__restrict__ y,
                                                             int32_t *status) {
  pdl_wait();
  constexpr int U = 8 / KM;
  const int64_t t0 = (int64_t)blockIdx.x * U;
  const T *src[U][KM];  // source row of each kept pick, or null
  float ksum[U];            // kept-gate sum (for MOE_FLAG_RENORM_SURVIVORS)
  bool live[U], renorm[U], ident[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t t = t0 + u;
    live[u] = t < T_;
    int nkept = 0;
    float kept_gate = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      int32_t r = (live[u] && j < k) ? __ldg(row_of + t * k + j) : -1;
      if (r >= R_max) {
        if (threadIdx.x == 0) report_error(status, MOE_ERR_BOUNDS, kKCombine, (int32_t)t);
        r = -1;
      }
      src[u][j] = r >= 0 ? y_perm + (int64_t)r * d : nullptr;
      if (r >= 0) {
        ++nkept;
        if (flags & MOE_FLAG_RENORM_SURVIVORS) kept_gate += __ldg(gate + t * k + j);
      }
    }
    ksum[u] = kept_gate;
    renorm[u] = (flags & MOE_FLAG_RENORM_SURVIVORS) && nkept > 0;
    ident[u] = (flags & MOE_FLAG_IDENTITY_FALLBACK) && nkept == 0;
  }
  static_assert(W * sizeof(T) == 16, "one 16-byte vector per source row and step");
  for (int64_t c = (int64_t)threadIdx.x * W; c < d; c += kC8Threads * W) {
    // raw 16-byte vectors (widened only when added: half the registers of
    // holding them as fp32, so more CTAs stay resident)
    uint4 raw[U][KM];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < KM; ++j)
        raw[u][j] = src[u][j] ? __ldg(reinterpret_cast<const uint4 *>(src[u][j] + c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!live[u]) continue;
      float a[W];
#pragma unroll
      for (int i = 0; i < W; ++i) a[i] = 0.f;
#pragma unroll
      for (int j = 0; j < KM; ++j)
        if (src[u][j]) {
          float v[W];
          widen<T, W>(raw[u][j], v);
#pragma unroll
          for (int i = 0; i < W; ++i) a[i] += v[i];
        }
      if (renorm[u])
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] /= ksum[u];
      if (ident[u]) ldv<W>(x + (t0 + u) * d + c, a);
      if (y_shared) {  // the shared expert, added last
        float sh[W];
        ldv<W>(y_shared + (t0 + u) * d + c, sh);
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] += sh[i];
      }
      stv<W>(y + (t0 + u) * d + c, a);
    }
  }
}

// Combine of many picks per token (k > 8: expert-choice routing, where every
// expert may take a token): a CTA owns one token, threads stride its columns;
// the picks are walked in order and most are -1. No flag variants apply.
template <typename T>
__global__ void __launch_bounds__(kCombineThreads) combine_many_kernel(const T *__restrict__ y_perm, int64_t d,
                                                                       const int32_t *__restrict__ row_of, int k,
                                                                       int64_t R_max, int64_t T_, T *__restrict__ y,
                                                                       int32_t *status) {
  pdl_wait();
  const int64_t t = blockIdx.x;
  if (t >= T_) return;
  for (int64_t c = (int64_t)threadIdx.x * 4; c < d; c += kCombineThreads * 4) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int32_t r = __ldg(row_of + t * k + j);
      if (r < 0) continue;
      if (r >= R_max) {
        if (c == 0) report_error(status, MOE_ERR_BOUNDS, kKCombine, (int32_t)t);
        continue;
      }
      const float4 v = Store4<T>::ld(y_perm + (int64_t)r * d + c);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    Store4<T>::st(y + t * d + c, a);
  }
}

__global__ void ec_pattern_kernel(int32_t *idx, int64_t T_, int N) {
  pdl_wait();
  const int64_t n = T_ * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    idx[i] = (int32_t)(i % N);
}

// Combine with the K slices of a decode-mode second GEMM: one thread per
// (token, 4 columns); the k x (1 + nsplit) source rows are walked as one flat
// list, 8 loads at a time. Per pick the slices are added in slice order, then
// the picks in pick order.
template <typename T>
__global__ void __launch_bounds__(kCombineThreads) combine_split_kernel(
    const T *__restrict__ y_perm, const float *__restrict__ y_split, int nsplit, int64_t d,
    const int32_t *__restrict__ row_of, const float *__restrict__ gate, const T *__restrict__ x,
    const T *__restrict__ y_shared, int64_t T_, int k, int64_t R_max, uint32_t flags, T *__restrict__ y,
    int32_t *status) {
  pdl_wait();
  const int64_t d4 = d >> 2;
  const int64_t i = (int64_t)blockIdx.x * kCombineThreads + threadIdx.x;
  if (i >= T_ * d4) return;
  const int64_t t = i / d4;
  const int64_t c = (i - t * d4) << 2;
  const int per = 1 + nsplit, nsrc = k * per;
  int nkept = 0;
  float kept_gate = 0.f;
  for (int j = 0; j < k; ++j) {
    const int32_t r = __ldg(row_of + t * k + j);
    if (r >= R_max && c == 0) report_error(status, MOE_ERR_BOUNDS, kKCombine, (int32_t)t);
    if (r >= 0 && r < R_max) {
      ++nkept;
      if (flags & MOE_FLAG_RENORM_SURVIVORS) kept_gate += __ldg(gate + t * k + j);
    }
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), part = acc;
  for (int q0 = 0; q0 < nsrc; q0 += 8) {
    float4 v[8];
    bool ok[8];  // the source's pick is kept
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int q = q0 + b;
      const int j = q / per, sl = q - j * per;
      int64_t r = 0;
      ok[b] = false;
      if (q < nsrc) {
        const int32_t rr = __ldg(row_of + t * k + j);
        ok[b] = rr >= 0 && rr < R_max;
        r = ok[b] ? rr : 0;
      }
      // slice 0 in y_perm (x's dtype), the others in y_split (fp32)
      v[b] = sl == 0 ? Store4<T>::ld(y_perm + r * d + c)
                     : __ldg(reinterpret_cast<const float4 *>(y_split + (int64_t)(sl - 1) * R_max * d + r * d + c));
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int q = q0 + b;
      if (q < nsrc) {
        const int j = q / per, sl = q - j * per;
        part.x += v[b].x;
        part.y += v[b].y;
        part.z += v[b].z;
        part.w += v[b].w;
        if (sl == nsplit) {
          if (ok[b]) {
            acc.x += part.x;
            acc.y += part.y;
            acc.z += part.z;
            acc.w += part.w;
          }
          part = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  if ((flags & MOE_FLAG_RENORM_SURVIVORS) && nkept > 0) {
    acc.x /= kept_gate;
    acc.y /= kept_gate;
    acc.z /= kept_gate;
    acc.w /= kept_gate;
  }
  if ((flags & MOE_FLAG_IDENTITY_FALLBACK) && nkept == 0) acc = Store4<T>::ld(x + t * d + c);
  if (y_shared) {  // the shared expert, added last
    const float4 sh = Store4<T>::ld(y_shared + t * d + c);
    acc.x += sh.x;
    acc.y += sh.y;
    acc.z += sh.z;
    acc.w += sh.w;
  }
  Store4<T>::st(y + t * d + c, acc);
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
  return launch_k(permute_kernel, dim3(grid_for(D.R_max, kWarps)), dim3(kWarps * 32), 0, s, 1u, (const uint4 *)x, vpr,
                  offsets, D.N, row_token, D.T, D.R_max, (uint4 *)x_perm, status);
}

namespace {
template <typename T>
cudaError_t launch_combine_t(const Dims &D, const T *y_perm, const float *y_split, int nsplit,
                             const int32_t *row_of, const float *gate, const T *x, const T *y_shared, T *y,
                             int32_t *status, cudaStream_t s) {
  const int64_t items = D.T * (D.d / 4);
  if (nsplit > 0) {
    const int64_t g = (items + kCombineThreads - 1) / kCombineThreads;
    return launch_k(combine_split_kernel<T>, dim3((unsigned)g), dim3(kCombineThreads), 0, s, 1u, y_perm, y_split,
                    nsplit, D.d, row_of, gate, x, y_shared, D.T, D.k, D.R_max, D.flags, y, status);
  }
  const int km = D.k <= 1 ? 1 : D.k <= 2 ? 2 : D.k <= 4 ? 4 : 8;
  const int64_t tok_per_block = 8 / km;
  const unsigned g = (unsigned)((D.T + tok_per_block - 1) / tok_per_block);
  // one 16-byte vector per thread and source row: 8 bf16 or 4 fp32 columns
  constexpr int W = 16 / (int)sizeof(T);
  auto kern = km == 1   ? combine_kernel<T, 1, W>
              : km == 2 ? combine_kernel<T, 2, W>
              : km == 4 ? combine_kernel<T, 4, W>
                        : combine_kernel<T, 8, W>;
  return launch_k(kern, dim3(g), dim3(kC8Threads), 0, s, 1u, y_perm, D.d, row_of, gate, x, y_shared, D.T, D.k,
                  D.R_max, D.flags, y, status);
}
}  // namespace

cudaError_t launch_combine(const Dims &D, const void *y_perm, const float *y_split, int nsplit,
                           const int32_t *row_of, const float *gate, const void *x, const void *y_shared, void *y,
                           int32_t *status, cudaStream_t s) {
  if (!y_split) nsplit = 0;
  if (nsplit > 7) return cudaErrorNotSupported;
  if (D.T == 0) return cudaSuccess;
  if (D.k > 8 && nsplit == 0) {
    if (y_shared || (D.flags & (MOE_FLAG_RENORM_SURVIVORS | MOE_FLAG_IDENTITY_FALLBACK))) return cudaErrorNotSupported;
    if (D.dt == MOE_DT_BF16)
      return launch_k(combine_many_kernel<__nv_bfloat16>, dim3((unsigned)D.T), dim3(kCombineThreads), 0, s, 1u,
                      (const __nv_bfloat16 *)y_perm, D.d, row_of, D.k, D.R_max, D.T, (__nv_bfloat16 *)y, status);
    return launch_k(combine_many_kernel<float>, dim3((unsigned)D.T), dim3(kCombineThreads), 0, s, 1u,
                    (const float *)y_perm, D.d, row_of, D.k, D.R_max, D.T, (float *)y, status);
  }
  if (D.dt == MOE_DT_BF16)
    return launch_combine_t<__nv_bfloat16>(D, (const __nv_bfloat16 *)y_perm, y_split, nsplit, row_of, gate,
                                           (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)y_shared,
                                           (__nv_bfloat16 *)y, status, s);
  return launch_combine_t<float>(D, (const float *)y_perm, y_split, nsplit, row_of, gate, (const float *)x,
                                 (const float *)y_shared, (float *)y, status, s);
}

namespace {
__global__ void shared_setup_kernel(int32_t *offsets, int64_t rows, int32_t *sync, int64_t n_sync) {
  pdl_wait();
  if (threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = (int32_t)rows;
  }
  for (int64_t i = threadIdx.x; i < n_sync; i += blockDim.x) sync[i] = 0;
}
}  // namespace

cudaError_t launch_ec_pattern(int32_t *idx, int64_t T, int N, cudaStream_t s) {
  int64_t g = (T * N + 255) / 256;
  if (g > 148 * 16) g = 148 * 16;
  return launch_k(ec_pattern_kernel, dim3((unsigned)g), dim3(256), 0, s, 1u, idx, T, N);
}

cudaError_t launch_shared_setup(int32_t *offsets, int64_t rows, int32_t *sync, int64_t n_sync, cudaStream_t s) {
  return launch_k(shared_setup_kernel, dim3(1), dim3(256), 0, s, 1u, offsets, rows, sync, n_sync);
}

}  // namespace moe
