// K2, expert capacity and capacity slots.
//
// "Mixture-of-Experts" (beta.fermi.ai wiki), step 4 and its worked example:
// an expert accepts at most C = ceil(cf*T*k/N) requests ("Communication cost
// in distributed settings"); when more arrive, the lowest-scoring requests are
// dropped for that expert. Equal scores keep the lower token index. The kept
// requests fill the expert's buffer in token order (the pseudocode's
// expert_buffer), which fixes each request's slot.
//
// Two launches, one CTA per expert each, no atomics on any output:
//   select: count the expert's requests; if the count exceeds C, radix-select
//           (4 passes of 8 bits over the fp32 score's bit pattern, which orders
//           non-negative floats) the C-th largest score and how many requests
//           equal to it must still be kept;
//   assign: the segment of expert e starts at the sum of the earlier experts'
//           kept counts, each rounded up to 128 rows; a block-wide scan in token
//           order over "kept" flags numbers the kept rows; ties at the
//           threshold are kept in token order until the quota is used.
#include <limits.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kItems = 8;  // consecutive requests per thread in the assign pass

__device__ __forceinline__ int64_t round_up_rows(int64_t v) { return (v + kRowAlign - 1) / kRowAlign * kRowAlign; }

__device__ __forceinline__ int block_sum(int v, int *s_red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) s_red[w] = v;
  __syncthreads();
  int t = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  __syncthreads();
  return t;
}

// Exclusive scan over the block in thread order; *total gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  if (w == 0) {
    int t = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += n;
    }
    s_warp[lane] = t;
  }
  __syncthreads();
  const int before = w > 0 ? s_warp[w - 1] : 0;
  *total = s_warp[31];
  __syncthreads();
  return before + incl - v;
}

__global__ void __launch_bounds__(kThreads) cap_select_kernel(const int32_t *__restrict__ idx,
                                                              const float *__restrict__ score, int64_t n, int64_t C,
                                                              int32_t *counts_raw, int32_t *counts_kept,
                                                              uint32_t *sel_thr, int32_t *sel_eq) {
  __shared__ int s_hist[256];
  __shared__ int s_red[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x;
  int cnt = 0;
  for (int64_t i = threadIdx.x; i < n; i += kThreads) cnt += (idx[i] == e);
  const int count = block_sum(cnt, s_red);
  if ((int64_t)count <= C) {
    if (threadIdx.x == 0) {
      counts_raw[e] = count;
      counts_kept[e] = count;
      sel_thr[e] = 0u;
      sel_eq[e] = INT_MAX;
    }
    return;
  }
  uint32_t prefix = 0u, mask = 0u;
  int need = (int)C;  // rank (from the top) of the wanted score among those matching prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) s_hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      if (idx[i] != e) continue;
      const uint32_t b = __float_as_uint(score[i]);
      if ((b & mask) == prefix) atomicAdd(&s_hist[(b >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int above = 0, D = 255;
      for (; D > 0; --D) {
        if (above + s_hist[D] >= need) break;
        above += s_hist[D];
      }
      s_prefix = prefix | ((uint32_t)D << shift);
      s_need = need - above;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    counts_raw[e] = count;
    counts_kept[e] = (int)C;
    sel_thr[e] = prefix;  // bit pattern of the C-th largest score
    sel_eq[e] = need;     // requests with exactly that score still kept, in token order
  }
}

__global__ void __launch_bounds__(kThreads) cap_assign_kernel(
    const int32_t *__restrict__ idx, const float *__restrict__ gate, const float *__restrict__ score, int64_t n,
    int k, int N, int64_t C, const int32_t *__restrict__ counts_raw, const int32_t *__restrict__ counts_kept,
    const uint32_t *__restrict__ sel_thr, const int32_t *__restrict__ sel_eq, int32_t *offsets, int32_t *row_of,
    int32_t *row_token, float *row_gate, int64_t R_max, int32_t *status) {
  __shared__ int s_warp[32];
  __shared__ int64_t s_off;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    int64_t off = 0;
    for (int j = 0; j < e; ++j) off += round_up_rows(counts_kept[j]);
    s_off = off;
    offsets[e] = (int32_t)off;
    if (e == N - 1) offsets[N] = (int32_t)(off + round_up_rows(counts_kept[e]));
  }
  __syncthreads();
  const int64_t off = s_off;
  const int kept_e = counts_kept[e];
  if (off + round_up_rows(kept_e) > R_max) {  // cannot happen for consistent inputs
    if (threadIdx.x == 0) report_error(status, MOE_ERR_BOUNDS, kKCapAssign, e);
    return;
  }
  const bool overflow = (int64_t)counts_raw[e] > C;
  const uint32_t thr = sel_thr[e];
  const int eq_keep = sel_eq[e];
  int run_eq = 0, run_kept = 0;
  for (int64_t base = 0; base < n; base += (int64_t)kThreads * kItems) {
    const int64_t i0 = base + (int64_t)threadIdx.x * kItems;
    int32_t ie[kItems];
    uint32_t b[kItems];
    int my_eq = 0;
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      const int64_t i = i0 + q;
      ie[q] = i < n ? idx[i] : -1;
      b[q] = (ie[q] == e) ? __float_as_uint(score[i]) : 0u;
      my_eq += (ie[q] == e && overflow && b[q] == thr);
    }
    int tot_eq;
    int eq_rank = block_exclusive_scan(my_eq, s_warp, &tot_eq) + run_eq;
    bool kept[kItems];
    int my_kept = 0;
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      bool kq = false;
      if (ie[q] == e) {
        if (!overflow || b[q] > thr) {
          kq = true;
        } else if (b[q] == thr) {
          kq = eq_rank < eq_keep;
          ++eq_rank;
        }
      }
      kept[q] = kq;
      my_kept += kq;
    }
    int tot_kept;
    int slot = block_exclusive_scan(my_kept, s_warp, &tot_kept) + run_kept;
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      if (ie[q] != e) continue;
      const int64_t i = i0 + q;
      if (kept[q] && slot >= kept_e) {  // inconsistent selection: never write past the segment
        report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 2000 + e);
        row_of[i] = -1;
      } else if (kept[q]) {
        const int64_t r = off + slot;
        row_of[i] = (int32_t)r;
        row_token[r] = (int32_t)(i / k);
        row_gate[r] = gate[i];
        ++slot;
      } else {
        row_of[i] = -1;
      }
    }
    run_eq += tot_eq;
    run_kept += tot_kept;
  }
  for (int64_t r = kept_e + threadIdx.x; r < round_up_rows(kept_e); r += kThreads) {
    row_token[off + r] = -1;
    row_gate[off + r] = 0.f;
  }
  if (threadIdx.x == 0 && run_kept != kept_e) report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 1000 + e);
}

}  // namespace

cudaError_t launch_capacity(const Dims &D, const int32_t *topk_idx, const float *gate, const float *score,
                            int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets, uint32_t *sel_thr,
                            int32_t *sel_eq, int32_t *row_of, int32_t *row_token, float *row_gate,
                            int32_t *status, cudaStream_t s) {
  const int64_t n = D.T * D.k;
  cap_select_kernel<<<D.N, kThreads, 0, s>>>(topk_idx, score, n, D.C, counts_raw, counts_kept, sel_thr, sel_eq);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  cap_assign_kernel<<<D.N, kThreads, 0, s>>>(topk_idx, gate, score, n, D.k, D.N, D.C, counts_raw, counts_kept,
                                             sel_thr, sel_eq, offsets, row_of, row_token, row_gate, D.R_max, status);
  return cudaGetLastError();
}

}  // namespace moe
