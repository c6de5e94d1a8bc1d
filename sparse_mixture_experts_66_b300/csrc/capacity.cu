// K2, expert capacity and capacity slots.
//
// "Mixture-of-Experts" (beta.fermi.ai wiki), step 4 and its worked example:
// an expert accepts at most C = ceil(cf*T*k/N) requests ("Communication cost
// in distributed settings"); when more arrive, the lowest-scoring requests are
// dropped for that expert. Equal scores keep the lower token index. The kept
// requests fill the expert's buffer in token order (the pseudocode's
// expert_buffer), which fixes each request's slot.
//
// One launch, no atomics deciding any output. Lists under 4096 requests: one
// CTA per expert with the list in registers. Up to 65 536 requests: a cluster
// of 2-8 CTAs per expert, each holding a slice in registers
// (capacity_cluster_kernel below: the same steps, the slices' counts added in
// rank order). Longer lists, or clusters that would not fit one wave of CTAs:
// one CTA per expert streaming the list in passes. The single-CTA form:
//   1. every CTA counts the requests of all N experts (warp-aggregated with
//      match_any into per-warp rows of a shared histogram), so each CTA can
//      compute every segment offset itself: offset[e] = sum over e' < e of
//      roundup(min(count[e'], C), A), A = 128 rows (the decode chunk, 32 or 64
//      rows, for decode-shaped batches). No CTA waits for another;
//   2. if its expert overflows, the CTA radix-selects (4 passes of 8 bits over
//      the fp32 score's bit pattern, which orders non-negative floats) the C-th
//      largest score and how many requests equal to it are still kept;
//   3. a block-wide scan in token order over "kept" flags numbers the kept
//      rows; ties at the threshold are kept in token order until the quota is
//      used. Padding rows of the segment get token -1 and gate 0.
#include <limits.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 8;  // consecutive requests per thread

__device__ __forceinline__ int64_t round_up_rows(int64_t v, int align) { return (v + align - 1) / align * align; }

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

// The requests [i0, i0 + kItems) of one thread: expert, score bits, gate.
struct Items {
  int32_t ie[kItems];
  uint32_t b[kItems];
  float g[kItems];
};

__device__ __forceinline__ void load_items(const int32_t *__restrict__ idx, const float *__restrict__ score,
                                           const float *__restrict__ gate, int64_t n, int64_t i0, Items &it) {
  if (i0 + kItems <= n) {  // i0 is a multiple of 8: 32-byte aligned vectors, all issued together
    const int4 a0 = __ldg(reinterpret_cast<const int4 *>(idx + i0));
    const int4 a1 = __ldg(reinterpret_cast<const int4 *>(idx + i0 + 4));
    const uint4 s0 = __ldg(reinterpret_cast<const uint4 *>(score + i0));
    const uint4 s1 = __ldg(reinterpret_cast<const uint4 *>(score + i0 + 4));
    const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gate + i0));
    const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gate + i0 + 4));
    it.ie[0] = a0.x; it.ie[1] = a0.y; it.ie[2] = a0.z; it.ie[3] = a0.w;
    it.ie[4] = a1.x; it.ie[5] = a1.y; it.ie[6] = a1.z; it.ie[7] = a1.w;
    it.b[0] = s0.x; it.b[1] = s0.y; it.b[2] = s0.z; it.b[3] = s0.w;
    it.b[4] = s1.x; it.b[5] = s1.y; it.b[6] = s1.z; it.b[7] = s1.w;
    it.g[0] = g0.x; it.g[1] = g0.y; it.g[2] = g0.z; it.g[3] = g0.w;
    it.g[4] = g1.x; it.g[5] = g1.y; it.g[6] = g1.z; it.g[7] = g1.w;
  } else {
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      const int64_t i = i0 + q;
      it.ie[q] = i < n ? idx[i] : -1;
      it.b[q] = i < n ? __float_as_uint(score[i]) : 0u;
      it.g[q] = i < n ? gate[i] : 0.f;
    }
  }
}

// kResident: all T*k requests fit one pass of kThreads * kItems, so they are
// loaded once and every phase works from registers.
template <bool kResident>
__global__ void __launch_bounds__(kThreads) capacity_kernel(
    const int32_t *__restrict__ idx, const float *__restrict__ gate, const float *__restrict__ score, int64_t n,
    int k, int N, int64_t C, int align, int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets,
    int32_t *row_of, int32_t *row_token, float *row_gate, int64_t R_max, int32_t *ffn_sync, int n_sync,
    int32_t *status) {
  pdl_wait();
  // the expert FFN's completion counters start every forward at zero
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_sync; i += kThreads) ffn_sync[i] = 0;
  extern __shared__ int s_hist[];  // [kWarps][N]
  __shared__ int s_warp[32];
  __shared__ int s_sel[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int64_t s_off, s_end;
  __shared__ int s_count;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int64_t kChunk = (int64_t)kThreads * kItems;
  const int64_t my0 = (int64_t)threadIdx.x * kItems;

  Items it;
  if (kResident) load_items(idx, score, gate, n, my0, it);

  // 1. histogram of every expert's requests
  for (int i = threadIdx.x; i < kWarps * N; i += kThreads) s_hist[i] = 0;
  __syncthreads();
  for (int64_t base = 0; base < n; base += kChunk) {
    if (!kResident) load_items(idx, score, gate, n, base + my0, it);
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      const int ex = it.ie[q];
      const unsigned peers = __match_any_sync(0xffffffffu, ex);
      if (ex >= 0 && ex < N && lane == __ffs(peers) - 1) s_hist[warp * N + ex] += __popc(peers);
    }
  }
  __syncthreads();
  int padded = 0, cnt = 0;
  if (threadIdx.x < N) {
    for (int w = 0; w < kWarps; ++w) cnt += s_hist[w * N + threadIdx.x];
    padded = (int)round_up_rows(cnt < C ? cnt : C, align);
  }
  int total_rows;
  const int excl = block_exclusive_scan(padded, s_warp, &total_rows);
  if (threadIdx.x == e) {
    s_off = excl;
    s_end = (int64_t)excl + padded;
    s_count = cnt;
  }
  __syncthreads();
  const int64_t off = s_off;
  const int count = s_count;
  const int kept_e = (int64_t)count < C ? count : (int)C;
  if (total_rows > R_max) {
    // Cannot happen for consistent inputs (R_max bounds every padded
    // segment). Leave an empty, well-formed dispatch rather than rows of an
    // earlier call: no kept rows, every request of this expert dropped.
    if (threadIdx.x == 0) {
      counts_raw[e] = count;
      counts_kept[e] = 0;
      offsets[e] = 0;
      if (e == N - 1) offsets[N] = 0;
      report_error(status, MOE_ERR_BOUNDS, kKCapAssign, e);
    }
    for (int64_t base = 0; base < n; base += kChunk) {
      if (!kResident) load_items(idx, score, gate, n, base + my0, it);
#pragma unroll
      for (int q = 0; q < kItems; ++q)
        if (it.ie[q] == e) row_of[base + my0 + q] = -1;
    }
    return;
  }
  if (threadIdx.x == 0) {
    counts_raw[e] = count;
    counts_kept[e] = kept_e;
    offsets[e] = (int32_t)off;
    if (e == N - 1) offsets[N] = total_rows;
  }

  // 2. the C-th largest score of this expert, when it overflows
  const bool overflow = (int64_t)count > C;
  uint32_t thr = 0u;
  int eq_keep = INT_MAX;
  if (overflow) {
    uint32_t prefix = 0u, mask = 0u;
    int need = (int)C;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) s_sel[i] = 0;
      __syncthreads();
      for (int64_t base = 0; base < n; base += kChunk) {
        if (!kResident) load_items(idx, score, gate, n, base + my0, it);
#pragma unroll
        for (int q = 0; q < kItems; ++q)
          if (it.ie[q] == e && (it.b[q] & mask) == prefix) atomicAdd(&s_sel[(it.b[q] >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // the digit D holding the need-th largest: lane L owns bins 8L..8L+7;
        // counts above each lane's bins come from a suffix scan across lanes
        int h[8], mine = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = s_sel[lane * 8 + j];
          mine += h[j];
        }
        int suffix = mine;  // inclusive sum over lanes >= this one
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_down_sync(0xffffffffu, suffix, o);
          if (lane + o < 32) suffix += v;
        }
        const int above = suffix - mine;  // requests in higher bins
        if (above < need && need <= suffix) {
          int run = above, D = lane * 8;
#pragma unroll
          for (int j = 7; j >= 0; --j) {
            if (run + h[j] >= need) {
              D = lane * 8 + j;
              break;
            }
            run += h[j];
          }
          s_prefix = prefix | ((uint32_t)D << shift);
          s_need = need - run;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      mask |= 255u << shift;
      __syncthreads();
    }
    thr = prefix;    // bit pattern of the C-th largest score
    eq_keep = need;  // requests with exactly that score still kept, in token order
  }

  // 3. slots in token order
  int run_eq = 0, run_kept = 0;
  for (int64_t base = 0; base < n; base += kChunk) {
    if (!kResident) load_items(idx, score, gate, n, base + my0, it);
    const int64_t i0 = base + my0;
    int my_eq = 0;
#pragma unroll
    for (int q = 0; q < kItems; ++q) my_eq += (it.ie[q] == e && overflow && it.b[q] == thr);
    int tot_eq = 0;
    int eq_rank = run_eq;
    if (overflow) eq_rank += block_exclusive_scan(my_eq, s_warp, &tot_eq);
    bool kept[kItems];
    int my_kept = 0;
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      bool kq = false;
      if (it.ie[q] == e) {
        if (!overflow || it.b[q] > thr) {
          kq = true;
        } else if (it.b[q] == thr) {
          kq = eq_rank < eq_keep;
          ++eq_rank;
        }
      }
      kept[q] = kq;
      my_kept += kq;
    }
    int tot_kept;
    int slot = block_exclusive_scan(my_kept, s_warp, &tot_kept) + run_kept;
    // token of each request: one division per thread, then steps (a division
    // per matching request would run once per item slot in a divergent warp)
    int64_t tq = i0 / k;
    int rq = (int)(i0 - tq * k);
    int32_t tok[kItems];
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      tok[q] = (int32_t)tq;
      if (++rq == k) {
        rq = 0;
        ++tq;
      }
    }
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      if (it.ie[q] != e) continue;
      const int64_t i = i0 + q;
      if (kept[q] && slot >= kept_e) {  // inconsistent selection: never write past the segment
        report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 2000 + e);
        row_of[i] = -1;
      } else if (kept[q]) {
        const int64_t r = off + slot;
        row_of[i] = (int32_t)r;
        row_token[r] = tok[q];
        row_gate[r] = it.g[q];
        ++slot;
      } else {
        row_of[i] = -1;
      }
    }
    run_eq += tot_eq;
    run_kept += tot_kept;
  }
  for (int64_t r = off + kept_e + threadIdx.x; r < s_end; r += kThreads) {
    row_token[r] = -1;
    row_gate[r] = 0.f;
  }
  if (threadIdx.x == 0 && run_kept != kept_e) report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 1000 + e);
}

// DSMEM helpers: a 32-bit / 4 x 32-bit load from a mapa'd shared address, and
// the split cluster barrier (arrive with release, wait with acquire).
// (no memory clobber: the cluster barrier before each read orders it, and the
// loads of several ranks can then be in flight together)
__device__ __forceinline__ int ld_cluster(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ int4 ld_cluster_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// The same selection with the S CTAs of a cluster sharing one expert: CTA r
// holds the requests [r*L, (r+1)*L) of the list in registers (L a multiple of
// kItems, at most one pass of kThreads * kItems) and the CTAs add up what each
// phase needs through distributed shared memory, in rank order:
//   1. each CTA counts its slice for every expert; summed over the ranks, the
//      counts give every CTA the same offsets;
//   2. the radix passes add the ranks' 256 digit counts (integers: the sums,
//      and so the C-th largest score, are exactly the single-CTA ones); a pass
//      whose chosen bin holds exactly the requests still to keep ends the
//      search early: every request of that bin is kept, the same set a full
//      search keeps;
//   3. each CTA counts its requests above the threshold and its ties; the ranks
//      before r give how many ties precede the slice and how many rows the
//      slice starts at, so slots and the tie quota follow token order across
//      the whole list as in the single-CTA kernel. An expert that does not
//      overflow keeps every request: its slice starts after the expert's
//      requests in the earlier slices, known from step 1, and no exchange runs.
// Every remote read is followed by a cluster barrier before any CTA leaves.
__global__ void __launch_bounds__(kThreads) capacity_cluster_kernel(
    const int32_t *__restrict__ idx, const float *__restrict__ gate, const float *__restrict__ score, int64_t n,
    int64_t L, int k, int N, int64_t C, int align, int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets,
    int32_t *row_of, int32_t *row_token, float *row_gate, int64_t R_max, int32_t *ffn_sync, int n_sync,
    int32_t *status) {
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_sync; i += kThreads) ffn_sync[i] = 0;
  extern __shared__ int s_hist[];  // [kWarps][N], then this slice's count per expert [N]
  int *s_cnt = s_hist + kWarps * N;
  __shared__ int s_warp[32];
  __shared__ __align__(16) int s_sel[4][256];  // digit counts of each radix pass
  __shared__ __align__(8) int s_x[2];          // this slice: requests above the threshold, ties
  __shared__ uint32_t s_prefix[4];
  __shared__ int s_need[4], s_last[4];
  __shared__ int64_t s_off, s_end;
  __shared__ int s_count, s_before;
  const int S = (int)tc::cluster_size();
  const int rank = (int)tc::cluster_rank();
  const int e = blockIdx.x / S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t lo = (int64_t)rank * L;
  const int64_t hi = lo + L < n ? lo + L : n;
  const int64_t i0 = lo + (int64_t)threadIdx.x * kItems;

  Items it;
  load_items(idx, score, gate, hi, i0, it);  // past the slice: expert -1

  // 1. this slice's histogram, then the cluster's
  for (int i = threadIdx.x; i < kWarps * N; i += kThreads) s_hist[i] = 0;
  for (int i = threadIdx.x; i < 4 * 256; i += kThreads) (&s_sel[0][0])[i] = 0;
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kItems; ++q) {
    const int ex = it.ie[q];
    const unsigned peers = __match_any_sync(0xffffffffu, ex);
    if (ex >= 0 && ex < N && lane == __ffs(peers) - 1) s_hist[warp * N + ex] += __popc(peers);
  }
  __syncthreads();
  if (threadIdx.x < N) {
    int c = 0;
    for (int w = 0; w < kWarps; ++w) c += s_hist[w * N + threadIdx.x];
    s_cnt[threadIdx.x] = c;
  }
  tc::cluster_sync_all();  // every slice's counts are visible to the cluster
  int padded = 0, cnt = 0, before = 0;
  if (threadIdx.x < N) {
    const uint32_t a = tc::saddr(s_cnt + threadIdx.x);
    int v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = q < S ? ld_cluster(tc::map_to_rank(a, (uint32_t)q)) : 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      before += q < rank ? v[q] : 0;
      cnt += v[q];
    }
    padded = (int)round_up_rows(cnt < C ? cnt : C, align);
  }
  // the counts were the last remote read unless the expert overflows: the
  // peers may leave once every CTA has arrived (the wait comes at the end, or
  // before the radix passes)
  cluster_arrive();
  int total_rows;
  const int excl = block_exclusive_scan(padded, s_warp, &total_rows);
  if (threadIdx.x == e) {
    s_off = excl;
    s_end = (int64_t)excl + padded;
    s_count = cnt;
    s_before = before;  // the expert's requests in the slices before this one
  }
  __syncthreads();
  const int64_t off = s_off;
  const int count = s_count;
  const int kept_e = (int64_t)count < C ? count : (int)C;
  if (total_rows > R_max) {  // the whole cluster takes this branch (same totals)
    // as the single-CTA kernel: an empty, well-formed dispatch
    if (rank == 0 && threadIdx.x == 0) {
      counts_raw[e] = count;
      counts_kept[e] = 0;
      offsets[e] = 0;
      if (e == N - 1) offsets[N] = 0;
      report_error(status, MOE_ERR_BOUNDS, kKCapAssign, e);
    }
#pragma unroll
    for (int q = 0; q < kItems; ++q)
      if (it.ie[q] == e) row_of[i0 + q] = -1;
    cluster_wait();  // no CTA leaves while a peer may read its counts
    return;
  }
  if (rank == 0 && threadIdx.x == 0) {
    counts_raw[e] = count;
    counts_kept[e] = kept_e;
    offsets[e] = (int32_t)off;
    if (e == N - 1) offsets[N] = total_rows;
  }

  // 2. the C-th largest score of this expert, when it overflows (the same
  // decision in every CTA of the cluster)
  const bool overflow = (int64_t)count > C;
  uint32_t thr = 0u, thr_mask = ~0u;  // kept: (score bits & thr_mask) above thr, or equal within the quota
  int eq_keep = INT_MAX;
  if (overflow) {
    cluster_wait();  // (completes the arrival after the counts)
    uint32_t prefix = 0u, mask = 0u;
    int need = (int)C;
    for (int shift = 24, p = 0; shift >= 0; shift -= 8, ++p) {
      int *sel = s_sel[p];  // zeroed in phase 1: no barrier before counting
#pragma unroll
      for (int q = 0; q < kItems; ++q)
        if (it.ie[q] == e && (it.b[q] & mask) == prefix) atomicAdd(&sel[(it.b[q] >> shift) & 255u], 1);
      tc::cluster_sync_all();  // the ranks' counts of this pass are visible
      if (warp == 0) {
        int h[8] = {0, 0, 0, 0, 0, 0, 0, 0}, mine = 0;
        const uint32_t a = tc::saddr(sel + lane * 8);
        int4 u[8], w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          u[q] = w[q] = make_int4(0, 0, 0, 0);
          if (q < S) {
            const uint32_t ra = tc::map_to_rank(a, (uint32_t)q);
            u[q] = ld_cluster_v4(ra);
            w[q] = ld_cluster_v4(ra + 16u);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          h[0] += u[q].x; h[1] += u[q].y; h[2] += u[q].z; h[3] += u[q].w;
          h[4] += w[q].x; h[5] += w[q].y; h[6] += w[q].z; h[7] += w[q].w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) mine += h[j];
        int suffix = mine;  // inclusive sum over lanes >= this one
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_down_sync(0xffffffffu, suffix, o);
          if (lane + o < 32) suffix += v;
        }
        const int above = suffix - mine;
        if (above < need && need <= suffix) {
          int run = above, D = lane * 8, hD = 0;
#pragma unroll
          for (int j = 7; j >= 0; --j) {
            if (run + h[j] >= need) {
              D = lane * 8 + j;
              hD = h[j];
              break;
            }
            run += h[j];
          }
          s_prefix[p] = prefix | ((uint32_t)D << shift);
          s_need[p] = need - run;
          s_last[p] = hD == need - run;  // the bin is kept whole
        }
      }
      __syncthreads();
      prefix = s_prefix[p];
      need = s_need[p];
      mask |= 255u << shift;
      if (s_last[p]) break;
    }
    thr = prefix;
    thr_mask = mask;
    eq_keep = need;
  }

  // 3. slots in token order across the slices
  int eq_before = 0, kept_before = 0, eq_rank = 0;
  if (overflow) {
    int my_gt = 0, my_eq = 0;  // this thread: kept without question, ties at the threshold
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      if (it.ie[q] != e) continue;
      const uint32_t bm = it.b[q] & thr_mask;
      if (bm > thr) ++my_gt;
      else if (bm == thr) ++my_eq;
    }
    // both counts in one scan: each is at most kThreads * kItems < 2^16
    int tot_pk;
    const int ex_pk = block_exclusive_scan(my_gt | (my_eq << 16), s_warp, &tot_pk);
    if (threadIdx.x == 0) {
      s_x[0] = tot_pk & 0xffff;
      s_x[1] = tot_pk >> 16;
    }
    tc::cluster_sync_all();
    // ties and kept rows of the slices before this one
    const uint32_t a = tc::saddr(s_x);
    int gt_q[8], eq_q[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // all loads in flight together
      gt_q[q] = eq_q[q] = 0;
      if (q < rank) {
        const uint32_t ra = tc::map_to_rank(a, (uint32_t)q);
        gt_q[q] = ld_cluster(ra);
        eq_q[q] = ld_cluster(ra + 4u);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      int eq_kept = eq_keep - eq_before;
      eq_kept = eq_kept < 0 ? 0 : (eq_kept > eq_q[q] ? eq_q[q] : eq_kept);
      kept_before += gt_q[q] + eq_kept;
      eq_before += eq_q[q];
    }
    cluster_arrive();  // the last remote read: the peers may leave once all arrive
    eq_rank = eq_before + (ex_pk >> 16);
  } else {
    kept_before = s_before;  // every request of the expert is kept
  }
  bool kept[kItems];
  int my_kept = 0;
#pragma unroll
  for (int q = 0; q < kItems; ++q) {
    bool kq = false;
    if (it.ie[q] == e) {
      const uint32_t bm = it.b[q] & thr_mask;
      if (!overflow || bm > thr) {
        kq = true;
      } else if (bm == thr) {
        kq = eq_rank < eq_keep;
        ++eq_rank;
      }
    }
    kept[q] = kq;
    my_kept += kq;
  }
  int tot_kept;
  int slot = block_exclusive_scan(my_kept, s_warp, &tot_kept) + kept_before;
  int tq = (int)i0 / k;  // at most 8 slices of 8192 requests: 32-bit division
  int rq = (int)i0 - tq * k;
  int32_t tok[kItems];
#pragma unroll
  for (int q = 0; q < kItems; ++q) {
    tok[q] = (int32_t)tq;
    if (++rq == k) {
      rq = 0;
      ++tq;
    }
  }
#pragma unroll
  for (int q = 0; q < kItems; ++q) {
    if (it.ie[q] != e) continue;
    const int64_t i = i0 + q;
    if (kept[q] && slot >= kept_e) {
      report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 2000 + e);
      row_of[i] = -1;
    } else if (kept[q]) {
      const int64_t r = off + slot;
      row_of[i] = (int32_t)r;
      row_token[r] = tok[q];
      row_gate[r] = it.g[q];
      ++slot;
    } else {
      row_of[i] = -1;
    }
  }
  if (rank == S - 1) {
    for (int64_t r = off + kept_e + threadIdx.x; r < s_end; r += kThreads) {
      row_token[r] = -1;
      row_gate[r] = 0.f;
    }
    if (threadIdx.x == 0 && kept_before + tot_kept != kept_e)
      report_error(status, MOE_ERR_BOUNDS, kKCapAssign, 1000 + e);
  }
  cluster_wait();
}

// CTAs per expert in the capacity launch: enough that every CTA holds its slice
// of the request list in registers (at most 8, the portable cluster size), then
// more while the launch stays one wave of CTAs and each slice keeps at least
// 2048 requests. 1 selects the single-CTA kernel (which streams the list in
// passes when it exceeds one CTA's registers).
int capacity_cluster(const Dims &D) {
  const int64_t n = D.T * D.k;
  constexpr int64_t kChunk = (int64_t)kThreads * kItems;
  int S = 1;
  while (S < 8 && n > S * kChunk) S *= 2;
  if (n > S * kChunk || (int64_t)D.N * S > num_sms()) return 1;
  while (S < 8 && (int64_t)D.N * S * 2 <= num_sms() && n >= (int64_t)S * 2 * 2048) S *= 2;
  return S;
}

}  // namespace

cudaError_t launch_capacity(const Dims &D, const int32_t *topk_idx, const float *gate, const float *score,
                            int32_t *counts_raw, int32_t *counts_kept, int32_t *offsets, uint32_t *sel_thr,
                            int32_t *sel_eq, int32_t *row_of, int32_t *row_token, float *row_gate,
                            int32_t *ffn_sync, int32_t *status, cudaStream_t s) {
  (void)sel_thr;
  (void)sel_eq;
  const int64_t n = D.T * D.k;
  const size_t smem = sizeof(int) * kWarps * D.N;
  const int n_sync = ffn_sync ? (int)ffn_sync_ints(D) : 0;
  const int S = capacity_cluster(D);
  if (S > 1) {
    // slices of whole kItems groups (aligned vector loads), the last one short
    const int64_t L = ((n + S - 1) / S + kItems - 1) / kItems * kItems;
    return launch_k(capacity_cluster_kernel, dim3((unsigned)(D.N * S)), dim3(kThreads), smem + sizeof(int) * D.N, s,
                    (unsigned)S, topk_idx, gate, score, n, L, D.k, D.N, D.C, row_align(D), counts_raw, counts_kept,
                    offsets, row_of, row_token, row_gate, D.R_max, ffn_sync, n_sync, status);
  }
  auto kern = n <= (int64_t)kThreads * kItems ? capacity_kernel<true> : capacity_kernel<false>;
  return launch_k(kern, dim3(D.N), dim3(kThreads), smem, s, 1u, topk_idx, gate, score, n, D.k, D.N, D.C,
                  row_align(D), counts_raw, counts_kept, offsets, row_of, row_token, row_gate, D.R_max, ffn_sync,
                  n_sync, status);
}

}  // namespace moe
