// K4 / K5: the expert FFNs of bf16 workloads as two grouped GEMMs on the
// 5th-generation tensor cores (tcgen05), fed by TMA, accumulating in tensor
// memory (TMEM).
//
// "Mixture of Experts (MoE): Architecture, Routing, and Scaling" (syntave.com),
// "Core Architecture": FFN(x) = W2 GELU(W1 x + b1) + b2 per expert; the gate
// scaling of the combine ("Mixture-of-Experts" wiki, step 7) is fused into the
// second GEMM's epilogue.
//   GEMM1: h[r, :]      = GELU(x_perm[r] . W1[e]^T + b1[e])         -> bf16
//          (GELU via the Abramowitz & Stegun 7.1.26 erf, |error| <= 1.5e-7)
//   GEMM2: y_perm[r, :] = row_gate[r] * (h[r] . W2[e]^T + b2[e])    -> bf16
// for the rows r of expert e's segment. Segments start on multiples of 128
// rows, so each 128-row half tile belongs to one expert and uses one weight
// matrix.
//
// One persistent launch on CTA pairs (clusters of 2, one CTA per SM) for both
// GEMMs: each pair walks 256 x 256 output tiles of all experts, first of
// GEMM1 and then of GEMM2 (per GEMM expert by expert; inside an expert n-tile
// by n-tile with the 256-row blocks fastest, so the expert's rows stay in L2
// while its weight tiles stream once). Warp roles in each CTA:
//   warp 0    TMA producer: this CTA's 128 rows of A and its half (128 rows)
//             of the B tile per 64-deep k-block (128-byte swizzle), a ring of
//             six 32 KB stages; completion is signalled on the leader's
//             barrier;
//   warp 1    TMEM owner (512 columns, allocated jointly by the pair); in the
//             leader CTA one thread issues tcgen05.mma.cta_group::2.kind::f16
//             (M=256, N=256, K=16) four times per stage into one of two TMEM
//             accumulators and multicasts the commits to both CTAs;
//   warps 2-9 epilogue: tcgen05.ld of the CTA's 128 finished rows (warp w
//             reads TMEM lanes 32*(w%4)...; two warps per lane quarter split
//             the columns), bias + GELU -> h (bf16 boxes staged in shared
//             memory, written by bulk tensor stores) or bias x gate -> y_perm
//             (bf16, 32-byte stores from registers);
//             then the accumulator is handed back to the leader, so the
//             epilogue of tile i overlaps the MMAs of tile i+1.
// Every wait is bounded: after kTimeoutNs the kernel records MOE_ERR_TIMEOUT,
// all roles leave their loops, in-flight copies and MMAs are drained (bounded
// again), TMEM is freed and the CTA exits.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16
constexpr int kEpiWarps = 8;  // a multiple of 4 (one group per TMEM lane quarter) dividing 32
constexpr int kThreads = 64 + kEpiWarps * 32;
static_assert(kEpiWarps % 4 == 0 && (256 / (kEpiWarps / 4)) % 32 == 0, "epilogue column split");
constexpr int kMaxExperts = 256;


struct Ctrl {
  unsigned long long full[8], empty[8], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int total1, total;  // GEMM1 tiles; GEMM1 + GEMM2 tiles
  int32_t offsets[kMaxExperts + 1];
  int32_t blk_start[kMaxExperts + 1];  // first 256-row block of each expert
  int32_t start1[kMaxExperts + 1];     // first GEMM1 tile of each expert
  int32_t start2[kMaxExperts + 1];     // first GEMM2 tile of each expert (counted from total1)
  uint4 bias[kEpiWarps][256 / (kEpiWarps / 4) / 8];  // each epilogue warp's bias columns of its current tile
};


// ---- CTA-pair (cluster of 2) forms --------------------------------------
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// 32-byte global store (one full sector per thread); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
// Bulk tensor store of a shared-memory box (issued by one thread), its group
// commit, and the waits for the group's shared-memory reads / for completion.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(saddr(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Ordinary shared-memory writes before a bulk copy reads them.
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// TMA load whose completion is signalled on an mbarrier of either CTA of the pair.

__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(saddr(dst)),
      "l"(map), "r"(mbar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(saddr(dst)),
      "l"(map), "r"(mbar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Arrive (once all prior MMAs of this thread complete) on the barrier at the
// same offset in every CTA of cta_mask.
__device__ __forceinline__ void umma_commit_pair(unsigned long long *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          saddr(bar)),
      "h"(cta_mask)
      : "memory");
}


// ---- CTA-pair kernel --------------------------------------------------------
// A cluster of 2 CTAs on the two SMs of a pair computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16): each CTA stages its own 128
// rows of A and one half (128 rows) of the B tile, so each SM moves 32 KB per
// 64-deep k-block instead of 48 KB, and six stages fit in shared memory. The
// leader (rank 0) issues the MMAs; D rows 0-127 land in its TMEM, rows
// 128-255 in the peer's. Both CTAs' TMA loads signal the leader's full
// barrier; MMA commits are multicast to both CTAs; the peer's epilogue warps
// arrive remotely on the leader's TMEM-empty barrier.
//
// One launch runs both GEMMs: the tile list holds every GEMM1 tile and then
// every GEMM2 tile, dealt round-robin to the pairs, so GEMM2 tiles start
// while the last GEMM1 tiles finish elsewhere and neither GEMM leaves a
// partly idle last wave. A GEMM2 tile of a 256-row block waits (bounded) until
// all GEMM1 tiles of that block have stored h: each of the 16 epilogue warps
// of a GEMM1 tile fences its stores for the async proxy and adds 1 (release)
// to the block's counter; the GEMM2 producers acquire it before loading h.
// The order is deadlock-free with all pairs resident: a tile only waits on
// tiles earlier in the list, and each pair walks its tiles in list order.
// (Handing tiles out through a global counter instead measured slower here:
// per-tile data waits grew more than the balance improved.)
//
// Tiles: per expert, pair tiles of 256 rows (two 128-row segment tiles). When
// an expert has an odd number of 128-row tiles, its last pair tile is a
// 128-row tail computed with the operands swapped: the 256 weight rows on M
// (128 per CTA, loaded exactly like the B half of a normal tile) and the 128
// tail rows on N (64 per CTA), tcgen05.mma M=256, N=128, so no padding rows
// are computed; its epilogue stores one feature per thread across the tokens.
constexpr int kStagesP = 6;
constexpr int kAP = BM * BK * 2;          // 16 KB: this CTA's 128 rows of A
constexpr int kBP = 128 * BK * 2;         // 16 KB: this CTA's half of the B tile
constexpr int kStageP = kAP + kBP;
constexpr int BNP = 256;                  // pair tile width
// GEMM1 output staging: per epilogue warp one 32-row x 32-column bf16 box
// (64 B rows, 64-byte swizzle) that a bulk tensor store writes to h
constexpr int kStageOut = 32 * 32 * 2;
constexpr size_t kSmemP = 1024 + (size_t)kStagesP * kStageP + (size_t)kEpiWarps * kStageOut + sizeof(Ctrl);

struct PTile {
  int phase;  // 0: GEMM1, 1: GEMM2
  int e;      // expert
  int m0;     // first row of the 256-row pair tile
  int ni;     // n-tile
  int blk;    // index of the 256-row block (dependency counter)
  int swap;   // a 128-row tail, computed with the operands swapped
};

__device__ __forceinline__ PTile decode_pair_tile(const Ctrl *c, int N_exp, int t) {
  PTile p;
  p.phase = t >= c->total1 ? 1 : 0;
  const int32_t *start = p.phase ? c->start2 : c->start1;
  const int tt = p.phase ? t - c->total1 : t;
  int lo = 0, hi = N_exp - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= tt) lo = mid; else hi = mid - 1;
  }
  p.e = lo;
  const int mp = c->blk_start[lo + 1] - c->blk_start[lo];
  const int local = tt - start[lo];
  p.ni = local / mp;
  const int pb = local - p.ni * mp;
  p.m0 = c->offsets[lo] + pb * (2 * BM);
  p.blk = c->blk_start[lo] + pb;
  p.swap = pb == mp - 1 && (((c->offsets[lo + 1] - c->offsets[lo]) / BM) & 1);
  return p;
}

__global__ void __launch_bounds__(kThreads, 1)
    ffn_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w2,
                    const __grid_constant__ CUtensorMap tm_hs,
                    const int32_t *__restrict__ offsets_g, int N_exp, int64_t R_max, int d, int d_ff,
                    const __nv_bfloat16 *__restrict__ b1, const __nv_bfloat16 *__restrict__ b2,
                    const float *__restrict__ row_gate, __nv_bfloat16 *__restrict__ h,
                    __nv_bfloat16 *__restrict__ y_perm,
                    int32_t *__restrict__ blk_done, int nblk_max, int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = base;
  uint8_t *sB = base + kStagesP * kAP;
  uint8_t *sOut = base + kStagesP * kStageP;  // 1024-byte aligned
  Ctrl *c = (Ctrl *)(sOut + kEpiWarps * kStageOut);
  volatile int *abort = &c->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int n1 = (d_ff + BNP - 1) / BNP, n2 = (d + BNP - 1) / BNP;
  const int kb1 = (d + BK - 1) / BK, kb2 = (d_ff + BK - 1) / BK;
  const int need = n1 * 2 * kEpiWarps;  // epilogue-warp arrivals that complete a 256-row block of h
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    pdl_wait();  // offsets come from the dispatch
    int nb[8];
    int sum = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      nb[i] = 0;
      if (e < N_exp) {
        const int o0 = offsets_g[e], o1 = offsets_g[e + 1];
        if (o1 < o0 || (o1 - o0) % BM != 0 || o1 > R_max) bad = true;
        else nb[i] = ((o1 - o0) / BM + 1) / 2;
      }
      sum += nb[i];
    }
    bad = __any_sync(0xffffffffu, bad);
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int excl = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < N_exp) {
        c->blk_start[e] = excl;
        c->start1[e] = excl * n1;
        c->start2[e] = excl * n2;
        c->offsets[e] = offsets_g[e];
      }
      excl += nb[i];
    }
    const int blocks = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      c->offsets[N_exp] = offsets_g[N_exp];
      c->blk_start[N_exp] = blocks;
      c->start1[N_exp] = blocks * n1;
      c->start2[N_exp] = blocks * n2;
      c->total1 = bad ? 0 : blocks * n1;
      c->total = bad ? 0 : blocks * (n1 + n2);
      c->abort = 0;
      if (bad && rank == 0) report_error(status, MOE_ERR_BOUNDS, kKGemmTc, 2);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < kStagesP; ++s) {
        mbar_init(&c->full[s], 1);
        mbar_init(&c->empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&c->tfull[a], 1);
        mbar_init(&c->tempty[a], 2 * kEpiWarps);
      }
      mbar_init(&c->drain, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&c->tmem_base)),
                 "r"(2 * BNP));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before anyone signals them
  tc_fence_after();
  pdl_wait();

  const int total = c->total;
  const uint32_t tmem = c->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, parity_mask = 0;  // stages with a copy issued, and its phase parity
      bool ok = true;
      // the leader's full barriers: consecutive 8-byte objects, mapped once
      const uint32_t full_leader0 = map_to_rank(saddr(&c->full[0]), 0);
      for (int t = pair; ok && t < total; t += npairs) {
        const PTile tl = decode_pair_tile(c, N_exp, t);
        // tokens: this CTA's 128 rows, or for a swapped tail its 64 (of a 128-row box)
        const int a_row = tl.m0 + (int)rank * (tl.swap ? BM / 2 : BM), b_row = tl.ni * BNP + (int)rank * 128;
        const CUtensorMap *ma = tl.phase ? &tm_h : &tm_x;
        const CUtensorMap *mb = tl.phase ? &tm_w2 : &tm_w1;
        const int kbn = tl.phase ? kb2 : kb1;
        if (tl.phase) {
          if (!wait_counter(blk_done + tl.blk, need, abort, status, kKGemmTc, 3)) break;
          fence_proxy_async_global();
        }
        for (int kb = 0; kb < kbn; ++kb) {
          if (!mbar_wait_fast(&c->empty[s], ph ^ 1u, abort, status, kKGemmTc, 50 + s)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(&c->full[s], 2 * kStageP);
          const uint32_t full_leader = full_leader0 + 8u * (uint32_t)s;
          tma_load_2d_pair(sA + s * kAP, ma, full_leader, kb * BK, a_row);
          tma_load_3d_pair(sB + s * kBP, mb, full_leader, kb * BK, b_row, tl.e);
          issued_mask |= 1u << s;
          parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
          if (++s == kStagesP) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (*abort && rank == 0) {  // the leader's full barriers track both CTAs' copies: drain them
        for (int i = 0; i < kStagesP; ++i)
          if (issued_mask & (1u << i)) {
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(&c->full[i], (parity_mask >> i) & 1u) && globaltimer() - t0 < kTimeoutNs) {
            }
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int s = 0;
      uint32_t ph = 0, aph = 0;
      int acc = 0;
      bool ok = true, any = false;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BNP >> 3) << 17) |
                             ((uint32_t)((2 * BM) >> 4) << 24);
      // swapped tail: weights on M (256 features), the 128 tail tokens on N
      const uint32_t idesc_swap = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BM >> 3) << 17) |
                                  ((uint32_t)((2 * BM) >> 4) << 24);
      // stage buffers are equally spaced: a stage's descriptor is the first one
      // advanced by the stage offset in 16-byte units (no carry out of the
      // 14-bit address field below 256 KB)
      const uint64_t adesc0 = smem_desc_sw128(saddr(sA)), bdesc0 = smem_desc_sw128(saddr(sB));
      for (int t = pair; ok && t < total; t += npairs) {
        const PTile tl = decode_pair_tile(c, N_exp, t);
        const int kbn = tl.phase ? kb2 : kb1;
        const uint32_t id = tl.swap ? idesc_swap : idesc;
        const uint64_t da0 = tl.swap ? bdesc0 : adesc0, db0 = tl.swap ? adesc0 : bdesc0;
        if (!mbar_wait_fast(&c->tempty[acc], aph ^ 1u, abort, status, kKGemmTc, 60 + acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BNP);
        for (int kb = 0; kb < kbn; ++kb) {
          if (!mbar_wait_fast(&c->full[s], ph, abort, status, kKGemmTc, 70 + s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          static_assert(kAP == kBP, "A and B stage buffers advance by the same stride");
          const uint64_t ad = da0 + (uint64_t)(s * (kAP >> 4)), bd = db0 + (uint64_t)(s * (kBP >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), id, (kb | kk) != 0 ? 1u : 0u);
          any = true;
          umma_commit_pair(&c->empty[s], (uint16_t)0x3);
          if (++s == kStagesP) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&c->tfull[acc], (uint16_t)0x3);
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if ((!ok || *abort) && any) {
        umma_commit_pair(&c->drain, (uint16_t)0x1);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&c->drain, 0) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else {
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;  // which share of the tile's columns (warps per lane quarter split them)
    constexpr int kCols = BNP / (kEpiWarps / 4);
    constexpr int kSwapCols = BM / (kEpiWarps / 4);  // token columns per warp of a swapped tail
    static_assert(kSwapCols == 32 || kSwapCols == 64, "swapped-tail column split");
    const int row_in_tile = (int)rank * BM + q * 32 + lane;
    const uint32_t tempty_leader0 = map_to_rank(saddr(&c->tempty[0]), 0);
    const uint32_t tempty_leader1 = map_to_rank(saddr(&c->tempty[1]), 0);
    int acc = 0;
    uint32_t aph = 0;
    uint4 *sbias = c->bias[warp - 2];
    for (int t = pair; t < total; t += npairs) {
      const PTile tl = decode_pair_tile(c, N_exp, t);
      // everything the tile's epilogue reads from memory is fetched before the
      // accumulator wait, so no load latency sits between TMEM and the stores
      const int N_out = tl.phase ? d : d_ff;
      const __nv_bfloat16 *bias = tl.phase ? b2 : b1;
      // normal tile: this thread's row, its gate, the warp's bias columns
      const int64_t row = (int64_t)tl.m0 + row_in_tile;
      const bool valid = row < c->offsets[tl.e + 1];
      float g = 1.0f;
      // swapped tail: this thread's feature, its bias, the gates of the warp's token columns
      const int f = tl.ni * BNP + (int)rank * 128 + q * 32 + lane;
      float bsw = 0.f, glo = 1.f, ghi = 1.f;
      if (!tl.swap) {
        if (tl.phase && row_gate && valid) g = row_gate[row];
        const int nb = tl.ni * BNP + part * kCols + lane * 8;
        __syncwarp();  // the previous tile's reads of sbias are done
        if (lane < kCols / 8)
          sbias[lane] = nb < N_out ? __ldg(reinterpret_cast<const uint4 *>(bias + (int64_t)tl.e * N_out + nb))
                                   : make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
      } else {
        if (f < N_out) bsw = __bfloat162float(bias[(int64_t)tl.e * N_out + f]);
        if (tl.phase && row_gate) {
          glo = row_gate[tl.m0 + part * kSwapCols + lane];
          if (kSwapCols > 32) ghi = row_gate[tl.m0 + part * kSwapCols + 32 + lane];
        }
      }
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&c->tfull[acc], aph, abort, status, kKGemmTc, 80 + acc) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      if (tl.swap) {
        // D^T: TMEM lane = feature f, column = token row m0 + column; the tail's
        // 128 rows all lie inside the expert's segment
        const bool fvalid = f < N_out;
#pragma unroll 1
        for (int cc = 0; cc < kSwapCols / 32; ++cc) {
          const int c0 = part * kSwapCols + cc * 32;
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BNP + c0), r);
          if (tl.phase == 0) {
            if (fvalid) {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float2 a = gelu_as2(
                    __fadd2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), make_float2(bsw, bsw)));
                const int64_t rr = (int64_t)tl.m0 + c0 + j;
                h[rr * d_ff + f] = __float2bfloat16_rn(a.x);
                h[(rr + 1) * d_ff + f] = __float2bfloat16_rn(a.y);
              }
            }
          } else {
            const float gsrc = cc == 0 ? glo : ghi;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float gj = __shfl_sync(0xffffffffu, gsrc, j);
              if (fvalid)
                y_perm[((int64_t)tl.m0 + c0 + j) * d + f] = __float2bfloat16_rn(gj * (__uint_as_float(r[j]) + bsw));
            }
          }
        }
      } else {
        // GEMM1: this warp's 32 rows x 32 columns (bf16) go through its staging
        // box in shared memory to a bulk tensor store into h: full 64-byte row
        // segments instead of 32 rows touched per store instruction (the h
        // epilogue paces GEMM1 otherwise)
        uint8_t *box = sOut + (warp - 2) * kStageOut;
        const int row0 = tl.m0 + (int)rank * BM + q * 32;
#pragma unroll 1
        for (int cc = 0; cc < kCols / 32; ++cc) {
          const int col0 = part * kCols + cc * 32;
          uint32_t r[32];
          __syncwarp();  // the TMEM load is warp-collective: reconverge after the row-masked stores
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BNP + col0), r);
          if (cc == kCols / 32 - 1) {  // the accumulator is read out: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0) mbar_arrive(&c->tempty[acc]);
              else mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
            }
          }
          const int n = tl.ni * BNP + col0;
          // GEMM1: GELU(acc + b1); GEMM2: gate * (acc + b2); both to bf16 (two
          // loops, so GEMM2 tiles never evaluate the GELU)
          uint32_t pk[16];
          if (tl.phase == 0) {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const uint4 braw = sbias[cc * 4 + g8];
              const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 a = gelu_as2(__fadd2_rn(
                    make_float2(__uint_as_float(r[g8 * 8 + 2 * j]), __uint_as_float(r[g8 * 8 + 2 * j + 1])),
                    make_float2(__uint_as_float(bw[j] << 16), __uint_as_float(bw[j] & 0xffff0000u))));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(a.x, a.y);
                pk[g8 * 4 + j] = *reinterpret_cast<uint32_t *>(&h2);
              }
            }
          } else {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const uint4 braw = sbias[cc * 4 + g8];
              const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 a = __fmul2_rn(
                    __fadd2_rn(make_float2(__uint_as_float(r[g8 * 8 + 2 * j]), __uint_as_float(r[g8 * 8 + 2 * j + 1])),
                               make_float2(__uint_as_float(bw[j] << 16), __uint_as_float(bw[j] & 0xffff0000u))),
                    make_float2(g, g));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(a.x, a.y);
                pk[g8 * 4 + j] = *reinterpret_cast<uint32_t *>(&h2);
              }
            }
          }
          if (tl.phase == 1) {
            // y_perm straight from registers: GEMM2 tiles wait on operand
            // delivery, and bulk stores would share the TMA unit with their
            // loads. One 32-byte store per 16 columns when the rows are 32-byte
            // aligned (base aligned, d a multiple of 16), else 16-byte stores.
            const bool wide_y = (d & 15) == 0 && ((uintptr_t)y_perm & 31) == 0;
            if (valid) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int nc = n + 16 * hf;
                __nv_bfloat16 *o = y_perm + row * d + nc;
                if (wide_y && nc + 16 <= N_out) {
                  st_global_v8(o, pk + 8 * hf);
                } else {
                  if (nc < N_out)
                    *reinterpret_cast<uint4 *>(o) = make_uint4(pk[8 * hf], pk[8 * hf + 1], pk[8 * hf + 2], pk[8 * hf + 3]);
                  if (nc + 8 < N_out)
                    *reinterpret_cast<uint4 *>(o + 8) = make_uint4(pk[8 * hf + 4], pk[8 * hf + 5], pk[8 * hf + 6], pk[8 * hf + 7]);
                }
              }
            }
            continue;
          }
          if (lane == 0) bulk_wait_read0();  // the previous box has left the staging buffer
          __syncwarp();
          // row `lane`, 16-byte chunk j at chunk j ^ ((row >> 1) & 3): the
          // 64-byte swizzle the store's tensor map names (and conflict-free)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0 && n < N_out) {  // columns past d_ff are clipped by the store
            tma_store_2d(&tm_hs, box, n, row0);
            bulk_commit();
          }
        }
      }
      if (tl.swap) {  // (normal tiles handed the accumulator back after their last TMEM load)
        if (tl.phase == 0) fence_proxy_async_global();  // h stores before the GEMM2 tiles' TMA loads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&c->tempty[acc]);
          else mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
          if (tl.phase == 0) red_release_add(blk_done + tl.blk, 1);
        }
      } else if (tl.phase == 0) {
        // the warp's bulk stores of h are complete before the block counter
        // lets GEMM2 tiles load them
        if (lane == 0) {
          bulk_wait0();
          fence_proxy_async_global();
          red_release_add(blk_done + tl.blk, 1);
        }
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    // the last boxes' bulk stores are complete (shared memory read, y_perm
    // and h written) before the CTA leaves
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  pdl_trigger();  // this CTA has no tiles left: the next kernel may launch
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BNP));
  }
  // The last CTA out resets the block counters (and the exit count) for the
  // next launch: every other CTA has finished all its counter accesses.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(blk_done + nblk_max, 1) == (int)gridDim.x - 1) {
      __threadfence();
      for (int i = 0; i <= nblk_max; ++i) blk_done[i] = 0;
    }
  }
}

// Clusters of 2 that can be resident at once on the current device (every
// pair must be, for the GEMM2 tiles' waits to end). The first call on a device
// also opts the kernel in to its shared-memory size there.
cudaError_t resident_pairs(int *out) {
  static PerDevice<int> cache;
  return cache.get(
      [](int *n) {
        cudaError_t e = cudaFuncSetAttribute(ffn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemP);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 256);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemP;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, ffn_pair_kernel, &cfg) != cudaSuccess || clusters < 1) {
          cudaGetLastError();
          clusters = num_sms() / 2;
        }
        *n = clusters < num_sms() / 2 ? clusters : num_sms() / 2;
        return cudaSuccess;
      },
      out);
}

}  // namespace

cudaError_t launch_ffn_tc(const Dims &D, const void *x_perm, int64_t a_rows, const int32_t *offsets, const void *w1,
                          const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                          void *y_perm, int32_t *blk_done, int32_t *status, cudaStream_t s) {
  if (D.dt != MOE_DT_BF16 || D.N > kMaxExperts || D.d > (1 << 30) || D.d_ff > (1 << 30) || !blk_done)
    return cudaErrorNotSupported;
  int pairs = 0;
  const cudaError_t pe = resident_pairs(&pairs);  // also sets the kernel's shared-memory size on this device
  if (pe != cudaSuccess) return pe;
  CUtensorMap tx, tw1, th, tw2, ths;
  const uint64_t dx[2] = {(uint64_t)D.d, (uint64_t)a_rows};  // rows past a_rows read as zeros
  const uint64_t dw1[3] = {(uint64_t)D.d, (uint64_t)D.d_ff, (uint64_t)D.N};
  const uint64_t dh[2] = {(uint64_t)D.d_ff, (uint64_t)D.R_max};
  const uint64_t dw2[3] = {(uint64_t)D.d_ff, (uint64_t)D.d, (uint64_t)D.N};
  if (!make_map(&tx, x_perm, 2, dx, BM) || !make_map(&tw1, w1, 3, dw1, 128) || !make_map(&th, h, 2, dh, BM) ||
      !make_map(&tw2, w2, 3, dw2, 128) || !make_map(&ths, h, 2, dh, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int64_t max_pairs = (int64_t)ffn_blocks_max(D) * (((D.d_ff + BNP - 1) / BNP) + ((D.d + BNP - 1) / BNP));
  if (max_pairs < pairs) pairs = (int)max_pairs;
  if (pairs < 1) pairs = 1;
  return launch_k(ffn_pair_kernel, dim3(2 * pairs), dim3(kThreads), kSmemP, s, 2u, tx, tw1, th, tw2, ths, offsets,
                  (int)D.N, (int64_t)D.R_max, (int)D.d, (int)D.d_ff, (const __nv_bfloat16 *)b1,
                  (const __nv_bfloat16 *)b2, row_gate, (__nv_bfloat16 *)h, (__nv_bfloat16 *)y_perm, blk_done,
                  (int)ffn_blocks_max(D), status);
}

}  // namespace moe
