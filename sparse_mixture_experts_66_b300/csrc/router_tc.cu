// K1 on the tensor cores: the fused router for bf16 inputs.
//
// "Mixture-of-Experts" (beta.fermi.ai wiki), step-by-step mechanism, steps
// 1-3: logits x W_g, softmax over the N experts, the k largest by score,
// renormalised to sum to 1. The projection is a [T x d] . [d x N] contraction;
// here it runs on tcgen05 with bf16 operands and fp32 accumulation in tensor
// memory, so every product is exact and the logits are fp32 sums, never
// rounded to bf16 ("Inside the Router", "Mixture of Experts: How Sparse
// Routing Scales Transformers": router logits at higher precision).
//
// S CTAs (a cluster of S) per 128 tokens, each over 1/S of d: warp 0 streams
// the token tile [128 x 64] and the W_g tile [NP x 64] per k-block with TMA
// (128-byte swizzle) through a small ring; warp 1 issues tcgen05.mma (M=128,
// N=NP, K=16) into one TMEM accumulator. With S > 1 the epilogue warps of ranks
// 1..S-1 copy their partial logits into rank 0's shared memory (distributed
// shared memory), and after a cluster barrier rank 0 forms each logit as its
// own partial plus ranks 1, 2, ... in that order: a fixed order, so the result
// is deterministic. Splitting d lets a small batch stream x on S times as many
// SMs. Rank 0's epilogue warps then do the softmax and the top-k in
// registers (TMEM lane = token; the k best kept by an unrolled insertion, ties
// to the lower expert, picks in rank order). Up to 32 experts one thread owns a
// token; from 64 on, 16 epilogue warps split each token's logits into four
// column groups, exchange the group maxima, partial sums (added in group order)
// and top-k candidates through shared memory, and group 0 merges the
// candidates: the same picks as one pass over all columns. NP is N rounded up
// to 16..256; the W_g rows past N are zero-filled by TMA and their columns are
// ignored.
#include <math.h>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRM = 128;  // tokens per CTA (MMA M)
constexpr int kRBK = 64;  // k-block: one 128-byte swizzle atom of bf16
template <int NP, int S> struct RCfg {
  // G column groups of epilogue warps: with many experts the per-token softmax
  // and top-k would be a long serial chain in one thread, so 4 warps share each
  // TMEM lane quadrant, a quarter of the logit columns each
  static constexpr int G = NP >= 64 ? 4 : 1;
  static constexpr int kCW = NP / G;  // logit columns per epilogue thread (a multiple of 16)
  static constexpr int kEpiThreads = 128 * G;
  static constexpr int kThreads = 64 + kEpiThreads;
  static constexpr int kXBytes = kRM * kRBK * 2;
  static constexpr int kWBytes = NP * kRBK * 2;
  static constexpr int kStageBytes = kXBytes + kWBytes;
  // rank 0's buffer for the partial logits of ranks 1..S-1: [S-1][128][NP + 4]
  // fp32 (rows 16-byte aligned; the +4 keeps a quarter-warp's 16-byte accesses
  // on distinct banks)
  static constexpr int kPartStride = NP + 4;
  static constexpr int kPartBytes = S > 1 ? (S - 1) * kRM * kPartStride * 4 : 0;
  // as many stages as fit 192 KB with the partials (2..12): few CTAs stream all
  // of x, so each needs many bytes in flight
  static constexpr int kFit = (192 * 1024 - kPartBytes) / kStageBytes;
  static constexpr int kStages = kFit < 2 ? 2 : (kFit > 12 ? 12 : kFit);
  static constexpr int kTmemCols = NP < 32 ? 32 : NP;  // a power of two >= 32
  // the column groups' exchange (per group and token: max, softmax partial sum,
  // 8 top-k candidates as value and expert), in the stage ring, idle by then
  static constexpr int kXchgBytes = G > 1 ? G * kRM * (4 + 4 + 8 * 8) : 0;
  static_assert(kCW % 16 == 0, "column groups are whole 16-column TMEM loads");
  static_assert(kXchgBytes <= kStages * kStageBytes, "exchange fits the stage ring");
};

// 16-byte store into another CTA's shared memory (a mapa'd address).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Named barrier 1 over the epilogue warps only.
template <int kCount> __device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCount) : "memory");
}

struct RCtrl {
  unsigned long long full[12], empty[12], tfull, drain;
  uint32_t tmem_base;
  int abort;
  float bias[256];  // the logit bias (0 when none), for every padded expert column
};

template <int NP, int S> constexpr size_t router_smem() {
  using C = RCfg<NP, S>;
  return 1024 + (size_t)C::kStages * C::kStageBytes + (size_t)C::kPartBytes + sizeof(RCtrl);
}

// KM: the top-k insertion's depth, k rounded up to 2 or 8 (each logit costs
// KM compare-and-swap steps, the epilogue's main work with many experts)
template <int NP, int S, int KM>
__global__ void __launch_bounds__(RCfg<NP, S>::kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const float *__restrict__ router_bias, int64_t T_, int d, int N, int k,
                     int32_t *__restrict__ topk_idx, float *__restrict__ gate, float *__restrict__ score,
                     float *__restrict__ probs, float *__restrict__ lse, int32_t *status) {
  using C = RCfg<NP, S>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sX = base;
  uint8_t *sW = base + C::kStages * C::kXBytes;
  float *part = (float *)(base + C::kStages * C::kStageBytes);
  RCtrl *c = (RCtrl *)(base + C::kStages * C::kStageBytes + C::kPartBytes);
  volatile int *abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  const int64_t t0 = (int64_t)(blockIdx.x / S) * kRM;
  // this rank's k-blocks: [r*kb/S, (r+1)*kb/S), at least two each (the host
  // splits only when kb >= 2S)
  const int kb_all = (d + kRBK - 1) / kRBK;
  const int kb_lo = (int)rank * kb_all / S, kb_hi = ((int)rank + 1) * kb_all / S;

  if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&c->full[s], 1);
        mbar_init(&c->empty[s], 1);
      }
      mbar_init(&c->tfull, 1);
      mbar_init(&c->drain, 1);
      c->abort = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&c->tmem_base)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  if (S > 1) cluster_sync_all();  // rank 0 runs before its peers write into its shared memory
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  pdl_wait();  // x and W_g may come from the previous kernel; the outputs may still be read by it
  int epi_ok = 0;  // epilogue warps: this CTA's accumulator is complete

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, parity_mask = 0;  // stages with a copy issued, and its phase parity
      bool ok = true;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!mbar_wait_fast(&c->empty[s], ph ^ 1u, abort, status, kKRouter, 10 + s)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&c->full[s], C::kStageBytes);
        tma_load_2d(sX + s * C::kXBytes, &tm_x, &c->full[s], kb * kRBK, (int)t0);
        tma_load_2d(sW + s * C::kWBytes, &tm_w, &c->full[s], kb * kRBK, 0);
        issued_mask |= 1u << s;
        parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) {
        for (int i = 0; i < C::kStages; ++i)
          if (issued_mask & (1u << i)) {
            const unsigned long long ts = globaltimer();
            while (!mbar_try_wait(&c->full[i], (parity_mask >> i) & 1u) && globaltimer() - ts < kTimeoutNs) {
            }
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true, any = false;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NP >> 3) << 17) |
                             ((uint32_t)(kRM >> 4) << 24);
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!mbar_wait_fast(&c->full[s], ph, abort, status, kKRouter, 20 + s)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(saddr(sX + s * C::kXBytes));
        const uint64_t bd = smem_desc_sw128(saddr(sW + s * C::kWBytes));
#pragma unroll
        for (int kk = 0; kk < kRBK / 16; ++kk)
          umma_bf16_cta1(tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc,
                         (kb != kb_lo || kk != 0) ? 1u : 0u);
        any = true;
        umma_commit_cta1(&c->empty[s]);
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) {
        umma_commit_cta1(&c->tfull);
      } else if (any) {
        umma_commit_cta1(&c->drain);
        const unsigned long long ts = globaltimer();
        while (!mbar_try_wait(&c->drain, 0) && globaltimer() - ts < kTimeoutNs) {
        }
      }
    }
  } else {
    const int q = warp & 3;     // TMEM lane quadrant: tokens 32q..32q+31
    const int g = (warp - 2) >> 2;  // column group: logit columns [g*CW, (g+1)*CW)
    const int row = q * 32 + lane;
    const int cb = g * C::kCW;
    // the epilogue warps stage the logit bias (0 when none) while the MMAs run
    for (int i = threadIdx.x - 64; i < NP; i += C::kEpiThreads)
      c->bias[i] = (router_bias && i < N) ? router_bias[i] : 0.f;
    epi_bar<C::kEpiThreads>();
    if (lane == 0) epi_ok = mbar_wait(&c->tfull, 0, abort, status, kKRouter, 30) ? 1 : 0;
    epi_ok = __shfl_sync(0xffffffffu, epi_ok, 0);
    // one outcome for all epilogue warps: a warp whose wait ran out raised the
    // abort flag before this barrier, so none of them joins the exchanges below
    epi_bar<C::kEpiThreads>();
    epi_ok = epi_ok && !*abort;
    if (S > 1 && rank != 0 && epi_ok) {
      // ranks 1..S-1: this thread's columns of its row's partial logits into
      // rank 0's slot
      tc_fence_after();
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      const uint32_t dst = map_to_rank(saddr(part + ((int)(rank - 1) * kRM + row) * C::kPartStride), 0);
#pragma unroll 1
      for (int c0 = cb; c0 < cb + C::kCW; c0 += 16) {
        uint32_t r[16];
        __syncwarp();
        tmem_ld16(lane_base + (uint32_t)c0, r);
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          st_cluster_v4(dst + (uint32_t)(c0 + j) * 4u, r[j], r[j + 1], r[j + 2], r[j + 3]);
      }
    }
  }
  if (S > 1) cluster_sync_all();  // the partials are in rank 0's shared memory

  if (warp >= 2 && rank == 0 && epi_ok) {
    const int q = warp & 3;
    const int g = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int cb = g * C::kCW;
    const int64_t t = t0 + row;
    tc_fence_after();
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    float *mine = part + row * C::kPartStride;  // rank 1's slot, reused for the summed logits
    if (S > 1) {
      // logit = own partial + rank 1 + rank 2 + ..., in that order
#pragma unroll 1
      for (int c0 = cb; c0 < cb + C::kCW; c0 += 16) {
        uint32_t r[16];
        __syncwarp();
        tmem_ld16(lane_base + (uint32_t)c0, r);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 a = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                 __uint_as_float(r[j + 3]));
#pragma unroll
          for (int src = 0; src < S - 1; ++src) {
            const float4 p = *reinterpret_cast<const float4 *>(part + (src * kRM + row) * C::kPartStride + c0 + j);
            a.x += p.x;
            a.y += p.y;
            a.z += p.z;
            a.w += p.w;
          }
          *reinterpret_cast<float4 *>(mine + c0 + j) = a;
        }
      }
    }
    // 16 logits of this token from column c0 (without the bias)
    auto load16 = [&](int c0, float(&v)[16]) {
      if (S == 1) {
        uint32_t r[16];
        __syncwarp();  // the TMEM load is warp-collective
        tmem_ld16(lane_base + (uint32_t)c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 a = *reinterpret_cast<const float4 *>(mine + c0 + j);
          v[j] = a.x;
          v[j + 1] = a.y;
          v[j + 2] = a.z;
          v[j + 3] = a.w;
        }
      }
    };
    // the k best so far (value desc, expert asc): a candidate goes after an
    // equal value, so ties keep the lower expert
    float tv[8];
    int te[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      tv[j] = -INFINITY;
      te[j] = 0x7fffffff;
    }
    auto insert = [&](float v, int e) {
#pragma unroll
      for (int s = 0; s < KM; ++s) {
        if (s < k && v > tv[s]) {
          const float fv = tv[s];
          const int fe = te[s];
          tv[s] = v;
          te[s] = e;
          v = fv;
          e = fe;
        }
      }
    };
    // pass 1: max and the k best of this thread's columns
    float m = -INFINITY;
#pragma unroll 1
    for (int c0 = cb; c0 < cb + C::kCW; c0 += 16) {
      float v16[16];
      load16(c0, v16);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = c0 + j;
        if (e >= N) break;  // padded expert columns
        const float v = v16[j] + c->bias[e];
        m = fmaxf(m, v);
        insert(v, e);
      }
    }
    // the groups' exchange (G > 1): group 0 of each token merges the others'
    // candidates; every group needs the row max and the full denominator
    float *xm = reinterpret_cast<float *>(base);  // [G][128] maxima
    float *xs = xm + C::G * kRM;                  // [G][128] partial sums
    float *xv = xs + C::G * kRM;                  // [G][8][128] candidate values
    int *xe = reinterpret_cast<int *>(xv + C::G * 8 * kRM);  // [G][8][128] candidate experts
    if (C::G > 1) {
      // the ring was last written and read by the async proxy (TMA, MMA), all
      // of it complete once the accumulator was
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      xm[g * kRM + row] = m;
      if (g > 0)
#pragma unroll
        for (int s = 0; s < KM; ++s)
          if (s < k) {
            xv[(g * 8 + s) * kRM + row] = tv[s];
            xe[(g * 8 + s) * kRM + row] = te[s];
          }
      epi_bar<C::kEpiThreads>();
      m = xm[row];
#pragma unroll
      for (int h = 1; h < C::G; ++h) m = fmaxf(m, xm[h * kRM + row]);
    }
    // pass 2: the softmax denominator, summed over groups in order
    float sum = 0.f;
#pragma unroll 1
    for (int c0 = cb; c0 < cb + C::kCW; c0 += 16) {
      float v16[16];
      load16(c0, v16);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = c0 + j;
        if (e >= N) break;
        sum += expf(v16[j] + c->bias[e] - m);
      }
    }
    if (C::G > 1) {
      xs[g * kRM + row] = sum;
      epi_bar<C::kEpiThreads>();
      sum = 0.f;
#pragma unroll
      for (int h = 0; h < C::G; ++h) sum += xs[h * kRM + row];
    }
    if (probs) {  // router statistics: the full probability row and the logsumexp
      // (the TMEM loads are warp-collective: every lane runs them, only lanes
      // of real tokens store)
#pragma unroll 1
      for (int c0 = cb; c0 < cb + C::kCW; c0 += 16) {
        float v16[16];
        load16(c0, v16);
        if (t < T_) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int e = c0 + j;
            if (e >= N) break;
            probs[t * N + e] = expf(v16[j] + c->bias[e] - m) / sum;
          }
        }
      }
      if (g == 0 && t < T_) lse[t] = m + logf(sum);
    }
    if (g == 0) {
      for (int h = 1; h < C::G; ++h)
#pragma unroll
        for (int s = 0; s < KM; ++s)
          if (s < k) insert(xv[(h * 8 + s) * kRM + row], xe[(h * 8 + s) * kRM + row]);
      if (t < T_) {
        float ex[8], sel = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          ex[s] = expf(tv[s] - m);
          if (s < k) sel += ex[s];
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if (s < k) {
            topk_idx[t * k + s] = te[s];
            score[t * k + s] = ex[s] / sum;
            gate[t * k + s] = ex[s] / sel;
          }
        }
      }
    }
  }

  pdl_trigger();  // the next kernel may launch while this one tears down
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  }
}

template <int NP, int S, int KM>
cudaError_t launch_npk(const Dims &D, const void *x, const void *w_g, const float *router_bias, int32_t *topk_idx,
                      float *gate, float *score, float *probs, float *lse, int32_t *status, cudaStream_t s) {
  static PerDevice<int> attr;  // this instance's shared-memory size, set once per device
  const size_t smem = router_smem<NP, S>();
  int set = 0;
  const cudaError_t ae = attr.get(
      [smem](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(router_tc_kernel<NP, S, KM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
      },
      &set);
  if (ae != cudaSuccess) return ae;
  CUtensorMap tx, tw;
  const uint64_t dx[2] = {(uint64_t)D.d, (uint64_t)D.T};
  const uint64_t dw[2] = {(uint64_t)D.d, (uint64_t)D.N};
  if (!make_map(&tx, x, 2, dx, kRM) || !make_map(&tw, w_g, 2, dw, NP)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)((D.T + kRM - 1) / kRM) * S;
  return launch_k(router_tc_kernel<NP, S, KM>, dim3(grid), dim3(RCfg<NP, S>::kThreads), smem, s, (unsigned)S, tx, tw, router_bias,
                  D.T, (int)D.d, D.N, D.k, topk_idx, gate, score, probs, lse, status);
}

template <int NP, int S>
cudaError_t launch_np(const Dims &D, const void *x, const void *w_g, const float *router_bias, int32_t *topk_idx,
                      float *gate, float *score, float *probs, float *lse, int32_t *status, cudaStream_t s) {
  if (D.k <= 2) return launch_npk<NP, S, 2>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  return launch_npk<NP, S, 8>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
}

// CTAs per 128-token tile: split d over a cluster of 4 or 2 while the tiles
// alone would leave most SMs idle and every rank keeps at least two k-blocks.
// Up to 64 experts: beyond, the per-token softmax and top-k, which rank 0
// alone runs, outweigh the faster stream of x.
int router_splits(const Dims &D, int NP) {
  const int64_t tiles = (D.T + kRM - 1) / kRM;
  const int kb = (int)((D.d + kRBK - 1) / kRBK);
  if (NP > 64) return 1;
  for (int S = 4; S >= 2; S >>= 1)
    if (tiles * S <= num_sms() && kb >= 2 * S) return S;
  return 1;
}

template <int NP>
cudaError_t launch_split(const Dims &D, const void *x, const void *w_g, const float *router_bias, int32_t *topk_idx,
                         float *gate, float *score, float *probs, float *lse, int32_t *status, cudaStream_t s) {
  switch (router_splits(D, NP)) {
    case 4: return launch_np<NP, 4>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
    case 2: return launch_np<NP, 2>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
    default: return launch_np<NP, 1>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  }
}

}  // namespace

cudaError_t launch_router_tc(const Dims &D, const void *x, const void *w_g, const float *router_bias,
                             int32_t *topk_idx, float *gate, float *score, float *probs, float *lse, int32_t *status,
                             cudaStream_t s) {
  if (D.dt != MOE_DT_BF16 || D.N > 256) return cudaErrorNotSupported;
  if (D.N <= 16) return launch_split<16>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  if (D.N <= 32) return launch_split<32>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  if (D.N <= 64) return launch_split<64>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  if (D.N <= 128) return launch_np<128, 1>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
  return launch_np<256, 1>(D, x, w_g, router_bias, topk_idx, gate, score, probs, lse, status, s);
}

}  // namespace moe
