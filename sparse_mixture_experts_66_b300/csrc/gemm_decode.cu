// K7: the expert FFNs of decode-shaped batches (few tokens per expert), as
// weight-streaming GEMMs with the operands swapped.
//
// Same mathematics as K4 / K5 ("Mixture of Experts (MoE): Architecture,
// Routing, and Scaling", "Core Architecture": FFN(x) = W2 GELU(W1 x + b1) +
// b2; the gate scaling of the wiki's step 7 fused into the second GEMM), but
// when an expert holds only a few dozen rows, a 128- or 256-row token tile
// would be mostly padding. Here the weights sit on the MMA's M side and the
// tokens on N:
//   D^T[f, j] = sum_k W[e][f, k] * A[off_e + j, k]   (M = 128 weight rows,
//                                                    N = 64 token rows)
// so every weight byte is streamed from HBM exactly once per 64-token chunk
// (one chunk per expert at decode sizes). Segments of the permuted buffer are
// aligned to 64 rows in this mode, so a chunk is never pure padding.
//
// Persistent, one CTA per SM: warp 0 streams the weight tile [128 x 64] and
// the token tile [64 x 64] per k-block with TMA (eight 24 KB stages); warp 1
// issues tcgen05.mma (M=128, N=64, K=16) into one of two TMEM accumulators;
// warps 2-5 read one accumulator lane each (TMEM lane = weight row f) and
// store the 64 token values of that row:
//   GEMM1: h[off_e + j, f]      = GELU(D^T[f, j] + b1[e][f])          (bf16)
//   GEMM2: y_s[off_e + j, o]    = g_j * (D^T[o, j] + [s == 0] b2[e][o]) (fp32)
// GEMM2 splits K into S slices (s = 0..S-1) to give every SM work; slice s
// writes its own partial buffer and the combine adds the S partials in a
// fixed order, so the result stays deterministic.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kDM = 128;  // weight rows per tile (MMA M)
constexpr int kDN = 64;   // token rows per chunk (MMA N)
constexpr int kDBK = 64;  // k-block
constexpr int kDStages = 8;
constexpr int kDWBytes = kDM * kDBK * 2;
constexpr int kDTBytes = kDN * kDBK * 2;
constexpr int kDStageBytes = kDWBytes + kDTBytes;
constexpr int kDThreads = 192;
constexpr int kDMaxExperts = 256;

struct DCtrl {
  unsigned long long full[kDStages], empty[kDStages], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int32_t offsets[kDMaxExperts + 1];
  int32_t tile_start[kDMaxExperts + 1];
};

constexpr size_t kDSmem = 1024 + (size_t)kDStages * kDStageBytes + sizeof(DCtrl);

// Tiles of expert e: chunks_e x splits x m_tiles, m fastest, then the slice.
__device__ __forceinline__ void decode_swap_tile(const DCtrl *c, int N_exp, int m_tiles, int splits, int t, int &e,
                                                 int &row0, int &m, int &s) {
  int lo = 0, hi = N_exp - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  e = lo;
  int local = t - c->tile_start[e];
  m = local % m_tiles;
  local /= m_tiles;
  s = local % splits;
  row0 = c->offsets[e] + (local / splits) * kDN;
}

template <int EPI>
__global__ void __launch_bounds__(kDThreads, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_t,
                     const int32_t *__restrict__ offsets_g, int N_exp, int64_t R_max, int K, int M_out, int splits,
                     const __nv_bfloat16 *__restrict__ bias, const float *__restrict__ row_gate,
                     void *__restrict__ out, float *__restrict__ out_split, int64_t split_stride, int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sW = base;
  uint8_t *sT = base + kDStages * kDWBytes;
  DCtrl *c = (DCtrl *)(base + kDStages * kDStageBytes);
  volatile int *abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M_out + kDM - 1) / kDM;
  const int kb_count = (K + kDBK - 1) / kDBK;
  const int kb_per_split = (kb_count + splits - 1) / splits;

  if (warp == 0) {
    int local[8];
    int sum = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      local[i] = 0;
      if (e < N_exp) {
        const int o0 = offsets_g[e], o1 = offsets_g[e + 1];
        if (o1 < o0 || (o1 - o0) % kDN != 0 || o1 > R_max) bad = true;
        else local[i] = (o1 - o0) / kDN * splits * m_tiles;
      }
      sum += local[i];
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
        c->tile_start[e] = excl;
        c->offsets[e] = offsets_g[e];
      }
      excl += local[i];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      c->offsets[N_exp] = offsets_g[N_exp];
      c->tile_start[N_exp] = total;
      c->total_tiles = bad ? 0 : total;
      c->abort = 0;
      if (bad) report_error(status, MOE_ERR_BOUNDS, kKGemmTcDecode, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < kDStages; ++s) {
        mbar_init(&c->full[s], 1);
        mbar_init(&c->empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&c->tfull[a], 1);
        mbar_init(&c->tempty[a], 4);
      }
      mbar_init(&c->drain, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&c->tmem_base)),
                 "r"(2 * kDN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int total = c->total_tiles;
  const uint32_t tmem = c->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool issued[kDStages];
      uint32_t issued_parity[kDStages];
      for (int i = 0; i < kDStages; ++i) issued[i] = false;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        int e, row0, m, sp;
        decode_swap_tile(c, N_exp, m_tiles, splits, t, e, row0, m, sp);
        const int kb0 = sp * kb_per_split;
        const int kb1 = min(kb_count, kb0 + kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_fast(&c->empty[s], ph ^ 1u, abort, status, kKGemmTcDecode, 10 + s)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&c->full[s], kDStageBytes);
          tma_load_3d(sW + s * kDWBytes, &tm_w, &c->full[s], kb * kDBK, m * kDM, e);
          tma_load_2d(sT + s * kDTBytes, &tm_t, &c->full[s], kb * kDBK, row0);
          issued[s] = true;
          issued_parity[s] = ph;
          if (++s == kDStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int i = 0; i < kDStages; ++i)
          if (issued[i]) {
            const unsigned long long ts = globaltimer();
            while (!mbar_try_wait(&c->full[i], issued_parity[i]) && globaltimer() - ts < kTimeoutNs) {
            }
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, aph = 0;
      int acc = 0;
      bool ok = true, any = false;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kDN >> 3) << 17) |
                             ((uint32_t)(kDM >> 4) << 24);
      uint64_t wdesc[kDStages], tdesc[kDStages];
      for (int i = 0; i < kDStages; ++i) {
        wdesc[i] = smem_desc_sw128(saddr(sW + i * kDWBytes));
        tdesc[i] = smem_desc_sw128(saddr(sT + i * kDTBytes));
      }
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        int e, row0, m, sp;
        decode_swap_tile(c, N_exp, m_tiles, splits, t, e, row0, m, sp);
        const int kb0 = sp * kb_per_split;
        const int kb1 = min(kb_count, kb0 + kb_per_split);
        if (!mbar_wait_fast(&c->tempty[acc], aph ^ 1u, abort, status, kKGemmTcDecode, 20 + acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * kDN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_fast(&c->full[s], ph, abort, status, kKGemmTcDecode, 30 + s)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kDBK / 16; ++kk)
            umma_bf16_cta1(d_tmem, wdesc[s] + (uint64_t)(2 * kk), tdesc[s] + (uint64_t)(2 * kk), idesc,
                           (kb != kb0 || kk != 0) ? 1u : 0u);
          any = true;
          umma_commit_cta1(&c->empty[s]);
          if (++s == kDStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_cta1(&c->tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if ((!ok || *abort) && any) {
        umma_commit_cta1(&c->drain);
        const unsigned long long ts = globaltimer();
        while (!mbar_try_wait(&c->drain, 0) && globaltimer() - ts < kTimeoutNs) {
        }
      }
    }
  } else {
    const int q = warp & 3;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, row0, m, sp;
      decode_swap_tile(c, N_exp, m_tiles, splits, t, e, row0, m, sp);
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&c->tfull[acc], aph, abort, status, kKGemmTcDecode, 40 + acc) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int f = m * kDM + q * 32 + lane;  // this thread's weight row (output feature)
      const bool fvalid = f < M_out;
      float b = 0.f;
      if (fvalid && (EPI == 1 || sp == 0)) b = __bfloat162float(bias[(int64_t)e * M_out + f]);
#pragma unroll 1
      for (int c0 = 0; c0 < kDN; c0 += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kDN + c0), r);
        if (fvalid) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t row = (int64_t)row0 + c0 + j;
            const float v = __uint_as_float(r[j]) + b;
            if (EPI == 1) {
              ((__nv_bfloat16 *)out)[row * M_out + f] = __float2bfloat16_rn(gelu_as(v));
            } else {
              const float g = row_gate ? row_gate[row] : 1.0f;
              float *dst = sp == 0 ? (float *)out : out_split + (int64_t)(sp - 1) * split_stride;
              dst[row * M_out + f] = g * v;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kDN));
  }
}

template <int EPI>
cudaError_t launch_swap(const Dims &D, const void *W, const void *A, int64_t K, int64_t M_out, int splits,
                        const void *bias, const float *row_gate, const int32_t *offsets, void *out,
                        float *out_split, int32_t *status, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_swap_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tw, tt;
  const uint64_t dw[3] = {(uint64_t)K, (uint64_t)M_out, (uint64_t)D.N};
  const uint64_t dt[2] = {(uint64_t)K, (uint64_t)D.R_max};
  if (!make_map(&tw, W, 3, dw, kDM) || !make_map(&tt, A, 2, dt, kDN)) return cudaErrorInvalidValue;
  const int64_t max_tiles = (D.R_max / kDN) * splits * ((M_out + kDM - 1) / kDM);
  int grid = num_sms();
  if (max_tiles < grid) grid = (int)max_tiles;
  if (grid < 1) grid = 1;
  gemm_swap_kernel<EPI><<<grid, kDThreads, kDSmem, s>>>(tw, tt, offsets, D.N, D.R_max, (int)K, (int)M_out, splits,
                                                         (const __nv_bfloat16 *)bias, row_gate, out, out_split,
                                                         D.R_max * M_out, status);
  return cudaGetLastError();
}

}  // namespace

int decode_splits(const Dims &D) {
  if (D.dt != MOE_DT_BF16 || D.T * (int64_t)D.k > (int64_t)kDecodeRowsPerExpert * D.N) return 0;
  // K slices of the second GEMM so that the tiles cover every SM about four times
  const int64_t tiles = (int64_t)D.N * ((D.d + kDM - 1) / kDM);
  int64_t s = (4 * 148 + tiles - 1) / tiles;
  const int64_t kb = (D.d_ff + kDBK - 1) / kDBK;
  if (s > kb / 4) s = kb / 4;
  if (s > 8) s = 8;
  if (s < 1) s = 1;
  return (int)s;
}

cudaError_t launch_ffn_decode(const Dims &D, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                              float *y_perm, float *y_split, int32_t *status, cudaStream_t s) {
  const int S = decode_splits(D);
  if (S < 1 || (S > 1 && !y_split)) return cudaErrorNotSupported;
  cudaError_t e = launch_swap<1>(D, w1, x_perm, D.d, D.d_ff, 1, b1, nullptr, offsets, h, nullptr, status, s);
  if (e != cudaSuccess) return e;
  // K slice 0 writes y_perm; slice s >= 1 writes y_split + (s - 1) * R_max * d
  return launch_swap<2>(D, w2, h, D.d_ff, D.d, S, b2, row_gate, offsets, y_perm, y_split, status, s);
}

}  // namespace moe
