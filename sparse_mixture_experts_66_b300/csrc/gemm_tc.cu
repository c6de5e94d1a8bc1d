// K4 / K5: the expert FFNs of bf16 workloads as two grouped GEMMs on the
// 5th-generation tensor cores (tcgen05), fed by TMA, accumulating in tensor
// memory (TMEM).
//
// "Mixture of Experts (MoE): Architecture, Routing, and Scaling" (syntave.com),
// "Core Architecture": FFN(x) = W2 GELU(W1 x + b1) + b2 per expert; the gate
// scaling of the combine ("Mixture-of-Experts" wiki, step 7) is fused into the
// second GEMM's epilogue.
//   GEMM1: h[r, :]      = GELU(x_perm[r] . W1[e]^T + b1[e])         -> bf16
//   GEMM2: y_perm[r, :] = row_gate[r] * (h[r] . W2[e]^T + b2[e])    -> fp32
// for the rows r of expert e's segment. Segments start on multiples of 128
// rows, so each 128-row tile belongs to one expert and uses one weight matrix.
//
// One persistent CTA per SM walks the tiles of all experts (expert by expert,
// within an expert n-tile by n-tile with the m-tiles fastest, so the expert's
// rows stay in L2 while its weight tiles stream once). Warp roles:
//   warp 0    TMA producer: A tile [128 x 64] and B tile [BN x 64] per stage
//             (128-byte swizzle), ring of kStages stages;
//   warp 1    TMEM owner and MMA issuer: one thread issues
//             tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16) four
//             times per stage into one of two TMEM accumulators, and commits
//             the stage back to the producer;
//   warps 2-9 epilogue: tcgen05.ld of the finished accumulator (warp w reads
//             TMEM lanes 32*(w%4)...; two warps per lane quarter split the
//             columns), bias + GELU or bias + gate scale, global stores; then
//             the accumulator is handed back, so the epilogue of tile i
//             overlaps the MMAs of tile i+1.
// Every wait is bounded: after kTimeoutNs the kernel records MOE_ERR_TIMEOUT,
// all roles leave their loops, in-flight copies and MMAs are drained (bounded
// again), TMEM is freed and the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr int kMaxExperts = 256;

template <int BN> struct TileCfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
};

struct Ctrl {
  unsigned long long full[8], empty[8], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int32_t offsets[kMaxExperts + 1];
  int32_t tile_start[kMaxExperts + 1];
};

template <int BN> constexpr size_t smem_bytes() {
  return 1024 + (size_t)TileCfg<BN>::kStages * TileCfg<BN>::kStageBytes + sizeof(Ctrl);
}

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity. Returns false (and raises
// the CTA's abort flag, recording MOE_ERR_TIMEOUT once) when the limit passes,
// or when another role has aborted.
__device__ __noinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity, volatile int *abort,
                                       int32_t *status, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        report_error(status, MOE_ERR_TIMEOUT, kKGemmTc, where);
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, unsigned long long *bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          saddr(dst)),
      "l"(map), "r"(saddr(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, unsigned long long *bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(saddr(dst)),
      "l"(map), "r"(saddr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile with 128-byte swizzle: rows of 128 bytes, 8-row atoms
// of 1024 bytes (the stride-dimension byte offset); the leading offset is
// unused for this layout. Bits 46-47 hold the descriptor version (1).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
template <int BN> __device__ __forceinline__ uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(unsigned long long *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- tile enumeration ----------------------------------------------------
// Tiles are numbered expert by expert; inside expert e (mt_e m-tiles), tile
// t_local = n * mt_e + m.
__device__ __forceinline__ void decode_tile(const Ctrl *c, int N_exp, int t, int &e, int &m0, int &n_idx) {
  int lo = 0, hi = N_exp - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int mt = (c->offsets[e + 1] - c->offsets[e]) / BM;
  const int local = t - c->tile_start[e];
  n_idx = local / mt;
  m0 = c->offsets[e] + (local - n_idx * mt) * BM;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const int32_t *__restrict__ offsets_g, int N_exp, int64_t R_max, int K, int N_out,
                   const __nv_bfloat16 *__restrict__ bias, const float *__restrict__ row_gate, void *__restrict__ out,
                   int32_t *status) {
  using C = TileCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = base;
  uint8_t *sB = base + C::kStages * C::kABytes;
  Ctrl *c = (Ctrl *)(base + C::kStages * C::kStageBytes);
  volatile int *abort = &c->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (N_out + BN - 1) / BN;
  const int kb_count = (K + BK - 1) / BK;

  if (warp == 0) {
    // per-expert tile counts and their exclusive prefix (lane l: experts 8l..8l+7)
    int local[8];
    int sum = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      local[i] = 0;
      if (e < N_exp) {
        const int o0 = offsets_g[e], o1 = offsets_g[e + 1];
        if (o1 < o0 || (o1 - o0) % BM != 0 || o1 > R_max) bad = true;
        else local[i] = (o1 - o0) / BM * n_tiles;
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
      if (bad) report_error(status, MOE_ERR_BOUNDS, kKGemmTc, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&c->full[s], 1);
        mbar_init(&c->empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&c->tfull[a], 1);
        mbar_init(&c->tempty[a], kEpiWarps);
      }
      mbar_init(&c->drain, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&c->tmem_base)),
                 "r"(C::kTmemCols));
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
      uint32_t issued_parity[8];
      bool issued[8];
      for (int i = 0; i < 8; ++i) issued[i] = false;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        int e, m0, ni;
        decode_tile(c, N_exp, t, e, m0, ni);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&c->empty[s], ph ^ 1u, abort, status, 10 + s)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&c->full[s], C::kStageBytes);
          tma_load_2d(sA + s * C::kABytes, &tm_a, &c->full[s], kb * BK, m0);
          tma_load_3d(sB + s * C::kBBytes, &tm_b, &c->full[s], kb * BK, ni * BN, e);
          issued[s] = true;
          issued_parity[s] = ph;
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // drain the copies still in flight before the CTA frees its shared memory
        for (int i = 0; i < C::kStages; ++i)
          if (issued[i]) {
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(&c->full[i], issued_parity[i]) && globaltimer() - t0 < kTimeoutNs) {
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
      const uint32_t idesc = idesc_bf16<BN>();
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        if (!mbar_wait(&c->tempty[acc], aph ^ 1u, abort, status, 20 + acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&c->full[s], ph, abort, status, 30 + s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(saddr(sA + s * C::kABytes));
          const uint64_t bd = smem_desc_sw128(saddr(sB + s * C::kBBytes));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, (kb | kk) != 0 ? 1u : 0u);
          any = true;
          umma_commit(&c->empty[s]);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&c->tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if (!ok || *abort) {  // wait for the MMAs already issued before TMEM is freed
        if (any) {
          umma_commit(&c->drain);
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&c->drain, 0) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else {
    const int q = warp & 3;                // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;      // which half of the tile's columns
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, m0, ni;
      decode_tile(c, N_exp, t, e, m0, ni);
      // one lane waits, the warp follows its verdict: the TMEM loads below are
      // warp-collective, so the warp must never split on a timeout
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&c->tfull[acc], aph, abort, status, 40 + acc) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int64_t row = (int64_t)m0 + row_in_tile;
      const float g = (EPI == 2 && row_gate) ? row_gate[row] : 1.0f;
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col0 = half * (BN / 2) + cc * 32;
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + col0), r);
        const int n = ni * BN + col0;
        const __nv_bfloat16 *bp = bias + (int64_t)e * N_out + n;
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          if (n + g8 * 8 >= N_out) break;
          const uint4 braw = __ldg(reinterpret_cast<const uint4 *>(bp + g8 * 8));
          const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
          float v[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(r[g8 * 8 + 2 * j]) + __uint_as_float(bw[j] << 16);
            v[2 * j + 1] = __uint_as_float(r[g8 * 8 + 2 * j + 1]) + __uint_as_float(bw[j] & 0xffff0000u);
          }
          if (EPI == 1) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(gelu_erf(v[2 * j]), gelu_erf(v[2 * j + 1]));
              p[j] = *reinterpret_cast<uint32_t *>(&h2);
            }
            __nv_bfloat16 *o = (__nv_bfloat16 *)out + row * N_out + n + g8 * 8;
            *reinterpret_cast<uint4 *>(o) = make_uint4(p[0], p[1], p[2], p[3]);
          } else {
            float *o = (float *)out + row * N_out + n + g8 * 8;
            *reinterpret_cast<float4 *>(o) = make_float4(g * v[0], g * v[1], g * v[2], g * v[3]);
            *reinterpret_cast<float4 *>(o + 4) = make_float4(g * v[4], g * v[5], g * v[6], g * v[7]);
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  }
}

// ---- host side ------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// bf16 tensor [outer..., inner] with a box of {64, box_rows(, 1)} and 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1}, es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gd[i] = dims[i];
  gs[0] = dims[0] * 2;
  if (rank == 3) gs[1] = dims[0] * dims[1] * 2;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), gd, gs, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int BN, int EPI>
cudaError_t launch_one(const Dims &D, const void *A, int64_t K, const void *B, const void *bias, int64_t N_out,
                       const float *row_gate, const int32_t *offsets, void *out, int32_t *status, cudaStream_t s) {
  static bool attr_set = false;
  const size_t smem = smem_bytes<BN>();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)D.R_max};
  const uint64_t db[3] = {(uint64_t)K, (uint64_t)N_out, (uint64_t)D.N};
  if (!make_map(&ta, A, 2, da, BM) || !make_map(&tb, B, 3, db, BN)) return cudaErrorInvalidValue;
  const int64_t max_tiles = D.R_max / BM * ((N_out + BN - 1) / BN);
  int grid = num_sms();
  if (max_tiles < grid) grid = (int)max_tiles;
  if (grid < 1) grid = 1;
  gemm_tc_kernel<BN, EPI><<<grid, kThreads, smem, s>>>(ta, tb, offsets, D.N, D.R_max, (int)K, (int)N_out,
                                                       (const __nv_bfloat16 *)bias, row_gate, out, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_tc(const Dims &D, const void *x_perm, const int32_t *offsets, const void *w1, const void *b1,
                          const void *w2, const void *b2, const float *row_gate, void *h, float *y_perm,
                          int32_t *status, cudaStream_t s) {
  if (D.dt != MOE_DT_BF16 || D.N > kMaxExperts || D.d > (1 << 30) || D.d_ff > (1 << 30))
    return cudaErrorNotSupported;
  cudaError_t e = launch_one<256, 1>(D, x_perm, D.d, w1, b1, D.d_ff, nullptr, offsets, h, status, s);
  if (e != cudaSuccess) return e;
  return launch_one<256, 2>(D, h, D.d_ff, w2, b2, D.d, row_gate, offsets, y_perm, status, s);
}

}  // namespace moe
