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
// One persistent launch, one CTA per SM, walks all GEMM1 tiles and then all
// GEMM2 tiles (so neither GEMM leaves a partly idle last wave): warp 0 streams
// the weight tile [128 x 64] and the token tile [64 x 64] per k-block with TMA
// (eight 24 KB stages); warp 1 issues tcgen05.mma (M=128, N=64, K=16) into
// one of two TMEM accumulators; warps 2-5 read one accumulator lane each
// (TMEM lane = weight row f) and store the 64 token values of that row:
//   GEMM1: h[off_e + j, f]      = GELU(D^T[f, j] + b1[e][f])          (bf16)
//   GEMM2: y_s[off_e + j, o]    = g_j * (D^T[o, j] + [s == 0] b2[e][o])
//          (slice 0 into y_perm as bf16, slices 1..S-1 into y_split as fp32)
// GEMM2 splits K into S slices (s = 0..S-1) to give every SM work; slice s
// writes its own partial buffer and the combine adds the S partials in a
// fixed order, so the result stays deterministic. A GEMM2 tile of expert e
// starts only when all of e's GEMM1 tiles have stored h: each epilogue warp
// fences its generic stores for the async proxy and then increments e's
// counter with release semantics; the producer acquires the counter (bounded
// wait) and fences before its TMA loads of h.
#include <vector>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kDM = 128;  // weight rows per tile (MMA M)
constexpr int kDAtom = 64;                // columns of one 128-byte swizzle atom (one TMA box)
constexpr int kDAtoms = 2;                // atoms per stage: each weight row is requested 256 B at a time
constexpr int kDBK = kDAtom * kDAtoms;    // k-block
constexpr int kDWAtomBytes = kDM * kDAtom * 2;
constexpr int kDWBytes = kDWAtomBytes * kDAtoms;
constexpr int kDThreads = 192;
constexpr int kDMaxExperts = 256;
constexpr int kDMaxStages = 5;

struct DCtrl {
  unsigned long long full[kDMaxStages], empty[kDMaxStages], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int total1, total2;  // GEMM1 tiles, GEMM1 + GEMM2 tiles
  int32_t offsets[kDMaxExperts + 1];
  int32_t start1[kDMaxExperts + 1];  // first GEMM1 tile of each expert
  int32_t start2[kDMaxExperts + 1];  // first GEMM2 tile of each expert (counted from total1)
};

struct DTile {
  int phase;  // 0: GEMM1, 1: GEMM2
  int e, row0, m, sp;
};

// Token chunks of DN rows (MMA N): 64, or 32 when experts hold few rows, which
// leaves room for a fifth stage (more weight bytes in flight per SM).
template <int DN> struct DCfg {
  static constexpr int kStages = DN == 32 ? 5 : 4;
  static constexpr int kTAtomBytes = DN * kDAtom * 2;
  static constexpr int kTBytes = kTAtomBytes * kDAtoms;
  static constexpr int kStageBytes = kDWBytes + kTBytes;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + sizeof(DCtrl);
  static_assert(kStages <= kDMaxStages, "barrier arrays");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Tiles of expert e: chunks_e x slices x m_tiles, m fastest, then the slice.
template <int DN>
__device__ __forceinline__ DTile decode_tile(const DCtrl *c, int N_exp, int m1, int m2, int S, int t) {
  DTile d;
  d.phase = t >= c->total1 ? 1 : 0;
  const int32_t *start = d.phase ? c->start2 : c->start1;
  const int tt = d.phase ? t - c->total1 : t;
  const int mt = d.phase ? m2 : m1, sl = d.phase ? S : 1;
  int lo = 0, hi = N_exp - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= tt) lo = mid; else hi = mid - 1;
  }
  d.e = lo;
  int local = tt - start[lo];
  d.m = local % mt;
  local /= mt;
  d.sp = local % sl;
  d.row0 = c->offsets[lo] + (local / sl) * DN;
  return d;
}

template <int DN>
__global__ void __launch_bounds__(kDThreads, 1)
    ffn_decode_kernel(const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_h,
                      const int32_t *__restrict__ offsets_g, int N_exp, int64_t R_max, int d, int d_ff, int S,
                      const __nv_bfloat16 *__restrict__ b1, const __nv_bfloat16 *__restrict__ b2,
                      const float *__restrict__ row_gate, __nv_bfloat16 *__restrict__ h,
                      __nv_bfloat16 *__restrict__ y_perm,
                      float *__restrict__ y_split, int32_t *__restrict__ h_done, int32_t *status) {
  using C = DCfg<DN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sW = base;
  uint8_t *sT = base + C::kStages * kDWBytes;
  DCtrl *c = (DCtrl *)(base + C::kStages * C::kStageBytes);
  volatile int *abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m1 = (d_ff + kDM - 1) / kDM, m2 = (d + kDM - 1) / kDM;
  const int kb1_count = (d + kDBK - 1) / kDBK, kb2_count = (d_ff + kDBK - 1) / kDBK;

  if (warp == 0) {
    pdl_wait();  // offsets come from the dispatch
    int n1[8], n2[8];
    int s1 = 0, s2 = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      n1[i] = n2[i] = 0;
      if (e < N_exp) {
        const int o0 = offsets_g[e], o1 = offsets_g[e + 1];
        if (o1 < o0 || (o1 - o0) % DN != 0 || o1 > R_max) bad = true;
        else {
          n1[i] = (o1 - o0) / DN * m1;
          n2[i] = (o1 - o0) / DN * S * m2;
        }
      }
      s1 += n1[i];
      s2 += n2[i];
    }
    bad = __any_sync(0xffffffffu, bad);
    int i1 = s1, i2 = s2;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v1 = __shfl_up_sync(0xffffffffu, i1, off);
      const int v2 = __shfl_up_sync(0xffffffffu, i2, off);
      if (lane >= off) {
        i1 += v1;
        i2 += v2;
      }
    }
    int x1 = i1 - s1, x2 = i2 - s2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < N_exp) {
        c->start1[e] = x1;
        c->start2[e] = x2;
        c->offsets[e] = offsets_g[e];
      }
      x1 += n1[i];
      x2 += n2[i];
    }
    const int t1 = __shfl_sync(0xffffffffu, i1, 31), t2 = __shfl_sync(0xffffffffu, i2, 31);
    if (lane == 0) {
      c->offsets[N_exp] = offsets_g[N_exp];
      c->start1[N_exp] = t1;
      c->start2[N_exp] = t2;
      c->total1 = bad ? 0 : t1;
      c->total2 = bad ? 0 : t1 + t2;
      c->abort = 0;
      if (bad) report_error(status, MOE_ERR_BOUNDS, kKGemmTcDecode, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
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
                 "r"(2 * DN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const int total = c->total2;
  const uint32_t tmem = c->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, parity_mask = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const DTile tl = decode_tile<DN>(c, N_exp, m1, m2, S, t);
        int kb0 = 0, kb1 = kb1_count;
        if (tl.phase) {
          kb0 = tl.sp * kb2_count / S;
          kb1 = (tl.sp + 1) * kb2_count / S;
          // every GEMM1 tile of this expert must have stored its rows of h
          const int need = (c->offsets[tl.e + 1] - c->offsets[tl.e]) / DN * m1 * 4;
          if (!wait_counter(h_done + tl.e, need, abort, status, kKGemmTcDecode, 5)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_fast(&c->empty[s], ph ^ 1u, abort, status, kKGemmTcDecode, 10 + s)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&c->full[s], C::kStageBytes);
          const CUtensorMap *mw = tl.phase ? &tm_w2 : &tm_w1;
          const CUtensorMap *mt = tl.phase ? &tm_h : &tm_x;
#pragma unroll
          for (int a = 0; a < kDAtoms; ++a)  // columns past K are zero-filled by TMA
            tma_load_3d(sW + s * kDWBytes + a * kDWAtomBytes, mw, &c->full[s], kb * kDBK + a * kDAtom, tl.m * kDM,
                        tl.e);
#pragma unroll
          for (int a = 0; a < kDAtoms; ++a)
            tma_load_2d(sT + s * C::kTBytes + a * C::kTAtomBytes, mt, &c->full[s], kb * kDBK + a * kDAtom, tl.row0);
          issued_mask |= 1u << s;
          parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
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
      uint32_t ph = 0, aph = 0;
      int acc = 0;
      bool ok = true, any = false;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(DN >> 3) << 17) |
                             ((uint32_t)(kDM >> 4) << 24);
      const uint64_t wdesc0 = smem_desc_sw128(saddr(sW)), tdesc0 = smem_desc_sw128(saddr(sT));
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const DTile tl = decode_tile<DN>(c, N_exp, m1, m2, S, t);
        int kb0 = 0, kb1 = kb1_count;
        if (tl.phase) {
          kb0 = tl.sp * kb2_count / S;
          kb1 = (tl.sp + 1) * kb2_count / S;
        }
        if (!mbar_wait_fast(&c->tempty[acc], aph ^ 1u, abort, status, kKGemmTcDecode, 20 + acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * DN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_fast(&c->full[s], ph, abort, status, kKGemmTcDecode, 30 + s)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kDBK / 16; ++kk)
            umma_bf16_cta1(d_tmem,
                           wdesc0 + (uint64_t)(s * (kDWBytes >> 4) + (kk >> 2) * (kDWAtomBytes >> 4) + 2 * (kk & 3)),
                           tdesc0 + (uint64_t)(s * (C::kTBytes >> 4) + (kk >> 2) * (C::kTAtomBytes >> 4) + 2 * (kk & 3)),
                           idesc,
                           (kb != kb0 || kk != 0) ? 1u : 0u);
          any = true;
          umma_commit_cta1(&c->empty[s]);
          if (++s == C::kStages) {
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
      const DTile tl = decode_tile<DN>(c, N_exp, m1, m2, S, t);
      // the bias and the chunk's row gates are fetched before the accumulator
      // wait, so no load latency sits between TMEM and the stores
      const int M_out = tl.phase ? d : d_ff;
      const int f = tl.m * kDM + q * 32 + lane;  // this thread's weight row (output feature)
      const bool fvalid = f < M_out;
      float b = 0.f;
      if (fvalid && (tl.phase == 0 || tl.sp == 0))
        b = __bfloat162float((tl.phase ? b2 : b1)[(int64_t)tl.e * M_out + f]);
      float gate_lo = 1.0f, gate_hi = 1.0f;  // row gates of chunk rows lane and 32 + lane
      if (tl.phase && row_gate) {
        gate_lo = row_gate[tl.row0 + lane];
        if (DN > 32) gate_hi = row_gate[tl.row0 + 32 + lane];
      }
      // K slice 0 goes to y_perm (bf16), slices 1..S-1 to y_split (fp32)
      float *dst = tl.phase && tl.sp > 0 ? y_split + (int64_t)(tl.sp - 1) * R_max * d : nullptr;
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&c->tfull[acc], aph, abort, status, kKGemmTcDecode, 40 + acc) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < DN; c0 += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * DN + c0), r);
        if (tl.phase == 0) {
          if (fvalid) {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int64_t row = (int64_t)tl.row0 + c0 + j;
              const float2 a = gelu_as2(__fadd2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                                                   make_float2(b, b)));
              h[row * d_ff + f] = __float2bfloat16_rn(a.x);
              h[(row + 1) * d_ff + f] = __float2bfloat16_rn(a.y);
            }
          }
        } else {
          const float gsrc = c0 == 0 ? gate_lo : gate_hi;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t row = (int64_t)tl.row0 + c0 + j;
            const float g = __shfl_sync(0xffffffffu, gsrc, j);
            if (fvalid) {
              const float v = g * (__uint_as_float(r[j]) + b);
              if (tl.sp == 0) y_perm[row * d + f] = __float2bfloat16_rn(v);
              else dst[row * d + f] = v;
            }
          }
        }
      }
      if (tl.phase == 0) {
        fence_proxy_async_global();  // h stores before the async-proxy loads of GEMM2 tiles
        __syncwarp();
        if (lane == 0) red_release_add(h_done + tl.e, 1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  pdl_trigger();  // this CTA has no tiles left: the next kernel may launch
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * DN));
  }
  // The last CTA out resets the expert counters (and the exit count) for the
  // next launch: every other CTA has finished all its counter accesses.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(h_done + N_exp, 1) == (int)gridDim.x - 1) {
      __threadfence();
      for (int i = 0; i <= N_exp; ++i) h_done[i] = 0;
    }
  }
}

}  // namespace

// Largest number of k-blocks one CTA streams when the tiles are dealt out
// round-robin (tile t to CTA t mod sms) in the kernel's order: all GEMM1
// tiles, then per chunk the S slices of m2 tiles each.
static int64_t max_cta_kblocks(int64_t chunks, int64_t m1, int64_t kb1, int64_t m2, int64_t kb2, int64_t S,
                               int64_t sms) {
  std::vector<int64_t> diff((size_t)sms + 1, 0);
  int64_t all = 0, p = 0;
  auto segment = [&](int64_t n, int64_t w) {
    all += n / sms * w;
    const int64_t rem = n % sms, a = (p + n - rem) % sms;
    if (rem > 0) {
      if (a + rem <= sms) {
        diff[(size_t)a] += w;
        diff[(size_t)(a + rem)] -= w;
      } else {
        diff[(size_t)a] += w;
        diff[(size_t)sms] -= w;
        diff[0] += w;
        diff[(size_t)(a + rem - sms)] -= w;
      }
    }
    p += n;
  };
  segment(chunks * m1, kb1);
  for (int64_t c = 0; c < chunks; ++c)
    for (int64_t sp = 0; sp < S; ++sp) segment(m2, (sp + 1) * kb2 / S - sp * kb2 / S);
  int64_t run = 0, mx = 0;
  for (int64_t i = 0; i < sms; ++i) {
    run += diff[(size_t)i];
    mx = run > mx ? run : mx;
  }
  return all + mx;
}

int decode_chunk_rows(const Dims &D) {
  return D.T * (int64_t)D.k <= (int64_t)kDecodeSmallRowsPerExpert * D.N ? 32 : 64;
}

int decode_splits(const Dims &D) {
  if (D.dt != MOE_DT_BF16 || D.T * (int64_t)D.k > (int64_t)kDecodeRowsPerExpert * D.N) return 0;
  // K slices of the second GEMM. The busiest CTA's weight stream sets the
  // time; every slice past the first adds a [rows, d] fp32 partial written
  // here and read by the combine. Pick the S (1..8, at least 4 k-blocks per
  // slice) that minimises the sum, for one token chunk per routed expert.
  const int64_t m1 = (D.d_ff + kDM - 1) / kDM, m2 = (D.d + kDM - 1) / kDM;
  const int64_t kb1 = (D.d + kDBK - 1) / kDBK, kb2 = (D.d_ff + kDBK - 1) / kDBK;
  const int64_t sms = num_sms();
  const int64_t tk = D.T * (int64_t)D.k;
  const int64_t chunks = tk < D.N ? (tk > 0 ? tk : 1) : D.N;
  const double tile_bytes = (double)kDM * kDBK * 2;
  int best = 1;
  double best_cost = 0.0;
  for (int64_t S = 1; S <= 8 && (S == 1 || S <= kb2 / 4); ++S) {
    const double cost = (double)max_cta_kblocks(chunks, m1, kb1, m2, kb2, S, sms) * tile_bytes * (double)sms +
                        (double)(S - 1) * 2.0 * (double)chunks * decode_chunk_rows(D) * (double)D.d * 4.0;
    if (S == 1 || cost < best_cost) {
      best_cost = cost;
      best = (int)S;
    }
  }
  return best;
}

namespace {
template <int DN>
cudaError_t launch_decode_t(const Dims &D, int S, const void *x_perm, const int32_t *offsets, const void *w1,
                            const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                            void *y_perm, float *y_split, int32_t *h_done, int32_t *status, cudaStream_t s) {
  using C = DCfg<DN>;
  static PerDevice<int> attr;  // the instance's shared-memory size, set once per device
  int set = 0;
  const cudaError_t ae = attr.get(
      [](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(ffn_decode_kernel<DN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::kSmem);
      },
      &set);
  if (ae != cudaSuccess) return ae;
  CUtensorMap tw1, tx, tw2, th;
  const uint64_t dw1[3] = {(uint64_t)D.d, (uint64_t)D.d_ff, (uint64_t)D.N};
  const uint64_t dx[2] = {(uint64_t)D.d, (uint64_t)D.R_max};
  const uint64_t dw2[3] = {(uint64_t)D.d_ff, (uint64_t)D.d, (uint64_t)D.N};
  const uint64_t dh[2] = {(uint64_t)D.d_ff, (uint64_t)D.R_max};
  if (!make_map(&tw1, w1, 3, dw1, kDM) || !make_map(&tx, x_perm, 2, dx, DN) || !make_map(&tw2, w2, 3, dw2, kDM) ||
      !make_map(&th, h, 2, dh, DN))
    return cudaErrorInvalidValue;
  const int64_t chunks = D.R_max / DN;
  const int64_t max_tiles = chunks * ((D.d_ff + kDM - 1) / kDM) + chunks * S * ((D.d + kDM - 1) / kDM);
  int grid = num_sms();
  if (max_tiles < grid) grid = (int)max_tiles;
  if (grid < 1) grid = 1;
  // One CTA per SM at most (shared memory) and no more CTAs than SMs, so all
  // are resident together: a GEMM2 tile never waits on a CTA that cannot run.
  return launch_k(ffn_decode_kernel<DN>, dim3((unsigned)grid), dim3(kDThreads), C::kSmem, s, 1u, tw1, tx, tw2, th,
                  offsets, (int)D.N, (int64_t)D.R_max, (int)D.d, (int)D.d_ff, S, (const __nv_bfloat16 *)b1,
                  (const __nv_bfloat16 *)b2, row_gate, (__nv_bfloat16 *)h, (__nv_bfloat16 *)y_perm, y_split, h_done,
                  status);
}
}  // namespace

cudaError_t launch_ffn_decode(const Dims &D, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *b1, const void *w2, const void *b2, const float *row_gate, void *h,
                              void *y_perm, float *y_split, int32_t *h_done, int32_t *status, cudaStream_t s) {
  const int S = decode_splits(D);
  if (S < 1 || (S > 1 && !y_split) || !h_done || D.N > kDMaxExperts) return cudaErrorNotSupported;
  return decode_chunk_rows(D) == 32
             ? launch_decode_t<32>(D, S, x_perm, offsets, w1, b1, w2, b2, row_gate, h, y_perm, y_split, h_done,
                                   status, s)
             : launch_decode_t<64>(D, S, x_perm, offsets, w1, b1, w2, b2, row_gate, h, y_perm, y_split, h_done,
                                   status, s);
}

}  // namespace moe
