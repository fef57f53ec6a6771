// bf16 GEMM on the sm_103a tensor cores for the MSR layer's projections
// (m0nads.wordpress.com, "Gated Multi-Scale Retention": Q = X W_Q,
// K = X W_K, V = X W_V, G = X W_G and the output projection Y W_O).
//
// C[M,N] = A[M,K] B[K,N]; A, B, C row-major bf16, fp32 accumulation.
// Persistent CTAs walk 128 x 256 output tiles.  Per CTA: warp 0 streams
// A (K-major) and B (MN-major) 64-deep slabs through a 4-stage TMA ring,
// warp 1 issues tcgen05 MMAs (M=128, N=256, K=16) into one of two TMEM
// accumulators, warps 2-5 drain the other accumulator (TMEM -> registers ->
// bf16 -> global) while the next tile is being computed.  Every wait is
// bounded (a timeout sets the status word and all roles leave).
//
// Gated form (the MSR layer's G = X W_G): C = swish(A B) (.) C, the gate
// applied in the epilogue to the retention output already in C, so G is
// never written.
#include <cudaTypedefs.h>

#include "ktimer.h"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace ret {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4, kNT = 192;
constexpr uint32_t kABytes = BM * BK * 2;   // 16 KB
constexpr uint32_t kBBytes = BK * BN * 2;   // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOffBar = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 5;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmem = kOffMisc + 16 + 1024;
constexpr uint32_t kBudget = 1u << 24;
constexpr int kGemmPlanSms = 152;  // the K split depends on the shape alone

__device__ __forceinline__ bool gwait(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                      unsigned *status) {
  for (uint32_t i = 0; i < kBudget; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

__device__ __forceinline__ void gdrain(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kBudget; ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

}  // namespace

// One work item: a 128 x 256 output tile of one matrix of the job, over one
// K slice.
struct GemmItem {
  int mat, m0, n0, kb0, kb1, ks;
};

__device__ __forceinline__ GemmItem gemm_item(const GemmJob &job, int t, int mtiles, int nk) {
  const int ntiles = job.ntile0[job.count];
  const int per = mtiles * ntiles;
  GemmItem it;
  it.ks = t / per;
  const int r = t % per, mt = r / ntiles, nt = r % ntiles;
  int mat = 0;
  while (mat + 1 < job.count && nt >= job.ntile0[mat + 1]) ++mat;
  it.mat = mat;
  it.m0 = mt * BM;
  it.n0 = (nt - job.ntile0[mat]) * BN;
  const int nkb = (nk + job.ksplit - 1) / job.ksplit;
  it.kb0 = it.ks * nkb;
  it.kb1 = min(nk, it.kb0 + nkb);
  return it;
}

// kMode 0: C = A B (bf16); 1: C <- swish(A B) (.) C; 2: fp32 partial
// products of each K slice into P[ks][M][ldc] at the matrix's columns.
template <int kMode>
__global__ void __launch_bounds__(kNT, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ GemmJob job,
               int M, int K, unsigned *status) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = tc::smem_align1024(smraw);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint64_t *empty = full + kStages;
  uint64_t *acc_full = empty + kStages;  // [2]
  uint64_t *acc_empty = acc_full + 2;    // [2]
  uint64_t *drain = acc_empty + 2;       // MMA completion marker
  uint32_t *tbase_p = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort_p = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // M may be ragged: the last row tile's missing rows of A are outside the
  // tensor map and arrive as zeros; their rows of C are not stored.
  const int mtiles = (M + BM - 1) / BM, nk = K / BK;
  const int tiles = mtiles * job.ntile0[job.count] * job.ksplit;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 1);
    }
    tc::mbar_init(drain, 1);
    *abort_p = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase_p, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = *tbase_p;

  // With early_b the producer sends the B tiles of the first stages before
  // waiting for the kernel before this one; their A tiles follow the wait.
  int pre = 0;
  if (job.early_b && warp == 0 && lane == 0) {
    for (int t = blockIdx.x; t < tiles && pre < kStages; t += gridDim.x) {
      const GemmItem w = gemm_item(job, t, mtiles, nk);
      const CUtensorMap *tmB = w.mat == 0   ? &job.tmB[0]
                               : w.mat == 1 ? &job.tmB[1]
                               : w.mat == 2 ? &job.tmB[2]
                                            : &job.tmB[3];
      for (int kb = w.kb0; kb < w.kb1 && pre < kStages; ++kb, ++pre) {
        uint8_t *st = sm + pre * kStageBytes;
        tc::mbar_arrive_expect_tx(&full[pre], kStageBytes);
#pragma unroll
        for (int j = 0; j < BN / 64; ++j)
          tc::tma_load_2d(st + kABytes + j * 8192, tmB, &full[pre], w.n0 + j * 64, kb * BK);
      }
    }
  }
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tmA);
#pragma unroll
      for (int i = 0; i < kGemmJobMax; ++i)
        if (i < job.count) tc::prefetch_tmap(&job.tmB[i]);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        const GemmItem w = gemm_item(job, t, mtiles, nk);
        const int m0 = w.m0, n0 = w.n0;
        // constant indices: each map's address stays the kernel parameter's own
        const CUtensorMap *tmB = w.mat == 0   ? &job.tmB[0]
                                 : w.mat == 1 ? &job.tmB[1]
                                 : w.mat == 2 ? &job.tmB[2]
                                              : &job.tmB[3];
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !gwait(&empty[s], ((it / kStages) - 1) & 1, abort_p, status)) {
            ok = false;
            break;
          }
          uint8_t *st = sm + s * kStageBytes;
          if (it >= pre) tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
          tc::tma_load_2d(st, &tmA, &full[s], kb * BK, m0);
          if (it >= pre) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tc::tma_load_2d(st + kABytes + j * 8192, tmB, &full[s], n0 + j * 64, kb * BK);
          }
        }
      }
      // Every load is issued: the next kernel may be scheduled (it waits
      // for this one to complete before touching its results).
      pdl_launch_dependents();
      for (int i = it > kStages ? it - kStages : 0; i < it; ++i)
        gdrain(&full[i % kStages], (i / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, BN, 0, 1);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++lt) {
        const int buf = lt & 1;
        if (lt >= 2 && !gwait(&acc_empty[buf], ((lt >> 1) - 1) & 1, abort_p, status)) break;
        tc::tc_fence_after();
        const uint32_t d = tb + buf * BN;
        const GemmItem w = gemm_item(job, t, mtiles, nk);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          if (!gwait(&full[s], (it / kStages) & 1, abort_p, status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(sm + s * kStageBytes), sb = sa + kABytes;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_ss(d, tc::smem_desc(sa + k * 32, 16, 1024, tc::kSw128),
                       tc::smem_desc(sb + k * 2048, 8192, 1024, tc::kSw128), idesc,
                       (kb > w.kb0) || k != 0);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&acc_full[buf]);
      }
      tc::mma_commit(drain);  // arrives once every MMA issued above is done
      gdrain(drain, 0);
    }
    __syncwarp();
  } else {
    // Epilogue: thread = one accumulator row (TMEM lane).
    const int q = warp & 3, row = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    int lt = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      bool ok = gwait(&acc_full[buf], (lt >> 1) & 1, abort_p, status);
      {  // all four epilogue warps leave together
        uint32_t r;
        asm volatile(
            "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
            " bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
            : "=r"(r)
            : "r"((uint32_t)ok)
            : "memory");
        ok = r != 0;
      }
      if (!ok) break;
      tc::tc_fence_after();
      const GemmItem w = gemm_item(job, t, mtiles, nk);
      const int m0 = w.m0, n0 = w.n0 + job.col0[w.mat];
      const bool live = m0 + row < M;  // the TMEM loads stay warp-wide
      const long long orow = (long long)(live ? m0 + row : 0);
      __nv_bfloat16 *crow = kMode == 2 ? nullptr : job.C + orow * job.ldc + n0;
      float *prow = kMode == 2 ? job.P + ((long long)w.ks * M + orow) * job.ldc + n0 : nullptr;
      for (int g = 0; g < BN / 32; ++g) {
        uint32_t r[32];
        tc::tmem_ld32(tb + lb + buf * BN + g * 32, r);
        tc::tmem_ld_wait();
        if (!live) continue;
        if constexpr (kMode == 2) {
          float4 *pd = reinterpret_cast<float4 *>(prow + g * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            pd[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          continue;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(crow + g * 32);
        if constexpr (kMode == 1) {
          // C <- swish(acc) (.) C: fast exponential and divide, a few ulp in
          // fp32 before the bf16 rounding; swish -> 0 as acc -> -inf.
          uint4 cur[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) cur[v] = dst[v];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t cw[4] = {cur[v].x, cur[v].y, cur[v].z, cur[v].w};
            uint32_t ow[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a0 = __uint_as_float(r[8 * v + 2 * e]);
              const float a1 = __uint_as_float(r[8 * v + 2 * e + 1]);
              const float y0 = __uint_as_float(cw[e] << 16), y1 = __uint_as_float(cw[e] & 0xffff0000u);
              ow[e] = tc::pack_bf16(y0 * __fdividef(a0, 1.f + __expf(-a0)),
                                    y1 * __fdividef(a1, 1.f + __expf(-a1)));
            }
            dst[v] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          }
        } else {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(
                tc::pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                tc::pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                tc::pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                tc::pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
        }
      }
      tc::tc_fence_before();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid == 64) tc::mbar_arrive(&acc_empty[buf]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

bool gemm_tc_supported(const void *A, const void *Bm, const void *C, int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return false;
  if (N % BN || K % BK) return false;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Bm) |
       reinterpret_cast<uintptr_t>(C)) & 15)
    return false;
  return tmap_available();
}

static bool encode_b(CUtensorMap *tm, const void *Bm, int N, int K) {
  const cuuint64_t db[2] = {(cuuint64_t)N, (cuuint64_t)K};
  const cuuint64_t sb[1] = {(cuuint64_t)N * 2};
  const cuuint32_t bb[2] = {64, BK};
  return tmap_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Bm, db, sb, bb,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int kMode>
static cudaError_t launch_job(const void *A, const GemmJob &job, int M, int K, unsigned *status,
                              cudaStream_t st) {
  CUtensorMap ta;
  const cuuint64_t da[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t sa[1] = {(cuuint64_t)K * 2};
  const cuuint32_t ba[2] = {BK, BM};
  if (!tmap_encode(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, da, sa, ba,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_tc_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int items = ((M + BM - 1) / BM) * job.ntile0[job.count] * job.ksplit;
  const int grid = items < sms ? items : sms;
  return launch_k(gemm_tc_kernel<kMode>, dim3(grid), dim3(kNT), kSmem, st, true, ta, job, M, K,
                  status);
}

cudaError_t launch_gemm_tc(const void *A, const void *Bm, void *C, int M, int N, int K,
                           unsigned *status, cudaStream_t st, bool gate) {
  GemmJob job;
  if (!encode_b(&job.tmB[0], Bm, N, K)) return cudaErrorInvalidValue;
  job.count = 1;
  job.ntile0[1] = N / BN;
  job.ldc = N;
  job.ksplit = 1;
  job.C = reinterpret_cast<__nv_bfloat16 *>(C);
  return gate ? launch_job<1>(A, job, M, K, status, st) : launch_job<0>(A, job, M, K, status, st);
}

int gemm_tc_split(int M, int Ntot, int K) {
  const int tiles = ((M + BM - 1) / BM) * (Ntot / BN), nk = K / BK;
  int ks = (2 * kGemmPlanSms + tiles - 1) / tiles;  // about two items per SM
  const int cap = K / (8 * (M > 0 ? M : 1));       // partials <= 1/4 of the weight bytes
  ks = ks < cap ? ks : cap;
  ks = ks < nk ? ks : nk;
  if (ks < 1) ks = 1;
  const int nkb = (nk + ks - 1) / ks;
  return (nk + nkb - 1) / nkb;  // every slice non-empty
}

cudaError_t launch_gemm_tc_partials(const void *A, int count, const void *const *Bs,
                                    const int *Ns, int M, int K, float *P, int ksplit,
                                    unsigned *status, cudaStream_t st, bool early_b) {
  if (count < 1 || count > kGemmJobMax || ksplit < 1) return cudaErrorInvalidValue;
  GemmJob job;
  job.count = count;
  job.early_b = early_b ? 1 : 0;
  int col = 0, nt = 0;
  for (int i = 0; i < count; ++i) {
    if (!encode_b(&job.tmB[i], Bs[i], Ns[i], K)) return cudaErrorInvalidValue;
    job.ntile0[i] = nt;
    job.col0[i] = col;
    nt += Ns[i] / BN;
    col += Ns[i];
  }
  job.ntile0[count] = nt;
  job.ldc = col;
  job.ksplit = ksplit;
  job.P = P;
  return launch_job<2>(A, job, M, K, status, st);
}

}  // namespace ret
