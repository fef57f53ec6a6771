// Tensor-core self-test: one CTA computes D = A * B^T (bf16 in, fp32
// accumulate) with one tcgen05 MMA chain, with A and B laid out in shared
// memory in the 128-byte-swizzled K-major or MN-major forms (or A in TMEM)
// that the retention kernels use.  All 128 TMEM lanes of D are written out,
// so the accumulator layout of M=64 can be checked as well as the values.
// The descriptor strides come from the caller, which lets one run check
// layout hypotheses side by side.
#include <cooperative_groups.h>

#include "tc.cuh"

namespace cg = cooperative_groups;

namespace ret {

namespace {
constexpr int kProbeSmem = 200 * 1024;
}

__global__ void __launch_bounds__(128)
tc_probe_kernel(int a_mode, int b_mode, int M, int N, int K, int a_lbo, int a_sbo, int b_lbo,
                int b_sbo, const __nv_bfloat16 *__restrict__ A,
                const __nv_bfloat16 *__restrict__ B, float *__restrict__ D,
                unsigned *status) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  uint8_t *sm = tc::smem_align1024(smraw);
  uint8_t *sA = sm;                 // up to 64 KB
  uint8_t *sB = sm + 64 * 1024;     // up to 64 KB
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tbase, 512);
    tc::tmem_relinquish();
  }
  // Fill shared memory.  K-major: region per 64-wide K block, rows of 128 B.
  // MN-major: region per 64-wide MN block, one 128-B row per k.
  auto put = [&](uint8_t *base, int mode, int rows, int r, int k, __nv_bfloat16 x) {
    uint32_t off;
    if (mode == 0)
      off = (uint32_t)(k / 64) * rows * 128 + tc::sw128_off(r, (k % 64) / 8) + (k % 8) * 2;
    else
      off = (uint32_t)(r / 64) * K * 128 + tc::sw128_off(k, (r % 64) / 8) + (r % 8) * 2;
    *reinterpret_cast<__nv_bfloat16 *>(base + off) = x;
  };
  if (a_mode != 2)
    for (int e = tid; e < M * K; e += 128) put(sA, a_mode, M, e / K, e % K, A[e]);
  for (int e = tid; e < N * K; e += 128) put(sB, b_mode, N, e / K, e % K, B[e]);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t t0 = tbase;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  // Sentinel in every D column of this warp's lanes, then A into TMEM.
  {
    uint32_t r[32];
    for (int i = 0; i < 32; ++i) r[i] = 0x7fc00000u;  // NaN
    for (int c = 0; c < N; c += 32) tc::tmem_st32(t0 + lane_base + c, r);
    if (a_mode == 2) {
      const int m = tid;
      for (int c0 = 0; c0 < K / 2; c0 += 32) {
        for (int i = 0; i < 32; ++i) {
          const int k = 2 * (c0 + i);
          r[i] = (m < M && k + 1 < K + 1 && k < K)
                     ? tc::pack_bf16(__bfloat162float(A[m * K + k]),
                                     __bfloat162float(A[m * K + k + 1]))
                     : 0u;
        }
        tc::tmem_st32(t0 + lane_base + 256 + c0, r);
      }
    }
    tc::tmem_st_wait();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16(M, N, a_mode == 1, b_mode == 1);
    for (int s = 0; s < K / 16; ++s) {
      const int k0 = s * 16;
      uint64_t bdesc;
      if (b_mode == 0)
        bdesc = tc::smem_desc(tc::smem_u32(sB) + (k0 / 64) * N * 128 + (k0 % 64) * 2, 16, 1024,
                              tc::kSw128);
      else
        bdesc = tc::smem_desc(tc::smem_u32(sB) + k0 * 128, b_lbo, b_sbo, tc::kSw128);
      if (a_mode == 2) {
        tc::mma_ts(t0, t0 + 256 + k0 / 2, bdesc, idesc, s > 0);
      } else {
        uint64_t adesc;
        if (a_mode == 0)
          adesc = tc::smem_desc(tc::smem_u32(sA) + (k0 / 64) * M * 128 + (k0 % 64) * 2, 16,
                                1024, tc::kSw128);
        else
          adesc = tc::smem_desc(tc::smem_u32(sA) + k0 * 128, a_lbo, a_sbo, tc::kSw128);
        tc::mma_ss(t0, adesc, bdesc, idesc, s > 0);
      }
    }
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, status, 1u << 22);
  tc::tc_fence_after();
  if (ok) {
    uint32_t r[32];
    for (int c = 0; c < N; c += 32) {
      tc::tmem_ld32(t0 + lane_base + c, r);
      tc::tmem_ld_wait();
      for (int i = 0; i < 32 && c + i < N; ++i)
        D[(warp * 32 + (tid & 31)) * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(t0, 512);
}

// D = A B^T with one MMA chain (K-major A and B, M = N = 128, K = 64), then
// the same chain again with the first MMA scaling the accumulator:
// D' = A B^T + D 2^-n.  Checks the scale-input-d operand of tcgen05.mma.
__global__ void __launch_bounds__(128)
tc_probe_scale_kernel(int n, const __nv_bfloat16 *__restrict__ A,
                      const __nv_bfloat16 *__restrict__ B, float *__restrict__ D,
                      unsigned *status) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  uint8_t *sm = tc::smem_align1024(smraw);
  uint8_t *sA = sm, *sB = sm + 16 * 1024;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int M = 128, N = 128, K = 64;
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tbase, 128);
    tc::tmem_relinquish();
  }
  for (int e = tid; e < M * K; e += 128) {
    const int r = e / K, k = e % K;
    *reinterpret_cast<__nv_bfloat16 *>(sA + tc::sw128_off(r, k / 8) + (k % 8) * 2) = A[e];
    *reinterpret_cast<__nv_bfloat16 *>(sB + tc::sw128_off(r, k / 8) + (k % 8) * 2) = B[e];
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t t0 = tbase;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16(M, N, 0, 0);
    for (int pass = 0; pass < 2; ++pass)
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t a = tc::smem_desc(tc::smem_u32(sA) + s * 32, 16, 1024, tc::kSw128);
        const uint64_t b = tc::smem_desc(tc::smem_u32(sB) + s * 32, 16, 1024, tc::kSw128);
        if (pass == 1 && s == 0)
          tc::mma_ss_scale_d(t0, a, b, idesc, n);
        else
          tc::mma_ss(t0, a, b, idesc, (pass | s) != 0);
      }
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, status, 1u << 22);
  tc::tc_fence_after();
  if (ok) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t r[32];
    for (int c = 0; c < N; c += 32) {
      tc::tmem_ld32(t0 + lane_base + c, r);
      tc::tmem_ld_wait();
      for (int i = 0; i < 32; ++i) D[(warp * 32 + (tid & 31)) * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(t0, 128);
}

// The CTA-pair MMA (cta_group::2): the two CTAs of a cluster compute D =
// A B^T for 256 rows, CTA r holding rows 128 r .. 128 r + 127 of A and
// columns N/2 r .. N/2 (r + 1) - 1 of B (both K-major, 128-byte swizzled)
// and receiving its 128 rows of D in its own TMEM.  The even CTA issues the
// MMAs; the commit arrives on the barrier of both.  Each CTA also writes
// the TMEM address its allocation returned to tbase_out[r].
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128)
tc_probe_pair_kernel(int N, int K, const __nv_bfloat16 *__restrict__ A,
                     const __nv_bfloat16 *__restrict__ B, float *__restrict__ D,
                     unsigned *__restrict__ tbase_out, unsigned *status) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  uint8_t *sm = tc::smem_align1024(smraw);
  uint8_t *sA = sm;              // 128 rows x K: K/64 blocks of 16 KB
  uint8_t *sB = sm + 32 * 1024;  // N/2 rows x K: K/64 blocks of N/2 x 128 B
  const int tid = threadIdx.x, warp = tid >> 5;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), nh = N / 2;
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc2(&tbase, 256);
    tc::tmem_relinquish2();
  }
  for (int e = tid; e < 128 * K; e += 128) {
    const int r = e / K, k = e % K;
    *reinterpret_cast<__nv_bfloat16 *>(sA + (k / 64) * 128 * 128 + tc::sw128_off(r, (k % 64) / 8) +
                                       (k % 8) * 2) = A[(rank * 128 + r) * K + k];
  }
  for (int e = tid; e < nh * K; e += 128) {
    const int r = e / K, k = e % K;
    *reinterpret_cast<__nv_bfloat16 *>(sB + (k / 64) * nh * 128 + tc::sw128_off(r, (k % 64) / 8) +
                                       (k % 8) * 2) = B[(rank * nh + r) * K + k];
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  cluster.sync();  // both CTAs' operands and barriers exist before the MMAs
  tc::tc_fence_after();
  const uint32_t t0 = tbase;
  if (tid == 0) tbase_out[rank] = t0;
  if (rank == 0 && tid == 0) {
    const uint32_t idesc = tc::idesc_bf16(256, N, 0, 0);
    for (int s = 0; s < K / 16; ++s) {
      const int k0 = s * 16;
      const uint64_t a = tc::smem_desc(tc::smem_u32(sA) + (k0 / 64) * 128 * 128 + (k0 % 64) * 2,
                                       16, 1024, tc::kSw128);
      const uint64_t b = tc::smem_desc(tc::smem_u32(sB) + (k0 / 64) * nh * 128 + (k0 % 64) * 2,
                                       16, 1024, tc::kSw128);
      tc::mma2_ss(t0, a, b, idesc, s > 0);
    }
    tc::mma2_commit_mc(&bar, 0x3);
  }
  const bool ok = tc::mbar_wait(&bar, 0, status, 1u << 22);
  tc::tc_fence_after();
  if (ok) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t r[32];
    for (int c = 0; c < N; c += 32) {
      tc::tmem_ld32(t0 + lane_base + c, r);
      tc::tmem_ld_wait();
      for (int i = 0; i < 32; ++i)
        D[(rank * 128 + warp * 32 + (tid & 31)) * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  cluster.sync();  // the pair's MMAs and TMEM reads are done in both CTAs
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc2(t0, 256);
}

}  // namespace ret

extern "C" int retention_tc_probe_pair(int N, int K, const void *A, const void *B, float *D,
                                       unsigned *tbase_out, unsigned *status,
                                       ret_stream_t stream) {
  using namespace ret;
  if ((N != 128 && N != 256) || (K != 64 && K != 128)) return RET_EINVAL;
  if (!A || !B || !D || !tbase_out || !status) return RET_EINVAL;
  const int smem = 32 * 1024 + 32 * 1024 + 1024;
  if (cudaFuncSetAttribute(tc_probe_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return RET_ECUDA;
  tc_probe_pair_kernel<<<2, 128, smem, (cudaStream_t)stream>>>(
      N, K, reinterpret_cast<const __nv_bfloat16 *>(A), reinterpret_cast<const __nv_bfloat16 *>(B),
      D, tbase_out, status);
  return cudaGetLastError() == cudaSuccess ? RET_OK : RET_ECUDA;
}

extern "C" int retention_tc_probe_scale_d(int n, const void *A, const void *B, float *D,
                                          unsigned *status, ret_stream_t stream) {
  using namespace ret;
  if (n < 0 || n > 15 || !A || !B || !D || !status) return RET_EINVAL;
  const int smem = 33 * 1024;
  if (cudaFuncSetAttribute(tc_probe_scale_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return RET_ECUDA;
  tc_probe_scale_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
      n, reinterpret_cast<const __nv_bfloat16 *>(A), reinterpret_cast<const __nv_bfloat16 *>(B),
      D, status);
  return cudaGetLastError() == cudaSuccess ? RET_OK : RET_ECUDA;
}

extern "C" int retention_tc_probe(int a_mode, int b_mode, int M, int N, int K, int a_lbo,
                                  int a_sbo, int b_lbo, int b_sbo, const void *A,
                                  const void *B, float *D, unsigned *status,
                                  ret_stream_t stream) {
  using namespace ret;
  if (a_mode < 0 || a_mode > 2 || b_mode < 0 || b_mode > 1) return RET_EINVAL;
  if ((M != 64 && M != 128) || N < 16 || N > 256 || N % 32 || K < 16 || K > 128 || K % 64)
    return RET_EINVAL;
  if (a_mode == 2 && M != 128) return RET_EINVAL;
  if (!A || !B || !D || !status) return RET_EINVAL;
  cudaError_t e = cudaFuncSetAttribute(tc_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return RET_ECUDA;
  tc_probe_kernel<<<1, 128, kProbeSmem, (cudaStream_t)stream>>>(
      a_mode, b_mode, M, N, K, a_lbo, a_sbo, b_lbo, b_sbo,
      reinterpret_cast<const __nv_bfloat16 *>(A), reinterpret_cast<const __nv_bfloat16 *>(B),
      D, status);
  return cudaGetLastError() == cudaSuccess ? RET_OK : RET_ECUDA;
}
