// CUDA-core GEMM C[M,N] = A[M,K] B[K,N] (bf16 row-major inputs, fp32
// accumulation): the fallback for projection shapes the tensor-core GEMM
// does not take.
#include "common.cuh"
#include "launch.h"

namespace ret {

namespace {
constexpr int BM = 64, BN = 64, BK = 16;
}

__global__ void __launch_bounds__(256)
gemm_simt_kernel(const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ Bm,
                 void *__restrict__ C, int M, int N, int K, int out_bf16) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int e = threadIdx.x; e < BM * BK; e += 256) {
      const int r = e / BK, c = e % BK;
      const int gm = m0 + r, gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? __bfloat162float(A[(long long)gm * K + gk]) : 0.f;
    }
    for (int e = threadIdx.x; e < BK * BN; e += 256) {
      const int r = e / BN, c = e % BN;
      const int gk = k0 + r, gn = n0 + c;
      Bs[r][c] = (gk < K && gn < N) ? __bfloat162float(Bm[(long long)gk * N + gn]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < M && gn < N) st_elem(C, (long long)gm * N + gn, acc[i][j], out_bf16);
    }
}

cudaError_t launch_gemm_bf16(const void *A, const void *Bm, void *C, int M, int N, int K,
                             int out_bf16, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  gemm_simt_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16 *>(A),
                                         reinterpret_cast<const __nv_bfloat16 *>(Bm), C, M,
                                         N, K, out_bf16);
  return cudaGetLastError();
}

}  // namespace ret
