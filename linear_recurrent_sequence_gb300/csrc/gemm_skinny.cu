// Weight-streaming GEMM for few rows: C[M,N] = A[M,K] B[K,N] with M <= 16
// (a decode batch), bf16 row-major operands, fp32 accumulation, bf16 result.
// At these M the product is bound by reading B once from HBM, so the kernel
// is built around that stream:
//   - a warp owns 256 columns of B and reads each of its rows as one 512-byte
//     run (16 bytes, eight columns, per lane); a CTA's eight warps own 2048
//     adjacent columns;
//   - K is split across CTAs (grid.y) so that about two CTAs run per SM;
//     each CTA keeps its K-slice of A in shared memory (fp32, MB rows) and
//     writes an fp32 partial tile; a second kernel adds the partials in
//     slice order (deterministic) and rounds to bf16;
//   - eight rows of B per lane are loaded before they are used, to keep
//     enough bytes in flight.
#include "common.cuh"
#include "launch.h"

namespace ret {

namespace {
constexpr int kSkWarps = 8;
constexpr int kSkCols = 256;                  // columns per warp (32 lanes x 8)
constexpr int kSkCtaCols = kSkWarps * kSkCols;  // 2048
constexpr int kSkUnroll = 8;                  // rows of B in flight per lane
constexpr int kSkMaxSplit = 128;
constexpr int kSkMaxRowsPerSlice = 512;       // K rows per CTA (A slice in shared memory)
}  // namespace

// grid: x = column block of 2048, y = K slice.  P: [split][M][N] fp32.
template <int MB>
__global__ void __launch_bounds__(kSkWarps * 32)
gemm_skinny_kernel(const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ Bm,
                   float *__restrict__ P, int M, int N, int K, int rows_per_slice) {
  __shared__ float As[kSkMaxRowsPerSlice][MB];
  const int k0 = blockIdx.y * rows_per_slice;
  const int kn = min(rows_per_slice, K - k0);
  for (int e = threadIdx.x; e < kn * MB; e += blockDim.x) {
    const int r = e / MB, m = e % MB;
    As[r][m] = m < M ? __bfloat162float(A[(long long)m * K + k0 + r]) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kSkCtaCols + warp * kSkCols + lane * 8;
  if (n0 >= N) return;  // N % 8 == 0: a lane's eight columns are all in or all out
  float acc[MB][8];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
  const __nv_bfloat16 *bcol = Bm + (long long)k0 * N + n0;
  for (int r0 = 0; r0 < kn; r0 += kSkUnroll) {
    uint4 w[kSkUnroll];
#pragma unroll
    for (int u = 0; u < kSkUnroll; ++u)
      w[u] = r0 + u < kn ? *reinterpret_cast<const uint4 *>(bcol + (long long)(r0 + u) * N)
                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kSkUnroll; ++u) {
      if (r0 + u >= kn) break;
      const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w[u]);
      float b[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        b[2 * t] = __low2float(h[t]);
        b[2 * t + 1] = __high2float(h[t]);
      }
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const float a = As[r0 + u][m];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[m][c] = fmaf(a, b[c], acc[m][c]);
      }
    }
  }
  float *pt = P + (long long)blockIdx.y * M * N + n0;
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m >= M) break;
    float4 *dst = reinterpret_cast<float4 *>(pt + (long long)m * N);
    dst[0] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    dst[1] = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
  }
}

// C[m][n] = bf16(sum over slices s, in order, of P[s][m][n]).
__global__ void __launch_bounds__(256)
skinny_reduce_kernel(const float *__restrict__ P, __nv_bfloat16 *__restrict__ C, long long MN,
                     int split) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= MN) return;
  float s = 0.f;
  for (int t = 0; t < split; ++t) s += P[(long long)t * MN + i];
  C[i] = __float2bfloat16_rn(s);
}

bool gemm_skinny_supported(const void *A, const void *Bm, const void *C, int M, int N, int K) {
  return M >= 1 && M <= 16 && N >= 8 && N % 8 == 0 && K >= 1 &&
         reinterpret_cast<uintptr_t>(Bm) % 16 == 0 && A && C;
}

// Slices of K: about two CTAs per SM of a 152-SM GB300, at most kSkMaxSplit
// slices, at most kSkMaxRowsPerSlice rows per slice, and at most K / (16 M)
// slices so that the fp32 partials (split * M * N * 4 bytes) stay near 1/8
// of B's bytes.  The plan depends on the shape alone (not on the device
// that happens to be current), so a workspace sized for a shape always fits
// the launch of that shape.
constexpr int kSkPlanSms = 152;
static void skinny_plan(int M, int N, int K, int &split, int &rows) {
  const int colblocks = (N + kSkCtaCols - 1) / kSkCtaCols;
  int s = (2 * kSkPlanSms + colblocks - 1) / colblocks;
  s = s < kSkMaxSplit ? s : kSkMaxSplit;
  const int sm = K / (16 * (M > 0 ? M : 1));
  s = s < sm ? s : sm;
  s = s < K ? s : K;
  if (s < 1) s = 1;
  rows = (K + s - 1) / s;
  if (rows > kSkMaxRowsPerSlice) rows = kSkMaxRowsPerSlice;
  split = (K + rows - 1) / rows;
}

size_t gemm_skinny_partial_bytes(int M, int N, int K) {
  int split = 1, rows = 1;
  skinny_plan(M, N, K, split, rows);
  return (size_t)split * M * N * sizeof(float);
}

cudaError_t launch_gemm_skinny(const void *A, const void *Bm, int M, int N, int K,
                               float *partial, cudaStream_t st) {
  int split = 1, rows = 1;
  skinny_plan(M, N, K, split, rows);
  dim3 grid((N + kSkCtaCols - 1) / kSkCtaCols, split);
  const auto *a = reinterpret_cast<const __nv_bfloat16 *>(A);
  const auto *b = reinterpret_cast<const __nv_bfloat16 *>(Bm);
  const int threads = kSkWarps * 32;
  if (M <= 1)
    gemm_skinny_kernel<1><<<grid, threads, 0, st>>>(a, b, partial, M, N, K, rows);
  else if (M <= 2)
    gemm_skinny_kernel<2><<<grid, threads, 0, st>>>(a, b, partial, M, N, K, rows);
  else if (M <= 4)
    gemm_skinny_kernel<4><<<grid, threads, 0, st>>>(a, b, partial, M, N, K, rows);
  else if (M <= 8)
    gemm_skinny_kernel<8><<<grid, threads, 0, st>>>(a, b, partial, M, N, K, rows);
  else
    gemm_skinny_kernel<16><<<grid, threads, 0, st>>>(a, b, partial, M, N, K, rows);
  return cudaGetLastError();
}

cudaError_t launch_skinny_reduce(const float *partial, void *C, int M, int N, int K,
                                 cudaStream_t st) {
  int split = 1, rows = 1;
  skinny_plan(M, N, K, split, rows);
  const long long MN = (long long)M * N;
  skinny_reduce_kernel<<<(unsigned)((MN + 255) / 256), 256, 0, st>>>(
      partial, reinterpret_cast<__nv_bfloat16 *>(C), MN, split);
  return cudaGetLastError();
}

}  // namespace ret
