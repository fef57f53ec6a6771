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
constexpr int kSkMaxSplit = 608;
constexpr int kSkMaxRowsPerSlice = 512;       // K rows per CTA (A slice in shared memory)
}  // namespace

// grid: x = column block of 2048 (over every matrix of the job), y = K
// slice.  P: [split][M][Ntot] fp32, matrix i's columns at col0[i].
template <int MB>
__global__ void __launch_bounds__(kSkWarps * 32)
gemm_skinny_kernel(const __nv_bfloat16 *__restrict__ A, const SkinnyJob job,
                   float *__restrict__ P, int M, int K, int rows_per_slice) {
  __shared__ float As[kSkMaxRowsPerSlice][MB];
  const int k0 = blockIdx.y * rows_per_slice;
  const int kn = min(rows_per_slice, K - k0);
  for (int e = threadIdx.x; e < kn * MB; e += blockDim.x) {
    const int r = e / MB, m = e % MB;
    As[r][m] = m < M ? __bfloat162float(A[(long long)m * K + k0 + r]) : 0.f;
  }
  __syncthreads();
  int mat = 0;
  while (mat + 1 < job.count && (int)blockIdx.x >= job.blk0[mat + 1]) ++mat;
  const int N = job.N[mat];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = ((int)blockIdx.x - job.blk0[mat]) * kSkCtaCols + warp * kSkCols + lane * 8;
  if (n0 >= N) return;  // N % 8 == 0: a lane's eight columns are all in or all out
  float acc[MB][8];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
  const __nv_bfloat16 *bcol = job.B[mat] + (long long)k0 * N + n0;
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
  float *pt = P + (long long)blockIdx.y * M * job.Ntot + job.col0[mat] + n0;
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m >= M) break;
    float4 *dst = reinterpret_cast<float4 *>(pt + (long long)m * job.Ntot);
    dst[0] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    dst[1] = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
  }
}

// C_i[m][n] = epilogue(bf16(sum over the slices of P[s][m][col0_i + n])):
// none; GELU x Phi(x) = x (1 + erf(x / sqrt 2)) / 2 of the rounded sum; or
// the rounded sum plus R[m][n] (the skip connection).  Each epilogue rounds
// to bf16 where the separate kernels it replaces would.  One warp per (row,
// 8 adjacent columns): lane l adds slices l, l + 32, ... in order, then the
// lanes' sums are combined by a fixed butterfly, so the result does not
// depend on timing (the partials were just written and are read from L2).
__global__ void __launch_bounds__(256)
skinny_reduce_kernel(const float *__restrict__ P, const SkinnyJob job, int M, int split) {
  const long long MN = (long long)M * job.Ntot;
  const long long g = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // 8-column group
  const int lane = threadIdx.x & 31;
  if (g * 8 >= MN) return;
  const long long i0 = g * 8;  // Ntot % 8 == 0: the group lies in one row and one matrix
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  int t = lane;
  for (; t + 96 < split; t += 128) {  // four slices' loads in flight, added in slice order
    float4 x[4], y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 *src = reinterpret_cast<const float4 *>(P + (long long)(t + 32 * u) * MN + i0);
      x[u] = src[0];
      y[u] = src[1];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a.x += x[u].x; a.y += x[u].y; a.z += x[u].z; a.w += x[u].w;
      b.x += y[u].x; b.y += y[u].y; b.z += y[u].z; b.w += y[u].w;
    }
  }
  for (; t < split; t += 32) {
    const float4 *src = reinterpret_cast<const float4 *>(P + (long long)t * MN + i0);
    const float4 x = src[0], y = src[1];
    a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
  }
  float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] += __shfl_xor_sync(0xffffffffu, v[e], o);
  if (lane >= 8) return;
  const int m = (int)(i0 / job.Ntot), n = (int)(i0 % job.Ntot) + lane;
  int mat = 0;
  while (mat + 1 < job.count && n >= job.col0[mat + 1]) ++mat;
  float sum = v[0];
#pragma unroll
  for (int e = 1; e < 8; ++e)
    if (lane == e) sum = v[e];
  float y = __bfloat162float(__float2bfloat16_rn(sum));
  const long long o = (long long)m * job.N[mat] + (n - job.col0[mat]);
  if (job.epi == kSkEpGelu)
    y = 0.5f * y * (1.f + erff(y * 0.70710678118654752f));
  else if (job.epi == kSkEpResidual)
    y = y + __bfloat162float(job.R[o]);
  job.C[mat][o] = __float2bfloat16_rn(y);
}

// The same reduce for few slices (the tensor-core GEMM's K split): one
// thread per (row, 8 adjacent columns) adds the slices in order.
__global__ void __launch_bounds__(256)
skinny_reduce_few_kernel(const float *__restrict__ P, const SkinnyJob job, int M, int split) {
  const long long MN = (long long)M * job.Ntot;
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g * 8 >= MN) return;
  const long long i0 = g * 8;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int t = 0; t < split; ++t) {
    const float4 *src = reinterpret_cast<const float4 *>(P + (long long)t * MN + i0);
    const float4 x = src[0], y = src[1];
    v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
    v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
  }
  const int m = (int)(i0 / job.Ntot), n0 = (int)(i0 % job.Ntot);
  int mat = 0;
  while (mat + 1 < job.count && n0 >= job.col0[mat + 1]) ++mat;
  const long long o = (long long)m * job.N[mat] + (n0 - job.col0[mat]);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float y = __bfloat162float(__float2bfloat16_rn(v[e]));
    if (job.epi == kSkEpGelu)
      y = 0.5f * y * (1.f + erff(y * 0.70710678118654752f));
    else if (job.epi == kSkEpResidual)
      y = y + __bfloat162float(job.R[o + e]);
    job.C[mat][o + e] = __float2bfloat16_rn(y);
  }
}

bool gemm_skinny_supported(const void *A, const void *Bm, const void *C, int M, int N, int K) {
  return M >= 1 && M <= 16 && N >= 8 && N % 8 == 0 && K >= 1 &&
         reinterpret_cast<uintptr_t>(Bm) % 16 == 0 && A && C;
}

// Slices of K: about four CTAs per SM of a 152-SM GB300 (each CTA keeps
// 32 KB of weight rows in flight, and the register budget allows four), at
// least kSkUnroll rows and at most kSkMaxRowsPerSlice rows per slice, and
// fp32 partials (split * M * N * 4 bytes) of at most 16 MB, which stay in
// L2 between the two kernels.  The plan depends on the shape alone (not on
// the device that happens to be current), so a workspace sized for a shape
// always fits the launch of that shape.
constexpr int kSkPlanSms = 152;
constexpr long long kSkMaxPartialBytes = 16LL << 20;
static void skinny_plan(int M, int N, int K, int &split, int &rows) {
  const int colblocks = (N + kSkCtaCols - 1) / kSkCtaCols;
  int s = (4 * kSkPlanSms + colblocks - 1) / colblocks;
  s = s < kSkMaxSplit ? s : kSkMaxSplit;
  const long long per_slice = 4LL * (M > 0 ? M : 1) * N;
  const long long cap = kSkMaxPartialBytes / (per_slice > 0 ? per_slice : 1);
  s = s < cap ? s : (int)cap;
  const int rmin = (K + kSkUnroll - 1) / kSkUnroll;  // slices of at least kSkUnroll rows
  s = s < rmin ? s : rmin;
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

bool skinny_job_init(SkinnyJob &job, int count, const void *const *Bs, void *const *Cs,
                     const int *Ns, int epi, const void *R) {
  if (count < 1 || count > kSkMaxMats) return false;
  job.count = count;
  job.epi = epi;
  job.R = reinterpret_cast<const __nv_bfloat16 *>(R);
  int col = 0, blk = 0;
  for (int i = 0; i < count; ++i) {
    if (Ns[i] < 8 || Ns[i] % 8 || !Bs[i] || !Cs[i] || reinterpret_cast<uintptr_t>(Bs[i]) % 16)
      return false;
    job.B[i] = reinterpret_cast<const __nv_bfloat16 *>(Bs[i]);
    job.C[i] = reinterpret_cast<__nv_bfloat16 *>(Cs[i]);
    job.N[i] = Ns[i];
    job.col0[i] = col;
    job.blk0[i] = blk;
    col += Ns[i];
    blk += (Ns[i] + kSkCtaCols - 1) / kSkCtaCols;
  }
  job.Ntot = col;
  job.blk0[count] = blk;
  return (epi != kSkEpResidual || (count == 1 && R));
}

cudaError_t launch_gemm_skinny_job(const void *A, const SkinnyJob &job, int M, int K,
                                   float *partial, cudaStream_t st) {
  int split = 1, rows = 1;
  skinny_plan(M, job.Ntot, K, split, rows);
  dim3 grid(job.blk0[job.count], split);
  const auto *a = reinterpret_cast<const __nv_bfloat16 *>(A);
  const int threads = kSkWarps * 32;
  if (M <= 1)
    gemm_skinny_kernel<1><<<grid, threads, 0, st>>>(a, job, partial, M, K, rows);
  else if (M <= 2)
    gemm_skinny_kernel<2><<<grid, threads, 0, st>>>(a, job, partial, M, K, rows);
  else if (M <= 4)
    gemm_skinny_kernel<4><<<grid, threads, 0, st>>>(a, job, partial, M, K, rows);
  else if (M <= 8)
    gemm_skinny_kernel<8><<<grid, threads, 0, st>>>(a, job, partial, M, K, rows);
  else
    gemm_skinny_kernel<16><<<grid, threads, 0, st>>>(a, job, partial, M, K, rows);
  return cudaGetLastError();
}

cudaError_t launch_skinny_reduce_job(const float *partial, const SkinnyJob &job, int M, int K,
                                     cudaStream_t st) {
  int split = 1, rows = 1;
  skinny_plan(M, job.Ntot, K, split, rows);
  return launch_skinny_reduce_split(partial, job, M, split, st);
}

cudaError_t launch_skinny_reduce_split(const float *partial, const SkinnyJob &job, int M,
                                       int split, cudaStream_t st) {
  const long long groups = (long long)M * job.Ntot / 8;
  if (split <= 16)  // one thread per group
    skinny_reduce_few_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(partial, job, M,
                                                                              split);
  else  // one warp per group
    skinny_reduce_kernel<<<(unsigned)((groups * 32 + 255) / 256), 256, 0, st>>>(partial, job, M,
                                                                               split);
  return cudaGetLastError();
}

// One matrix, no epilogue.
static SkinnyJob single_job(const void *Bm, void *C, int N) {
  SkinnyJob job;
  job.count = 1;
  job.B[0] = reinterpret_cast<const __nv_bfloat16 *>(Bm);
  job.C[0] = reinterpret_cast<__nv_bfloat16 *>(C);
  job.N[0] = N;
  job.Ntot = N;
  job.blk0[1] = (N + kSkCtaCols - 1) / kSkCtaCols;
  return job;
}

cudaError_t launch_gemm_skinny(const void *A, const void *Bm, int M, int N, int K,
                               float *partial, cudaStream_t st) {
  return launch_gemm_skinny_job(A, single_job(Bm, nullptr, N), M, K, partial, st);
}

cudaError_t launch_skinny_reduce(const float *partial, void *C, int M, int N, int K,
                                 cudaStream_t st) {
  return launch_skinny_reduce_job(partial, single_job(nullptr, C, N), M, K, st);
}

}  // namespace ret
