// Weight-streaming GEMM for few rows: C[M,N] = A[M,K] B[K,N] with M <= 16
// (a decode batch), bf16 row-major operands, fp32 accumulation, bf16 result.
// At these M the product is bound by reading B once from HBM, so the kernel
// is built around that stream:
//   - a warp owns 256 columns of B and reads each of its rows as one 512-byte
//     run (16 bytes, eight columns, per lane); a CTA's eight warps own 2048
//     adjacent columns;
//   - K is split across CTAs (grid.y) so that about three CTAs (up to four
//     rows) or two (more rows) run per SM;
//     each CTA keeps its K-slice of A in shared memory (fp32, MB rows) and
//     writes an fp32 partial tile; a second kernel adds the partials in
//     slice order (deterministic) and rounds to bf16;
//   - each thread keeps D - 1 rows of its columns of B in flight with
//     asynchronous copies into its own slots of a shared-memory ring (no
//     registers held by loads in flight; each thread reads back only what
//     it copied, so its own copy-group waits order everything).
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace ret {

namespace {
constexpr int kSkWarps = 8;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkCols = 256;                  // columns per warp (32 lanes x 8)
constexpr int kSkCtaCols = kSkWarps * kSkCols;  // 2048
constexpr int kSkMaxSplit = 608;
constexpr int kSkMaxRowsPerSlice = 512;       // K rows per CTA (A slice in shared memory)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
}  // namespace

// Ring depth (rows of B per thread, D - 1 of them in flight): with three
// CTAs per SM (up to four rows) about 180 KB of copies in flight per SM.
// Measured per layer of the 6.7B-scale decode stack at B = 1 / 2 (CTAs per
// SM x depth): 3 x 16 95.8 / 102.5 us, 2 x 24 97.9 / 104.8, 4 x 12
// 95.6 / 104.6, 6 x 8 100.7 / 111.6, 1 x 48 108.1 / 119.0.
template <int MB>
__host__ __device__ constexpr int sk_depth() { return 16; }

// grid: x = column block of 2048 (over every matrix of the job), y = K
// slice.  P: [split][M][Ntot] fp32, matrix i's columns at col0[i].
template <int MB>
__global__ void __launch_bounds__(kSkThreads)
gemm_skinny_kernel(const __nv_bfloat16 *__restrict__ A, const SkinnyJob job,
                   float *__restrict__ P, int M, int K, int rows_per_slice, int early_b) {
  constexpr int D = sk_depth<MB>();
  __shared__ float As[kSkMaxRowsPerSlice][MB];
  extern __shared__ __align__(16) uint4 ring[];  // [D][kSkThreads]
  const int k0 = blockIdx.y * rows_per_slice;
  const int kn = min(rows_per_slice, K - k0);
  int mat = 0;
  while (mat + 1 < job.count && (int)blockIdx.x >= job.blk0[mat + 1]) ++mat;
  const int N = job.N[mat];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = ((int)blockIdx.x - job.blk0[mat]) * kSkCtaCols + warp * kSkCols + lane * 8;
  const bool live = n0 < N;  // N % 8 == 0: a lane's eight columns are all in or all out
  const __nv_bfloat16 *brow = job.B[mat] + (long long)k0 * N + n0;
  const uint32_t slot0 = tc::smem_u32(ring + threadIdx.x), sstride = kSkThreads * 16u;
  if (!early_b) pdl_wait();
  // Rows 0 .. D-2 of B in flight first (one copy group per row): they do
  // not depend on A, so staging A overlaps them (and, with early_b, the
  // end of the kernel before this one).
  const __nv_bfloat16 *bnext = brow;
#pragma unroll 1
  for (int r = 0; r < D - 1; ++r, bnext += N) {
    if (live && r < kn) cp_async16(slot0 + (uint32_t)r * sstride, bnext);
    cp_async_commit();
  }
  if (early_b) pdl_wait();
  for (int e = threadIdx.x; e < kn * MB; e += blockDim.x) {
    const int r = e / MB, m = e % MB;
    As[r][m] = m < M ? __bfloat162float(A[(long long)m * K + k0 + r]) : 0.f;
  }
  __syncthreads();
  if (!live) {
    cp_async_wait<0>();
    pdl_launch_dependents();
    return;
  }
  float2 acc[MB][4];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = make_float2(0.f, 0.f);
  int sl = 0, sn = D - 1;  // ring slots of rows r and r + D - 1
#pragma unroll 1
  for (int r = 0; r < kn; ++r, bnext += N) {
    // Refill the slot of row r - 1 (read in the previous iteration) with
    // row r + D - 1, then wait for row r (at most D - 1 groups pending).
    if (r + D - 1 < kn) cp_async16(slot0 + (uint32_t)sn * sstride, bnext);
    cp_async_commit();
    cp_async_wait<D - 1>();
    const uint4 w = ring[sl * kSkThreads + threadIdx.x];
    sl = sl + 1 == D ? 0 : sl + 1;
    sn = sn + 1 == D ? 0 : sn + 1;
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float2 b2[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      b2[t] = make_float2(__uint_as_float(wv[t] << 16), __uint_as_float(wv[t] & 0xffff0000u));
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      const float a = As[r][m];
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[m][t] = tc::fma2(a2, b2[t], acc[m][t]);
    }
  }
  cp_async_wait<0>();
  // The stream is read: the reduce may be scheduled (it waits for this
  // kernel to complete before reading the partials).
  pdl_launch_dependents();
  float *pt = P + (long long)blockIdx.y * M * job.Ntot + job.col0[mat] + n0;
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m >= M) break;
    float4 *dst = reinterpret_cast<float4 *>(pt + (long long)m * job.Ntot);
    dst[0] = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
    dst[1] = make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
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
  pdl_launch_dependents();
  pdl_wait();
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
  pdl_launch_dependents();
  pdl_wait();
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

// Slices of K: about three CTAs per SM of a 152-SM GB300 for up to four
// rows, two beyond (the 16-row kernel's registers allow fewer; the
// shared-memory ring of each CTA holds its copies in flight), at least
// eight rows and at
// most kSkMaxRowsPerSlice rows per slice, and
// fp32 partials (split * M * N * 4 bytes) of at most 16 MB, which stay in
// L2 between the two kernels.  The plan depends on the shape alone (not on
// the device that happens to be current), so a workspace sized for a shape
// always fits the launch of that shape.
constexpr int kSkPlanSms = 152;
constexpr long long kSkMaxPartialBytes = 16LL << 20;
static void skinny_plan(int M, int N, int K, int &split, int &rows) {
  const int colblocks = (N + kSkCtaCols - 1) / kSkCtaCols;
  const int per_sm = M <= 4 ? 3 : 2;
  int s = (per_sm * kSkPlanSms + colblocks - 1) / colblocks;
  s = s < kSkMaxSplit ? s : kSkMaxSplit;
  const long long per_slice = 4LL * (M > 0 ? M : 1) * N;
  const long long cap = kSkMaxPartialBytes / (per_slice > 0 ? per_slice : 1);
  s = s < cap ? s : (int)cap;
  const int rmin = (K + 7) / 8;  // slices of at least eight rows
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

template <int MB>
static cudaError_t launch_skinny_mb(dim3 grid, const __nv_bfloat16 *a, const SkinnyJob &job,
                                    float *partial, int M, int K, int rows, int early_b,
                                    cudaStream_t st) {
  const int smem = sk_depth<MB>() * kSkThreads * 16;
  cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<MB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_k(gemm_skinny_kernel<MB>, grid, dim3(kSkThreads), smem, st, true, a, job,
                  partial, M, K, rows, early_b);
}

cudaError_t launch_gemm_skinny_job(const void *A, const SkinnyJob &job, int M, int K,
                                   float *partial, cudaStream_t st, bool early_b) {
  int split = 1, rows = 1;
  skinny_plan(M, job.Ntot, K, split, rows);
  dim3 grid(job.blk0[job.count], split);
  const auto *a = reinterpret_cast<const __nv_bfloat16 *>(A);
  const int eb = early_b ? 1 : 0;
  if (M <= 1) return launch_skinny_mb<1>(grid, a, job, partial, M, K, rows, eb, st);
  if (M <= 2) return launch_skinny_mb<2>(grid, a, job, partial, M, K, rows, eb, st);
  if (M <= 4) return launch_skinny_mb<4>(grid, a, job, partial, M, K, rows, eb, st);
  if (M <= 8) return launch_skinny_mb<8>(grid, a, job, partial, M, K, rows, eb, st);
  return launch_skinny_mb<16>(grid, a, job, partial, M, K, rows, eb, st);
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
    return launch_k(skinny_reduce_few_kernel, dim3((unsigned)((groups + 255) / 256)), dim3(256),
                    0, st, true, partial, job, M, split);
  // one warp per group
  return launch_k(skinny_reduce_kernel, dim3((unsigned)((groups * 32 + 255) / 256)), dim3(256),
                  0, st, true, partial, job, M, split);
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
