// Operand preparation for the tensor-core backward of chunkwise retention.
//
// The backward is assembled from runs of the forward tensor-core kernel
// (the recurrence is linear, and its adjoint is the same recurrence run in
// reversed time; hwhale.com/article/285883, recurrent form
// S_n = gamma S_{n-1} + K_n^T V_n, O_n = Q_n S_n).  With s_t the row factor
// of the first two normalisations (O_t = s_t q'_t S_t):
//   U_t = dL/dS_t = gamma U_{t+1} + s_t q'_t^T dO_t,   U_{N-1} = dS_out + s q'^T dO,
//   dv_t = k'_t U_t,   dk'_t = v_t U_t^T,   dq'_t = s_t dO_t S_t^T,   dS_in = gamma U_0,
// so
//   - dv is the forward on (k', s q', dO) in reversed time from the entry
//     state dS_out/gamma (the forward decays its entry state once more
//     than its last token);
//   - dq' / s is the forward on (dO, v, k') from S_in^T;
//   - dk' is the forward on (v, dO, s q') in reversed time from
//     (dS_out/gamma)^T;
// and the last two have d_v as their score dimension, which is split into
// pieces of at most 256 (the forward's widest), the results being linear in
// the scores.  The kernels here write the operands those runs read (bf16,
// contiguous [B*H][N][d], rotated, scaled, reversed in time), transpose the
// entry states, and fold the runs' fp32 results back into the caller's
// gradients.  Both streaming kernels move 8 elements (16 bytes of bf16) per
// thread and row.
#include "ktimer.h"
#include "launch.h"

namespace ret {

constexpr int kBwdThreads = 256;
constexpr int kBwdVec = 8;  // elements per thread

// Loads 8 consecutive elements (bf16 or fp32) at x[off]; vec: the address
// allows one 16-byte (bf16) or two 16-byte (fp32) loads.
__device__ __forceinline__ void ld8(const void *x, long long off, int bf16, int vec, float *f) {
  if (bf16) {
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(x) + off;
    if (vec) {
      const uint4 u = *reinterpret_cast<const uint4 *>(b);
      const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __bfloat162float(b[i]);
    }
  } else {
    const float *s = reinterpret_cast<const float *>(x) + off;
    if (vec) {
      const float4 a = *reinterpret_cast<const float4 *>(s);
      const float4 c = *reinterpret_cast<const float4 *>(s + 4);
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
      f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = s[i];
    }
  }
}

__device__ __forceinline__ uint4 pack8(const float *f) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// The rotation frequencies (hi and lo parts) staged in shared memory: read
// from the parameters with a lane-dependent index, they would be served one
// address at a time.
struct ThetaSmem {
  float hi[kMaxPairs], lo[kMaxPairs];
};

__device__ __forceinline__ void stage_theta(const KParams &p, int pairs, ThetaSmem &th) {
  for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
    th.hi[j] = p.th_hi[j];
    th.lo[j] = p.th_lo[j];
  }
  __syncthreads();
}

// cos and sin of t theta for operands that are rounded to bf16 afterwards:
// the reduced angle, then the hardware approximation, whose absolute error
// (about 2^-21) is far below bf16's 2^-9.
__device__ __forceinline__ void rot_cs_bf16(long long t, float th_hi, float th_lo, float &c,
                                            float &s) {
  __sincosf(rot_angle(t, th_hi, th_lo), &s, &c);
}

// Rotates the 4 pairs starting at pair j0 by +t theta (dir = 1) or back by
// -t theta (dir = -1).
__device__ __forceinline__ void rotate8(const ThetaSmem &th, long long t, int j0, float dir,
                                        float *f) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float cs, sn;
    rot_cs_bf16(t, th.hi[j0 + i], th.lo[j0 + i], cs, sn);
    sn *= dir;
    const float a = f[2 * i], c = f[2 * i + 1];
    f[2 * i] = a * cs - c * sn;
    f[2 * i + 1] = a * sn + c * cs;
  }
}

// One CTA covers kBwdRowsPer * kBwdThreads * 8 / d rows of one (b, h) for
// job blockIdx.z (each thread loads its rows before it works on them, for
// more bytes in flight): row t of the source is read once and written to
// fwd[bh][t] and/or rev[bh][N-1-t].
constexpr int kBwdRowsPer = 2;

__global__ void __launch_bounds__(kBwdThreads)
bwd_prep_kernel(const __grid_constant__ KParams p, const __grid_constant__ BwdPrepJobs jobs) {
  __shared__ ThetaSmem th;
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
  const BwdPrepJob &J = jobs.job[blockIdx.z];
  const int per_row = J.d / kBwdVec, rows = kBwdThreads / per_row;
  const int t0 = blockIdx.x * rows * kBwdRowsPer;
  if (t0 >= p.N) return;
  if (J.rotate) stage_theta(p, J.d / 2, th);
  if (threadIdx.x >= rows * per_row) return;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int c0 = (threadIdx.x % per_row) * kBwdVec;
  const int r0 = t0 + threadIdx.x / per_row;
  float f[kBwdRowsPer][kBwdVec];
#pragma unroll
  for (int i = 0; i < kBwdRowsPer; ++i) {
    const int t = r0 + i * rows;
    if (t < p.N)
      ld8(J.src, b * J.s[0] + h * J.s[1] + (long long)t * J.s[2] + c0, J.bf16, J.vec, f[i]);
  }
  const long long base = (long long)bh * p.N;
#pragma unroll
  for (int i = 0; i < kBwdRowsPer; ++i) {
    const int t = r0 + i * rows;
    if (t >= p.N) break;
    if (J.rotate) rotate8(th, p.pos0 + t, c0 / 2, 1.f, f[i]);
    if (J.rowscale) {
      const float s = row_scale(p, h, p.pos0 + t + 1);
#pragma unroll
      for (int e = 0; e < kBwdVec; ++e) f[i][e] *= s;
    }
    const uint4 u = pack8(f[i]);
    if (J.fwd) *reinterpret_cast<uint4 *>(J.fwd + (base + t) * J.d + c0) = u;
    if (J.rev) *reinterpret_cast<uint4 *>(J.rev + (base + p.N - 1 - t) * J.d + c0) = u;
  }
}

// T_j[bh][e][a] = S[bh][a][j*w + e] for the column blocks j of width w:
// the entry state seen by the runs whose score dimension is d_v.
__global__ void __launch_bounds__(256)
bwd_transpose_kernel(const float *__restrict__ S, int BH, int dk, int dv, int w,
                     float *__restrict__ T) {
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
  const long long n = (long long)BH * dk * dv;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int a = (int)(i % dk);
    const long long rest = i / dk;
    const int e = (int)(rest % dv), bh = (int)(rest / dv);
    const int j = e / w, ej = e % w;
    T[(((long long)j * BH + bh) * w + ej) * dk + a] = S[((long long)bh * dk + a) * dv + e];
  }
}

// out[b,h,t,:] (caller's strides and dtype) = the sum of the fp32 inputs
// [B*H][N][d] at row (reverse ? N-1-t : t), times s_t when rowscale is set,
// turned back by -t theta when unrotate is set (the transpose of the
// rotation).
__global__ void __launch_bounds__(kBwdThreads)
bwd_finish_kernel(const __grid_constant__ KParams p, const __grid_constant__ BwdFinish F) {
  __shared__ ThetaSmem th;
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
  if (F.unrotate) stage_theta(p, F.d / 2, th);
  const int per_row = F.d / kBwdVec, rows = kBwdThreads / per_row;
  const int t = blockIdx.x * rows + threadIdx.x / per_row;
  if (t >= p.N || threadIdx.x >= rows * per_row) return;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int c0 = (threadIdx.x % per_row) * kBwdVec;
  const int r = F.reverse ? p.N - 1 - t : t;
  const long long src = ((long long)bh * p.N + r) * F.d + c0;
  float f[kBwdVec] = {};
#pragma unroll
  for (int i = 0; i < kBwdFinishMax; ++i) {
    if (i < F.n_in) {
      float g[kBwdVec];
      ld8(F.x[i], src, 0, 1, g);
#pragma unroll
      for (int e = 0; e < kBwdVec; ++e) f[e] += g[e];
    }
  }
  if (F.rowscale) {
    const float s = row_scale(p, h, p.pos0 + t + 1);
#pragma unroll
    for (int e = 0; e < kBwdVec; ++e) f[e] *= s;
  }
  if (F.unrotate) rotate8(th, p.pos0 + t, c0 / 2, -1.f, f);
  const long long dst = b * F.s[0] + h * F.s[1] + (long long)t * F.s[2] + c0;
  if (F.out_bf16 && F.vec) {
    *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(F.out) + dst) = pack8(f);
  } else {
#pragma unroll
    for (int e = 0; e < kBwdVec; ++e) st_elem(F.out, dst + e, f[e], F.out_bf16);
  }
}

static bool aligned16(const void *x, const long long s[3], int elem) {
  if (reinterpret_cast<uintptr_t>(x) & 15) return false;
  for (int i = 0; i < 3; ++i)
    if ((s[i] * elem) % 16) return false;
  return true;
}

cudaError_t launch_bwd_prep(const KParams &p, BwdPrepJobs jobs, cudaStream_t st) {
  if (p.N == 0 || p.B == 0 || p.H == 0 || jobs.count == 0) return cudaSuccess;
  if (jobs.count > kBwdPrepMax) return cudaErrorInvalidValue;
  int gx = 0;
  for (int i = 0; i < jobs.count; ++i) {
    BwdPrepJob &J = jobs.job[i];
    if (J.d % kBwdVec || J.d > kBwdThreads * kBwdVec) return cudaErrorInvalidValue;
    if (J.rotate && J.d / 2 > kMaxPairs) return cudaErrorInvalidValue;
    if ((J.fwd && (reinterpret_cast<uintptr_t>(J.fwd) & 15)) ||
        (J.rev && (reinterpret_cast<uintptr_t>(J.rev) & 15)))
      return cudaErrorInvalidValue;
    J.vec = aligned16(J.src, J.s, J.bf16 ? 2 : 4);
    const int rows = kBwdRowsPer * (kBwdThreads / (J.d / kBwdVec));
    const int x = (p.N + rows - 1) / rows;
    gx = x > gx ? x : gx;
  }
  dim3 grid((unsigned)gx, (unsigned)(p.B * p.H), (unsigned)jobs.count);
  return launch_k(bwd_prep_kernel, grid, dim3(kBwdThreads), 0, st, true, p, jobs);
}

cudaError_t launch_bwd_transpose(const float *S, int BH, int dk, int dv, int w, float *T,
                                 cudaStream_t st) {
  const long long n = (long long)BH * dk * dv;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_k(bwd_transpose_kernel, dim3((unsigned)blocks), dim3(256), 0, st, true, S, BH, dk,
                  dv, w, T);
}

cudaError_t launch_bwd_finish(const KParams &p, BwdFinish F, cudaStream_t st) {
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  if (F.n_in < 1 || F.n_in > kBwdFinishMax) return cudaErrorInvalidValue;
  if (F.d % kBwdVec || F.d > kBwdThreads * kBwdVec) return cudaErrorInvalidValue;
  if (F.unrotate && F.d / 2 > kMaxPairs) return cudaErrorInvalidValue;
  for (int i = 0; i < F.n_in; ++i)
    if (reinterpret_cast<uintptr_t>(F.x[i]) & 15) return cudaErrorInvalidValue;
  F.vec = aligned16(F.out, F.s, F.out_bf16 ? 2 : 4);
  const int rows = kBwdThreads / (F.d / kBwdVec);
  dim3 grid((unsigned)((p.N + rows - 1) / rows), (unsigned)(p.B * p.H));
  return launch_k(bwd_finish_kernel, grid, dim3(kBwdThreads), 0, st, true, p, F);
}

}  // namespace ret
