// Rotate-and-scale prologue: Q = (X W_Q) (.) Theta, K = (X W_K) (.) conj(Theta)
// (hwhale.com/article/285883, equation of Q, K, V and Theta_n = e^{i n theta};
// m0nads.wordpress.com "A dubious successor to Transformer", xPos rotation).
// Pair j of a row is read as x_2j + i x_2j+1 and multiplied by e^{i t theta_j};
// the key's conjugate is taken by the real dot product downstream.
//
// Optionally each row is also multiplied by a decay that depends on its
// position inside its chunk, which lets the tensor-core chunk kernel fold the
// chunkwise form's xi and zeta factors into its operands:
//   kScaleXi:   row i of a chunk  * gamma^(i+1)        (queries)
//   kScaleZeta: row j of a chunk  * gamma^(L-1-j)      (keys; L = chunk length)
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"
#include <cuda_fp16.h>
#include <string.h>

namespace ret {

__global__ void __launch_bounds__(256)
rotate_scale_kernel(KParams p, const void *__restrict__ x, long long s0, long long s1,
                    long long s2, int d, void *__restrict__ out, int out_bf16,
                    const float *__restrict__ scale, int mode) {
  __shared__ float th[2][kMaxPairs];  // per-pair frequencies (indexed per thread)
  const int b = blockIdx.z, h = blockIdx.y;
  const int P = d / 2;
  for (int t = threadIdx.x; t < P; t += blockDim.x) {
    th[0][t] = p.th_hi[t];
    th[1][t] = p.th_lo[t];
  }
  __syncthreads();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)p.N * P) return;
  const int tau = (int)(idx / P), j = (int)(idx % P);
  const long long src = b * s0 + h * s1 + tau * s2 + 2 * j;
  float a = ld_elem(x, src, p.in_bf16), c2 = ld_elem(x, src + 1, p.in_bf16);
  if (p.rotate) {
    float cs, sn;
    rot_cs(p.pos0 + tau, th[0][j], th[1][j], cs, sn);
    const float ra = a * cs - c2 * sn;
    const float rb = a * sn + c2 * cs;
    a = ra;
    c2 = rb;
  }
  float f = 1.f;
  if (mode == kScaleArray) {
    f = scale[tau];
  } else if (mode == kScaleXi || mode == kScaleZeta) {
    const int i = tau % p.chunk;
    const int L = min(p.chunk, p.N - (tau - i));
    f = gpow(p.lng[h], mode == kScaleXi ? i + 1 : L - 1 - i);
  }
  const long long dst = (((long long)b * p.H + h) * p.N + tau) * d + 2 * j;
  st_elem(out, dst, a * f, out_bf16);
  st_elem(out, dst + 1, c2 * f, out_bf16);
}

// fp16 operand prologue of the tensor-core chunk kernel: one CTA per
// (batch*head, chunk).  Each chunk's rows are rotated and scaled by xi
// (queries) or zeta (keys) in fp32, then written as fp16 times a power of
// two 2^-e chosen from the chunk's largest scaled magnitude m
// (m 2^-e < 2^14), so no value can overflow and every value keeps fp16's
// 11-bit precision.  e goes to exps[bh*nch + c]; the largest magnitude of
// the rotated rows BEFORE the decay factor goes to maxs[bh*nch + c] (it
// bounds the scores and the state update downstream).  For keys, the
// column sums of the scaled rows (sum_j zeta_j rot(k_j), fp32) go to
// colsum[(bh*nch + c)*dk + col]: the chunk's contribution to z.
//
// Angles: a thread keeps one pair column j and walks rows i0, i0+s, ...;
// e^{i t theta_j} is advanced by the rotation e^{i s theta_j} and re-anchored
// with the accurate reduction every 8 rows, so the angle error stays near
// 1e-6 rad while most rows cost four FMAs instead of a sine and cosine.
template <bool kTma>
__global__ void __launch_bounds__(256)
rotate_chunk_f16_kernel(KParams p, const void *__restrict__ x, long long s0, long long s1,
                        long long s2, const __grid_constant__ CUtensorMap tmx,
                        __half *__restrict__ out, int *__restrict__ exps,
                        float *__restrict__ maxs, float *__restrict__ colsum, int mode) {
  // kTma: the chunk's rows arrive in shared memory by one TMA copy (row-major
  // [C][dk] bf16); otherwise each thread loads its pairs from global memory.
  extern __shared__ __align__(128) uint8_t xtile[];
  __shared__ __align__(8) uint64_t tbar;
  constexpr int kPer = 32;  // pairs per thread: 64 rows * 128 pairs / 256 threads
  __shared__ float wmax[8], wraw[8];
  __shared__ float th[2][kMaxPairs];  // per-pair frequencies (indexed per thread)
  __shared__ float2 csum[256];
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int C = p.chunk, P = p.dk / 2, tid = threadIdx.x;
  if (tid < P) {
    th[0][tid] = p.th_hi[tid];
    th[1][tid] = p.th_lo[tid];
  }
  if (kTma && tid == 0) {
    tc::mbar_init(&tbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (kTma) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(&tbar, (uint32_t)(C * p.dk * 2));
      tc::tma_load_4d(xtile, &tmx, &tbar, 0, c * C, h, b);
    }
    // Bounded wait; if it ever ran out, wait (bounded) again for the copy
    // to land before reading or leaving.
    if (!tc::mbar_wait(&tbar, 0, p.status, 1u << 24)) tc::mbar_wait(&tbar, 0, nullptr, 1u << 24);
  }
  const int t0 = c * C, L = min(C, p.N - t0);
  // Pair (i, j) of element e = tid + 256 u; when P divides 256 the thread
  // keeps column jp and walks rows ip + u*istep.
  const bool walk = (256 % P) == 0;
  const int jp = tid % P, ip = tid / P, istep = 256 / P;
  const int U = walk ? (C + istep - 1) / istep : kPer;
  const bool pair_ld = p.in_bf16 && ((reinterpret_cast<uintptr_t>(x) & 3) == 0) &&
                       !(s0 & 1) && !(s1 & 1) && !(s2 & 1);
  float2 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    v[u] = make_float2(0.f, 0.f);
    const int e = tid + u * 256;
    const int i = walk ? ip + u * istep : e / P, j = walk ? jp : e % P;
    if (u < U && i < L && (walk || e < L * P)) {
      const long long src = b * s0 + h * s1 + (long long)(t0 + i) * s2 + 2 * j;
      if (kTma) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(xtile + ((size_t)i * p.dk + 2 * j) * 2);
        v[u] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
      } else if (pair_ld) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(
            reinterpret_cast<const __nv_bfloat16 *>(x) + src));
        v[u] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
      } else {
        v[u] = make_float2(ld_elem(x, src, p.in_bf16), ld_elem(x, src + 1, p.in_bf16));
      }
    }
  }
  const float lng = p.lng[h];
  float m = 0.f, mraw = 0.f;
  float2 cs_acc = make_float2(0.f, 0.f);
  // Angle and decay recurrences (walk mode).
  float cs = 1.f, sn = 0.f, dcs = 1.f, dsn = 0.f;
  if (walk && p.rotate) rot_cs(istep, th[0][jp], th[1][jp], dcs, dsn);
  const float dstep = gpow(lng, istep);
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * 256;
    const int i = walk ? ip + u * istep : e / P, j = walk ? jp : e % P;
    if (u < U && i < L && (walk || e < L * P)) {
      float a0 = v[u].x, a1 = v[u].y;
      if (p.rotate) {
        if (!walk || (u & 7) == 0) {
          rot_cs(p.pos0 + t0 + i, th[0][j], th[1][j], cs, sn);
        } else {
          const float nc = cs * dcs - sn * dsn, ns = sn * dcs + cs * dsn;
          cs = nc;
          sn = ns;
        }
        const float r0 = a0 * cs - a1 * sn, r1 = a0 * sn + a1 * cs;
        a0 = r0;
        a1 = r1;
      }
      mraw = fmaxf(mraw, fmaxf(fabsf(a0), fabsf(a1)));
      const float f = gpow(lng, mode == kScaleXi ? i + 1 : L - 1 - i);
      v[u] = make_float2(a0 * f, a1 * f);
      m = fmaxf(m, fmaxf(fabsf(v[u].x), fabsf(v[u].y)));
      cs_acc.x += v[u].x;
      cs_acc.y += v[u].y;
    }
  }
  (void)dstep;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, o));
  }
  if ((tid & 31) == 0) {
    wmax[tid >> 5] = m;
    wraw[tid >> 5] = mraw;
  }
  if (colsum && walk) csum[tid] = cs_acc;
  __syncthreads();
  m = wmax[0];
  mraw = wraw[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) {
    m = fmaxf(m, wmax[w]);
    mraw = fmaxf(mraw, wraw[w]);
  }
  int ex = 0;
  if (m > 0.f && m < INFINITY) {
    frexpf(m, &ex);
    ex -= 14;
  }
  const float sc = exp2f((float)-ex);
  __half2 *o2 = reinterpret_cast<__half2 *>(out + ((long long)bh * p.N + t0) * p.dk);
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * 256;
    const int i = walk ? ip + u * istep : e / P, j = walk ? jp : e % P;
    if (u < U && i < L && (walk || e < L * P))
      o2[i * P + j] = __floats2half2_rn(v[u].x * sc, v[u].y * sc);
  }
  const int nch = (p.N + C - 1) / C;
  if (colsum) {
    float *cdst = colsum + ((long long)bh * nch + c) * p.dk;
    if (walk) {
      if (tid < P) {
        float2 acc = csum[tid];
        for (int r = 1; r < istep; ++r) {
          acc.x += csum[tid + r * P].x;
          acc.y += csum[tid + r * P].y;
        }
        cdst[2 * tid] = acc.x;
        cdst[2 * tid + 1] = acc.y;
      }
    } else {
      // General pair count: sum the columns from the fp32 values via shared
      // memory atomics (this path is only taken for d_k = 192).
      __shared__ float cacc[2 * kMaxPairs];
      for (int t = tid; t < p.dk; t += 256) cacc[t] = 0.f;
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = tid + u * 256;
        if (e < L * P) {
          atomicAdd(&cacc[2 * (e % P)], v[u].x);
          atomicAdd(&cacc[2 * (e % P) + 1], v[u].y);
        }
      }
      __syncthreads();
      for (int t = tid; t < p.dk; t += 256) cdst[t] = cacc[t];
    }
  }
  if (tid == 0) {
    exps[bh * nch + c] = ex;
    maxs[bh * nch + c] = mraw;
  }
}

cudaError_t launch_rotate_chunk_f16(const KParams &p, const void *x, const long long s[3],
                                    void *out, int *exps, float *maxs, float *colsum, int mode,
                                    cudaStream_t st) {
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  if (p.chunk * (p.dk / 2) > 256 * 32) return cudaErrorInvalidValue;
  dim3 grid((p.N + p.chunk - 1) / p.chunk, p.B * p.H);
  // TMA source when the rows are 16-byte aligned bf16 with 16-byte strides.
  CUtensorMap tm;
  memset(&tm, 0, sizeof(tm));
  bool tma = p.in_bf16 && (reinterpret_cast<uintptr_t>(x) % 16 == 0) && s[0] % 8 == 0 &&
             s[1] % 8 == 0 && s[2] % 8 == 0 && p.dk <= 256 && p.chunk <= 256;
  if (tma) {
    const cuuint64_t dims[4] = {(cuuint64_t)p.dk, (cuuint64_t)p.N, (cuuint64_t)p.H,
                                (cuuint64_t)p.B};
    const cuuint64_t strides[3] = {(cuuint64_t)s[2] * 2, (cuuint64_t)s[1] * 2,
                                   (cuuint64_t)s[0] * 2};
    const cuuint32_t box[4] = {(cuuint32_t)p.dk, (cuuint32_t)p.chunk, 1, 1};
    tma = tmap_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (tma) {
    const size_t smem = (size_t)p.chunk * p.dk * 2;
    cudaError_t e = cudaFuncSetAttribute(rotate_chunk_f16_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    rotate_chunk_f16_kernel<true><<<grid, 256, smem, st>>>(
        p, x, s[0], s[1], s[2], tm, reinterpret_cast<__half *>(out), exps, maxs, colsum, mode);
  } else {
    rotate_chunk_f16_kernel<false><<<grid, 256, 0, st>>>(
        p, x, s[0], s[1], s[2], tm, reinterpret_cast<__half *>(out), exps, maxs, colsum, mode);
  }
  return cudaGetLastError();
}

cudaError_t launch_rotate(const KParams &p, const void *x, const long long s[3], int d,
                          void *out, int out_bf16, const float *scale, int mode,
                          cudaStream_t st) {
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  const long long pairs = (long long)p.N * (d / 2);
  dim3 grid((unsigned)((pairs + 255) / 256), p.H, p.B);
  rotate_scale_kernel<<<grid, 256, 0, st>>>(p, x, s[0], s[1], s[2], d, out, out_bf16,
                                            scale, mode);
  return cudaGetLastError();
}

}  // namespace ret
