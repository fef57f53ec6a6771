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
#include <cuda_fp16.h>

namespace ret {

__global__ void __launch_bounds__(256)
rotate_scale_kernel(KParams p, const void *__restrict__ x, long long s0, long long s1,
                    long long s2, int d, void *__restrict__ out, int out_bf16,
                    const float *__restrict__ scale, int mode) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int P = d / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)p.N * P) return;
  const int tau = (int)(idx / P), j = (int)(idx % P);
  const long long src = b * s0 + h * s1 + tau * s2 + 2 * j;
  float a = ld_elem(x, src, p.in_bf16), c2 = ld_elem(x, src + 1, p.in_bf16);
  if (p.rotate) {
    float cs, sn;
    rot_cs(p.pos0 + tau, p.th_hi[j], p.th_lo[j], cs, sn);
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
// bounds the scores and the state update downstream).
__global__ void __launch_bounds__(256)
rotate_chunk_f16_kernel(KParams p, const void *__restrict__ x, long long s0, long long s1,
                        long long s2, __half *__restrict__ out, int *__restrict__ exps,
                        float *__restrict__ maxs, int mode) {
  constexpr int kPer = 32;  // pairs per thread: 64 rows * 128 pairs / 256 threads
  __shared__ float wmax[8], wraw[8];
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int C = p.chunk, P = p.dk / 2, tid = threadIdx.x;
  const int t0 = c * C, L = min(C, p.N - t0);
  const int npairs = L * P;
  float2 v[kPer];
  float m = 0.f, mraw = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * 256;
    v[u] = make_float2(0.f, 0.f);
    if (e < npairs) {
      const int i = e / P, j = e % P;
      const long long src = b * s0 + h * s1 + (long long)(t0 + i) * s2 + 2 * j;
      float a0 = ld_elem(x, src, p.in_bf16), a1 = ld_elem(x, src + 1, p.in_bf16);
      if (p.rotate) {
        float cs, sn;
        rot_cs(p.pos0 + t0 + i, p.th_hi[j], p.th_lo[j], cs, sn);
        const float r0 = a0 * cs - a1 * sn, r1 = a0 * sn + a1 * cs;
        a0 = r0;
        a1 = r1;
      }
      mraw = fmaxf(mraw, fmaxf(fabsf(a0), fabsf(a1)));
      const float f = gpow(p.lng[h], mode == kScaleXi ? i + 1 : L - 1 - i);
      v[u] = make_float2(a0 * f, a1 * f);
      m = fmaxf(m, fmaxf(fabsf(v[u].x), fabsf(v[u].y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, o));
  }
  if ((tid & 31) == 0) {
    wmax[tid >> 5] = m;
    wraw[tid >> 5] = mraw;
  }
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
    if (e < npairs) o2[e] = __floats2half2_rn(v[u].x * sc, v[u].y * sc);
  }
  if (tid == 0) {
    const int nch = (p.N + C - 1) / C;
    exps[bh * nch + c] = ex;
    maxs[bh * nch + c] = mraw;
  }
}

cudaError_t launch_rotate_chunk_f16(const KParams &p, const void *x, const long long s[3],
                                    void *out, int *exps, float *maxs, int mode,
                                    cudaStream_t st) {
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  if (p.chunk * (p.dk / 2) > 256 * 32) return cudaErrorInvalidValue;
  dim3 grid((p.N + p.chunk - 1) / p.chunk, p.B * p.H);
  rotate_chunk_f16_kernel<<<grid, 256, 0, st>>>(p, x, s[0], s[1], s[2],
                                                reinterpret_cast<__half *>(out), exps, maxs,
                                                mode);
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
