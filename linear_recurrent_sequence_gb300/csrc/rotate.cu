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
