// Per-head GroupNorm (+ swish gate) epilogue for the CUDA-core forms.
// GroupNorm per (token, head) over d_v, biased variance, no affine
// (hwhale.com/article/285883: heads use different gamma, so their variances
// differ and each head is normalised on its own).  The gate is
// swish(g) = g sigmoid(g) (m0nads.wordpress.com, "Gated Multi-Scale
// Retention").  Input rows are F[row] * Oraw[row, :].
#include "common.cuh"
#include "launch.h"

namespace ret {

constexpr int kGnMaxPerLane = 32;  // d_v <= 1024

__global__ void __launch_bounds__(256)
groupnorm_kernel(KParams p, const float *__restrict__ Oraw, const float *__restrict__ F,
                 void *__restrict__ o, Gate gate) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.H * p.N;
  if (warp >= rows) return;
  const long long row = warp;  // row = (b*H + h)*N + n
  const int n = (int)(row % p.N);
  const int bh = (int)(row / p.N), b = bh / p.H, h = bh % p.H;
  const int dv = p.dv;
  const float f = F[row];
  float x[kGnMaxPerLane];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kGnMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    x[i] = (e < dv) ? f * Oraw[row * dv + e] : 0.f;
    sum += x[i];
  }
  float mu = 0.f, inv = 1.f;
  if (p.gn_eps >= 0.f) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    mu = sum / dv;
    float var = 0.f;
#pragma unroll
    for (int i = 0; i < kGnMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      const float d = (e < dv) ? x[i] - mu : 0.f;
      var = fmaf(d, d, var);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) var += __shfl_xor_sync(0xffffffffu, var, s);
    inv = rsqrtf(var / dv + p.gn_eps);
  }
  const long long obase = b * p.so[0] + h * p.so[1] + (long long)n * p.so[2];
  const long long gbase = b * gate.s[0] + h * gate.s[1] + (long long)n * gate.s[2];
#pragma unroll
  for (int i = 0; i < kGnMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    if (e >= dv) break;
    float y = (x[i] - mu) * inv;
    if (gate.ptr) {
      const float g = ld_elem(gate.ptr, gbase + e, 1);
      y *= g / (1.f + expf(-g));
    }
    st_elem(o, obase + e, y, p.out_bf16);
  }
}

cudaError_t launch_groupnorm(const KParams &p, const float *Oraw, const float *F, void *o,
                             Gate gate, cudaStream_t st) {
  const long long rows = (long long)p.B * p.H * p.N;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows * 32 + 255) / 256;
  groupnorm_kernel<<<(unsigned)blocks, 256, 0, st>>>(p, Oraw, F, o, gate);
  return cudaGetLastError();
}

}  // namespace ret
