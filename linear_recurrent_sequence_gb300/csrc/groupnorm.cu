// Per-head GroupNorm epilogue for the CUDA-core forms, and the MSR layer's
// swish gate as a separate pass.  GroupNorm per (token, head) over d_v,
// biased variance, no affine (hwhale.com/article/285883: heads use
// different gamma, so their variances differ and each head is normalised on
// its own); input rows are F[row] * Oraw[row, :].  The gate is
// swish(g) = g sigmoid(g) (m0nads.wordpress.com, "Gated Multi-Scale
// Retention").
#include "common.cuh"
#include "launch.h"

namespace ret {

constexpr int kGnMaxPerLane = 32;  // d_v <= 1024

__global__ void __launch_bounds__(256)
groupnorm_kernel(KParams p, const float *__restrict__ Oraw, const float *__restrict__ F,
                 void *__restrict__ o) {
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
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
#pragma unroll
  for (int i = 0; i < kGnMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    if (e >= dv) break;
    st_elem(o, obase + e, (x[i] - mu) * inv, p.out_bf16);
  }
}

cudaError_t launch_groupnorm(const KParams &p, const float *Oraw, const float *F, void *o,
                             cudaStream_t st) {
  const long long rows = (long long)p.B * p.H * p.N;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows * 32 + 255) / 256;
  return launch_k(groupnorm_kernel, dim3((unsigned)blocks), dim3(256), 0, st, true, p, Oraw, F, o);
}

// The MSR layer's gate on the retention output, y <- y * swish(g), bf16
// in and out, fp32 arithmetic (fast exponential and divide: a few ulp before
// the bf16 rounding).  Eight values per thread when both pointers are
// 16-byte aligned; a scalar pass covers the rest.
__global__ void __launch_bounds__(256)
swish_gate_kernel(__nv_bfloat16 *__restrict__ y, const __nv_bfloat16 *__restrict__ g,
                  long long n, int vec) {
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
  const long long nv = vec ? n / 8 : 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    uint4 yu = reinterpret_cast<const uint4 *>(y)[i];
    const uint4 gu = reinterpret_cast<const uint4 *>(g)[i];
    uint32_t *yw = reinterpret_cast<uint32_t *>(&yu);
    const uint32_t *gw = reinterpret_cast<const uint32_t *>(&gu);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 yv = *reinterpret_cast<const __nv_bfloat162 *>(&yw[e]);
      const __nv_bfloat162 gv = *reinterpret_cast<const __nv_bfloat162 *>(&gw[e]);
      const float g0 = __low2float(gv), g1 = __high2float(gv);
      const float a = __low2float(yv) * __fdividef(g0, 1.f + __expf(-g0));
      const float c = __high2float(yv) * __fdividef(g1, 1.f + __expf(-g1));
      yv = __floats2bfloat162_rn(a, c);
      yw[e] = *reinterpret_cast<const uint32_t *>(&yv);
    }
    reinterpret_cast<uint4 *>(y)[i] = yu;
  }
  for (long long i = nv * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float gi = __bfloat162float(g[i]);
    y[i] = __float2bfloat16_rn(__bfloat162float(y[i]) * __fdividef(gi, 1.f + __expf(-gi)));
  }
}

cudaError_t launch_swish_gate(void *y, const void *g, long long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int vec = (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(g) % 16 == 0);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  const long long work = vec ? (n + 7) / 8 : n;
  long long blocks = (work + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  return launch_k(swish_gate_kernel, dim3((unsigned)blocks), dim3(256), 0, st, true,
                  reinterpret_cast<__nv_bfloat16 *>(y), reinterpret_cast<const __nv_bfloat16 *>(g),
                  n, vec);
}

}  // namespace ret
