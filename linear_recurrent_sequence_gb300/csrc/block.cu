// The element-wise and row-wise steps of the RetNet block around the MSR
// layer and the FFN's two GEMMs (m0nads.wordpress.com "A dubious successor
// to Transformer", section "Overall architecture": a LayerNorm before MSR
// and before the FFN, a skip connection around each):
//   LayerNorm over d_model, biased variance, fp32 gain and bias;
//   the skip connection y <- y + r;
//   GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2 on the FFN's hidden
//   activations (the pages name the FFN but not its activation; GELU is the
//   reading taken).
// bf16 in and out, fp32 arithmetic.
#include "common.cuh"
#include "launch.h"

namespace ret {

namespace {
constexpr int kLnThreads = 256;

__device__ __forceinline__ float block_sum(float x, float *red) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] of an earlier call has been read
  if (lane == 0) red[w] = x;
  __syncthreads();
  float t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) t += __shfl_xor_sync(0xffffffffu, t, s);
  return t;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return sms;
}
}  // namespace

// One CTA per row of d values: the row is kept in shared memory (fp32), the
// mean and then the variance of the deviations are block sums.
__global__ void __launch_bounds__(kLnThreads)
layernorm_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ w,
                 const float *__restrict__ b, __nv_bfloat16 *__restrict__ y, int d, float eps) {
  extern __shared__ float row[];
  __shared__ float red[kLnThreads / 32];
  pdl_launch_dependents();
  pdl_wait();
  const long long base = (long long)blockIdx.x * d;
  float s = 0.f;
  for (int i = threadIdx.x; i < d; i += kLnThreads) {
    const float v = __bfloat162float(x[base + i]);
    row[i] = v;
    s += v;
  }
  const float mu = block_sum(s, red) / d;
  float q = 0.f;
  for (int i = threadIdx.x; i < d; i += kLnThreads) {
    const float dv = row[i] - mu;
    q = fmaf(dv, dv, q);
  }
  const float inv = rsqrtf(block_sum(q, red) / d + eps);
  for (int i = threadIdx.x; i < d; i += kLnThreads)
    y[base + i] = __float2bfloat16_rn(fmaf((row[i] - mu) * inv, w[i], b[i]));
}

// kOp 0: y <- y + r (skip connection); kOp 1: y <- gelu(y) (r unused).
// Eight values per thread where the pointers are 16-byte aligned, then a
// scalar pass over the rest.
template <int kOp>
__device__ __forceinline__ float elem_op(float yv, float rv) {
  if (kOp == 0) return yv + rv;
  return 0.5f * yv * (1.f + erff(yv * 0.70710678118654752f));
}

template <int kOp>
__global__ void __launch_bounds__(256)
elementwise_kernel(__nv_bfloat16 *__restrict__ y, const __nv_bfloat16 *__restrict__ r,
                   long long n, int vec) {
  pdl_launch_dependents();
  pdl_wait();
  const long long nv = vec ? n / 8 : 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    uint4 yu = reinterpret_cast<const uint4 *>(y)[i];
    uint4 ru = make_uint4(0u, 0u, 0u, 0u);
    if (kOp == 0) ru = reinterpret_cast<const uint4 *>(r)[i];
    uint32_t *yw = reinterpret_cast<uint32_t *>(&yu);
    const uint32_t *rw = reinterpret_cast<const uint32_t *>(&ru);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 yv = *reinterpret_cast<const __nv_bfloat162 *>(&yw[e]);
      const __nv_bfloat162 rv = *reinterpret_cast<const __nv_bfloat162 *>(&rw[e]);
      yv = __floats2bfloat162_rn(elem_op<kOp>(__low2float(yv), __low2float(rv)),
                                 elem_op<kOp>(__high2float(yv), __high2float(rv)));
      yw[e] = *reinterpret_cast<const uint32_t *>(&yv);
    }
    reinterpret_cast<uint4 *>(y)[i] = yu;
  }
  for (long long i = nv * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float rv = kOp == 0 ? __bfloat162float(r[i]) : 0.f;
    y[i] = __float2bfloat16_rn(elem_op<kOp>(__bfloat162float(y[i]), rv));
  }
}

cudaError_t launch_layernorm(const void *x, const float *w, const float *b, void *y, long long rows,
                             int d, float eps, cudaStream_t st, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)d;
  cudaError_t e = cudaFuncSetAttribute(layernorm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(layernorm_kernel, dim3((unsigned)rows), dim3(kLnThreads), smem, st, pdl,
                  reinterpret_cast<const __nv_bfloat16 *>(x), w, b,
                  reinterpret_cast<__nv_bfloat16 *>(y), d, eps);
}

static cudaError_t launch_elementwise(int op, void *y, const void *r, long long n,
                                      cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int vec = (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                  (op != 0 || reinterpret_cast<uintptr_t>(r) % 16 == 0);
  const long long work = vec ? (n + 7) / 8 : n;
  long long blocks = (work + 255) / 256;
  const long long cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  auto *yp = reinterpret_cast<__nv_bfloat16 *>(y);
  auto *rp = reinterpret_cast<const __nv_bfloat16 *>(r);
  return launch_k(op == 0 ? elementwise_kernel<0> : elementwise_kernel<1>,
                  dim3((unsigned)blocks), dim3(256), 0, st, true, yp, rp, n, vec);
}

cudaError_t launch_residual_add(void *y, const void *r, long long n, cudaStream_t st) {
  return launch_elementwise(0, y, r, n, st);
}

cudaError_t launch_gelu(void *y, long long n, cudaStream_t st) {
  return launch_elementwise(1, y, nullptr, n, st);
}

}  // namespace ret
