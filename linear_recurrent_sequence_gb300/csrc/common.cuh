// Shared device-side definitions of the retention library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/retention.h"

namespace ret {

constexpr int kMaxPairs = 128;  // d_k <= 256

// Status word codes written by kernels into the workspace (first 256 bytes).
enum : unsigned { kDevOk = 0u, kDevTimeout = 1u, kDevBounds = 2u };
constexpr size_t kStatusBytes = 256;

// Everything a kernel needs to know about one retention call.  Per-head
// constants and the rotation frequencies are computed on the host in
// float64 and rounded once.
struct KParams {
  int B, H, N, dk, dv, chunk;
  long long sq[3], sk[3], sv[3], so[3];
  long long pos0;
  int norm_flags, rotate, in_bf16, out_bf16;
  float gn_eps, inv_sqrt_dk;
  float gam[RET_MAX_HEADS];  // gamma_h
  float lng[RET_MAX_HEADS];  // ln(gamma_h); -inf for gamma_h = 0
  float omg[RET_MAX_HEADS];  // 1 - gamma_h
  float th_hi[kMaxPairs];    // theta_j rounded to float
  float th_lo[kMaxPairs];    // theta_j - th_hi[j]
  unsigned *status;          // device status word (workspace start)
  unsigned report_budget;    // tries of a reporting wait (see retention.h)
};

// ---------------------------------------------------------------- numbers
__device__ __forceinline__ float gpow(float lng, int k) {
  // gamma^k for integer k >= 0 (gamma = 0 gives 0^0 = 1, 0^k = 0).
  return k == 0 ? 1.f : expf((float)k * lng);
}

// sum_{i=1}^{n} gamma^(n-i) = (1 - gamma^n)/(1 - gamma), n for gamma = 1.
__device__ __forceinline__ float decay_row_sum(float lng, float omg, long long n) {
  if (omg == 0.f) return (float)n;
  return -expm1f((float)n * lng) / omg;
}

// Product of the first two normalisations for 1-based position n.
__device__ __forceinline__ float row_scale(const KParams &p, int h, long long n) {
  float s = 1.f;
  if (p.norm_flags & RET_NORM_SCALE) s *= p.inv_sqrt_dk;
  if (p.norm_flags & RET_NORM_DROW) s *= rsqrtf(decay_row_sum(p.lng[h], p.omg[h], n));
  return s;
}

__device__ __forceinline__ float rsum_scale(const KParams &p, float rowsum) {
  return (p.norm_flags & RET_NORM_RSUM) ? 1.f / fmaxf(fabsf(rowsum), 1.f) : 1.f;
}

// t * theta_j reduced to [-pi, pi].  The product is kept as a float pair and
// reduced modulo 2 pi with a two-part 2 pi (Cody-Waite), so the angle error
// stays near 1e-6 rad for every position below 2^24.
__device__ __forceinline__ float rot_angle(long long t, float th_hi, float th_lo) {
  const float tf = (float)t;
  const float p_hi = tf * th_hi;
  const float p_lo = fmaf(tf, th_hi, -p_hi) + tf * th_lo;
  const float k = rintf(p_hi * 0.159154943091895336f);
  float r = fmaf(-k, 6.28318548202514648f, p_hi);
  r = fmaf(-k, -1.74845553146951725e-07f, r);
  return r + p_lo;
}

// cos/sin of t * theta_j.
__device__ __forceinline__ void rot_cs(long long t, float th_hi, float th_lo,
                                       float &c, float &s) {
  sincosf(rot_angle(t, th_hi, th_lo), &s, &c);
}

// ---------------------------------------------------------------- memory
__device__ __forceinline__ float ld_elem(const void *p, long long i, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  return reinterpret_cast<const float *>(p)[i];
}

__device__ __forceinline__ void st_elem(void *p, long long i, float x, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float *>(p)[i] = x;
}

__device__ __forceinline__ void report(unsigned *status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream still
// runs: pdl_wait() blocks until every kernel it depends on has completed and
// their memory operations are visible, so each such kernel calls it before
// its first access to global memory that an earlier kernel may write or
// read.  Since every kernel in such a chain waits before it touches shared
// data, a kernel past its wait knows all earlier kernels complete.
// pdl_launch_dependents() lets the next kernel be scheduled now (it takes
// effect once every CTA has called it or exited).  Without programmatic
// serialization both return at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ret
