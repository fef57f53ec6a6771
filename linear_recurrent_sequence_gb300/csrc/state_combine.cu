// The recurrent state as a linear function of the tokens.
//
// hwhale.com/article/285883, recurrent form S_n = gamma S_{n-1} + K_n^T V_n:
// the recurrence is linear, so the state after a run of tokens is the state
// before it decayed by gamma^(run length) plus the state the run produces
// from zero, and a state carried over t further tokens with no input
// becomes gamma^t S.  Two kernels use that:
//   - state_combine_kernel: S_out = sum_i gamma_h^(t_i) S_i (and z likewise),
//     the decayed sum that joins partial states (pieces of one sequence, or
//     segments held by different ranks);
//   - state_simt_kernel / zstate_simt_kernel: the state a run of tokens
//     produces, S = gamma^N S_in + sum_m gamma^(N-1-m) K'_m^T V_m, by the
//     recurrence itself on CUDA cores (fp32 inputs and shapes the
//     tensor-core state kernel does not take).
#include "ktimer.h"
#include "launch.h"

namespace ret {

// Weight gamma^t of one part, per head (t = 0 gives 1 for every gamma).
__device__ __forceinline__ float part_weight(float lng, long long t) {
  return t == 0 ? 1.f : expf((float)t * lng);
}

// Grid-stride over the n = B*H*per_head values (coalesced scalar accesses:
// the callers' states need no particular alignment).
__global__ void __launch_bounds__(256)
state_combine_kernel(const CombineParts parts, const KParams p, float *__restrict__ out,
                     long long per_head, int is_z) {
  pdl_wait();  // the kernel before this one is complete (programmatic launch)
  pdl_launch_dependents();
  const long long n = (long long)p.B * p.H * per_head;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float lng = p.lng[(int)((i / per_head) % p.H)];
    float acc = 0.f;
    for (int j = 0; j < parts.count; ++j) {
      const float *src = is_z ? parts.z[j] : parts.S[j];
      if (src) acc = fmaf(part_weight(lng, parts.t[j]), src[i], acc);
    }
    out[i] = acc;
  }
}

cudaError_t launch_state_combine(const KParams &p, const CombineParts &parts, float *S_out,
                                 float *z_out, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  const long long BH = (long long)p.B * p.H;
  for (int which = 0; which < 2; ++which) {
    float *out = which ? z_out : S_out;
    if (!out) continue;
    const long long per = which ? (long long)p.dk : (long long)p.dk * p.dv;
    const long long blocks = (BH * per + 255) / 256;
    const int grid = (int)(blocks < 8LL * sms ? blocks : 8LL * sms);
    cudaError_t e = launch_k(state_combine_kernel, dim3(grid), dim3(256), 0, st, true, parts, p,
                             out, per, which);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// One CTA per (bh, 16 state rows, 128 value columns); thread = one value
// column, 16 rows of the state in registers, advanced token by token:
//   S_row <- gamma S_row + K'_m[row] v_m[col].
// The rotated keys come contiguous fp32 [B*H][N][d_k] (K'); v through the
// strides sv[] in the input dtype.  Tokens are staged 32 at a time.
constexpr int kSsRows = 16, kSsCols = 128, kSsTok = 32;

__global__ void __launch_bounds__(kSsCols)
state_simt_kernel(const KParams p, const float *__restrict__ Kr, const void *__restrict__ v,
                  const float *__restrict__ S_in, float *__restrict__ S_out) {
  __shared__ float ks[kSsTok][kSsRows];
  const int bh = blockIdx.z, b = bh / p.H, h = bh % p.H;
  const int a0 = blockIdx.y * kSsRows, e = blockIdx.x * kSsCols + threadIdx.x;
  const bool live = e < p.dv;
  const float g = p.gam[h];
  float acc[kSsRows];
#pragma unroll
  for (int r = 0; r < kSsRows; ++r) {
    const int a = a0 + r;
    acc[r] = (S_in && live && a < p.dk) ? S_in[((long long)bh * p.dk + a) * p.dv + e] : 0.f;
  }
  for (int m0 = 0; m0 < p.N; m0 += kSsTok) {
    const int nt = min(kSsTok, p.N - m0);
    __syncthreads();
    for (int i = threadIdx.x; i < kSsTok * kSsRows; i += kSsCols) {
      const int t = i / kSsRows, r = i % kSsRows;
      ks[t][r] = (t < nt && a0 + r < p.dk)
                     ? Kr[((long long)bh * p.N + m0 + t) * p.dk + a0 + r] : 0.f;
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      const float x = live ? ld_elem(v, b * p.sv[0] + h * p.sv[1] + (long long)(m0 + t) * p.sv[2] + e,
                                     p.in_bf16) : 0.f;
#pragma unroll
      for (int r = 0; r < kSsRows; ++r) acc[r] = fmaf(g, acc[r], ks[t][r] * x);
    }
  }
  if (!live) return;
#pragma unroll
  for (int r = 0; r < kSsRows; ++r) {
    const int a = a0 + r;
    if (a < p.dk) S_out[((long long)bh * p.dk + a) * p.dv + e] = acc[r];
  }
}

// z <- gamma z + K'_m, one thread per (bh, row).
__global__ void __launch_bounds__(128)
zstate_simt_kernel(const KParams p, const float *__restrict__ Kr, const float *__restrict__ z_in,
                   float *__restrict__ z_out) {
  const int bh = blockIdx.y, h = bh % p.H, a = blockIdx.x * 128 + threadIdx.x;
  if (a >= p.dk) return;
  const float g = p.gam[h];
  float z = z_in ? z_in[(long long)bh * p.dk + a] : 0.f;
  for (int m = 0; m < p.N; ++m) z = fmaf(g, z, Kr[((long long)bh * p.N + m) * p.dk + a]);
  z_out[(long long)bh * p.dk + a] = z;
}

cudaError_t launch_state_simt(const KParams &p, const float *Kr, const void *v,
                              const float *S_in, const float *z_in, float *S_out, float *z_out,
                              cudaStream_t st) {
  const int BH = p.B * p.H;
  if (S_out) {
    dim3 grid((p.dv + kSsCols - 1) / kSsCols, (p.dk + kSsRows - 1) / kSsRows, BH);
    state_simt_kernel<<<grid, kSsCols, 0, st>>>(p, Kr, v, S_in, S_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (z_out) {
    dim3 grid((p.dk + 127) / 128, BH);
    zstate_simt_kernel<<<grid, 128, 0, st>>>(p, Kr, z_in, z_out);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace ret
