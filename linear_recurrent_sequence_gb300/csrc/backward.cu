// Backward of retention on CUDA cores, fp32: the gradients of q, k, v and of
// the entry state, given the gradients of the outputs and of the final state.
//
// Forward (hwhale.com/article/285883, recurrent and chunkwise equations):
//   S_n = gamma S_{n-1} + K'_n^T V_n,   O_n = s_n Q'_n S_n,
// Q', K' the rotated rows (xPos/RoPE phase) and s_n the row factor of the
// first two normalisations, which does not depend on the data.  Reverse mode
// of that recurrence, written per chunk of L tokens with dO~_n = s_n dO_n,
// S_c the state entering the chunk and U_c the gradient with respect to the
// state after its last token:
//   dQ'_i = sum_{j<=i} gamma^(i-j) (dO~_i . V_j) K'_j + gamma^(i+1) S_c dO~_i
//   dK'_i = sum_{j>=i} gamma^(j-i) (dO~_j . V_i) Q'_j + gamma^(L-1-i) U_c V_i
//   dV_i  = sum_{j>=i} gamma^(j-i) (Q'_j . K'_i) dO~_j + gamma^(L-1-i) K'_i U_c
//   S_{c+1} = gamma^L S_c + sum_j gamma^(L-1-j) K'_j^T V_j            (S_0 = S_in)
//   U_{c-1} = gamma^L U_c + sum_j gamma^(j+1) Q'_j^T dO~_j   (U_last = dS_out)
//   dS_in = U_{-1};  dQ, dK = dQ', dK' turned back by e^{-i t theta}.
//
// dQ' and dK' sum over d_v and are computed by CTAs that own a slice of d_k
// (bwd_rows_kernel, forward and reverse sweep); dV sums over d_k and is
// computed by CTAs that own a slice of d_v (bwd_values_kernel, reverse
// sweep), which also write dS_in.
#include "common.cuh"
#include "launch.h"

namespace ret {

namespace {
constexpr int NT = 256;  // threads per CTA
constexpr int RA = 16;   // d_k columns per CTA of the row kernel
constexpr int RC = 16;   // tokens per step of the row kernel (RC * RC == NT)
constexpr int VW = 32;   // d_v columns per CTA of the value kernel
constexpr int VC = 32;   // tokens per step of the value kernel

size_t rows_smem(int dv) {
  const size_t ld = (size_t)dv + 1;
  return sizeof(float) * (RA * ld + 2 * RC * ld + RC * RA + RC * (RC + 1) + (RC + 1) + RC);
}

size_t values_smem(int dk) {
  const size_t ld = (size_t)dk + 1;
  return sizeof(float) * ((size_t)dk * VW + 2 * VC * ld + VC * VW + VC * (VC + 1) +
                          (VC + 1) + VC);
}
}  // namespace

// Row gradients dQ' (kRev = false, forward sweep over the states S_c) or
// dK' (kRev = true, reverse sweep over the gradients U_c), for RA columns
// a0.. of d_k.  Per chunk, X holds the rows that own the outputs and Y, Z
// the partner rows:
//   forward:  X = dO~, Y = V, Z = K'[:, a0..];  reverse: X = V, Y = dO~, Z = Q'[:, a0..]
// and T the slice [a0..][0, d_v) of S_c or U_c.
template <bool kRev>
__global__ void __launch_bounds__(NT)
bwd_rows_kernel(KParams p, const float *__restrict__ Zsrc, const void *__restrict__ v,
                const void *__restrict__ dO, const float *__restrict__ T0,
                float *__restrict__ out) {
  extern __shared__ float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N, ld = dv + 1;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int a0 = blockIdx.x * RA;
  float *T = sm;                  // [RA][ld]
  float *X = T + RA * ld;         // [RC][ld]
  float *Y = X + RC * ld;         // [RC][ld]
  float *Z = Y + RC * ld;         // [RC][RA]
  float *A = Z + RC * RA;         // [RC][RC+1]
  float *gp = A + RC * (RC + 1);  // [RC+1] gamma^k
  float *sr = gp + RC + 1;        // [RC] row factors of the chunk
  const int tid = threadIdx.x;
  const float lng = p.lng[h];
  const long long vb = b * p.sv[0] + h * p.sv[1];
  const long long ob = b * p.so[0] + h * p.so[1];

  for (int e = tid; e < RA * dv; e += NT) {
    const int a = e / dv, c = e % dv;
    T[a * ld + c] = (T0 && a0 + a < dk) ? T0[((long long)bh * dk + a0 + a) * dv + c] : 0.f;
  }
  if (tid <= RC) gp[tid] = gpow(lng, tid);

  const int nch = (N + RC - 1) / RC;
  for (int s = 0; s < nch; ++s) {
    const int c0 = (kRev ? nch - 1 - s : s) * RC;
    const int L = min(RC, N - c0);
    __syncthreads();  // the previous step's readers of X, Y, Z, sr are done
    if (tid < RC) sr[tid] = tid < L ? row_scale(p, h, p.pos0 + c0 + tid + 1) : 0.f;
    __syncthreads();
    for (int e = tid; e < RC * dv; e += NT) {
      const int i = e / dv, c = e % dv;
      float dov = 0.f, vv = 0.f;
      if (i < L) {
        dov = sr[i] * ld_elem(dO, ob + (c0 + i) * p.so[2] + c, p.out_bf16);
        vv = ld_elem(v, vb + (c0 + i) * p.sv[2] + c, p.in_bf16);
      }
      X[i * ld + c] = kRev ? vv : dov;
      Y[i * ld + c] = kRev ? dov : vv;
    }
    for (int e = tid; e < RC * RA; e += NT) {
      const int j = e / RA, a = e % RA;
      Z[e] = (j < L && a0 + a < dk) ? Zsrc[((long long)bh * N + c0 + j) * dk + a0 + a] : 0.f;
    }
    __syncthreads();
    {  // A[i][j] = gamma^|i-j| (X_i . Y_j) on the causal side, else 0
      const int i = tid / RC, j = tid % RC;
      float acc = 0.f;
      const bool on = i < L && j < L && (kRev ? j >= i : j <= i);
      if (on) {
        const float *xi = X + i * ld, *yj = Y + j * ld;
        for (int c = 0; c < dv; ++c) acc = fmaf(xi[c], yj[c], acc);
        acc *= gp[kRev ? j - i : i - j];
      }
      A[i * (RC + 1) + j] = acc;
    }
    __syncthreads();
    {  // outputs: intra-chunk part + the state term
      const int i = tid / RA, a = tid % RA;
      if (i < L && a0 + a < dk) {
        float intra = 0.f;
#pragma unroll
        for (int j = 0; j < RC; ++j) intra = fmaf(A[i * (RC + 1) + j], Z[j * RA + a], intra);
        float cross = 0.f;
        const float *ta = T + a * ld, *xi = X + i * ld;
        for (int c = 0; c < dv; ++c) cross = fmaf(ta[c], xi[c], cross);
        const float wc = gp[kRev ? L - 1 - i : i + 1];
        out[((long long)bh * N + c0 + i) * dk + a0 + a] = fmaf(wc, cross, intra);
      }
    }
    __syncthreads();
    // State (forward) or gradient (reverse) carry across the chunk.
    const float gL = gp[L];
    for (int e = tid; e < RA * dv; e += NT) {
      const int a = e / dv, c = e % dv;
      float acc = gL * T[a * ld + c];
      for (int j = 0; j < L; ++j)
        acc = fmaf(gp[kRev ? j + 1 : L - 1 - j] * Z[j * RA + a], Y[j * ld + c], acc);
      T[a * ld + c] = acc;
    }
  }
}

// Value gradients dV for VW columns v0.. of d_v (reverse sweep), and dS_in.
// Per chunk: Kc = K' rows (the output owners), Qc = Q' rows, Dc = dO~ slice,
// U the slice [0, d_k)[v0..] of U_c.
__global__ void __launch_bounds__(NT)
bwd_values_kernel(KParams p, const float *__restrict__ Qr, const float *__restrict__ Kr,
                  const void *__restrict__ dO, const float *dS_out, void *__restrict__ dv_out,
                  float *dS_in) {
  extern __shared__ float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N, ld = dk + 1;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int v0 = blockIdx.x * VW;
  float *U = sm;                  // [dk][VW]
  float *Kc = U + dk * VW;        // [VC][ld]
  float *Qc = Kc + VC * ld;       // [VC][ld]
  float *Dc = Qc + VC * ld;       // [VC][VW]
  float *A = Dc + VC * VW;        // [VC][VC+1]
  float *gp = A + VC * (VC + 1);  // [VC+1]
  float *sr = gp + VC + 1;        // [VC]
  const int tid = threadIdx.x;
  const float lng = p.lng[h];
  const long long vb = b * p.sv[0] + h * p.sv[1];
  const long long ob = b * p.so[0] + h * p.so[1];

  for (int e = tid; e < dk * VW; e += NT) {
    const int a = e / VW, c = e % VW;
    U[e] = (dS_out && v0 + c < dv) ? dS_out[((long long)bh * dk + a) * dv + v0 + c] : 0.f;
  }
  if (tid <= VC) gp[tid] = gpow(lng, tid);

  const int nch = (N + VC - 1) / VC;
  for (int s = nch - 1; s >= 0; --s) {
    const int c0 = s * VC, L = min(VC, N - c0);
    __syncthreads();
    if (tid < VC) sr[tid] = tid < L ? row_scale(p, h, p.pos0 + c0 + tid + 1) : 0.f;
    __syncthreads();
    for (int e = tid; e < VC * dk; e += NT) {
      const int i = e / dk, a = e % dk;
      const long long g = ((long long)bh * N + c0 + i) * dk + a;
      Kc[i * ld + a] = i < L ? Kr[g] : 0.f;
      Qc[i * ld + a] = i < L ? Qr[g] : 0.f;
    }
    for (int e = tid; e < VC * VW; e += NT) {
      const int i = e / VW, c = e % VW;
      Dc[e] = (i < L && v0 + c < dv)
                  ? sr[i] * ld_elem(dO, ob + (c0 + i) * p.so[2] + v0 + c, p.out_bf16)
                  : 0.f;
    }
    __syncthreads();
    // A[i][j] = gamma^(j-i) (Q'_j . K'_i) for j >= i
    for (int e = tid; e < VC * VC; e += NT) {
      const int i = e / VC, j = e % VC;
      float acc = 0.f;
      if (j >= i && j < L) {
        const float *ki = Kc + i * ld, *qj = Qc + j * ld;
        for (int a = 0; a < dk; ++a) acc = fmaf(ki[a], qj[a], acc);
        acc *= gp[j - i];
      }
      A[i * (VC + 1) + j] = acc;
    }
    __syncthreads();
    for (int e = tid; e < VC * VW; e += NT) {
      const int i = e / VW, c = e % VW;
      if (i >= L || v0 + c >= dv) continue;
      float intra = 0.f;
      for (int j = i; j < L; ++j) intra = fmaf(A[i * (VC + 1) + j], Dc[j * VW + c], intra);
      float cross = 0.f;
      const float *ki = Kc + i * ld;
      for (int a = 0; a < dk; ++a) cross = fmaf(ki[a], U[a * VW + c], cross);
      st_elem(dv_out, vb + (c0 + i) * p.sv[2] + v0 + c, fmaf(gp[L - 1 - i], cross, intra),
              p.in_bf16);
    }
    __syncthreads();
    const float gL = gp[L];
    for (int e = tid; e < dk * VW; e += NT) {
      const int a = e / VW, c = e % VW;
      float acc = gL * U[e];
      for (int j = 0; j < L; ++j) acc = fmaf(gp[j + 1] * Qc[j * ld + a], Dc[j * VW + c], acc);
      U[e] = acc;
    }
  }
  __syncthreads();
  if (dS_in)
    for (int e = tid; e < dk * VW; e += NT) {
      const int a = e / VW, c = e % VW;
      if (v0 + c < dv) dS_in[((long long)bh * dk + a) * dv + v0 + c] = U[e];
    }
}

// out = x turned back by e^{-i t theta_j} (the transpose of the prologue's
// rotation), or copied when the call does not rotate.  x: contiguous fp32
// [B*H][N][d_k]; out through the strides s (b, h, n).
__global__ void __launch_bounds__(256)
unrotate_kernel(KParams p, const float *__restrict__ x, long long s0, long long s1,
                long long s2, void *__restrict__ out, int out_bf16) {
  const int b = blockIdx.z, h = blockIdx.y, P = p.dk / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)p.N * P) return;
  const int tau = (int)(idx / P), j = (int)(idx % P);
  const float *xr = x + (((long long)b * p.H + h) * p.N + tau) * p.dk + 2 * j;
  float a = xr[0], c2 = xr[1];
  if (p.rotate) {
    float cs, sn;
    rot_cs(p.pos0 + tau, p.th_hi[j], p.th_lo[j], cs, sn);
    const float ra = a * cs + c2 * sn;
    const float rb = c2 * cs - a * sn;
    a = ra;
    c2 = rb;
  }
  const long long dst = b * s0 + h * s1 + tau * s2 + 2 * j;
  st_elem(out, dst, a, out_bf16);
  st_elem(out, dst + 1, c2, out_bf16);
}

cudaError_t launch_bwd_rows(const KParams &p, bool rev, const float *Z, const void *v,
                            const void *dO, const float *T0, float *out, cudaStream_t st) {
  const size_t smem = rows_smem(p.dv);
  dim3 grid((p.dk + RA - 1) / RA, p.B * p.H);
  cudaError_t e;
  if (rev) {
    e = cudaFuncSetAttribute(bwd_rows_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_rows_kernel<true><<<grid, NT, smem, st>>>(p, Z, v, dO, T0, out);
  } else {
    e = cudaFuncSetAttribute(bwd_rows_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_rows_kernel<false><<<grid, NT, smem, st>>>(p, Z, v, dO, T0, out);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_values(const KParams &p, const float *Qr, const float *Kr,
                              const void *dO, const float *dS_out, void *dv, float *dS_in,
                              cudaStream_t st) {
  const size_t smem = values_smem(p.dk);
  cudaError_t e = cudaFuncSetAttribute(bwd_values_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.dv + VW - 1) / VW, p.B * p.H);
  bwd_values_kernel<<<grid, NT, smem, st>>>(p, Qr, Kr, dO, dS_out, dv, dS_in);
  return cudaGetLastError();
}

cudaError_t launch_unrotate(const KParams &p, const float *x, const long long s[3], void *out,
                            int out_bf16, cudaStream_t st) {
  const long long pairs = (long long)p.N * (p.dk / 2);
  dim3 grid((unsigned)((pairs + 255) / 256), p.H, p.B);
  unrotate_kernel<<<grid, 256, 0, st>>>(p, x, s[0], s[1], s[2], out, out_bf16);
  return cudaGetLastError();
}

}  // namespace ret
