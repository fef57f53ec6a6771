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
constexpr int RM = 4;    // value columns per thread in the row kernel's carry (d_v <= RM * NT)
constexpr int VW = 32;   // d_v columns per CTA of the value kernel
constexpr int VC = 32;   // tokens per step of the value kernel
constexpr int VLU = VW + 1;  // row stride of the value kernel's U
constexpr int kLoadBatch = 8;  // global loads a thread issues before storing them

// Row stride of the d_v-wide rows of the row kernel: d_v + 2 keeps the
// 2x2-tiled loads of its score phase free of bank conflicts (d_v % 32 == 0).
int rows_ld(int dv) { return dv + 2; }

size_t rows_smem(int dv) {
  const size_t ld = (size_t)rows_ld(dv);
  return sizeof(float) * (RA * ld + 2 * RC * ld + 2 * RC * RA + RC * (RC + 1) + RC * (RA + 1) +
                          (RC + 1) + RC);
}

__host__ __device__ inline size_t round4(size_t x) { return (x + 3) & ~(size_t)3; }

size_t values_smem(int dk) {
  const size_t ld = (size_t)dk + 1;
  return sizeof(float) * (round4((size_t)dk * VLU) + 2 * VC * ld + 2 * VC * VW +
                          VC * (VC + 1) + (VC + 1) + VC);
}
}  // namespace

// Row gradients dQ' (kRev = false, forward sweep over the states S_c) or
// dK' (kRev = true, reverse sweep over the gradients U_c), for RA columns
// a0.. of d_k.  Per chunk, X holds the rows that own the outputs and Y, Z
// the partner rows:
//   forward:  X = dO~, Y = V, Z = K'[:, a0..];  reverse: X = V, Y = dO~, Z = Q'[:, a0..]
// and T the slice [a0..][0, d_v) of S_c or U_c.  Each chunk takes three
// phases: the scores A = X Y^T and the state term X T^T over d_v (2x2 tiles
// per thread, d_v split four ways across neighbouring lanes); the outputs;
// and the carry T <- gamma^L T + Zw^T Y (Zw = Z with the carry weights), a
// thread holding all RA rows of its value columns in registers.
template <bool kRev>
__global__ void __launch_bounds__(NT)
bwd_rows_kernel(KParams p, const float *__restrict__ Zsrc, const void *__restrict__ v,
                const void *__restrict__ dO, const float *__restrict__ T0,
                float *__restrict__ out) {
  extern __shared__ __align__(16) float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N, ld = dv + 2;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int a0 = blockIdx.x * RA;
  float *T = sm;                   // [RA][ld]
  float *X = T + RA * ld;          // [RC][ld]
  float *Y = X + RC * ld;          // [RC][ld]
  float *Z = Y + RC * ld;          // [RC][RA]
  float *Zw = Z + RC * RA;         // [RC][RA] Z times the carry weight of its row
  float *A = Zw + RC * RA;         // [RC][RC+1]
  float *Cr = A + RC * (RC + 1);   // [RC][RA+1] X T^T
  float *gp = Cr + RC * (RA + 1);  // [RC+1] gamma^k
  float *sr = gp + RC + 1;         // [RC] row factors of the chunk
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
    __syncthreads();  // the previous step's readers are done
    if (tid < RC) sr[tid] = tid < L ? row_scale(p, h, p.pos0 + c0 + tid + 1) : 0.f;
    __syncthreads();
    // Rows i0..i0+kLoadBatch-1 of a column: independent loads in flight
    // before their stores, and no division by d_v.
    for (int c = tid; c < dv; c += NT) {
#pragma unroll 1
      for (int i0 = 0; i0 < RC; i0 += kLoadBatch) {
        float dov[kLoadBatch], vv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
          const int i = i0 + u;
          dov[u] = vv[u] = 0.f;
          if (i < L) {
            dov[u] = ld_elem(dO, ob + (c0 + i) * p.so[2] + c, p.out_bf16);
            vv[u] = ld_elem(v, vb + (c0 + i) * p.sv[2] + c, p.in_bf16);
          }
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
          const int i = i0 + u;
          const float d = sr[i] * dov[u];
          X[i * ld + c] = kRev ? vv[u] : d;
          Y[i * ld + c] = kRev ? d : vv[u];
        }
      }
    }
    for (int e = tid; e < RC * RA; e += NT) {
      const int j = e / RA, a = e % RA;
      const float z =
          (j < L && a0 + a < dk) ? Zsrc[((long long)bh * N + c0 + j) * dk + a0 + a] : 0.f;
      Z[e] = z;
      Zw[e] = j < L ? gp[kRev ? j + 1 : L - 1 - j] * z : 0.f;
    }
    __syncthreads();
    {  // A[i][j] = gamma^|i-j| (X_i . Y_j) on the causal side, and Cr = X T^T
      const int p4 = tid & 3, q = (tid >> 2) & 7, ip = tid >> 5;
      const int i0 = 2 * ip, r0 = 2 * q;
      const float *x0 = X + i0 * ld, *x1 = x0 + ld;
      const float *y0 = Y + r0 * ld, *y1 = y0 + ld;
      const float *t0 = T + r0 * ld, *t1 = t0 + ld;
      float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
      float u00 = 0.f, u01 = 0.f, u10 = 0.f, u11 = 0.f;
      for (int c = p4; c < dv; c += 4) {
        const float xa = x0[c], xb = x1[c];
        const float ya = y0[c], yb = y1[c];
        const float ta = t0[c], tb = t1[c];
        s00 = fmaf(xa, ya, s00); s01 = fmaf(xa, yb, s01);
        s10 = fmaf(xb, ya, s10); s11 = fmaf(xb, yb, s11);
        u00 = fmaf(xa, ta, u00); u01 = fmaf(xa, tb, u01);
        u10 = fmaf(xb, ta, u10); u11 = fmaf(xb, tb, u11);
      }
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        s00 += __shfl_xor_sync(0xffffffffu, s00, m);
        s01 += __shfl_xor_sync(0xffffffffu, s01, m);
        s10 += __shfl_xor_sync(0xffffffffu, s10, m);
        s11 += __shfl_xor_sync(0xffffffffu, s11, m);
        u00 += __shfl_xor_sync(0xffffffffu, u00, m);
        u01 += __shfl_xor_sync(0xffffffffu, u01, m);
        u10 += __shfl_xor_sync(0xffffffffu, u10, m);
        u11 += __shfl_xor_sync(0xffffffffu, u11, m);
      }
      if (p4 == 0) {
        const float sv[2][2] = {{s00, s01}, {s10, s11}};
        const float uv[2][2] = {{u00, u01}, {u10, u11}};
#pragma unroll
        for (int di = 0; di < 2; ++di)
#pragma unroll
          for (int dj = 0; dj < 2; ++dj) {
            const int i = i0 + di, j = r0 + dj;
            const bool on = i < L && j < L && (kRev ? j >= i : j <= i);
            A[i * (RC + 1) + j] = on ? sv[di][dj] * gp[kRev ? j - i : i - j] : 0.f;
            Cr[i * (RA + 1) + j] = uv[di][dj];
          }
      }
    }
    __syncthreads();
    {  // outputs: intra-chunk part + the state term (reads A, Z, Cr)
      const int i = tid / RA, a = tid % RA;
      if (i < L && a0 + a < dk) {
        float intra = 0.f;
#pragma unroll
        for (int j = 0; j < RC; ++j) intra = fmaf(A[i * (RC + 1) + j], Z[j * RA + a], intra);
        const float wc = gp[kRev ? L - 1 - i : i + 1];
        out[((long long)bh * N + c0 + i) * dk + a0 + a] = fmaf(wc, Cr[i * (RA + 1) + a], intra);
      }
    }
    {  // carry across the chunk (reads Zw, Y, T; writes T)
      const float gL = gp[L];
      float acc[RM][RA];
#pragma unroll
      for (int m = 0; m < RM; ++m) {
        const int c = tid + NT * m;
#pragma unroll
        for (int a = 0; a < RA; ++a) acc[m][a] = c < dv ? gL * T[a * ld + c] : 0.f;
      }
      for (int j = 0; j < L; ++j) {
        float zw[RA];
        const float4 *zr = reinterpret_cast<const float4 *>(Zw + j * RA);
#pragma unroll
        for (int t = 0; t < RA / 4; ++t) {
          const float4 z4 = zr[t];
          zw[4 * t] = z4.x; zw[4 * t + 1] = z4.y; zw[4 * t + 2] = z4.z; zw[4 * t + 3] = z4.w;
        }
#pragma unroll
        for (int m = 0; m < RM; ++m) {
          const int c = tid + NT * m;
          if (c < dv) {
            const float y = Y[j * ld + c];
#pragma unroll
            for (int a = 0; a < RA; ++a) acc[m][a] = fmaf(zw[a], y, acc[m][a]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < RM; ++m) {
        const int c = tid + NT * m;
        if (c < dv)
#pragma unroll
          for (int a = 0; a < RA; ++a) T[a * ld + c] = acc[m][a];
      }
    }
  }
}

// Value gradients dV for VW columns v0.. of d_v (reverse sweep), and dS_in.
// Per chunk: Kc = K' rows (the output owners), Qc = Q' rows, Dc = dO~ slice,
// Dw = Dc with the carry weights, U the slice [0, d_k)[v0..] of U_c.  The
// scores A = Kc Qc^T and the state term Kc U run together over d_k (2x2
// tiles of each per thread); the thread then finishes its own 2x2 output
// tile; the carry U <- gamma^L U + Qc^T Dw gives each thread one row of U.
__global__ void __launch_bounds__(NT)
bwd_values_kernel(KParams p, const float *__restrict__ Qr, const float *__restrict__ Kr,
                  const void *__restrict__ dO, const float *dS_out, void *__restrict__ dv_out,
                  float *dS_in) {
  extern __shared__ __align__(16) float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N, ldk = dk + 1;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int v0 = blockIdx.x * VW;
  float *U = sm;                                  // [dk][VLU]
  float *Kc = U + round4((size_t)dk * VLU);       // [VC][ldk]
  float *Qc = Kc + VC * ldk;                      // [VC][ldk]
  float *Dc = Qc + VC * ldk;                      // [VC][VW]
  float *Dw = Dc + VC * VW;                       // [VC][VW]
  float *A = Dw + VC * VW;                        // [VC][VC+1]
  float *gp = A + VC * (VC + 1);                  // [VC+1]
  float *sr = gp + VC + 1;                        // [VC]
  const int tid = threadIdx.x;
  const float lng = p.lng[h];
  const long long vb = b * p.sv[0] + h * p.sv[1];
  const long long ob = b * p.so[0] + h * p.so[1];

  for (int e = tid; e < dk * VW; e += NT) {
    const int a = e / VW, c = e % VW;
    U[a * VLU + c] =
        (dS_out && v0 + c < dv) ? dS_out[((long long)bh * dk + a) * dv + v0 + c] : 0.f;
  }
  if (tid <= VC) gp[tid] = gpow(lng, tid);

  const int ip = tid >> 4, q = tid & 15;  // 2x2 tile: rows 2ip.., columns 2q..
  const int i0 = 2 * ip, r0 = 2 * q;
  const int nch = (N + VC - 1) / VC;
  for (int s = nch - 1; s >= 0; --s) {
    const int c0 = s * VC, L = min(VC, N - c0);
    __syncthreads();
    if (tid < VC) sr[tid] = tid < L ? row_scale(p, h, p.pos0 + c0 + tid + 1) : 0.f;
    __syncthreads();
    // Rows i0..i0+kLoadBatch-1 of a column: independent loads in flight
    // before their stores, and no division by d_k.
    for (int a = tid; a < dk; a += NT) {
#pragma unroll 1
      for (int i0 = 0; i0 < VC; i0 += kLoadBatch) {
        float kv[kLoadBatch], qv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
          const int i = i0 + u;
          kv[u] = qv[u] = 0.f;
          if (i < L) {
            const long long g = ((long long)bh * N + c0 + i) * dk + a;
            kv[u] = Kr[g];
            qv[u] = Qr[g];
          }
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
          Kc[(i0 + u) * ldk + a] = kv[u];
          Qc[(i0 + u) * ldk + a] = qv[u];
        }
      }
    }
    {
      constexpr int kPer = VC * VW / NT;  // 4 values of dO~ per thread
      float dd[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = tid + u * NT, i = e / VW, c = e % VW;
        dd[u] = (i < L && v0 + c < dv)
                    ? ld_elem(dO, ob + (c0 + i) * p.so[2] + v0 + c, p.out_bf16)
                    : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = tid + u * NT, i = e / VW;
        const float d = sr[i] * dd[u];
        Dc[e] = d;
        Dw[e] = i < L ? gp[i + 1] * d : 0.f;
      }
    }
    __syncthreads();
    float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;  // Kc U (state term)
    {
      float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
      const float *k0 = Kc + i0 * ldk, *k1 = k0 + ldk;
      const float *q0 = Qc + r0 * ldk, *q1 = q0 + ldk;
      for (int a = 0; a < dk; ++a) {
        const float ka = k0[a], kb = k1[a];
        const float qa = q0[a], qb = q1[a];
        const float ua = U[a * VLU + r0], ub = U[a * VLU + r0 + 1];
        s00 = fmaf(ka, qa, s00); s01 = fmaf(ka, qb, s01);
        s10 = fmaf(kb, qa, s10); s11 = fmaf(kb, qb, s11);
        x00 = fmaf(ka, ua, x00); x01 = fmaf(ka, ub, x01);
        x10 = fmaf(kb, ua, x10); x11 = fmaf(kb, ub, x11);
      }
      const float sv[2][2] = {{s00, s01}, {s10, s11}};
#pragma unroll
      for (int di = 0; di < 2; ++di)
#pragma unroll
        for (int dj = 0; dj < 2; ++dj) {
          const int i = i0 + di, j = r0 + dj;
          A[i * (VC + 1) + j] = (j >= i && j < L) ? sv[di][dj] * gp[j - i] : 0.f;
        }
    }
    __syncthreads();
    {  // the thread's own 2x2 output tile (reads A, Dc)
      const float xv[2][2] = {{x00, x01}, {x10, x11}};
#pragma unroll
      for (int di = 0; di < 2; ++di) {
        const int i = i0 + di;
        if (i >= L) continue;
#pragma unroll
        for (int dc = 0; dc < 2; ++dc) {
          const int c = r0 + dc;
          if (v0 + c >= dv) continue;
          float intra = 0.f;
          for (int j = i; j < L; ++j) intra = fmaf(A[i * (VC + 1) + j], Dc[j * VW + c], intra);
          st_elem(dv_out, vb + (c0 + i) * p.sv[2] + v0 + c,
                  fmaf(gp[L - 1 - i], xv[di][dc], intra), p.in_bf16);
        }
      }
    }
    if (tid < dk) {  // carry: row a = tid of U (reads Qc, Dw, U; writes U)
      const int a = tid;
      const float gL = gp[L];
      float acc[VW];
#pragma unroll
      for (int c = 0; c < VW; ++c) acc[c] = gL * U[a * VLU + c];
      for (int j = 0; j < L; ++j) {
        const float qa = Qc[j * ldk + a];
        const float4 *dr = reinterpret_cast<const float4 *>(Dw + j * VW);
#pragma unroll
        for (int t = 0; t < VW / 4; ++t) {
          const float4 d4 = dr[t];
          acc[4 * t] = fmaf(qa, d4.x, acc[4 * t]);
          acc[4 * t + 1] = fmaf(qa, d4.y, acc[4 * t + 1]);
          acc[4 * t + 2] = fmaf(qa, d4.z, acc[4 * t + 2]);
          acc[4 * t + 3] = fmaf(qa, d4.w, acc[4 * t + 3]);
        }
      }
#pragma unroll
      for (int c = 0; c < VW; ++c) U[a * VLU + c] = acc[c];
    }
  }
  __syncthreads();
  if (dS_in)
    for (int e = tid; e < dk * VW; e += NT) {
      const int a = e / VW, c = e % VW;
      if (v0 + c < dv) dS_in[((long long)bh * dk + a) * dv + v0 + c] = U[a * VLU + c];
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
