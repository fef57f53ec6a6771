// fp32 CUDA-core retention: the chunkwise and parallel forms for any shape
// and any gamma in [0, 1].  They write the unnormalised rows Oraw and the
// per-row factor F = s(n) r(n) of the normalisations; GroupNorm follows in
// groupnorm.cu.  These kernels carry the fp32 inputs (true fp32 FMAs) and
// every shape the tensor-core kernel does not take.
//
// Chunkwise form (hwhale.com/article/285883, chunkwise equation and
// ChunkwiseRetention; m0nads.wordpress.com, chunkwise representation):
//   O_[c] = (Q_[c] K_[c]^T (.) D) V_[c] + (Q_[c] S_c) (.) xi,  xi_i = gamma^(i+1)
//   S_{c+1} = gamma^L S_c + sum_j gamma^(L-1-j) K_j^T V_j
// with the row sum of the third normalisation carried by
//   z_{c+1} = gamma^L z_c + sum_j gamma^(L-1-j) K_j.
// Parallel form (same page, Retention(X) = (Q K^T (.) D) V).
#include "common.cuh"
#include "launch.h"

namespace ret {

namespace {
constexpr int WS = 32;   // value columns per CTA
constexpr int CS = 32;   // tokens per step (the result does not depend on it)
constexpr int NT = 256;  // threads per CTA

size_t chunk_smem(int dk) {
  return sizeof(float) * ((size_t)dk * WS + dk + 2 * (size_t)CS * dk + CS * WS +
                          CS * (CS + 1) + 2 * CS);
}
}  // namespace

__global__ void __launch_bounds__(NT)
chunk_simt_kernel(KParams p, const float *__restrict__ Qr, const float *__restrict__ Kr,
                  const void *__restrict__ v, const float *S_in, const float *z_in,
                  float *S_out, float *z_out, float *__restrict__ Oraw,
                  float *__restrict__ F) {
  extern __shared__ float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int v0 = blockIdx.x * WS;
  float *S = sm;                      // [dk][WS]
  float *z = S + dk * WS;             // [dk]
  float *Q = z + dk;                  // [CS][dk]
  float *K = Q + CS * dk;             // [CS][dk]
  float *V = K + CS * dk;             // [CS][WS]
  float *A = V + CS * WS;             // [CS][CS+1]
  float *fr = A + CS * (CS + 1);      // [CS] row factor
  float *xi = fr + CS;                // [CS] gamma^(i+1)
  const float lng = p.lng[h];
  const int tid = threadIdx.x;

  for (int e = tid; e < dk * WS; e += NT) {
    const int a = e / WS, c = e % WS;
    const int col = v0 + c;
    S[e] = (S_in && col < dv) ? S_in[((long long)bh * dk + a) * dv + col] : 0.f;
  }
  for (int a = tid; a < dk; a += NT) z[a] = z_in ? z_in[(long long)bh * dk + a] : 0.f;
  __syncthreads();

  const long long vbase = b * p.sv[0] + h * p.sv[1];
  for (int c0 = 0; c0 < N; c0 += CS) {
    const int L = min(CS, N - c0);
    for (int e = tid; e < CS * dk; e += NT) {
      const int i = e / dk;
      const long long g = ((long long)bh * N + c0 + i) * dk + (e % dk);
      Q[e] = i < L ? Qr[g] : 0.f;
      K[e] = i < L ? Kr[g] : 0.f;
    }
    for (int e = tid; e < CS * WS; e += NT) {
      const int i = e / WS, c = e % WS;
      V[e] = (i < L && v0 + c < dv) ? ld_elem(v, vbase + (c0 + i) * p.sv[2] + v0 + c, p.in_bf16)
                                    : 0.f;
    }
    if (tid < CS) xi[tid] = gpow(lng, tid + 1);
    __syncthreads();
    // Intra-chunk scores with the decay mask D.
    for (int e = tid; e < CS * CS; e += NT) {
      const int i = e / CS, j = e % CS;
      float acc = 0.f;
      if (j <= i && i < L) {
        for (int a = 0; a < dk; ++a) acc = fmaf(Q[i * dk + a], K[j * dk + a], acc);
        acc *= gpow(lng, i - j);
      }
      A[i * (CS + 1) + j] = acc;
    }
    __syncthreads();
    // Row factors: s(n) r(n) with sum_{m<=n} R_nm = s(n) (sum_j A_ij + xi_i Q_i.z).
    if (tid < L) {
      float rs = 0.f;
      for (int j = 0; j <= tid; ++j) rs += A[tid * (CS + 1) + j];
      float qz = 0.f;
      for (int a = 0; a < dk; ++a) qz = fmaf(Q[tid * dk + a], z[a], qz);
      rs = fmaf(xi[tid], qz, rs);
      const float s = row_scale(p, h, p.pos0 + c0 + tid + 1);
      const float f = s * rsum_scale(p, s * rs);
      fr[tid] = f;
      if (blockIdx.x == 0) F[(long long)bh * N + c0 + tid] = f;
    }
    // Outputs: intra + cross (unnormalised).
    for (int e = tid; e < CS * WS; e += NT) {
      const int i = e / WS, c = e % WS;
      if (i >= L || v0 + c >= dv) continue;
      float inner = 0.f;
      for (int j = 0; j <= i; ++j) inner = fmaf(A[i * (CS + 1) + j], V[j * WS + c], inner);
      float cross = 0.f;
      for (int a = 0; a < dk; ++a) cross = fmaf(Q[i * dk + a], S[a * WS + c], cross);
      Oraw[((long long)bh * N + c0 + i) * dv + v0 + c] = fmaf(xi[i], cross, inner);
    }
    __syncthreads();
    // State carry.
    const float gL = gpow(lng, L);
    for (int e = tid; e < dk * WS; e += NT) {
      const int a = e / WS, c = e % WS;
      float acc = gL * S[e];
      for (int j = 0; j < L; ++j)
        acc = fmaf(gpow(lng, L - 1 - j) * K[j * dk + a], V[j * WS + c], acc);
      S[e] = acc;
    }
    for (int a = tid; a < dk; a += NT) {
      float acc = gL * z[a];
      for (int j = 0; j < L; ++j) acc = fmaf(gpow(lng, L - 1 - j), K[j * dk + a], acc);
      z[a] = acc;
    }
    __syncthreads();
  }
  if (S_out)
    for (int e = tid; e < dk * WS; e += NT) {
      const int a = e / WS, c = e % WS;
      if (v0 + c < dv) S_out[((long long)bh * dk + a) * dv + v0 + c] = S[e];
    }
  if (z_out && blockIdx.x == 0)
    for (int a = tid; a < dk; a += NT) z_out[(long long)bh * dk + a] = z[a];
}

// Parallel form, tiled over (query tile, key tile).
__global__ void __launch_bounds__(NT)
parallel_simt_kernel(KParams p, const float *__restrict__ Qr, const float *__restrict__ Kr,
                     const void *__restrict__ v, float *__restrict__ Oraw,
                     float *__restrict__ F) {
  extern __shared__ float sm[];
  const int dk = p.dk, dv = p.dv, N = p.N;
  const int bh = blockIdx.z, b = bh / p.H, h = bh % p.H;
  const int v0 = blockIdx.x * WS, i0 = blockIdx.y * CS;
  float *Q = sm;                  // [CS][dk]
  float *K = Q + CS * dk;         // [CS][dk]
  float *V = K + CS * dk;         // [CS][WS]
  float *A = V + CS * WS;         // [CS][CS+1]
  float *rs = A + CS * (CS + 1);  // [CS]
  const float lng = p.lng[h];
  const int tid = threadIdx.x;
  const long long vbase = b * p.sv[0] + h * p.sv[1];

  for (int e = tid; e < CS * dk; e += NT) {
    const int i = e / dk;
    Q[e] = (i0 + i < N) ? Qr[((long long)bh * N + i0 + i) * dk + (e % dk)] : 0.f;
  }
  if (tid < CS) rs[tid] = 0.f;
  // Each thread owns output (i, c) pairs e = tid + k*NT, k < CS*WS/NT.
  constexpr int PER = CS * WS / NT;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;

  for (int j0 = 0; j0 <= i0 && j0 < N; j0 += CS) {
    __syncthreads();
    for (int e = tid; e < CS * dk; e += NT) {
      const int j = e / dk;
      K[e] = (j0 + j < N) ? Kr[((long long)bh * N + j0 + j) * dk + (e % dk)] : 0.f;
    }
    for (int e = tid; e < CS * WS; e += NT) {
      const int j = e / WS, c = e % WS;
      V[e] = (j0 + j < N && v0 + c < dv)
                 ? ld_elem(v, vbase + (j0 + j) * p.sv[2] + v0 + c, p.in_bf16)
                 : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < CS * CS; e += NT) {
      const int i = e / CS, j = e % CS;
      const int n = i0 + i, m = j0 + j;
      float a = 0.f;
      if (m <= n && n < N && m < N) {
        for (int t = 0; t < dk; ++t) a = fmaf(Q[i * dk + t], K[j * dk + t], a);
        a *= gpow(lng, n - m);  // D_nm
      }
      A[i * (CS + 1) + j] = a;
    }
    __syncthreads();
    if (tid < CS) {
      float s = 0.f;
      for (int j = 0; j < CS; ++j) s += A[tid * (CS + 1) + j];
      rs[tid] += s;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = tid + k * NT, i = e / WS, c = e % WS;
      float o = acc[k];
      for (int j = 0; j < CS; ++j) o = fmaf(A[i * (CS + 1) + j], V[j * WS + c], o);
      acc[k] = o;
    }
  }
  __syncthreads();
  if (tid < CS && i0 + tid < N && blockIdx.x == 0) {
    const float s = row_scale(p, h, p.pos0 + i0 + tid + 1);
    F[(long long)bh * N + i0 + tid] = s * rsum_scale(p, s * rs[tid]);
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = tid + k * NT, i = e / WS, c = e % WS;
    if (i0 + i < N && v0 + c < dv) Oraw[((long long)bh * N + i0 + i) * dv + v0 + c] = acc[k];
  }
}

cudaError_t launch_chunk_simt(const KParams &p, const float *Qr, const float *Kr,
                              const void *v, const float *S_in, const float *z_in,
                              float *S_out, float *z_out, float *Oraw, float *F,
                              cudaStream_t st) {
  const size_t smem = chunk_smem(p.dk);
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.dv + WS - 1) / WS, p.B * p.H);
  chunk_simt_kernel<<<grid, NT, smem, st>>>(p, Qr, Kr, v, S_in, z_in, S_out, z_out, Oraw, F);
  return cudaGetLastError();
}

cudaError_t launch_parallel_simt(const KParams &p, const float *Qr, const float *Kr,
                                 const void *v, float *Oraw, float *F, cudaStream_t st) {
  const size_t smem = sizeof(float) * (2 * (size_t)CS * p.dk + CS * WS + CS * (CS + 1) + CS);
  cudaError_t e = cudaFuncSetAttribute(parallel_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.dv + WS - 1) / WS, (p.N + CS - 1) / CS, p.B * p.H);
  parallel_simt_kernel<<<grid, NT, smem, st>>>(p, Qr, Kr, v, Oraw, F);
  return cudaGetLastError();
}

}  // namespace ret
