// One recurrent decode step (hwhale.com/article/285883, recurrent form
// S_n = gamma S_{n-1} + K_n^T V_n, Retention(X_n) = Q_n S_n, and the
// RecurrentRetention pseudocode: the output is read after the state update
// and summed over the key dimension; m0nads.wordpress.com, recurrent
// representation).  Followed by the per-head GroupNorm.
//
// Memory-bound: every step reads and writes the fp32 state S once
// (8 bytes per element).  Layout of work:
//   * a cluster of KS CTAs per (batch, head); CTA r owns rows
//     [r*dk/KS, (r+1)*dk/KS) of S (and of z);
//   * each thread streams 16-byte chunks of its rows (float4 along d_v),
//     updates them in registers, writes them back and accumulates its
//     share of q.S;
//   * partial outputs are summed across the cluster in a fixed order through
//     distributed shared memory (deterministic, no atomics, no waits other
//     than the cluster barrier), then GroupNorm statistics are exchanged the
//     same way and each CTA normalises and stores its d_v/KS outputs.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace ret {

namespace {
constexpr int NT = 128;   // threads per CTA
constexpr int UNR = 8;    // rows in flight per thread

// Sum `val` over the CTA into *dst (all threads must call).
__device__ __forceinline__ void block_sum(float val, float *dst, float *wsum, int tid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
  if ((tid & 31) == 0) wsum[tid >> 5] = val;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < NT / 32; ++w) t += wsum[w];
    *dst = t;
  }
  __syncthreads();
}
}  // namespace

__global__ void __launch_bounds__(NT)
recurrent_step_kernel(KParams p, int KS, const void *__restrict__ q,
                      const void *__restrict__ k, const void *__restrict__ v,
                      float *__restrict__ S, float *__restrict__ z, void *__restrict__ o) {
  extern __shared__ float sm[];
  __shared__ float wsum[NT / 32];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int bh = blockIdx.x / KS;
  const int b = bh / p.H, h = bh % p.H;
  const int dk = p.dk, dv = p.dv;
  const int R = dk / KS, k0 = rank * R;
  const int tid = threadIdx.x;
  const float g = p.gam[h];

  float *qr = sm;             // [R]
  float *kr = qr + R;         // [R]
  float *vs = kr + R;         // [dv]
  float *opart = vs + dv;     // [dv] this CTA's partial q.S
  float *red = opart + dv;    // [8]: [0] partial q.z, [1] sum x, [2] sum (x-mu)^2, warp scratch
  __shared__ float th[2][kMaxPairs];  // per-pair frequencies (indexed per thread)
  for (int t = tid; t < R / 2; t += NT) {
    th[0][t] = p.th_hi[k0 / 2 + t];
    th[1][t] = p.th_lo[k0 / 2 + t];
  }
  __syncthreads();

  // Rotated q, k rows of this CTA (positions: the token sits at pos0).
  const long long qb = b * p.sq[0] + h * p.sq[1];
  const long long kb = b * p.sk[0] + h * p.sk[1];
  for (int t = tid; t < R / 2; t += NT) {
    const int j = k0 / 2 + t;
    float q0 = ld_elem(q, qb + 2 * j, p.in_bf16), q1 = ld_elem(q, qb + 2 * j + 1, p.in_bf16);
    float c0 = ld_elem(k, kb + 2 * j, p.in_bf16), c1 = ld_elem(k, kb + 2 * j + 1, p.in_bf16);
    if (p.rotate) {
      float cs, sn;
      rot_cs(p.pos0, th[0][t], th[1][t], cs, sn);
      const float a = q0 * cs - q1 * sn, bq = q0 * sn + q1 * cs;
      const float c = c0 * cs - c1 * sn, d = c0 * sn + c1 * cs;
      q0 = a; q1 = bq; c0 = c; c1 = d;
    }
    qr[2 * t] = q0; qr[2 * t + 1] = q1;
    kr[2 * t] = c0; kr[2 * t + 1] = c1;
  }
  const long long vb = b * p.sv[0] + h * p.sv[1];
  for (int e = tid; e < dv; e += NT) vs[e] = ld_elem(v, vb + e, p.in_bf16);
  __syncthreads();

  // z <- gamma z + k (rows of this CTA) and the partial q.z of the row sum.
  const bool rsum = (p.norm_flags & RET_NORM_RSUM) != 0;
  if (tid < 32) {
    float part = 0.f;
    if (rsum && z)
      for (int t = tid; t < R; t += 32) {
        float *zp = z + (long long)bh * dk + k0 + t;
        const float zn = fmaf(g, *zp, kr[t]);
        *zp = zn;
        part = fmaf(qr[t], zn, part);
      }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
    if (tid == 0) red[0] = part;
  }

  // Stream the rows: S <- gamma S + k_a v ; acc += q_a S.
  const int nvec = dv / 4;
  float4 *Srow0 = reinterpret_cast<float4 *>(S + ((long long)bh * dk + k0) * dv);
  for (int c = tid; c < nvec; c += NT) {
    const float4 vv = reinterpret_cast<const float4 *>(vs)[c];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int a0 = 0; a0 < R; a0 += UNR) {
      float4 s[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        if (a0 + u < R) s[u] = Srow0[(long long)(a0 + u) * nvec + c];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (a0 + u >= R) break;
        const float ka = kr[a0 + u], qa = qr[a0 + u];
        s[u].x = fmaf(g, s[u].x, ka * vv.x);
        s[u].y = fmaf(g, s[u].y, ka * vv.y);
        s[u].z = fmaf(g, s[u].z, ka * vv.z);
        s[u].w = fmaf(g, s[u].w, ka * vv.w);
        Srow0[(long long)(a0 + u) * nvec + c] = s[u];
        acc.x = fmaf(qa, s[u].x, acc.x);
        acc.y = fmaf(qa, s[u].y, acc.y);
        acc.z = fmaf(qa, s[u].z, acc.z);
        acc.w = fmaf(qa, s[u].w, acc.w);
      }
    }
    reinterpret_cast<float4 *>(opart)[c] = acc;
  }
  cluster.sync();

  // Fixed-order sum of the KS partials for this CTA's output columns
  // e0 + tid + NT*i (span = dv/KS <= 1024 columns, so i < 8).
  const int span = dv / KS, e0 = rank * span;
  float qz = 0.f;
  for (int r = 0; r < KS; ++r) qz += cluster.map_shared_rank(red, r)[0];
  const float s = row_scale(p, h, p.pos0 + 1);
  const float f = s * rsum_scale(p, s * qz);
  float x[8];
  float lsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = tid + NT * i;
    x[i] = 0.f;
    if (e < span) {
      float acc = 0.f;
      for (int r = 0; r < KS; ++r) acc += cluster.map_shared_rank(opart, r)[e0 + e];
      x[i] = f * acc;
      lsum += x[i];
    }
  }
  float mu = 0.f, inv = 1.f;
  if (p.gn_eps >= 0.f) {
    block_sum(lsum, red + 1, wsum, tid);
    cluster.sync();
    float tot = 0.f;
    for (int r = 0; r < KS; ++r) tot += cluster.map_shared_rank(red, r)[1];
    mu = tot / dv;
    float lvar = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (tid + NT * i < span) lvar = fmaf(x[i] - mu, x[i] - mu, lvar);
    block_sum(lvar, red + 2, wsum, tid);
    cluster.sync();
    float var = 0.f;
    for (int r = 0; r < KS; ++r) var += cluster.map_shared_rank(red, r)[2];
    inv = rsqrtf(var / dv + p.gn_eps);
  }
  const long long ob = b * p.so[0] + h * p.so[1] + e0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (tid + NT * i < span) st_elem(o, ob + tid + NT * i, (x[i] - mu) * inv, p.out_bf16);
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

cudaError_t launch_recurrent_step(const KParams &p, const void *q, const void *k,
                                  const void *v, float *S, float *z, void *o,
                                  cudaStream_t st) {
  if (p.B == 0 || p.H == 0) return cudaSuccess;
  // Cluster size: up to 8 CTAs per head, each keeping an even number of
  // rows and an equal share of the outputs (<= NT columns).
  int KS = 8;
  while (KS > 1 && (p.dk % KS || (p.dk / KS) % 2 || p.dv % KS)) KS >>= 1;
  const int R = p.dk / KS;
  const size_t smem = sizeof(float) * (2 * R + 2 * p.dv + 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.H * KS));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, recurrent_step_kernel, p, KS, q, k, v, S, z, o);
}

}  // namespace ret
