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
#include "tc.cuh"
#include "tmap.h"
#include <cuda_fp16.h>
#include <string.h>

namespace ret {

__global__ void __launch_bounds__(256)
rotate_scale_kernel(KParams p, const void *__restrict__ x, long long s0, long long s1,
                    long long s2, int d, void *__restrict__ out, int out_bf16,
                    const float *__restrict__ scale, int mode) {
  __shared__ float th[2][kMaxPairs];  // per-pair frequencies (indexed per thread)
  const int b = blockIdx.z, h = blockIdx.y;
  const int P = d / 2;
  for (int t = threadIdx.x; t < P; t += blockDim.x) {
    th[0][t] = p.th_hi[t];
    th[1][t] = p.th_lo[t];
  }
  __syncthreads();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)p.N * P) return;
  const int tau = (int)(idx / P), j = (int)(idx % P);
  const long long src = b * s0 + h * s1 + tau * s2 + 2 * j;
  float a = ld_elem(x, src, p.in_bf16), c2 = ld_elem(x, src + 1, p.in_bf16);
  if (p.rotate) {
    float cs, sn;
    rot_cs(p.pos0 + tau, th[0][j], th[1][j], cs, sn);
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

// fp16 operand prologue of the tensor-core chunk kernel, queries and keys in
// one launch.  A tile is the 64 rows of one (batch*head, chunk) of q or k.
// Its rows are rotated and scaled by xi (queries) or zeta (keys) in fp32,
// then written as fp16 times a power of two 2^-e, e chosen from a bound m of
// the scaled values (m 2^-e < 2^14): a rotation keeps each pair's norm, which
// is at most sqrt(2) max|x| over the tile's raw elements, and the decay is at
// most gamma (xi) or 1 (zeta).  So no value can overflow and every normal
// value keeps fp16's 11-bit precision.  e and the pair-norm bound before the
// decay go to the tile's ChunkMeta record; for keys the column sums of the
// scaled rows (sum_j zeta_j rot(k_j), fp32) go to colsum[(bh*nch + c)*dk + col],
// the chunk's contribution to z.
//
// Persistent CTAs walk the tiles; the next tile's rows arrive by TMA into the
// second of two shared-memory buffers while the current one is processed.
// A thread keeps two adjacent pair columns and walks rows i0, i0+s, ...; the
// angles start from e^{i (pos0+t0) theta_j} (one per column and tile, shared
// through shared memory) times the thread's fixed offset e^{i i0 theta_j} and
// advance by e^{i s theta_j}; the decay advances by gamma^(+-s).  A walk is at
// most 16 steps, so the rounding it accumulates stays near 1e-6.
struct RotQK {
  const void *x[2];         // q, k (bf16)
  long long s[2][3];        // element strides (b, h, n)
  __half *out[2];           // Q', K' contiguous [B*H][N][dk] fp16
  ChunkMeta *meta;          // [B*H][nch]
  float *colsum;            // [B*H][nch][dk] or null
  int ntiles;               // kinds * B*H * nch
  int kinds;                // 2: queries and keys; 1: keys only
};

// Tile t: which tensor (0 queries, 1 keys) and which (batch*head, chunk).
__device__ __forceinline__ void tile_of(const RotQK &a, int t, int &which, int &r) {
  which = a.kinds == 2 ? (t & 1) : 1;
  r = a.kinds == 2 ? (t >> 1) : t;
}

template <bool kTma>
__global__ void __launch_bounds__(256)
rotate_qk_kernel(const __grid_constant__ KParams p, const __grid_constant__ RotQK a,
                 const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk) {
  constexpr int C = 64;
  extern __shared__ __align__(128) uint8_t xt[];  // [2][C][dk] bf16
  __shared__ __align__(8) uint64_t tbar[2];
  __shared__ unsigned red[8];
  __shared__ __align__(16) float2 anc[kMaxPairs];  // e^{i (pos0+t0) theta_j}
  __shared__ __align__(16) float4 csum[256];
  const int tid = threadIdx.x, P = p.dk / 2, Q2 = p.dk / 4;
  const int istep = 256 / Q2, jq = tid % Q2, ip = tid / Q2;
  const bool active = tid < Q2 * istep;
  const int nch = (p.N + C - 1) / C;
  const uint32_t tile_bytes = (uint32_t)(C * p.dk * 2);
  // The thread's fixed angle offsets: e^{i ip theta} and e^{i istep theta}
  // for its pair columns 2jq and 2jq+1.
  float oc[2] = {1.f, 1.f}, os[2] = {0.f, 0.f}, dc[2] = {1.f, 1.f}, ds[2] = {0.f, 0.f};
  if (p.rotate && active)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      rot_cs(ip, p.th_hi[2 * jq + e], p.th_lo[2 * jq + e], oc[e], os[e]);
      rot_cs(istep, p.th_hi[2 * jq + e], p.th_lo[2 * jq + e], dc[e], ds[e]);
    }
  if (kTma && tid == 0) {
    tc::mbar_init(&tbar[0], 1);
    tc::mbar_init(&tbar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();  // global memory only once the kernel before this one is complete
  auto issue = [&](int t, int buf) {
    int which, r;
    tile_of(a, t, which, r);
    const int bh = r / nch, c = r % nch;
    tc::mbar_arrive_expect_tx(&tbar[buf], tile_bytes);
    tc::tma_load_4d(xt + buf * tile_bytes, which ? &tmk : &tmq, &tbar[buf], 0, c * C,
                    bh % p.H, bh / p.H);
  };
  if (kTma && tid == 0 && (int)blockIdx.x < a.ntiles) issue(blockIdx.x, 0);
  int k = 0;
  for (int t = blockIdx.x; t < a.ntiles; t += gridDim.x, ++k) {
    if (t + (int)gridDim.x >= a.ntiles) pdl_launch_dependents();  // this CTA's last tile
    int which, r;
    tile_of(a, t, which, r);
    const int bh = r / nch, c = r % nch;
    const int b = bh / p.H, h = bh % p.H;
    const int buf = kTma ? (k & 1) : 0;
    const uint8_t *tile = xt + buf * tile_bytes;
    const int t0 = c * C, L = min(C, p.N - t0);
    const float lng = p.lng[h];
    const bool xi = which == 0;
    if (kTma) {
      if (tid == 0 && t + (int)gridDim.x < a.ntiles) issue(t + gridDim.x, buf ^ 1);
      // Bounded wait; if it ever ran out, wait (bounded) again for the copy
      // to land before reading or leaving.
      if (!tc::mbar_wait(&tbar[buf], (k >> 1) & 1, p.status, p.report_budget))
        tc::mbar_wait(&tbar[buf], (k >> 1) & 1, nullptr, 1u << 24);
    } else {
      const long long *sx = a.s[which];
      const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a.x[which]);
      for (int e = tid; e < L * P; e += 256) {
        const int i = e / P, j = e % P;
        const long long src = b * sx[0] + h * sx[1] + (long long)(t0 + i) * sx[2] + 2 * j;
        __nv_bfloat162 w;
        w.x = x[src];
        w.y = x[src + 1];
        *reinterpret_cast<__nv_bfloat162 *>(xt + ((size_t)i * p.dk + 2 * j) * 2) = w;
      }
      __syncthreads();
    }
    // Pass 1: max |x| over the tile's rows (bf16 magnitudes compare as
    // unsigned 16-bit integers); the tile's angle anchors.
    unsigned mb = 0;
    {
      const uint4 *t4 = reinterpret_cast<const uint4 *>(tile);
      const int n4 = L * p.dk / 8;
      for (int e = tid; e < n4; e += 256) {
        const uint4 u = t4[e];
        mb = __vmaxu2(mb, __vmaxu2(__vmaxu2(u.x & 0x7fff7fffu, u.y & 0x7fff7fffu),
                                   __vmaxu2(u.z & 0x7fff7fffu, u.w & 0x7fff7fffu)));
      }
    }
    if (p.rotate && tid < P) {
      float cs, sn;
      rot_cs(p.pos0 + t0, p.th_hi[tid], p.th_lo[tid], cs, sn);
      anc[tid] = make_float2(cs, sn);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = __vmaxu2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    if ((tid & 31) == 0) red[tid >> 5] = mb;
    __syncthreads();
    mb = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mb = __vmaxu2(mb, red[w]);
    const float xmax = fmaxf(__uint_as_float(mb << 16), __uint_as_float(mb & 0xffff0000u));
    const float nb = xmax * 1.41421366f;  // >= sqrt(2) max|x|: bound of every pair norm
    const float m = xi ? nb * p.gam[h] : nb;
    int ex = 0;
    if (m > 0.f && m < INFINITY) {
      frexpf(m, &ex);
      ex -= 14;
    }
    const float sc = exp2f((float)-ex);
    // Pass 2: rotate, scale, round to fp16, store; key column sums.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && ip < L) {
      // Decay of row i: xi = gamma^(i+1) (queries), zeta = gamma^(L-1-i) (keys).
      const float fstep = xi ? gpow(lng, istep) : expf(-(float)istep * lng);
      float fs = gpow(lng, xi ? ip + 1 : L - 1 - ip) * sc;
      float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;
      if (p.rotate) {
        const float4 an = *reinterpret_cast<const float4 *>(&anc[2 * jq]);
        c0 = an.x * oc[0] - an.y * os[0];
        s0 = an.x * os[0] + an.y * oc[0];
        c1 = an.z * oc[1] - an.w * os[1];
        s1 = an.z * os[1] + an.w * oc[1];
      }
      const uint8_t *src = tile + ((size_t)ip * p.dk + 4 * jq) * 2;
      uint2 *dst = reinterpret_cast<uint2 *>(a.out[which] + ((long long)bh * p.N + t0 + ip) * p.dk +
                                             4 * jq);
      const size_t sstep = (size_t)istep * p.dk * 2, dstep = (size_t)istep * p.dk / 4;
      for (int i = ip; i < L; i += istep, src += sstep, dst += dstep) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        const float a0 = __uint_as_float(w.x << 16), a1 = __uint_as_float(w.x & 0xffff0000u);
        const float a2 = __uint_as_float(w.y << 16), a3 = __uint_as_float(w.y & 0xffff0000u);
        const float r0 = (a0 * c0 - a1 * s0) * fs, r1 = (a0 * s0 + a1 * c0) * fs;
        const float r2 = (a2 * c1 - a3 * s1) * fs, r3 = (a2 * s1 + a3 * c1) * fs;
        acc.x += r0;
        acc.y += r1;
        acc.z += r2;
        acc.w += r3;
        *dst = make_uint2(tc::pack_f16(r0, r1), tc::pack_f16(r2, r3));
        fs *= fstep;
        const float n0 = c0 * dc[0] - s0 * ds[0], m0 = s0 * dc[0] + c0 * ds[0];
        const float n1 = c1 * dc[1] - s1 * ds[1], m1 = s1 * dc[1] + c1 * ds[1];
        c0 = n0;
        s0 = m0;
        c1 = n1;
        s1 = m1;
      }
    }
    if (!xi && a.colsum) csum[tid] = acc;
    __syncthreads();
    if (!xi && a.colsum && tid < Q2) {
      float4 s4 = csum[tid];
      for (int rr = 1; rr < istep; ++rr) {
        const float4 o4 = csum[tid + rr * Q2];
        s4.x += o4.x;
        s4.y += o4.y;
        s4.z += o4.z;
        s4.w += o4.w;
      }
      const float back = exp2f((float)ex);  // the sums were taken in units of 2^ex
      float4 *cdst = reinterpret_cast<float4 *>(a.colsum + ((long long)bh * nch + c) * p.dk) + tid;
      *cdst = make_float4(s4.x * back, s4.y * back, s4.z * back, s4.w * back);
    }
    if (tid == 0) {
      ChunkMeta *mt = a.meta + (long long)bh * nch + c;
      if (xi) {
        mt->qexp = ex;
        mt->qmax = nb;
      } else {
        mt->kexp = ex;
        mt->kmax = nb;
      }
    }
    __syncthreads();  // buffer, csum, anc and red are free for the next tile
  }
}

cudaError_t launch_rotate_qk(const KParams &p, const void *q, const void *k, __half *Qp,
                             __half *Kp, ChunkMeta *meta, float *colsum, cudaStream_t st,
                             bool keys_only) {
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  if (p.chunk != 64 || p.dk < 4 || p.dk > 256 || p.dk % 4 || !p.in_bf16)
    return cudaErrorInvalidValue;
  RotQK a;
  a.x[0] = q;
  a.x[1] = k;
  for (int i = 0; i < 3; ++i) {
    a.s[0][i] = p.sq[i];
    a.s[1][i] = p.sk[i];
  }
  a.out[0] = Qp;
  a.out[1] = Kp;
  a.meta = meta;
  a.colsum = colsum;
  const int nch = (p.N + 63) / 64;
  a.kinds = keys_only ? 1 : 2;
  a.ntiles = a.kinds * p.B * p.H * nch;
  // TMA source when both inputs are 16-byte aligned with 16-byte strides.
  CUtensorMap tm[2];
  memset(tm, 0, sizeof(tm));
  bool tma = p.dk % 8 == 0;
  for (int w = keys_only ? 1 : 0; w < 2 && tma; ++w) {
    const long long *s = a.s[w];
    tma = (reinterpret_cast<uintptr_t>(a.x[w]) % 16 == 0) && s[0] % 8 == 0 && s[1] % 8 == 0 &&
          s[2] % 8 == 0;
    if (!tma) break;
    const cuuint64_t dims[4] = {(cuuint64_t)p.dk, (cuuint64_t)p.N, (cuuint64_t)p.H,
                                (cuuint64_t)p.B};
    const cuuint64_t strides[3] = {(cuuint64_t)s[2] * 2, (cuuint64_t)s[1] * 2,
                                   (cuuint64_t)s[0] * 2};
    const cuuint32_t box[4] = {(cuuint32_t)p.dk, 64, 1, 1};
    tma = tmap_encode(&tm[w], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.x[w], dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t tile = (size_t)64 * p.dk * 2;
  if (tma) {
    const size_t smem = 2 * tile;
    cudaError_t e = cudaFuncSetAttribute(rotate_qk_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = a.ntiles < 3 * sms ? a.ntiles : 3 * sms;
    return launch_k(rotate_qk_kernel<true>, dim3(grid), dim3(256), smem, st, true, p, a, tm[0],
                    tm[1]);
  }
  cudaError_t e = cudaFuncSetAttribute(rotate_qk_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tile);
  if (e != cudaSuccess) return e;
  const int grid = a.ntiles < 6 * sms ? a.ntiles : 6 * sms;
  return launch_k(rotate_qk_kernel<false>, dim3(grid), dim3(256), tile, st, true, p, a, tm[0],
                  tm[1]);
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
