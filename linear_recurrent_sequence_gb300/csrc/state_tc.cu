// State-only pass of the chunkwise form on the tensor cores.  It lets the
// chunk kernel run several segments of one sequence at once: the state that
// enters a segment is a decayed sum of partial states, each the state after
// one "piece" of whole chunks started from zero,
//   P_i = sum_{c in piece i} gamma^(L (b_i - 1 - c)) K'_[c]^T V_[c],
// where K'_[c] already carries zeta_j = gamma^(L-1-j) (hwhale.com/article/285883,
// chunkwise equation: S_{c+1} = gamma^L S_c + K_[c]^T (V_[c] (.) zeta); the
// recurrence is linear, so a sum of shifted pieces equals the sequential
// result up to rounding order).  Alongside, zP_i = the same sum of the key
// column sums, for the third normalisation's z.
//
// One CTA per (piece, batch, head, 128-wide slice of d_v).  Warp 0 streams K'
// and V through a 2-stage TMA ring, warp 1 issues the state-update MMAs
// (S^T += V^T K', M=128 v, N=d_k, K=64 tokens, fp32 accumulator in TMEM),
// warps 2-5 convert V to fp16.  The decay never touches the accumulator:
// TMEM holds D = S 2^-sigma with a real-valued sigma, and
//   S_{c+1} = gamma^L S_c + U_c   becomes   D_{c+1} = A B + D_c 2^-n_c,
// the MMA's own accumulator scale (an integer n_c in 0..15) with
// sigma_{c+1} = sigma_c + n_c + L log2(gamma): the gamma^L of every chunk
// goes into the bookkeeping, and V of chunk c is converted with the factor
// 2^(kexp_c - sigma_{c+1}) that puts A B = U_c 2^-sigma_{c+1} in the same
// units.  n_c keeps the converted V below 2^15 (fp16's range); a chunk that
// would need n_c > 15 has its accumulator rescaled on the CUDA cores first.
// So the MMAs of consecutive chunks follow each other with no CUDA-core
// step in between.  Every wait is bounded; a wait that runs out sets the
// status word and an abort flag, and every role leaves after draining its
// own asynchronous work.
#include "ktimer.h"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace ret {

namespace {

constexpr int kC = 64, kW = 128, kNT = 192;
// Stage: K' 32K | V 16K | key column sums (d_k fp32) | ChunkMeta.
constexpr uint32_t kOffK = 0, kOffV = 32 * 1024, kOffKs = 48 * 1024, kOffMeta = kOffKs + 1024;
constexpr uint32_t kStage = 50 * 1024;
constexpr uint32_t kOffRed = 2 * kStage;
constexpr uint32_t kOffN = kOffRed + 64;   // [2] int: the accumulator scale of each stage's MMA
constexpr uint32_t kOffBar = kOffN + 16;
constexpr int kNumBars = 8;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmem = kOffMisc + 16 + 1024;
constexpr uint32_t kBudget = 1u << 24;
enum { FULL0 = 0, FULL1, EMPTY0, EMPTY1, CONV0, CONV1, SFULL, DRAIN };

__device__ __forceinline__ bool swait(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                      unsigned *status) {
  for (uint32_t i = 0; i < kBudget; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

__device__ __forceinline__ void sdrain(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kBudget; ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

// AND over the 128 threads of the scaling group (named barrier 1).
__device__ __forceinline__ bool grp_all4(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// e such that m * 2^-e < 2^14 (0 for m = 0).
__device__ __forceinline__ int expo14s(float m) {
  int e = 0;
  if (m > 0.f && m < INFINITY) {
    frexpf(m, &e);
    e -= 14;
  }
  return e;
}

__device__ __forceinline__ float bfl(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bfh(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

__global__ void __launch_bounds__(kNT, 1)
state_tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const ChunkMeta *__restrict__ meta,
                const float *__restrict__ ksum, int piece_len, float *Part, float *zPart,
                int need_z) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = tc::smem_align1024(smraw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  float *red = reinterpret_cast<float *>(sm + kOffRed);
  uint32_t *tbase_p = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort_p = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NV = p.dv / kW, BH = p.B * p.H;
  const int piece = blockIdx.x / (BH * NV), rem = blockIdx.x % (BH * NV);
  const int bh = rem / NV, rank = rem % NV, b = bh / p.H, h = bh % p.H;
  const int v0 = rank * kW, DK = p.dk, NKB = DK / 64, N = p.N;
  const int nch = (N + kC - 1) / kC;
  const int c0 = piece * piece_len, ncl = max(0, min(piece_len, nch - c0));
  const float lng = p.lng[h];

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) tc::mbar_init(&bars[i], 1);
    *abort_p = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase_p, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = *tbase_p;
  pdl_wait();  // global memory only once the kernel before this one is complete

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      const uint32_t bytes =
          (uint32_t)NKB * 8192u + 16384u + 16u + (need_z ? (uint32_t)DK * 4u : 0u);
      int issued = 0;
      for (int lc = 0; lc < ncl; ++lc) {
        const int s = lc & 1, c = c0 + lc;
        if (lc >= 2 && !swait(&bars[EMPTY0 + s], ((lc >> 1) - 1) & 1, abort_p, p.status)) break;
        uint8_t *st = sm + s * kStage;
        tc::mbar_arrive_expect_tx(&bars[FULL0 + s], bytes);
        for (int kb = 0; kb < NKB; ++kb)
          tc::tma_load_3d(st + kOffK + kb * 8192, &tmK, &bars[FULL0 + s], kb * 64, c * kC, bh);
        for (int vb = 0; vb < 2; ++vb)
          tc::tma_load_4d(st + kOffV + vb * 8192, &tmV, &bars[FULL0 + s], v0 + vb * 64, c * kC,
                          h, b);
        tc::bulk_load(st + kOffMeta, meta + (long long)bh * nch + c, 16u, &bars[FULL0 + s]);
        if (need_z)
          tc::bulk_load(st + kOffKs, ksum + ((long long)bh * nch + c) * DK, (uint32_t)DK * 4u,
                        &bars[FULL0 + s]);
        ++issued;
      }
      pdl_launch_dependents();  // every load is issued
      for (int lc = issued > 2 ? issued - 2 : 0; lc < issued; ++lc)
        sdrain(&bars[FULL0 + (lc & 1)], (lc >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    // D = A B + D 2^-n: the first K-step of a chunk applies the chunk's
    // accumulator scale (the first chunk starts from zero), the others add.
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_f16(128, DK, 1, 1);
      const int *nsm = reinterpret_cast<const int *>(sm + kOffN);
      for (int lc = 0; lc < ncl; ++lc) {
        const int s = lc & 1;
        if (!swait(&bars[CONV0 + s], (lc >> 1) & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        const uint32_t sk = tc::smem_u32(sm + s * kStage + kOffK), sv = sk + kOffV;
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t da = tc::smem_desc(sv + ks * 2048, 8192, 1024, tc::kSw128);
          const uint64_t db = tc::smem_desc(sk + ks * 2048, 8192, 1024, tc::kSw128);
          if (ks == 0 && lc > 0)
            tc::mma_ss_scale_d(tb, da, db, id_s, nsm[s]);
          else
            tc::mma_ss(tb, da, db, id_s, (lc | ks) != 0);
        }
        tc::mma_commit(&bars[SFULL]);
        tc::mma_commit(&bars[EMPTY0 + s]);
      }
      tc::mma_commit(&bars[DRAIN]);  // every MMA issued above is finished
      sdrain(&bars[DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ scaling group
    const int q = warp & 3, et = tid - 64, vrow = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const long long vglob = v0 + vrow;
    int *nsm = reinterpret_cast<int *>(sm + kOffN);
    int rslot = 0;
    // TMEM holds D = S u with u = um 2^-ue (um in [1, 2)), i.e. u = 2^-sigma.
    float um = 1.f;
    int ue = 0;
    const bool zown = need_z && rank == 0 && 2 * et < DK;
    float zr0 = 0.f, zr1 = 0.f;  // z entries 2 et, 2 et + 1
    bool ok = true;
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      const float gL = gpow(lng, L);
      uint8_t *st = sm + s * kStage;
      ok = grp_all4(swait(&bars[FULL0 + s], (lc >> 1) & 1, abort_p, p.status));
      if (!ok) break;
      const int bk = reinterpret_cast<const ChunkMeta *>(st + kOffMeta)->kexp;
      // (0) z over the piece: z <- gamma^L z + sum_j K'_j (read before the
      // stage is released).
      if (zown) {
        const float *ks = reinterpret_cast<const float *>(st + kOffKs);
        zr0 = fmaf(gL, zr0, ks[2 * et]);
        zr1 = fmaf(gL, zr1, ks[2 * et + 1]);
      }
      // (1) max |V| of the tile (1024 16-byte words).
      uint4 vv[8];
      float vm = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        vv[u] = reinterpret_cast<const uint4 *>(st + kOffV)[et + 128 * u];
        const uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) vm = fmaxf(vm, fmaxf(fabsf(bfl(w[e])), fabsf(bfh(w[e]))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      float *r4 = red + 4 * rslot;
      rslot ^= 1;
      if (lane == 0) r4[et >> 5] = vm;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const float vmx = fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3]));
      // (2) units of this chunk.  V is converted with f = u' 2^kexp, u' the
      // accumulator's units after the chunk; u' = u gamma^-L 2^-n, n chosen
      // so that max|V| f < 2^15.  The first chunk starts from zero: its
      // units are free, taken so that max|V| f is about 2^14.
      int n = 0, extra = 0;
      if (lc == 0) {
        const int e = expo14s(vmx);  // vmx 2^-e < 2^14
        um = 1.f;
        ue = e + bk;                 // f = 2^(bk - ue) = 2^-e
      } else {
        // u gamma^-L as (mantissa, exponent)
        int d = 0;
        float m = frexpf(um * __frcp_rn(gL), &d);  // in [0.5, 1)
        m *= 2.f;
        int e = ue - d + 1;
        // f0 = m 2^(bk - e): need vmx f0 2^-n < 2^15
        const int need = vmx > 0.f ? expo14s(vmx * ldexpf(m, bk - e)) : 0;  // vmx f0 2^-need < 2^14
        // at least the decay's own exponent, d - 1, so that the units u do
        // not drift upward over chunks whose V is small or zero (D then
        // shrinks with the true state instead of growing)
        n = max(max(need, d - 1), 0);
        if (n > 15) {
          extra = n - 15;
          n = 15;
        }
        um = m;
        ue = e + n + extra;
      }
      const float f = ldexpf(um, bk - ue);
      if (et == 0) nsm[s] = n;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o4[e] = tc::pack_f16(bfl(w[e]) * f, bfh(w[e]) * f);
        reinterpret_cast<uint4 *>(st + kOffV)[et + 128 * u] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      tc::fence_proxy_async_smem();
      // (3) rare: a chunk far larger than the state so far needs the
      // accumulator scaled down by more than the MMA's 2^-15; the rest,
      // 2^-extra, is applied here once the previous chunk's MMAs are done.
      if (grp_all4(extra == 0) == false) {
        ok = grp_all4(swait(&bars[SFULL], (lc - 1) & 1, abort_p, p.status));
        if (!ok) break;
        tc::tc_fence_after();
        const float sc = exp2f((float)-extra);
        for (int g0 = 0; g0 < DK / 32; ++g0) {
          uint32_t r[32];
          tc::tmem_ld32(tb + lb + g0 * 32, r);
          tc::tmem_ld_wait_on(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * sc);
          tc::tmem_st32(tb + lb + g0 * 32, r);
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (et == 0) tc::mbar_arrive(&bars[CONV0 + s]);
    }
    if (ok && ncl > 0) {
      ok = grp_all4(swait(&bars[SFULL], (ncl - 1) & 1, abort_p, p.status));
      if (ok) {
        tc::tc_fence_after();
        const float back = ldexpf(__frcp_rn(um), ue);  // S = D / u
        float *dst = Part + (((long long)piece * BH + bh) * DK) * p.dv + vglob;
        for (int g = 0; g < DK / 32; ++g) {
          uint32_t r[32];
          tc::tmem_ld32(tb + lb + g * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            dst[(long long)(g * 32 + i) * p.dv] = __uint_as_float(r[i]) * back;
        }
        if (zown) {
          float *zd = zPart + ((long long)piece * BH + bh) * DK;
          zd[2 * et] = zr0;
          zd[2 * et + 1] = zr1;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 256);
  }
}

cudaError_t launch_state_tc(const KParams &p, const void *Kp, const void *v,
                            const ChunkMeta *meta, const float *ksum, int npieces,
                            int piece_len, float *Part, float *zPart, int need_z,
                            cudaStream_t st) {
  const int BH = p.B * p.H;
  CUtensorMap tk, tv;
  const cuuint64_t dq[3] = {(cuuint64_t)p.dk, (cuuint64_t)p.N, (cuuint64_t)BH};
  const cuuint64_t sq[2] = {(cuuint64_t)p.dk * 2, (cuuint64_t)p.N * p.dk * 2};
  const cuuint32_t bq[3] = {64, (cuuint32_t)kC, 1};
  const cuuint64_t dv4[4] = {(cuuint64_t)p.dv, (cuuint64_t)p.N, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t sv4[3] = {(cuuint64_t)p.sv[2] * 2, (cuuint64_t)p.sv[1] * 2,
                             (cuuint64_t)p.sv[0] * 2};
  const cuuint32_t bv[4] = {64, (cuuint32_t)kC, 1, 1};
  if (!tmap_encode(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, Kp, dq, sq, bq,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dv4, sv4, bv,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int grid = npieces * BH * (p.dv / kW);
  return launch_k(state_tc_kernel, dim3(grid), dim3(kNT), kSmem, st, true, p, tk, tv, meta, ksum,
                  piece_len, Part, zPart, need_z);
}

}  // namespace ret
