// Chunkwise retention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, per head and chunk of 64 tokens (hwhale.com/article/285883,
// chunkwise equation and ChunkwiseRetention; m0nads.wordpress.com,
// chunkwise representation):
//   O_[c] = (Q_[c] K_[c]^T (.) D) V_[c] + (Q_[c] S_c) (.) xi,  xi_i = gamma^(i+1)
//   S_{c+1} = gamma^L S_c + K_[c]^T (V_[c] (.) zeta),          zeta_j = gamma^(L-1-j)
// then the three normalisations and the per-head GroupNorm (+ swish gate).
//
// Operands.  The prologue writes Q' = xi (.) rot(q) and K' = zeta (.) rot(k)
// per chunk as fp16 times a power of two.  Then Q'_i . K'_j =
// gamma^(L+i-j) q_i . k_j, so the decay mask is the constant gamma^(-L) on
// the causal triangle, the cross term is Q' S_c and the state update K'^T V.
// Every MMA operand is fp16 (11-bit significand) with an exact power-of-two
// block scale chosen from a rigorous upper bound of its magnitude, so no
// operand can overflow: Q', K' per chunk (prologue), V per tile, and one
// joint exponent per chunk for R and the 16-bit copy of the state (the two
// share the O accumulator).  The fp32 state in TMEM carries its own power of
// two, folded into the per-chunk rescale it needs anyway (gamma^L).
//
// Work split.  One CTA per (batch, head, 128-wide slice of d_v); the d_v/128
// CTAs of a head form a cluster that exchanges GroupNorm statistics through
// distributed shared memory.  Everything is transposed so the v-slice is
// the MMA's M=128 dimension:
//   T   = Q' K'^T            (M=64 i, N=64 j, K=d_k)       -> TMEM (M=64 layout)
//   O^T = V^T R^T            (M=128 v, N=64 i, K=64 j)     -> TMEM
//   O^T += S^T Q'^T          (A = fp16 copy of S^T in TMEM, K=d_k)
//   S^T += V^T K'            (M=128 v, N=d_k, K=64 j)      -> TMEM fp32 state
//
// Warp roles (12 warps): warp 0 issues TMA loads (2-stage ring), warp 1
// issues MMAs (one thread) and owns TMEM, warps 2-3 ("helper" group)
// convert V to fp16, compute Q'.z for the third normalisation and carry z,
// warps 4-7 ("state" group) build R and the row factors, then refresh the
// state copy, warps 8-11 ("output" group) drain O^T and run GroupNorm and
// the stores.  The MMA order per chunk c is O^T = V^T R^T (once R is built),
// the scores of chunk c+1, then (once the state copy is refreshed) the cross
// term and the state update, so R of chunk c+1 is built while the state MMAs
// of chunk c run.  Every wait is bounded; a wait that runs out sets the
// status word and an abort flag, and every role leaves after draining its
// own asynchronous work.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "ktimer.h"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace cg = cooperative_groups;

namespace ret {

namespace {

constexpr int kC = 64;    // tokens per chunk
constexpr int kW = 128;   // value columns per CTA
constexpr int kNT = 384;  // threads per CTA

// Shared-memory map (offsets from a 1024-byte aligned base).
// Stage: Q' 32K | K' 32K | V 16K | key column sums (d_k fp32) | ChunkMeta.
constexpr uint32_t kOffQ = 0, kOffK = 32 * 1024, kOffV = 64 * 1024;
constexpr uint32_t kOffKs = 80 * 1024, kOffMeta = kOffKs + 1024;
constexpr uint32_t kStage = 82 * 1024;
constexpr uint32_t kOffR = 2 * kStage;                  // 64 x 128 B, fp16
constexpr uint32_t kOTPitch = 132;                      // floats per O^T row
constexpr uint32_t kOffOT = kOffR + 8 * 1024;           // [64][132] fp32
constexpr uint32_t kOffZ = kOffOT + 64 * kOTPitch * 4;  // [256] fp32
constexpr uint32_t kOffF = kOffZ + 256 * 4;             // [2][64] fp32 row factors
constexpr uint32_t kOffE = kOffF + 2 * 64 * 4;          // [2] int chunk exponents
constexpr uint32_t kOffRed = kOffE + 16;                // [2 groups][8] fp32 scratch
constexpr uint32_t kOffGN = kOffRed + 64;               // [2][8][64][2] fp32
constexpr uint32_t kOffNrm = kOffGN + 2 * 8 * 64 * 2 * 4;  // [64][2] fp32 shift, scale
constexpr uint32_t kOffVX = kOffNrm + 64 * 2 * 4;          // [2] int vx, [2] float max|V|
constexpr uint32_t kOffQZ = kOffVX + 16;                   // [2][64] fp32 Q'_i . z
constexpr uint32_t kOffHRed = kOffQZ + 2 * 64 * 4;         // [2][2] fp32 helper scratch
constexpr uint32_t kOffBar = kOffHRed + 16;
constexpr int kNumBars = 17;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

enum Bar {
  FULL0 = 0, FULL1, EMPTY0, EMPTY1, QK, RRDY, OFULL, SFULL, OFREE, GN0, GN1, DRAIN,
  VRDY0, VRDY1, QZRDY0, QZRDY1,  // per parity: the helper may run one chunk ahead
  SRDY
};

// TMEM column map.
constexpr uint32_t kTS = 0, kTSh = 256, kTO = 384, kTQK = 448;

constexpr uint32_t kBudget = 1u << 24;

struct TcArgs {
  const float *S_in, *z_in;
  float *S_out, *z_out;
  void *o;
  Gate gate;
  const ChunkMeta *meta;       // per (bh, chunk): exponents and magnitudes of Q', K'
  const float *ksum;           // per (bh, chunk) column sums of K' (d_k floats)
  // Sequence segments: segment k (blockIdx.x / (B H NV)) runs chunks
  // [k seg_len, (k+1) seg_len).  Its entry state is gamma^(64 c0) S_in plus
  // the pieces (piece_len whole chunks each, [piece][bh][d_k][d_v] fp32 and
  // [piece][bh][d_k]) that end at or before its first chunk, each decayed
  // from its end to c0.
  const float *Part, *zPart;
  int seg_len, piece_len;
  int NV;        // CTAs per head (d_v / 128)
  int need_z;    // carry z (third normalisation or z_out)
  int vec_out;   // o rows are 16-byte aligned: vector stores
};

// Named barrier among the n threads of group g (1 = state, 2 = output,
// 3 = helper).
__device__ __forceinline__ void grp_sync(int g, int n = 128) {
  asm volatile("bar.sync %0, %1;" ::"r"(g), "r"(n) : "memory");
}

// AND of `v` over the n threads of group g; also a barrier among them.
__device__ __forceinline__ bool grp_all(int g, bool v, int n = 128) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %2, 0;\n"
      " bar.red.and.pred q, %1, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(g), "r"((uint32_t)v), "r"(n)
      : "memory");
  return r != 0;
}

// Max of `v` over the 128 threads of group g.  `red` holds two 4-float
// slots used alternately (`slot` flips every call), so one barrier suffices:
// a slot is rewritten only after the next call's barrier, which every
// thread passes after reading it.
__device__ __forceinline__ float grp_max(int g, float v, float *red, int &slot, int et) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  float *r = red + 4 * slot;
  slot ^= 1;
  if ((et & 31) == 0) r[et >> 5] = v;
  grp_sync(g);
  return fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                         unsigned *status) {
  for (uint32_t i = 0; i < kBudget; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity,
                                                 volatile int *abort_p, unsigned *status) {
  for (uint32_t i = 0; i < kBudget; ++i) {
    if (tc::mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

// Wait used only while draining: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kBudget; ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

// e such that m * 2^-e < 2^14 (0 for m = 0).
__device__ __forceinline__ int expo14(float m) {
  int e = 0;
  if (m > 0.f && m < INFINITY) {
    frexpf(m, &e);
    e -= 14;
  }
  return e;
}

__device__ __forceinline__ float2 h2f(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

__global__ void __launch_bounds__(kNT, 1)
chunk_tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const TcArgs a) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = tc::smem_align1024(smraw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tbase_p = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort_p = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  float *zsm = reinterpret_cast<float *>(sm + kOffZ);
  float *fsm = reinterpret_cast<float *>(sm + kOffF);
  int *Esm = reinterpret_cast<int *>(sm + kOffE);
  float *red = reinterpret_cast<float *>(sm + kOffRed);
  float *OT = reinterpret_cast<float *>(sm + kOffOT);
  float *gns = reinterpret_cast<float *>(sm + kOffGN);
  float *nrm = reinterpret_cast<float *>(sm + kOffNrm);
  int *vxs = reinterpret_cast<int *>(sm + kOffVX);
  float *vmxs = reinterpret_cast<float *>(sm + kOffVX + 8);
  float *qzs = reinterpret_cast<float *>(sm + kOffQZ);
  float *hred = reinterpret_cast<float *>(sm + kOffHRed);

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NV = a.NV;
  const int rank = (int)cluster.block_rank();
  const int BHNV = p.B * p.H * NV;
  const int seg = blockIdx.x / BHNV;
  const int bh = (blockIdx.x % BHNV) / NV, b = bh / p.H, h = bh % p.H;
  const int v0 = rank * kW;
  const int DK = p.dk, NKB = DK / 64, N = p.N;
  const int nch = (N + kC - 1) / kC;
  // This CTA's chunks: global c = c0 + lc; barrier phases follow lc.
  const int c0 = seg * a.seg_len;
  const int ncl = min(nch, c0 + a.seg_len) - c0;
  const bool last_seg = c0 + ncl >= nch;
  const int npc = seg > 0 ? c0 / a.piece_len : 0;  // pieces before c0
  const float lng = p.lng[h];

  if (tid == 0) {
    tc::mbar_init(&bars[FULL0], 1);
    tc::mbar_init(&bars[FULL1], 1);
    tc::mbar_init(&bars[EMPTY0], 2);
    tc::mbar_init(&bars[EMPTY1], 2);
    tc::mbar_init(&bars[QK], 1);
    tc::mbar_init(&bars[RRDY], 1);
    tc::mbar_init(&bars[SRDY], 1);
    tc::mbar_init(&bars[OFULL], 1);
    tc::mbar_init(&bars[SFULL], 1);
    tc::mbar_init(&bars[OFREE], 1);
    tc::mbar_init(&bars[GN0], 1);
    tc::mbar_init(&bars[GN1], 1);
    tc::mbar_init(&bars[DRAIN], 1);
    tc::mbar_init(&bars[VRDY0], 1);
    tc::mbar_init(&bars[VRDY1], 1);
    tc::mbar_init(&bars[QZRDY0], 1);
    tc::mbar_init(&bars[QZRDY1], 1);
    *abort_p = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase_p, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  cluster.sync();  // every CTA's barriers exist before any remote arrive
  tc::tc_fence_after();
  const uint32_t tb = *tbase_p;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      const uint32_t bytes = (uint32_t)NKB * 8192u * 2u + 16384u + 16u +
                             (a.need_z ? (uint32_t)DK * 4u : 0u);
      int issued = 0;
      for (int lc = 0; lc < ncl; ++lc) {
        const int s = lc & 1, c = c0 + lc;
        if (lc >= 2 && !wait_bar(&bars[EMPTY0 + s], ((lc >> 1) - 1) & 1, abort_p, p.status)) break;
        uint8_t *st = sm + s * kStage;
        tc::mbar_arrive_expect_tx(&bars[FULL0 + s], bytes);
        for (int kb = 0; kb < NKB; ++kb)
          tc::tma_load_3d(st + kOffQ + kb * 8192, &tmQ, &bars[FULL0 + s], kb * 64, c * kC, bh);
        for (int kb = 0; kb < NKB; ++kb)
          tc::tma_load_3d(st + kOffK + kb * 8192, &tmK, &bars[FULL0 + s], kb * 64, c * kC, bh);
        for (int vb = 0; vb < 2; ++vb)
          tc::tma_load_4d(st + kOffV + vb * 8192, &tmV, &bars[FULL0 + s], v0 + vb * 64, c * kC,
                          h, b);
        tc::bulk_load(st + kOffMeta, a.meta + (long long)bh * nch + c, 16u, &bars[FULL0 + s]);
        if (a.need_z)
          tc::bulk_load(st + kOffKs, a.ksum + ((long long)bh * nch + c) * DK, (uint32_t)DK * 4u,
                        &bars[FULL0 + s]);
        ++issued;
      }
      // Let every issued copy land before the CTA can leave.
      for (int lc = issued > 2 ? issued - 2 : 0; lc < issued; ++lc)
        drain_wait(&bars[FULL0 + (lc & 1)], (lc >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16(64, 64, 0, 0);
      const uint32_t id_o = tc::idesc_f16(128, 64, 1, 0);
      const uint32_t id_x = tc::idesc_f16(128, 64, 0, 0);
      const uint32_t id_s = tc::idesc_f16(128, DK, 1, 1);
      const uint32_t sr = tc::smem_u32(sm + kOffR);
      auto mma_qk = [&](int lc) {  // T = Q' K'^T
        const uint32_t sq = tc::smem_u32(sm + (lc & 1) * kStage + kOffQ), sk = sq + kOffK;
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
          tc::mma_ss(tb + kTQK, tc::smem_desc(sq + off, 16, 1024, tc::kSw128),
                     tc::smem_desc(sk + off, 16, 1024, tc::kSw128), id_qk, ks > 0);
        }
        tc::mma_commit(&bars[QK]);
      };
      bool go = ncl > 0 && wait_bar(&bars[FULL0], 0, abort_p, p.status);
      if (go) {
        tc::tc_fence_after();
        mma_qk(0);
      }
      // Per chunk: O^T = V^T R^T once R is built and O^T of the previous
      // chunk is drained; then the next chunk's scores, so the state group
      // can build the next R while this chunk's state MMAs run; then, once
      // the state copy is refreshed, the cross term and the state update.
      for (int lc = 0; go && lc < ncl; ++lc) {
        const int s = lc & 1;
        const uint32_t sq = tc::smem_u32(sm + s * kStage + kOffQ);
        const uint32_t sk = sq + kOffK, sv = sq + kOffV;
        if (!wait_bar(&bars[RRDY], lc & 1, abort_p, p.status)) break;
        if (lc > 0 && !wait_bar(&bars[OFREE], (lc - 1) & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        for (int ks = 0; ks < 4; ++ks)  // O^T = V^T R^T
          tc::mma_ss(tb + kTO, tc::smem_desc(sv + ks * 2048, 8192, 1024, tc::kSw128),
                     tc::smem_desc(sr + ks * 32, 16, 1024, tc::kSw128), id_o, ks > 0);
        if (lc + 1 < ncl) {
          if (!wait_bar(&bars[FULL0 + (s ^ 1)], ((lc + 1) >> 1) & 1, abort_p, p.status)) break;
          tc::tc_fence_after();
          mma_qk(lc + 1);
        }
        if (!wait_bar(&bars[SRDY], lc & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        for (int ks = 0; ks < DK / 16; ++ks)  // O^T += S^T Q'^T
          tc::mma_ts(tb + kTO, tb + kTSh + ks * 8,
                     tc::smem_desc(sq + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, tc::kSw128),
                     id_x, 1);
        tc::mma_commit(&bars[OFULL]);
        for (int ks = 0; ks < 4; ++ks)  // S^T += V^T K'
          tc::mma_ss(tb + kTS, tc::smem_desc(sv + ks * 2048, 8192, 1024, tc::kSw128),
                     tc::smem_desc(sk + ks * 2048, 8192, 1024, tc::kSw128), id_s, 1);
        tc::mma_commit(&bars[SFULL]);
        tc::mma_commit(&bars[EMPTY0 + s]);
      }
      tc::mma_commit(&bars[DRAIN]);  // every MMA issued above is finished
      drain_wait(&bars[DRAIN], 0);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ helper group
    const int G = 3, NT = 64;
    const int ht = tid - 64;  // 0..63
    const bool rsum = (p.norm_flags & RET_NORM_RSUM) != 0;
    int hslot = 0;
    bool ok = true;
    if (a.need_z)
      for (int k2 = ht; k2 < DK; k2 += NT) {
        float z = a.z_in ? a.z_in[(long long)bh * DK + k2] : 0.f;
        if (seg > 0) {  // entry z of a later segment
          z *= gpow(lng, kC * c0);
          for (int i = 0; i < npc; ++i)
            z = fmaf(gpow(lng, kC * (c0 - (i + 1) * a.piece_len)),
                     a.zPart[((long long)i * p.B * p.H + bh) * DK + k2], z);
        }
        zsm[k2] = z;
      }
    grp_sync(G, NT);
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      uint8_t *st = sm + s * kStage;
      ok = grp_all(G, wait_bar(&bars[FULL0 + s], (lc >> 1) & 1, abort_p, p.status), NT);
      if (!ok) break;
      // (1) V tile: bf16 -> fp16 * 2^-vx in place (1024 16-byte words).
      uint4 vv[16];
      float vm = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        vv[u] = reinterpret_cast<const uint4 *>(st + kOffV)[ht + NT * u];
        const uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) vm = fmaxf(vm, fmaxf(fabsf(bf_lo(w[e])), fabsf(bf_hi(w[e]))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      float *hr = hred + 2 * hslot;
      hslot ^= 1;
      if ((ht & 31) == 0) hr[ht >> 5] = vm;
      grp_sync(G, NT);
      const float vmx = fmaxf(hr[0], hr[1]);
      const int vx = expo14(vmx);
      const float vsc = exp2f((float)-vx);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o4[e] = tc::pack_f16(bf_lo(w[e]) * vsc, bf_hi(w[e]) * vsc);
        reinterpret_cast<uint4 *>(st + kOffV)[ht + NT * u] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (ht == 0) {
        vxs[s] = vx;
        vmxs[s] = vmx;
      }
      tc::fence_proxy_async_smem();
      grp_sync(G, NT);
      if (ht == 0) tc::mbar_arrive(&bars[VRDY0 + s]);
      // (2) Q'_i . z_c for the row sums of the third normalisation.
      if (rsum) {
        const int i = ht;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const uint4 u =
                *reinterpret_cast<const uint4 *>(st + kOffQ + kb * 8192 + tc::sw128_off(i, cc));
            const float4 z0 = *reinterpret_cast<const float4 *>(zsm + kb * 64 + cc * 8);
            const float4 z1 = *reinterpret_cast<const float4 *>(zsm + kb * 64 + cc * 8 + 4);
            const float2 a0 = h2f(u.x), a1 = h2f(u.y), a2 = h2f(u.z), a3 = h2f(u.w);
            acc[0] = fmaf(a0.x, z0.x, fmaf(a0.y, z0.y, acc[0]));
            acc[1] = fmaf(a1.x, z0.z, fmaf(a1.y, z0.w, acc[1]));
            acc[2] = fmaf(a2.x, z1.x, fmaf(a2.y, z1.y, acc[2]));
            acc[3] = fmaf(a3.x, z1.z, fmaf(a3.y, z1.w, acc[3]));
          }
        qzs[s * 64 + i] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) *
                          exp2f((float)reinterpret_cast<const ChunkMeta *>(st + kOffMeta)->qexp);
        grp_sync(G, NT);
        if (ht == 0) tc::mbar_arrive(&bars[QZRDY0 + s]);
      }
      // (3) z_{c+1} = gamma^L z_c + sum_j K'_j (column sums from the prologue).
      if (a.need_z) {
        const int L = min(kC, N - c * kC);
        const float gL = gpow(lng, L);
        const float *ks = reinterpret_cast<const float *>(st + kOffKs);
        for (int k2 = ht; k2 < DK; k2 += NT) zsm[k2] = fmaf(gL, zsm[k2], ks[k2]);
      }
      grp_sync(G, NT);
      if (ht == 0) tc::mbar_arrive(&bars[EMPTY0 + s]);
    }
    if (ok && a.z_out && rank == 0 && last_seg)
      for (int k2 = ht; k2 < DK; k2 += NT) a.z_out[(long long)bh * DK + k2] = zsm[k2];
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ state group
    const int G = 1;
    const int q = warp & 3;                 // TMEM lane quarter
    const int et = tid - 128;               // 0..127
    const int vrow = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const long long vglob = v0 + vrow;
    const bool rsum = (p.norm_flags & RET_NORM_RSUM) != 0;
    float *rd = red;
    int rslot = 0;
    bool ok = true;
    // Entry state (S_in, or for a later segment the decayed sum of S_in and
    // the pieces before it) goes to the TMEM state columns; s_bound = max |S|.
    const bool has_state = a.S_in != nullptr || npc > 0;
    float m0 = 0.f;
    if (has_state) {
      const float w_in = seg > 0 ? gpow(lng, kC * c0) : 1.f;
      for (int g = 0; g < DK / 32; ++g) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const long long e = ((long long)bh * DK + g * 32 + i) * p.dv + vglob;
          r[i] = __float_as_uint(a.S_in ? w_in * a.S_in[e] : 0.f);
        }
        for (int pi = 0; pi < npc; ++pi) {
          const float w = gpow(lng, kC * (c0 - (pi + 1) * a.piece_len));
          const float *src = a.Part + (long long)pi * p.B * p.H * DK * p.dv;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const long long e = ((long long)bh * DK + g * 32 + i) * p.dv + vglob;
            r[i] = __float_as_uint(fmaf(w, src[e], __uint_as_float(r[i])));
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) m0 = fmaxf(m0, fabsf(__uint_as_float(r[i])));
        tc::tmem_st32(tb + lb + kTS + g * 32, r);
      }
      tc::tmem_st_wait();
    }
    float s_bound = grp_max(G, m0, rd, rslot, et);
    int sigma = 0;  // TMEM state holds S * 2^-sigma
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      const float gL = gpow(lng, L);
      const float ginvL = expf(-(float)L * lng);
      ok = grp_all(G, wait_bar(&bars[VRDY0 + s], (lc >> 1) & 1, abort_p, p.status));
      if (!ok) break;
      const ChunkMeta mt = *reinterpret_cast<const ChunkMeta *>(sm + s * kStage + kOffMeta);
      const int aq = mt.qexp, bk = mt.kexp;
      const float qmx = mt.qmax, kmx = mt.kmax;
      const int vx = vxs[s];
      const float vmx = vmxs[s];
      // (2) exponents: R and the state copy share the O accumulator's scale.
      // |R_ij| = gamma^(i-j) |q_i . k_j| <= (d_k/2) max|pair of rot q| max|pair of rot k|
      // (j <= i; a dot product is a sum of d_k/2 pair products).
      const int rr_nat = expo14((float)(DK / 2) * qmx * kmx);
      int E = rr_nat + vx;
      if (s_bound > 0.f) E = max(E, expo14(s_bound) + aq);
      const int rr = E - vx, ss = E - aq;
      const int sigma_next = vx + bk;
      // (3) R (fp16, * 2^-rr) as K-major rows; row factors.  The scores'
      // completion (QK) means every earlier MMA is finished: MMA2 of the
      // previous chunk, the last reader of R, and, through MMA2's wait on
      // OFREE two chunks back, the output group's reads of slot s.
      ok = grp_all(G, wait_bar(&bars[QK], lc & 1, abort_p, p.status) &&
                          (!rsum || wait_bar(&bars[QZRDY0 + s], (lc >> 1) & 1, abort_p, p.status)));
      if (!ok) break;
      tc::tc_fence_after();
      if (et == 0) Esm[s] = E;
      {
        uint32_t t0[32], t1[32];
        tc::tmem_ld32(tb + lb + kTQK, t0);
        tc::tmem_ld32(tb + lb + kTQK + 32, t1);
        tc::tmem_ld_wait();
        if (lane < 16) {
          const int i = q * 16 + lane;  // M=64 accumulator: row i in lane 32(i/16) + i%16
          const float tsc = exp2f((float)(aq + bk)) * ginvL;
          const float rsc = exp2f((float)-rr);
          float rs = 0.f;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = cc * 8 + 2 * e;
              const float x0 = __uint_as_float(j < 32 ? t0[j] : t1[j - 32]);
              const float x1 = __uint_as_float(j + 1 < 32 ? t0[j + 1] : t1[j + 1 - 32]);
              const float r0 = (j <= i && i < L) ? x0 * tsc : 0.f;
              const float r1 = (j + 1 <= i && i < L) ? x1 * tsc : 0.f;
              rs += r0 + r1;
              w[e] = tc::pack_f16(r0 * rsc, r1 * rsc);
            }
            *reinterpret_cast<uint4 *>(sm + kOffR + tc::sw128_off(i, cc)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          float f = 0.f;
          if (i < L) {
            if (rsum) rs += qzs[s * 64 + i];
            const float sn = row_scale(p, h, p.pos0 + (long long)c * kC + i + 1);
            f = sn * rsum_scale(p, sn * rs);
          }
          fsm[s * 64 + i] = f;
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[RRDY]);
      // (4) state pass: fp16 copy of S_c * 2^-ss; S_acc <- gamma^L S_c * 2^-sigma_next
      if (lc > 0) {
        ok = grp_all(G, wait_bar(&bars[SFULL], (lc - 1) & 1, abort_p, p.status));
        if (!ok) break;
        tc::tc_fence_after();
      }
      {
        const float f_cp = exp2f((float)(sigma - ss));
        const float f_pre = gL * exp2f((float)(sigma - sigma_next));
        for (int g0 = 0; g0 < DK / 32; g0 += 2) {
          uint32_t r[2][32];
          if (lc == 0 && !has_state) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int i = 0; i < 32; ++i) r[hh][i] = 0u;
          } else {
            tc::tmem_ld32(tb + lb + kTS + g0 * 32, r[0]);
            tc::tmem_ld32(tb + lb + kTS + g0 * 32 + 32, r[1]);
            tc::tmem_ld_wait();
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float x0 = __uint_as_float(r[hh][2 * i]), x1 = __uint_as_float(r[hh][2 * i + 1]);
              pk[i] = tc::pack_f16(x0 * f_cp, x1 * f_cp);
            }
            tc::tmem_st16(tb + lb + kTSh + (g0 + hh) * 16, pk);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[hh][i] = __float_as_uint(__uint_as_float(r[hh][i]) * f_pre);
            tc::tmem_st32(tb + lb + kTS + (g0 + hh) * 32, r[hh]);
          }
        }
        tc::tmem_st_wait();
      }
      tc::tc_fence_before();
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[SRDY]);
      // Upper bound of max |S_{c+1}|: |S_{c+1}| <= gamma^L |S_c| + sum_j |K'_j||V_j|
      // with zeta <= 1 (a pair norm bounds each component of its pair).  It is
      // loose by the ratio of a sum of L terms to their random-sign size,
      // which costs nothing in floating point.
      s_bound = gL * s_bound + (float)L * kmx * vmx;
      sigma = sigma_next;
    }
    if (ok && a.S_out && last_seg) {
      ok = grp_all(G, wait_bar(&bars[SFULL], (ncl - 1) & 1, abort_p, p.status));
      if (ok) {
        tc::tc_fence_after();
        const float back = exp2f((float)sigma);
        for (int g = 0; g < DK / 32; ++g) {
          uint32_t r[32];
          tc::tmem_ld32(tb + lb + kTS + g * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            a.S_out[((long long)bh * DK + g * 32 + i) * p.dv + vglob] = __uint_as_float(r[i]) * back;
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ output group
    const int G = 2;
    const int q = warp & 3;
    const int et = tid - 256;  // 0..127
    const int vrow = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const bool gn = p.gn_eps >= 0.f;
    // Statistics: 4 threads per token, interleaved columns (conflict-free
    // with a row pitch of 132 floats); 32 tokens per pass, two passes.
    const int sq4 = et & 3, st0 = et >> 2;
    bool ok = true;
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      ok = grp_all(G, wait_bar(&bars[OFULL], lc & 1, abort_p, p.status));
      if (!ok) break;
      tc::tc_fence_after();
      const float osc = exp2f((float)Esm[s]);
      float fr[2];
      fr[0] = fsm[s * 64 + st0];
      fr[1] = fsm[s * 64 + st0 + 32];
      {
        uint32_t t0[32], t1[32];
        tc::tmem_ld32(tb + lb + kTO, t0);
        tc::tmem_ld32(tb + lb + kTO + 32, t1);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          OT[i * kOTPitch + vrow] = __uint_as_float(t0[i]);
          OT[(32 + i) * kOTPitch + vrow] = __uint_as_float(t1[i]);
        }
      }
      tc::tc_fence_before();
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[OFREE]);
      float mloc[2], M2loc[2];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const float *row = OT + (st0 + 32 * pass) * kOTPitch + sq4;
        float sm0 = 0.f, sm1 = 0.f;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          sm0 += row[4 * e];
          sm1 += row[4 * e + 4];
        }
        float m = sm0 + sm1;
        m += __shfl_xor_sync(0xffffffffu, m, 1);
        m += __shfl_xor_sync(0xffffffffu, m, 2);
        m *= (1.f / kW);
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float d0 = row[4 * e] - m, d1 = row[4 * e + 4] - m;
          q0 = fmaf(d0, d0, q0);
          q1 = fmaf(d1, d1, q1);
        }
        float M2 = q0 + q1;
        M2 += __shfl_xor_sync(0xffffffffu, M2, 1);
        M2 += __shfl_xor_sync(0xffffffffu, M2, 2);
        mloc[pass] = m * osc;  // O^T holds O * 2^-E; osc = 2^E
        M2loc[pass] = M2 * osc * osc;
      }
      float mean[2] = {mloc[0], mloc[1]};
      float var[2] = {M2loc[0] * (1.f / kW), M2loc[1] * (1.f / kW)};
      if (gn && NV > 1) {
        // Every CTA of the head sends its per-token (mean, M2) to every CTA;
        // each copy completes 8 bytes on the receiver's barrier, which
        // expects NV*64*8 bytes for this chunk.
        const int par = lc & 1;
        if (et == 0) tc::mbar_arrive_expect_tx(&bars[GN0 + par], (uint32_t)(NV * 64 * 8));
        if (sq4 == 0)
#pragma unroll
          for (int pass = 0; pass < 2; ++pass) {
            const float *slot = gns + ((par * 8 + rank) * 64 + st0 + 32 * pass) * 2;
            for (int r2 = 0; r2 < NV; ++r2)
              tc::st_async_v2(slot, &bars[GN0 + par], r2, mloc[pass], M2loc[pass]);
          }
        ok = grp_all(G, wait_bar_cluster(&bars[GN0 + par], (lc >> 1) & 1, abort_p, p.status));
        if (!ok) break;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const int ti = st0 + 32 * pass;
          float msum = 0.f;
          for (int r2 = 0; r2 < NV; ++r2) msum += gns[((par * 8 + r2) * 64 + ti) * 2];
          const float mu = msum / NV;
          float M2t = 0.f;
          for (int r2 = 0; r2 < NV; ++r2) {
            const float *sl = gns + ((par * 8 + r2) * 64 + ti) * 2;
            const float d = sl[0] - mu;
            M2t += sl[1] + (float)kW * d * d;
          }
          mean[pass] = mu;
          var[pass] = M2t / (float)(kW * NV);
        }
      }
      // GroupNorm of x = f o: y = (o - mean) f / sqrt(f^2 var + eps); no
      // GroupNorm: y = f o.
      // Stored O^T is O * 2^-E: fold 2^E into the per-token shift and scale.
      if (sq4 == 0)
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const float f = fr[pass];
          nrm[(st0 + 32 * pass) * 2] = gn ? mean[pass] / osc : 0.f;
          nrm[(st0 + 32 * pass) * 2 + 1] =
              (gn ? f * rsqrtf(f * f * var[pass] + p.gn_eps) : f) * osc;
        }
      grp_sync(G);
      // Stores: warp q writes token rows 2q + 8k and 2q + 8k + 1; half-warp
      // per row, 8 columns per lane (one 16-byte bf16 store).
      {
        const int rsel = lane >> 4, col = 8 * (lane & 15);
        const long long rstride = 8 * p.so[2];
        long long ob = b * p.so[0] + h * p.so[1] + ((long long)c * kC + 2 * q + rsel) * p.so[2] +
                       v0 + col;
        long long gb = b * a.gate.s[0] + h * a.gate.s[1] +
                       ((long long)c * kC + 2 * q + rsel) * a.gate.s[2] + v0 + col;
#pragma unroll 2
        for (int it = 0; it < 8; ++it, ob += rstride, gb += 8 * a.gate.s[2]) {
          const int ti = 2 * q + 8 * it + rsel;
          if (ti < L) {
            const float shift = nrm[ti * 2], scale = nrm[ti * 2 + 1];
            const float4 x0 = *reinterpret_cast<const float4 *>(OT + ti * kOTPitch + col);
            const float4 x1 = *reinterpret_cast<const float4 *>(OT + ti * kOTPitch + col + 4);
            float y[8] = {(x0.x - shift) * scale, (x0.y - shift) * scale, (x0.z - shift) * scale,
                          (x0.w - shift) * scale, (x1.x - shift) * scale, (x1.y - shift) * scale,
                          (x1.z - shift) * scale, (x1.w - shift) * scale};
            if (a.gate.ptr) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float g = ld_elem(a.gate.ptr, gb + e, 1);
                y[e] *= g / (1.f + expf(-g));
              }
            }
            if (a.vec_out && p.out_bf16) {
              *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.o) + ob) =
                  make_uint4(tc::pack_bf16(y[0], y[1]), tc::pack_bf16(y[2], y[3]),
                             tc::pack_bf16(y[4], y[5]), tc::pack_bf16(y[6], y[7]));
            } else if (a.vec_out) {
              float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + ob);
              dst[0] = make_float4(y[0], y[1], y[2], y[3]);
              dst[1] = make_float4(y[4], y[5], y[6], y[7]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) st_elem(a.o, ob + e, y[e], p.out_bf16);
            }
          }
        }
      }
      grp_sync(G);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  cluster.sync();  // no CTA leaves while a peer may still write to it
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

// ------------------------------------------------------------------ host
bool chunk_tc_supported(const KParams &p, const void *v, const long long sv[3]) {
  if (!p.in_bf16 || p.chunk != kC) return false;
  if (p.dk % 64 || p.dk < 64 || p.dk > 256) return false;
  if (p.dv % kW || p.dv / kW > 8) return false;
  if (reinterpret_cast<uintptr_t>(v) & 15) return false;
  for (int i = 0; i < 3; ++i)
    if (sv[i] % 8) return false;
  // Folding the decays into fp16 rows spans gamma^(L-1) inside one chunk:
  // keep it within fp16's normal range (gamma^64 >= 2^-16, gamma >= 0.841).
  for (int h = 0; h < p.H; ++h)
    if (!(p.lng[h] * kC >= -16.f * 0.69314718f)) return false;
  return tmap_available();
}

cudaError_t launch_chunk_tc(const KParams &p, const void *Qp, const void *Kp, const void *v,
                            const ChunkMeta *meta, const float *ksum, const float *S_in,
                            const float *z_in, float *S_out, float *z_out, void *o, Gate gate,
                            int need_z, const SegPlan &seg, cudaStream_t st) {
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv;
  const cuuint64_t dq[3] = {(cuuint64_t)p.dk, (cuuint64_t)p.N, (cuuint64_t)BH};
  const cuuint64_t sq[2] = {(cuuint64_t)p.dk * 2, (cuuint64_t)p.N * p.dk * 2};
  const cuuint32_t bq[3] = {64, (cuuint32_t)kC, 1};
  const cuuint64_t dv4[4] = {(cuuint64_t)p.dv, (cuuint64_t)p.N, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t sv4[3] = {(cuuint64_t)p.sv[2] * 2, (cuuint64_t)p.sv[1] * 2,
                             (cuuint64_t)p.sv[0] * 2};
  const cuuint32_t bv[4] = {64, (cuuint32_t)kC, 1, 1};
  if (!tmap_encode(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, Qp, dq, sq, bq,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, Kp, dq, sq, bq,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dv4, sv4, bv,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.S_in = S_in;
  a.z_in = z_in;
  a.S_out = S_out;
  a.z_out = z_out;
  a.o = o;
  a.gate = gate;
  a.meta = meta;
  a.ksum = ksum;
  a.NV = p.dv / kW;
  a.need_z = need_z;
  const int nch = (p.N + kC - 1) / kC;
  a.seg_len = seg.P > 1 ? seg.seg_len : nch;
  a.piece_len = seg.P > 1 ? seg.piece_len : 1;
  a.Part = seg.Part;
  a.zPart = seg.zPart;
  const int P = seg.P > 1 ? seg.P : 1;
  // Row-vector stores: 8 columns per lane (16 bytes bf16, 2 x 16 bytes fp32).
  const int al = p.out_bf16 ? 8 : 4;  // elements per aligned vector
  const uintptr_t abytes = 16;
  a.vec_out = (reinterpret_cast<uintptr_t>(o) % abytes == 0) && p.so[0] % al == 0 &&
              p.so[1] % al == 0 && p.so[2] % al == 0;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P * BH * a.NV));
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.NV;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_tc_kernel, p, tq, tk, tv, a);
}

}  // namespace ret
