// Parallel form of retention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, per head (hwhale.com/article/285883, parallel form
// Retention(X) = (Q K^T (.) D) V with D_nm = gamma^(n-m) for n >= m, else 0;
// ParallelRetention), the raw rows O_n = sum_{m<=n} (q'_n . k'_m) gamma^(n-m) v_m
// and their sums r_n = sum_{m<=n} (q'_n . k'_m) gamma^(n-m), from which the
// row factor of the three normalisations follows.  Where one CTA holds a
// whole row (d_v <= 256) it also applies GroupNorm and writes the output;
// otherwise a GroupNorm pass does, from the raw rows.  The full causal score
// matrix is walked block by block, 128 queries against KT = 128 keys at a
// time (64 when d_k = 256, whose operands leave no room for two 128-key
// stages), without the recurrent state.
//
// Operands.  The chunkwise path's prologue writes Q' = xi (.) rot(q) and
// K' = zeta (.) rot(k) per 64-token chunk (xi_i = gamma^(i+1), zeta_j =
// gamma^(L-1-j)) as fp16 times a power of two, and the chunk's exponents and
// magnitude bounds.  For query chunk cq and key chunk ck,
//   Q'_i . K'_j = rot(q_n) . rot(k_m) gamma^(i+1+L-1-j) 2^-(qexp+kexp),
// so the block's scores times g = gamma^(64 (cq-ck) - L) 2^(qexp+kexp) carry
// the exact decay gamma^(n-m); one factor per (row, key block).  The scaled
// scores P~ = P 2^-E go to TMEM as bf16 (the A operand of O += P~ V, V in
// bf16 as the caller stores it), with E per CTA from the rigorous bound
// |P_nm| <= (d_k/2) max pair norm of q' * max pair norm of k' (the
// prologue's magnitudes), so P~ < 2^15 whatever the inputs' scale.
//
// Work split.  One CTA per (batch, head, 128 queries, W value columns), W =
// 256 or 128; the heaviest query blocks (most key blocks) are launched
// first.  TMEM: KT-column score buffers (two for KT = 128, three for 64;
// each reused for its bf16 P~ in place) and the O accumulator (W columns,
// 128 lanes = queries).
//   S   = Q' K'^T     (M=128 queries, N=KT keys, K=d_k; fp16)  -> TMEM
//   O  += P~ V        (M=128 queries, N=W, K=KT keys; A = P~ in TMEM, bf16)
// One thread issues every MMA, and an MMA takes about as long to issue as
// a 128x256x16 one takes to run, so wide key blocks (fewer, larger score
// MMAs) are what keeps the tensor pipe busy.
// Warp roles (12 warps): warp 0 TMA (Q' once, then K' and V per key block in
// a ring), warp 1 MMA issue, warps 4-7 and 8-11 two converter groups taking
// alternate key blocks (scores -> P~, one query row per thread; the time of
// one block's TMEM round trips overlaps the other's), the first of them also
// the final drain of O.  Every wait is bounded; a wait that runs
// out sets the status word and an abort flag, and each role leaves after
// draining its own asynchronous work.
#include <cudaTypedefs.h>

#include "ktimer.h"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace ret {

namespace {

constexpr int kPQ = 128;         // queries per CTA
constexpr int kPK = 64;          // tokens per prologue chunk
constexpr int kPThreads = 384;
constexpr int kPMaxStages = 4;
constexpr uint32_t kPSmemLimit = 232448;
constexpr uint32_t kPSpin = 1u << 24;  // polls without progress before a role gives up

constexpr int kPSB = 3;          // score buffers in TMEM, at most

enum PBar {
  PB_FULLQ = 0,
  PB_FULLK = 1,
  PB_EMPTYK = PB_FULLK + kPMaxStages,
  PB_FULLV = PB_EMPTYK + kPMaxStages,
  PB_EMPTYV = PB_FULLV + kPMaxStages,
  PB_SFULL = PB_EMPTYV + kPMaxStages,
  PB_PRDY = PB_SFULL + kPSB,
  PB_PVDONE = PB_PRDY + kPSB,
  PB_ODONE = PB_PVDONE + kPSB,
  PB_DRAIN,
  PB_COUNT
};

struct ParArgs {
  const ChunkMeta *meta;  // per (bh, chunk): exponents and magnitudes of Q', K'
  float *Oraw;            // [B*H][N][d_v] raw rows (NVS > 1)
  float *F;               // [B*H][N] row factors (NVS > 1)
  void *o;                // the output (NVS == 1: GroupNorm in this kernel)
  int W, NVS, nst;        // value columns per CTA, CTAs per head, ring stages
  int vec_out;            // o rows 16-byte aligned: vector stores
  uint32_t off_k, kstage;  // K' ring: offset, bytes per stage
  uint32_t off_v, vstage;  // V ring
  uint32_t off_bar, tmem_cols;
};

// Bounded wait that also gives up once another role has aborted.
__device__ __noinline__ bool par_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                           unsigned *status) {
  for (uint32_t i = 0; i < (1u << 20); ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

__device__ __forceinline__ bool par_wait(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                         unsigned *status) {
  return tc::mbar_try_wait(bar, parity) || par_wait_slow(bar, parity, abort_p, status);
}

// Wait used only while draining: ignores the abort flag, still bounded.
__device__ __forceinline__ void par_drain(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
}

// K-step ks (16 elements) of a K-major SW128 operand stored in blocks of
// `rows` rows x 64 elements, in the descriptor's 16-byte units.
__device__ __forceinline__ uint64_t kstep(int ks, uint32_t rows) {
  return (uint64_t)(((uint32_t)(ks >> 2) * rows * 128u + (uint32_t)(ks & 3) * 32u) >> 4);
}

}  // namespace

template <int KT>
__global__ void __launch_bounds__(kPThreads, 1)
parallel_tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ ParArgs a) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = tc::smem_align1024(smraw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.off_bar);
  uint32_t *tbase_p = reinterpret_cast<uint32_t *>(sm + a.off_bar + PB_COUNT * 8);
  volatile int *abort_p = reinterpret_cast<volatile int *>(sm + a.off_bar + PB_COUNT * 8 + 4);
  float *red = reinterpret_cast<float *>(sm + a.off_bar + PB_COUNT * 8 + 16);  // [2][8]
  float *rsx = reinterpret_cast<float *>(sm + a.off_bar + PB_COUNT * 8 + 80);  // [128]

  constexpr int NSB = KT == 128 ? 2 : 3;  // score buffers
  constexpr int CPT = KT / kPK;            // prologue chunks per key block
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H, N = p.N, DK = p.dk, NKB = DK / 64, W = a.W, NVB = W / 64;
  const int nch = (N + kPK - 1) / kPK, nqt = (N + kPQ - 1) / kPQ;
  const int per_qt = BH * a.NVS;
  const int qt = nqt - 1 - (int)(blockIdx.x / per_qt);
  const int rem = (int)(blockIdx.x % per_qt);
  const int bh = rem / a.NVS, vs = rem % a.NVS, b = bh / p.H, h = bh % p.H;
  const int q0 = qt * kPQ, v0 = vs * W;
  const int nkc = min(2 * qt + 2, nch);  // key chunks up to the diagonal
  const int nkt = (nkc + CPT - 1) / CPT;  // key blocks
  const int nst = a.nst;

  if (tid == 0) {
    for (int i = 0; i < PB_COUNT; ++i)
      tc::mbar_init(&bars[i], (i >= PB_PRDY && i < PB_PRDY + NSB) ? 128 : 1);
    *abort_p = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase_p, a.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = *tbase_p;
  const uint32_t tO = tb + NSB * KT;  // O accumulator after the score buffers
  pdl_wait();  // global memory only once the kernel before this one is complete

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    // K' and V of a key block come in separate rings: K' is free once the
    // scores are done, V once O += P~ V is, so each refills as early as it
    // can.  One thread issues both, whichever has a free stage.
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      tc::mbar_arrive_expect_tx(&bars[PB_FULLQ], (uint32_t)NKB * kPQ * 128u);
      for (int kb = 0; kb < NKB; ++kb)
        tc::tma_load_3d(sm + kb * kPQ * 128, &tmQ, &bars[PB_FULLQ], kb * 64, q0, bh);
      int tk = 0, tv = 0;
      for (uint32_t spin = 0; tk < nkt || tv < nkt;) {
        bool moved = false;
        if (tk < nkt &&
            (tk < nst || tc::mbar_test_wait(&bars[PB_EMPTYK + tk % nst], ((tk / nst) - 1) & 1))) {
          const int s = tk % nst;
          uint8_t *st = sm + a.off_k + s * a.kstage;
          tc::mbar_arrive_expect_tx(&bars[PB_FULLK + s], a.kstage);
          for (int kb = 0; kb < NKB; ++kb)
            tc::tma_load_3d(st + kb * KT * 128, &tmK, &bars[PB_FULLK + s], kb * 64, tk * KT, bh);
          ++tk;
          moved = true;
        }
        if (tv < nkt &&
            (tv < nst || tc::mbar_test_wait(&bars[PB_EMPTYV + tv % nst], ((tv / nst) - 1) & 1))) {
          const int s = tv % nst;
          uint8_t *st = sm + a.off_v + s * a.vstage;
          tc::mbar_arrive_expect_tx(&bars[PB_FULLV + s], a.vstage);
          for (int vb = 0; vb < NVB; ++vb)
            tc::tma_load_4d(st + vb * KT * 128, &tmV, &bars[PB_FULLV + s], v0 + vb * 64, tv * KT,
                            h, b);
          ++tv;
          moved = true;
        }
        if (!moved) {
          if (++spin >= kPSpin) {
            report(p.status, kDevTimeout);
            *abort_p = 1;
            break;
          }
          if ((spin & 255u) == 255u && *abort_p) break;
        }
      }
      pdl_launch_dependents();  // every load is issued
      // Every issued copy lands before the CTA can leave.
      par_drain(&bars[PB_FULLQ], 0);
      for (int u = tk > nst ? tk - nst : 0; u < tk; ++u)
        par_drain(&bars[PB_FULLK + u % nst], (u / nst) & 1);
      for (int u = tv > nst ? tv - nst : 0; u < tv; ++u)
        par_drain(&bars[PB_FULLV + u % nst], (u / nst) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // Whatever is ready first: O += P~ V of block tp once its P~ and V are
    // in place (first, as it frees a V stage and a score buffer), the scores
    // of block ts once its K' has landed and its buffer's previous P~ has
    // been consumed.
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_f16(kPQ, KT, 0, 0);
      const uint32_t id_o = tc::idesc_bf16(kPQ, W, 0, 1);
      const uint32_t sq = tc::smem_u32(sm);
      const uint64_t dq = tc::smem_desc(sq, 16, 1024, tc::kSw128);  // Q' K-major
      const int nks = DK / 16;
      bool ok = par_wait(&bars[PB_FULLQ], 0, abort_p, p.status);
      int ts = 0, tp = 0;
      for (uint32_t spin = 0; ok && tp < nkt;) {
        bool moved = false;
        if (tp < ts && tc::mbar_test_wait(&bars[PB_PRDY + tp % NSB], (tp / NSB) & 1) &&
            tc::mbar_test_wait(&bars[PB_FULLV + tp % nst], (tp / nst) & 1)) {
          tc::tc_fence_after();
          const int bb = tp % NSB;
          // V MN-major: 64-column blocks KT * 128 bytes apart, 8-key groups
          // 1 KB apart.
          const uint64_t dv = tc::smem_desc(sq + a.off_v + (tp % nst) * a.vstage, KT * 128, 1024,
                                            tc::kSw128);
#pragma unroll 1
          for (int ks = 0; ks < KT / 16; ++ks)
            tc::mma_ts(tO, tb + KT * bb + ks * 8, dv + ks * 128, id_o,
                       (tp > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(&bars[PB_PVDONE + bb]);
          tc::mma_commit(&bars[PB_EMPTYV + tp % nst]);
          ++tp;
          moved = true;
        }
        if (ts < nkt && ts - tp < NSB &&
            tc::mbar_test_wait(&bars[PB_FULLK + ts % nst], (ts / nst) & 1) &&
            (ts < NSB ||
             tc::mbar_test_wait(&bars[PB_PVDONE + ts % NSB], ((ts / NSB) - 1) & 1))) {
          tc::tc_fence_after();
          const int bb = ts % NSB;
          const uint64_t dk =
              tc::smem_desc(sq + a.off_k + (ts % nst) * a.kstage, 16, 1024, tc::kSw128);
#pragma unroll 1
          for (int ks = 0; ks < nks; ++ks)
            tc::mma_ss(tb + KT * bb, dq + kstep(ks, kPQ), dk + kstep(ks, KT), id_s, ks > 0);
          tc::mma_commit(&bars[PB_SFULL + bb]);
          tc::mma_commit(&bars[PB_EMPTYK + ts % nst]);
          ++ts;
          moved = true;
        }
        if (!moved) {
          if (++spin >= kPSpin) {
            report(p.status, kDevTimeout);
            *abort_p = 1;
            ok = false;
          } else if ((spin & 255u) == 255u && *abort_p) {
            ok = false;
          }
        }
      }
      if (ok) tc::mma_commit(&bars[PB_ODONE]);
      tc::mma_commit(&bars[PB_DRAIN]);
      par_drain(&bars[PB_DRAIN], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ scores -> P~, O drain
    const int q = warp & 3;                               // TMEM lane quarter
    const int et = (tid - 128) & 127, wg = (tid - 128) >> 7;  // query row; group
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const int n = q0 + et;
    const int cq = n / kPK, cqm = min(cq, nch - 1), ri = n - cq * kPK;
    const ChunkMeta *meta = a.meta + (long long)bh * nch;
    // E: P~ = P 2^-E < 2^15 for every score of the CTA (bound from the
    // prologue's magnitudes: |q'_n . k'_m| <= (d_k/2) qmax kmax).
    float km = 0.f, qm = 0.f;
    for (int c = et; c < nkc; c += 128) km = fmaxf(km, meta[c].kmax);
    if (et < 2 && 2 * qt + et < nch) qm = meta[2 * qt + et].qmax;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
      qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
    }
    float *rd = red + 8 * wg;
    if (lane == 0) {
      rd[q] = km;
      rd[4 + q] = qm;
    }
    asm volatile("bar.sync %0, 128;" ::"r"(1 + wg) : "memory");
    km = fmaxf(fmaxf(rd[0], rd[1]), fmaxf(rd[2], rd[3]));
    qm = fmaxf(fmaxf(rd[4], rd[5]), fmaxf(rd[6], rd[7]));
    const float bound = 0.5f * (float)DK * qm * km;
    int E = 0;
    if (bound > 0.f && bound < INFINITY) {
      frexpf(bound, &E);
      E -= 15;
    }
    const float lg2 = p.lng[h] * 1.44269504088896341f;  // log2 gamma
    const int qe = meta[cqm].qexp;
    float2 rs2 = make_float2(0.f, 0.f);
    // Key exponents of the group's next block, read one block ahead.
    int ke_next[CPT];
#pragma unroll
    for (int h2 = 0; h2 < CPT; ++h2) {
      const int ck = wg * CPT + h2;
      ke_next[h2] = ck < nkc ? meta[ck].kexp : 0;
    }
    bool ok = true;
    for (int j = wg; j < nkt && ok; j += 2) {
      int ke[CPT];
#pragma unroll
      for (int h2 = 0; h2 < CPT; ++h2) {
        ke[h2] = ke_next[h2];
        const int ck = (j + 2) * CPT + h2;
        if (ck < nkc) ke_next[h2] = meta[ck].kexp;
      }
      const int bb = j % NSB;
      ok = par_wait(&bars[PB_SFULL + bb], (j / NSB) & 1, abort_p, p.status);
      if (!ok) break;
      tc::tc_fence_after();
#pragma unroll
      for (int h2 = 0; h2 < CPT; ++h2) {
        // 64 keys of chunk ck: scores from columns 64 h2.., P~ to 32 h2..
        // (the score columns already read).
        const int ck = j * CPT + h2;
        uint32_t r0[32], r1[32];
        tc::tmem_ld32(tb + lb + KT * bb + 64 * h2, r0);
        tc::tmem_ld32(tb + lb + KT * bb + 64 * h2 + 32, r1);
        tc::tmem_ld_wait_on(r0);
        tc::tmem_ld_wait_on(r1);
        // g carries the decay gamma^(n-m) not folded into the operands and
        // the exponents; keys after the row's own position are masked.
        const int Lc = min(kPK, N - ck * kPK);
        const float g = (ck <= cq && ck < nkc)
                            ? exp2f((float)(kPK * (cq - ck) - Lc) * lg2 + (float)(qe + ke[h2] - E))
                            : 0.f;
        const float2 g2 = make_float2(g, g);
        uint32_t w[32];
        if (ck < cq) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 x = tc::mul2(make_float2(__uint_as_float(r0[2 * c]),
                                                  __uint_as_float(r0[2 * c + 1])), g2);
            rs2 = tc::add2(rs2, x);
            w[c] = tc::pack_bf16(x.x, x.y);
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 x = tc::mul2(make_float2(__uint_as_float(r1[2 * c]),
                                                  __uint_as_float(r1[2 * c + 1])), g2);
            rs2 = tc::add2(rs2, x);
            w[16 + c] = tc::pack_bf16(x.x, x.y);
          }
        } else {
          const int lim = ck == cq ? ri : -1;  // keys c <= lim are kept
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float x0 = 2 * c <= lim ? __uint_as_float(r0[2 * c]) * g : 0.f;
            const float x1 = 2 * c + 1 <= lim ? __uint_as_float(r0[2 * c + 1]) * g : 0.f;
            rs2 = tc::add2(rs2, make_float2(x0, x1));
            w[c] = tc::pack_bf16(x0, x1);
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float x0 = 32 + 2 * c <= lim ? __uint_as_float(r1[2 * c]) * g : 0.f;
            const float x1 = 33 + 2 * c <= lim ? __uint_as_float(r1[2 * c + 1]) * g : 0.f;
            rs2 = tc::add2(rs2, make_float2(x0, x1));
            w[16 + c] = tc::pack_bf16(x0, x1);
          }
        }
        tc::tmem_st32(tb + lb + KT * bb + 32 * h2, w);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[PB_PRDY + bb]);
    }
    // The second group hands its row sums to the first, which drains O.
    // Both groups pass this barrier exactly once, aborted or not.
    if (wg == 1) rsx[et] = rs2.x + rs2.y;
    asm volatile("bar.sync 3, 256;" ::: "memory");
    if (wg == 1) ok = false;
    const float rs = (rs2.x + rs2.y) + (wg == 0 ? rsx[et] : 0.f);
    if (ok) ok = par_wait(&bars[PB_ODONE], 0, abort_p, p.status);
    if (ok && a.NVS > 1) {
      // Raw rows and row factors for the GroupNorm pass.
      tc::tc_fence_after();
      const float back = exp2f((float)E);
      for (int g32 = 0; g32 < W / 32; ++g32) {
        uint32_t r[32];
        tc::tmem_ld32(tO + lb + 32 * g32, r);
        tc::tmem_ld_wait_on(r);
        if (n < N) {
          float4 *dst = reinterpret_cast<float4 *>(a.Oraw + ((long long)bh * N + n) * p.dv + v0 +
                                                   32 * g32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * back, __uint_as_float(r[4 * i + 1]) * back,
                                 __uint_as_float(r[4 * i + 2]) * back,
                                 __uint_as_float(r[4 * i + 3]) * back);
        }
      }
      if (vs == 0 && n < N) {
        const float s = row_scale(p, h, p.pos0 + n + 1);
        a.F[(long long)bh * N + n] = s * rsum_scale(p, s * rs * back);
      }
    } else if (ok) {
      // The whole row is in this thread's TMEM lane: row factor, GroupNorm
      // (mean, then the variance about it, as the GroupNorm pass computes
      // them) and the store, reading the accumulator once per pass.
      tc::tc_fence_after();
      const float back = exp2f((float)E);
      const float s = row_scale(p, h, p.pos0 + n + 1);
      const float f = s * rsum_scale(p, s * rs * back) * back;
      float mu = 0.f, inv = 1.f;
      if (p.gn_eps >= 0.f) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f};
        for (int g32 = 0; g32 < W / 32; ++g32) {
          uint32_t r[32];
          tc::tmem_ld32(tO + lb + 32 * g32, r);
          tc::tmem_ld_wait_on(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) sa[i & 3] += f * __uint_as_float(r[i]);
        }
        mu = ((sa[0] + sa[1]) + (sa[2] + sa[3])) / (float)W;
        float va[4] = {0.f, 0.f, 0.f, 0.f};
        for (int g32 = 0; g32 < W / 32; ++g32) {
          uint32_t r[32];
          tc::tmem_ld32(tO + lb + 32 * g32, r);
          tc::tmem_ld_wait_on(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float dlt = f * __uint_as_float(r[i]) - mu;
            va[i & 3] = fmaf(dlt, dlt, va[i & 3]);
          }
        }
        inv = rsqrtf(((va[0] + va[1]) + (va[2] + va[3])) / (float)W + p.gn_eps);
      }
      const long long ob = b * p.so[0] + h * p.so[1] + (long long)n * p.so[2];
      for (int g32 = 0; g32 < W / 32; ++g32) {
        uint32_t r[32];
        tc::tmem_ld32(tO + lb + 32 * g32, r);
        tc::tmem_ld_wait_on(r);
        const long long e0 = ob + 32 * g32;
        if (n >= N) {
        } else if (a.vec_out && p.out_bf16) {
          uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.o) + e0);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = tc::pack_bf16((f * __uint_as_float(r[8 * i + 2 * e]) - mu) * inv,
                                    (f * __uint_as_float(r[8 * i + 2 * e + 1]) - mu) * inv);
            dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        } else if (a.vec_out) {
          float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + e0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4((f * __uint_as_float(r[4 * i]) - mu) * inv,
                                 (f * __uint_as_float(r[4 * i + 1]) - mu) * inv,
                                 (f * __uint_as_float(r[4 * i + 2]) - mu) * inv,
                                 (f * __uint_as_float(r[4 * i + 3]) - mu) * inv);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            st_elem(a.o, e0 + i, (f * __uint_as_float(r[i]) - mu) * inv, p.out_bf16);
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, a.tmem_cols);
  }
}

// ------------------------------------------------------------------ host
cudaError_t launch_parallel_tc(const KParams &p, const __half *Qp, const __half *Kp, const void *v,
                               const ChunkMeta *meta, float *Oraw, float *F, void *o,
                               bool *fused, cudaStream_t st) {
  *fused = false;
  if (p.N == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  if (p.dk % 64 || p.dk > 256 || p.dv % 128 || p.dv > 1024) return cudaErrorInvalidValue;
  const int BH = p.B * p.H;
  ParArgs a;
  a.meta = meta;
  a.Oraw = Oraw;
  a.F = F;
  a.W = p.dv % 256 == 0 ? 256 : 128;
  a.NVS = p.dv / a.W;
  a.o = o;
  const int al = p.out_bf16 ? 8 : 4;  // elements per 16 bytes
  a.vec_out = (reinterpret_cast<uintptr_t>(o) % 16 == 0) && p.so[0] % al == 0 &&
              p.so[1] % al == 0 && p.so[2] % al == 0;
  const uint32_t NKB = (uint32_t)p.dk / 64, NVB = (uint32_t)a.W / 64;
  const uint32_t qbytes = NKB * kPQ * 128u;
  const uint32_t tail = PB_COUNT * 8 + 608 + 1024;  // barriers, misc, alignment slack
  // 128-key blocks where two stages of them fit, else 64-key blocks.
  int KT = 128, nst = 0;
  for (; KT >= 64; KT /= 2) {
    nst = (int)((kPSmemLimit - tail - qbytes) / ((NKB + NVB) * (uint32_t)KT * 128u));
    if (nst >= 2) break;
  }
  if (nst > kPMaxStages) nst = kPMaxStages;
  if (nst < 2) return cudaErrorInvalidValue;
  a.nst = nst;
  a.off_k = qbytes;
  a.kstage = NKB * (uint32_t)KT * 128u;
  a.off_v = a.off_k + (uint32_t)nst * a.kstage;
  a.vstage = NVB * (uint32_t)KT * 128u;
  a.off_bar = a.off_v + (uint32_t)nst * a.vstage;
  a.tmem_cols = 512;
  const uint32_t smem = a.off_bar + tail;

  CUtensorMap tq, tk, tv;
  const cuuint64_t dq[3] = {(cuuint64_t)p.dk, (cuuint64_t)p.N, (cuuint64_t)BH};
  const cuuint64_t sq[2] = {(cuuint64_t)p.dk * 2, (cuuint64_t)p.N * p.dk * 2};
  const cuuint32_t bq[3] = {64, (cuuint32_t)kPQ, 1};
  const cuuint32_t bk[3] = {64, (cuuint32_t)KT, 1};
  const cuuint64_t dv4[4] = {(cuuint64_t)p.dv, (cuuint64_t)p.N, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t sv4[3] = {(cuuint64_t)p.sv[2] * 2, (cuuint64_t)p.sv[1] * 2,
                             (cuuint64_t)p.sv[0] * 2};
  const cuuint32_t bv[4] = {64, (cuuint32_t)KT, 1, 1};
  if (!tmap_encode(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, Qp, dq, sq, bq,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, Kp, dq, sq, bk,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dv4, sv4, bv,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  void (*kern)(KParams, CUtensorMap, CUtensorMap, CUtensorMap, ParArgs) =
      KT == 128 ? parallel_tc_kernel<128> : parallel_tc_kernel<64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)((p.N + kPQ - 1) / kPQ) * BH * a.NVS;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  *fused = a.NVS == 1;
  return launch_k(kern, dim3((unsigned)grid), dim3(kPThreads), smem, st, true, p, tq, tk, tv, a);
}

}  // namespace ret
