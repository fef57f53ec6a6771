// Chunkwise retention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, per head and chunk of 64 tokens (hwhale.com/article/285883,
// chunkwise equation and ChunkwiseRetention; m0nads.wordpress.com,
// chunkwise representation):
//   O_[c] = (Q_[c] K_[c]^T (.) D) V_[c] + (Q_[c] S_c) (.) xi,  xi_i = gamma^(i+1)
//   S_{c+1} = gamma^L S_c + K_[c]^T (V_[c] (.) zeta),          zeta_j = gamma^(L-1-j)
// then the three normalisations and the per-head GroupNorm.
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
// O^T is double-buffered in TMEM (chunk parity); the scores of chunk c live
// in O^T buffer c&1 until the R group has read them.
//
// Warp roles (16 warps):
//   warp 0       TMA loads (2-stage ring) and the scores MMAs
//   warp 1       O^T = V^T R^T, then per half of d_k the cross term and the
//                state update (two issuing threads keep the tensor pipe fed:
//                one thread issues at most about one MMA per 28 ns)
//   warps 2-3    helper: max |V|, the chunk's block exponents, V -> fp16
//   warps 4-7    R group: scores -> masked fp16 R, Q'.z, row factors, z carry
//   warps 8-11   state group: fp16 copy of the state and gamma^L, per half
//                of d_k, so it overlaps the MMAs of the other half
//   warps 12-15  output group: drain O^T, GroupNorm, stores
// Every wait is bounded; a wait that runs out sets the status word and an
// abort flag, and every role leaves after draining its own asynchronous work.
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
constexpr int kNT = 512;  // threads per CTA

// Shared-memory map (offsets from a 1024-byte aligned base).
// Stage: Q' 32K | K' 32K | V 16K | key column sums (d_k fp32) | ChunkMeta.
constexpr uint32_t kOffQ = 0, kOffK = 32 * 1024, kOffV = 64 * 1024;
constexpr uint32_t kOffKs = 80 * 1024, kOffMeta = kOffKs + 1024;
constexpr uint32_t kStage = 82 * 1024;
constexpr uint32_t kOffR = 2 * kStage;                  // 64 x 128 B, fp16
constexpr uint32_t kOTPitch = 144;                      // floats per O^T row
constexpr uint32_t kOffOT = kOffR + 8 * 1024;           // [64][144] fp32
constexpr uint32_t kOffZ = kOffOT + 64 * kOTPitch * 4;  // [256] fp32
constexpr uint32_t kOffF = kOffZ + 256 * 4;             // [2][64] fp32 row factors
constexpr uint32_t kOffOS = kOffF + 2 * 64 * 4;         // [2] fp32 2^E for the output group
constexpr uint32_t kOffSc = kOffOS + 16;                // [2] Scales (helper -> R, state)
constexpr uint32_t kOffRed = kOffSc + 2 * 32;           // [4 groups][8] fp32 scratch
constexpr uint32_t kOffGN = kOffRed + 128;              // [2][8][64][2] fp32
constexpr uint32_t kOffVX = kOffGN + 2 * 8 * 64 * 2 * 4;   // [2] float max|V|, s_bound entry
constexpr uint32_t kOffQZ = kOffVX + 16;                   // [64] fp32 R row sums, scratch
constexpr uint32_t kOffBar = kOffQZ + 2 * 64 * 4;
constexpr int kNumBars = 29;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Barriers with a 0/1 pair exist per stage or per O^T buffer (chunk parity),
// so a producer may run one chunk ahead of a consumer without two phases of
// one barrier completing before the consumer looks.
enum Bar {
  FULLQ0 = 0, FULLQ1, FULLV0, FULLV1, EMPTY0, EMPTY1, QK0, QK1, RRDY, RFREE, OFULL0, OFULL1, OFREE0, OFREE1,
  SFULL0, SFULL1, SRDY0, SRDY1, GN0, GN1, DRAIN, DRAIN2, VRDY0, VRDY1, VCONV0, VCONV1,
  FRDY0, FRDY1, SB0
};

// Per-chunk block exponents and state factors, chosen by the helper from
// rigorous magnitude bounds (see the helper group) and read by the R and
// state groups.
struct Scales {
  int E;           // O^T accumulator holds O * 2^-E
  int rr;          // R is stored as fp16 R * 2^-rr
  float f_cp;      // fp16 state copy = TMEM state * f_cp
  float f_pre;     // TMEM state <- TMEM state * f_pre before the update
  int sigma_next;  // TMEM state holds S * 2^-sigma_next after the update
  int pad[3];
};
static_assert(sizeof(Scales) == 32, "Scales record");

// TMEM column map: fp32 state, its fp16 copy, two O^T buffers (chunk
// parity).  The scores T of chunk c (M=64 layout) live in O^T buffer c&1
// until the R group has read them; O^T of chunk c then overwrites them.
constexpr uint32_t kTS = 0, kTSh = 256, kTO0 = 384;
__device__ __forceinline__ uint32_t tcol_o(int c) { return kTO0 + 64u * (uint32_t)(c & 1); }

constexpr uint32_t kBudget = 1u << 24;

struct TcArgs {
  const float *S_in, *z_in;
  float *S_out, *z_out;
  void *o;
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
// 3 = helper, 4 = R).
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

// K-step ks (16 elements) of a K-major operand stored as 64-element swizzled
// rows in 8 KB blocks of 64 rows, in the 16-byte units of a descriptor's
// start-address field.  Descriptors are built once; a K-step adds this
// offset (every shared-memory address stays below 256 KB, so the 14-bit
// field never carries).
__device__ __forceinline__ uint64_t kmaj_off(int ks) {
  return (uint64_t)(((ks >> 2) * 8192 + (ks & 3) * 32) >> 4);
}

// Bounded wait that also gives up when another role has aborted.  The
// first try_wait (which already suspends the thread for a while) is inline;
// the bounded retry loop is out of line, since the kernel's speed depends on
// its instruction footprint (all roles run on every SM sub-partition).
__device__ __noinline__ bool wait_bar_slow(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                           unsigned *status) {
  // Each try suspends the thread for the hardware's own time limit unless
  // the phase completes first (measured slightly faster than a 20 us or
  // 1 us suspend hint); 2^20 tries bound the wait to well under seconds
  // beyond any legitimate wait, and the abort flag is checked every 16.
  for (uint32_t i = 0; i < (1u << 20); ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && *abort_p) return false;
  }
  report(status, kDevTimeout);
  *abort_p = 1;
  return false;
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_p,
                                         unsigned *status) {
  return tc::mbar_try_wait(bar, parity) || wait_bar_slow(bar, parity, abort_p, status);
}

__device__ __noinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity,
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

// e such that m * 2^-e < 2^14 (0 for m = 0, infinite or NaN): read off the
// exponent field, m = f 2^(be - 126) with f in [0.5, 1) for normal m; a
// subnormal m < 2^-126 takes the exponent of 2^-126, which still bounds it.
__device__ __forceinline__ int expo14(float m) {
  const int be = (int)((__float_as_uint(m) >> 23) & 0xffu);
  return (m > 0.f && be < 255) ? max(be, 1) - 126 - 14 : 0;
}

__device__ __forceinline__ float2 h2f(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

// Store variants, fixed at compile time so the hot loop carries no unused
// paths: kStoreAny handles every output dtype and alignment; kStoreBf16 is
// 16-byte aligned bf16 rows.
enum StoreMode { kStoreAny = 0, kStoreBf16 = 1 };

// Entry state of this CTA's value columns into the TMEM state columns at
// `ts` (one warp, its 32 lanes), 32-row groups [g0, g1) of d_k: S_in, or for
// a later segment the decayed sum of S_in and the pieces before it.  Returns
// the lane's max |S| over those rows.
__device__ __noinline__ float load_entry_state(const KParams &p, const TcArgs &a, uint32_t ts,
                                               int bh, long long vglob, int seg, int c0, int npc,
                                               float lng, int g0, int g1) {
  const int DK = p.dk;
  const float w_in = seg > 0 ? gpow(lng, kC * c0) : 1.f;
  float m0 = 0.f;
  for (int g = g0; g < g1; ++g) {
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
    tc::tmem_st32(ts + g * 32, r);
  }
  tc::tmem_st_wait();
  return m0;
}

// The TMEM state columns at `ts` (one warp, its 32 lanes) times `back` to
// S_out.
__device__ __noinline__ void store_state(const KParams &p, float *S_out, uint32_t ts, int bh,
                                         long long vglob, float back) {
  const int DK = p.dk;
  for (int g = 0; g < DK / 32; ++g) {
    uint32_t r[32];
    tc::tmem_ld32(ts + g * 32, r);
    tc::tmem_ld_wait_on(r);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      S_out[((long long)bh * DK + g * 32 + i) * p.dv + vglob] = __uint_as_float(r[i]) * back;
  }
}

// Entry z of this head (z_in, or for a later segment the decayed sum of
// z_in and the pieces before it) into zsm; thread et of 128.
__device__ __noinline__ void load_entry_z(const KParams &p, const TcArgs &a, float *zsm, int et,
                                          int bh, int seg, int c0, int npc, float lng) {
  const int DK = p.dk;
  for (int k2 = et; k2 < DK; k2 += 128) {
    float z = a.z_in ? a.z_in[(long long)bh * DK + k2] : 0.f;
    if (seg > 0) {
      z *= gpow(lng, kC * c0);
      for (int i = 0; i < npc; ++i)
        z = fmaf(gpow(lng, kC * (c0 - (i + 1) * a.piece_len)),
                 a.zPart[((long long)i * p.B * p.H + bh) * DK + k2], z);
    }
    zsm[k2] = z;
  }
}

template <int kStore>
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
  float *oss = reinterpret_cast<float *>(sm + kOffOS);
  Scales *scs = reinterpret_cast<Scales *>(sm + kOffSc);
  float *red = reinterpret_cast<float *>(sm + kOffRed);
  float *OT = reinterpret_cast<float *>(sm + kOffOT);
  float *gns = reinterpret_cast<float *>(sm + kOffGN);
  float *vmxs = reinterpret_cast<float *>(sm + kOffVX);  // [0] max|V| scratch, [1] entry bound
  float *qzs = reinterpret_cast<float *>(sm + kOffQZ);

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
  const bool rsum = (p.norm_flags & RET_NORM_RSUM) != 0;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      tc::mbar_init(&bars[i], (i == EMPTY0 || i == EMPTY1) ? 2 : 1);
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
  // Launched with programmatic serialization: the setup above overlaps the
  // kernel before this one; global memory only after it has completed.
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA and scores
    // One thread issues the stage loads and the scores T = Q' K'^T of each
    // chunk, into O^T buffer c&1 once the output group has drained that
    // buffer's previous chunk (c-2).
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      // V and the chunk's record land first (FULLV, for the helper); Q', K'
      // and the key sums after them (FULLQ, for the scores).
      const uint32_t bytes_v = 16384u + 16u;
      const uint32_t bytes_q = (uint32_t)NKB * 8192u * 2u + (a.need_z ? (uint32_t)DK * 4u : 0u);
      const uint32_t id_qk = tc::idesc_f16(64, 64, 0, 0);
      const int nks = DK / 16;
      const uint32_t sq0 = tc::smem_u32(sm + kOffQ);
      const uint64_t dq0 = tc::smem_desc(sq0, 16, 1024, tc::kSw128);          // Q' K-major
      const uint64_t dk0 = tc::smem_desc(sq0 + kOffK, 16, 1024, tc::kSw128);  // K' K-major
      int t_ld = 0, t_qk = 0;  // next chunk to load / to score
      for (uint32_t spin = 0; t_qk < ncl;) {
        bool moved = false;
        if (t_ld < ncl &&
            (t_ld < 2 || tc::mbar_test_wait(&bars[EMPTY0 + (t_ld & 1)], ((t_ld >> 1) - 1) & 1))) {
          const int s = t_ld & 1, c = c0 + t_ld;
          uint8_t *st = sm + s * kStage;
          tc::mbar_arrive_expect_tx(&bars[FULLV0 + s], bytes_v);
          for (int vb = 0; vb < 2; ++vb)
            tc::tma_load_4d(st + kOffV + vb * 8192, &tmV, &bars[FULLV0 + s], v0 + vb * 64, c * kC,
                            h, b);
          tc::bulk_load(st + kOffMeta, a.meta + (long long)bh * nch + c, 16u, &bars[FULLV0 + s]);
          tc::mbar_arrive_expect_tx(&bars[FULLQ0 + s], bytes_q);
          for (int kb = 0; kb < NKB; ++kb)
            tc::tma_load_3d(st + kOffQ + kb * 8192, &tmQ, &bars[FULLQ0 + s], kb * 64, c * kC, bh);
          for (int kb = 0; kb < NKB; ++kb)
            tc::tma_load_3d(st + kOffK + kb * 8192, &tmK, &bars[FULLQ0 + s], kb * 64, c * kC, bh);
          if (a.need_z)
            tc::bulk_load(st + kOffKs, a.ksum + ((long long)bh * nch + c) * DK, (uint32_t)DK * 4u,
                          &bars[FULLQ0 + s]);
          ++t_ld;
          moved = true;
        }
        const int bq = t_qk & 1;
        if (t_qk < t_ld && tc::mbar_test_wait(&bars[FULLQ0 + bq], (t_qk >> 1) & 1) &&
            (t_qk < 2 || tc::mbar_test_wait(&bars[OFREE0 + bq], ((t_qk >> 1) - 1) & 1))) {
          tc::tc_fence_after();
          const uint64_t so = bq ? (uint64_t)(kStage >> 4) : 0ull;
#pragma unroll 1
          for (int ks = 0; ks < nks; ++ks)  // T = Q' K'^T
            tc::mma_ss(tb + tcol_o(t_qk), dq0 + so + kmaj_off(ks), dk0 + so + kmaj_off(ks), id_qk,
                       ks > 0);
          tc::mma_commit(&bars[QK0 + bq]);
          ++t_qk;
          moved = true;
        }
        if (!moved) {
          if (++spin >= kBudget) {
            report(p.status, kDevTimeout);
            *abort_p = 1;
            break;
          }
          if ((spin & 255u) == 255u && *abort_p) break;
          // No back-off: a sleep here (32 or 128 ns) measured slower.
        }
      }
      // Every load and score is issued: the next kernel may be scheduled
      // (it waits for this one to complete in its own pdl_wait).
      pdl_launch_dependents();
      // Let every issued copy and MMA finish before the CTA can leave.
      // (Earlier stages were reused, so only the last two loads can be
      // outstanding.)
      for (int t = t_ld > 2 ? t_ld - 2 : 0; t < t_ld; ++t) {
        drain_wait(&bars[FULLV0 + (t & 1)], (t >> 1) & 1);
        drain_wait(&bars[FULLQ0 + (t & 1)], (t >> 1) & 1);
      }
      tc::mma_commit(&bars[DRAIN]);
      drain_wait(&bars[DRAIN], 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ O^T and state MMAs
    // Per chunk: O^T = V^T R^T (starts the accumulator in buffer c&1, after
    // the R group has read the scores there), then per half of d_k, as soon
    // as the state group has refreshed it: O^T += S^T Q'^T over the half's
    // K-steps and S^T[:, half] += V^T K'[:, half].  SFULL0/SFULL1 tell the
    // state group that the half's copy has been read and its state updated.
    if (lane == 0) {
      const uint32_t id_o = tc::idesc_f16(128, 64, 1, 0);
      const uint32_t id_x = tc::idesc_f16(128, 64, 0, 0);
      const uint32_t id_s = tc::idesc_f16(128, DK == 256 ? 128 : DK, 1, 1);
      const int nh = DK == 256 ? 2 : 1;  // d_k = 256 runs in two halves of 128
      const int nkh = DK / 16 / nh;     // K-steps of the cross term per half
      const uint32_t sq0 = tc::smem_u32(sm + kOffQ);
      const uint64_t dq0 = tc::smem_desc(sq0, 16, 1024, tc::kSw128);             // Q' K-major
      const uint64_t dkm0 = tc::smem_desc(sq0 + kOffK, 8192, 1024, tc::kSw128);  // K' MN-major
      const uint64_t dv0 = tc::smem_desc(sq0 + kOffV, 8192, 1024, tc::kSw128);   // V^T MN-major
      const uint64_t dr = tc::smem_desc(tc::smem_u32(sm + kOffR), 16, 1024, tc::kSw128);
      bool ok = true;
      for (int lc = 0; lc < ncl && ok; ++lc) {
        const int s = lc & 1;
        const uint64_t so = s ? (uint64_t)(kStage >> 4) : 0ull;
        const uint32_t to = tb + tcol_o(lc);
        ok = wait_bar(&bars[FULLQ0 + s], (lc >> 1) & 1, abort_p, p.status) &&
             wait_bar(&bars[VCONV0 + s], (lc >> 1) & 1, abort_p, p.status) &&
             wait_bar(&bars[RRDY], lc & 1, abort_p, p.status);
        if (!ok) break;
        tc::tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks)  // O^T = V^T R^T
          tc::mma_ss(to, dv0 + so + ks * 128, dr + ks * 2, id_o, ks > 0);
        tc::mma_commit(&bars[RFREE]);
        for (int hh = 0; hh < nh; ++hh) {
          if (!wait_bar(&bars[SRDY0 + hh], lc & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll 1
          for (int ks = hh * nkh; ks < (hh + 1) * nkh; ++ks)  // O^T += S^T Q'^T, this half
            tc::mma_ts(to, tb + kTSh + ks * 8, dq0 + so + kmaj_off(ks), id_x, 1);
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks)  // S^T[:, half] += V^T K'[:, half]
            tc::mma_ss(tb + kTS + hh * 128, dv0 + so + ks * 128,
                       dkm0 + so + ks * 128 + (uint64_t)hh * 1024, id_s, 1);
          tc::mma_commit(&bars[nh == 1 ? SFULL1 : SFULL0 + hh]);
        }
        if (!ok) break;
        tc::mma_commit(&bars[OFULL0 + s]);
        tc::mma_commit(&bars[EMPTY0 + s]);
      }
      tc::mma_commit(&bars[DRAIN2]);
      drain_wait(&bars[DRAIN2], 0);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ helper group
    const int G = 3, NT = 64;
    const int ht = tid - 64;  // 0..63
    float *hred = red;        // [2 slots][2 warps]
    int hslot = 0;
    // Bound of max |S| entering the first chunk, from the state group.
    bool ok = grp_all(G, wait_bar(&bars[SB0], 0, abort_p, p.status), NT);
    float s_bound = vmxs[1];
    int sigma = 0;  // the TMEM state holds S * 2^-sigma
    const float g64 = gpow(lng, kC);
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      uint8_t *st = sm + s * kStage;
      ok = grp_all(G, wait_bar(&bars[FULLV0 + s], (lc >> 1) & 1, abort_p, p.status), NT);
      if (!ok) break;
      // (1) max |V| of the tile (1024 16-byte words), on bf16 pairs.
      const uint4 *vt = reinterpret_cast<const uint4 *>(st + kOffV);
      __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll 4
      for (int u = 0; u < 16; ++u) {
        const uint4 v4 = vt[ht + NT * u];
        const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e])));
      }
      float vm = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      float *hr = hred + 2 * hslot;
      hslot ^= 1;
      if ((ht & 31) == 0) hr[ht >> 5] = vm;
      grp_sync(G, NT);
      const float vmx = fmaxf(hr[0], hr[1]);
      // (2) block exponents of the chunk.  R is stored at its own scale
      // 2^-rr, rr from the bound |R_ij| = gamma^(i-j) |q_i . k_j| <= (d_k/2)
      // max|pair of rot q| max|pair of rot k| (j <= i; a dot product is a sum
      // of d_k/2 pair products), so the R group needs nothing from here.  R
      // and the state copy share the O accumulator's scale 2^-E, E = rr + vx
      // = ss + aq; V takes the larger exponent when the state bound s_bound
      // >= max |S_c| needs it, which keeps every fp16 operand below 2^15.
      const ChunkMeta mt = *reinterpret_cast<const ChunkMeta *>(st + kOffMeta);
      const float gL = L == kC ? g64 : gpow(lng, L);
      const int rr = expo14((float)(DK / 2) * mt.qmax * mt.kmax);
      int vx = expo14(vmx);
      if (s_bound > 0.f) vx = max(vx, expo14(s_bound) + mt.qexp - rr);
      {
        const int E = rr + vx, ss = E - mt.qexp, sigma_next = vx + mt.kexp;
        if (ht == 0) {
          Scales sc;
          sc.E = E;
          sc.rr = rr;
          sc.f_cp = exp2f((float)(sigma - ss));
          sc.f_pre = gL * exp2f((float)(sigma - sigma_next));
          sc.sigma_next = sigma_next;
          sc.pad[0] = sc.pad[1] = sc.pad[2] = 0;
          scs[s] = sc;
          tc::mbar_arrive(&bars[VRDY0 + s]);
        }
        sigma = sigma_next;
        // |S_{c+1}| <= gamma^L |S_c| + sum_j |K'_j||V_j| with zeta <= 1 (a
        // pair norm bounds each component of its pair).  Loose by the ratio
        // of a sum of L terms to their random-sign size, which costs nothing
        // in floating point.
        s_bound = gL * s_bound + (float)L * mt.kmax * vmx;
      }
      // (3) V tile: bf16 -> fp16 * 2^-vx in place.
      const float vsc = exp2f((float)-vx);
      const float2 vsc2 = make_float2(vsc, vsc);
#pragma unroll 4
      for (int u = 0; u < 16; ++u) {
        const uint4 v4 = vt[ht + NT * u];
        const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = tc::mul2(make_float2(bf_lo(w[e]), bf_hi(w[e])), vsc2);
          o4[e] = tc::pack_f16(f.x, f.y);
        }
        reinterpret_cast<uint4 *>(st + kOffV)[ht + NT * u] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      tc::fence_proxy_async_smem();
      grp_sync(G, NT);
      if (ht == 0) tc::mbar_arrive(&bars[VCONV0 + s]);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ R group
    const int G = 4;
    const int q = warp & 3;                 // TMEM lane quarter
    const int et = tid - 128;               // 0..127
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    float *rsm = qzs;                       // [64] R row sums
    float *tbl = qzs + 64;                  // [64] 1 - gamma^i
    bool ok = true;
    // Second normalisation: the decay row sum of 1-based position n is
    // (1 - gamma^n)/(1 - gamma) (n for gamma = 1).  With n0 the position of a
    // chunk's first row, 1 - gamma^(n0+i) = A + B (1 - gamma^i), A = 1 -
    // gamma^n0, B = gamma^n0: a sum of non-negative terms, so no
    // cancellation; A and B advance by 64 positions per chunk the same way.
    const float omg = p.omg[h], inv_omg = omg > 0.f ? 1.f / omg : 0.f;
    const float g64 = gpow(lng, kC), t64 = -expm1f((float)kC * lng);
    const float gi64 = expf(-(float)kC * lng);
    float rowA, rowB;
    {
      const float n0 = (float)(p.pos0 + (long long)c0 * kC + 1);
      rowA = -expm1f(n0 * lng);
      rowB = expf(n0 * lng);
      if (et < 64) tbl[et] = et == 0 ? 0.f : -expm1f((float)et * lng);
    }
    if (a.need_z) {
      load_entry_z(p, a, zsm, et, bh, seg, c0, npc, lng);
      grp_sync(G);
    }
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      uint8_t *st = sm + s * kStage;
      // RFREE: the previous chunk's O^T = V^T R^T has read R.
      ok = grp_all(G, wait_bar(&bars[QK0 + s], (lc >> 1) & 1, abort_p, p.status) &&
                          wait_bar(&bars[FULLV0 + s], (lc >> 1) & 1, abort_p, p.status) &&
                          wait_bar(&bars[FULLQ0 + s], (lc >> 1) & 1, abort_p, p.status) &&
                          (lc == 0 || wait_bar(&bars[RFREE], (lc - 1) & 1, abort_p, p.status)));
      if (!ok) break;
      tc::tc_fence_after();
      const ChunkMeta mt = *reinterpret_cast<const ChunkMeta *>(st + kOffMeta);
      // (1) R (fp16, * 2^-rr) as K-major rows, and its row sums; rr is the
      // exponent of R's magnitude bound (the helper uses the same one).
      const int rr = expo14((float)(DK / 2) * mt.qmax * mt.kmax);
      // Row i of the M=64 accumulator is in lane 32(i/16) + i%16: lanes 0-15
      // of each warp hold rows, lanes 16-31 only join the warp-wide loads
      // (tcgen05.ld is warp-collective, so every lane executes the same one).
      const int i = q * 16 + (lane & 15);
      const float ginvL = L == kC ? gi64 : expf(-(float)L * lng);
      // R_ij = T_ij 2^(aq+bk) gamma^-L on the causal triangle (j <= i < L).
      const float tsc = exp2f((float)(mt.qexp + mt.kexp)) * ginvL;
      const float k1 = tsc * exp2f((float)-rr);
      const float2 k2 = make_float2(k1, k1);
      const int lim = i < L ? i : -1;  // last unmasked column of the row
      float2 xs = make_float2(0.f, 0.f);
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // 32 columns at a time
        uint32_t t[32];
        tc::tmem_ld32(tb + lb + tcol_o(lc) + 32 * half, t);
        tc::tmem_ld_wait_on(t);
        if (lane < 16) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int jl = cc * 8 + 2 * e, j = 32 * half + jl;
              float2 x = make_float2(__uint_as_float(t[jl]), __uint_as_float(t[jl + 1]));
              x.x = j <= lim ? x.x : 0.f;
              x.y = j + 1 <= lim ? x.y : 0.f;
              xs = tc::add2(xs, x);
              const float2 r = tc::mul2(x, k2);
              w[e] = tc::pack_f16(r.x, r.y);
            }
            *reinterpret_cast<uint4 *>(sm + kOffR + tc::sw128_off(i, 4 * half + cc)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (lane < 16) rsm[i] = (xs.x + xs.y) * tsc;
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();  // the scores are read; O^T may overwrite them
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[RRDY]);
      // O's scale 2^E for the output group, once the helper has chosen it
      // (the helper rewrites this stage's record only after EMPTY, which
      // this group gives below).
      ok = grp_all(G, wait_bar(&bars[VRDY0 + s], (lc >> 1) & 1, abort_p, p.status));
      if (!ok) break;
      if (et == 0) oss[s] = exp2f((float)scs[s].E);
      // (2) row factors f(n) = s1 s2(n) r(n).  The third normalisation adds
      // gamma^(i+1) s1 s2(n) Q_i . z_c to the row sum: Q'_i . z_c, two
      // threads per row.
      {
        const int i = et >> 1, half = et & 1;
        float qz = 0.f;
        if (rsum) {
          float2 p01 = make_float2(0.f, 0.f), p23 = p01, p45 = p01, p67 = p01;
#pragma unroll 4
          for (int t = 0; t < NKB * 4; ++t) {
            const int kb = t >> 2, cc = (t & 3) + 4 * half;
            const uint4 u =
                *reinterpret_cast<const uint4 *>(st + kOffQ + kb * 8192 + tc::sw128_off(i, cc));
            const float4 z0 = *reinterpret_cast<const float4 *>(zsm + kb * 64 + cc * 8);
            const float4 z1 = *reinterpret_cast<const float4 *>(zsm + kb * 64 + cc * 8 + 4);
            const float2 a0 = h2f(u.x), a1 = h2f(u.y), a2 = h2f(u.z), a3 = h2f(u.w);
            p01 = tc::fma2(a0, make_float2(z0.x, z0.y), p01);
            p23 = tc::fma2(a1, make_float2(z0.z, z0.w), p23);
            p45 = tc::fma2(a2, make_float2(z1.x, z1.y), p45);
            p67 = tc::fma2(a3, make_float2(z1.z, z1.w), p67);
          }
          const float2 ps = tc::add2(tc::add2(p01, p23), tc::add2(p45, p67));
          qz = ps.x + ps.y;
          qz += __shfl_xor_sync(0xffffffffu, qz, 1);
          qz *= exp2f((float)mt.qexp);
        }
        if (half == 0) {
          float f = 0.f;
          if (i < L) {
            float sn = (p.norm_flags & RET_NORM_SCALE) ? p.inv_sqrt_dk : 1.f;
            if (p.norm_flags & RET_NORM_DROW)
              sn *= rsqrtf(omg > 0.f ? fmaf(rowB, tbl[i], rowA) * inv_omg
                                     : (float)(p.pos0 + (long long)c * kC + i + 1));
            f = rsum ? sn * __frcp_rn(fmaxf(fabsf(sn * (rsm[i] + qz)), 1.f)) : sn;
          }
          fsm[s * 64 + i] = f;
        }
      }
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[FRDY0 + s]);
      // (3) z_{c+1} = gamma^L z_c + sum_j K'_j (column sums from the prologue).
      rowA = fmaf(rowB, t64, rowA);  // next chunk's first row is 64 positions on
      rowB *= g64;
      if (a.need_z) {
        const float gL = L == kC ? g64 : gpow(lng, L);
        const float *ks = reinterpret_cast<const float *>(st + kOffKs);
        for (int k2 = et; k2 < DK; k2 += 128) zsm[k2] = fmaf(gL, zsm[k2], ks[k2]);
      }
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[EMPTY0 + s]);  // done with Q' and the key sums
    }
    if (ok && a.z_out && rank == 0 && last_seg)
      for (int k2 = et; k2 < DK; k2 += 128) a.z_out[(long long)bh * DK + k2] = zsm[k2];
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ state group
    const int G = 1;
    const int q = warp & 3;                 // TMEM lane quarter
    const int et = tid - 256;               // 0..127
    const int vrow = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const long long vglob = v0 + vrow;
    float *rd = red + 16;
    int rslot = 0;
    bool ok = true;
    // Entry state (S_in, or for a later segment the decayed sum of S_in and
    // the pieces before it) goes to the TMEM state columns; its max |S| is
    // the helper's first state bound.
    // The first half of the entry state's rows here, the second half in the
    // output group (idle until the first chunk's O^T): both halves are in
    // TMEM, and the output group's bounds in OT (unused until then), after
    // the two groups' join barrier.
    const bool has_state = a.S_in != nullptr || npc > 0;
    float m0 = has_state ? load_entry_state(p, a, tb + lb + kTS, bh, vglob, seg, c0, npc, lng, 0,
                                            DK / 64)
                         : 0.f;
    if (has_state) {
      tc::tc_fence_before();
      asm volatile("bar.sync 5, 256;" ::: "memory");
      tc::tc_fence_after();
      m0 = fmaxf(m0, OT[et]);
    }
    {
      const float sb = grp_max(G, m0, rd, rslot, et);
      if (et == 0) {
        vmxs[1] = sb;
        tc::mbar_arrive(&bars[SB0]);
      }
    }
    int sigma = 0;  // TMEM state holds S * 2^-sigma
    // d_k = 256 runs in two halves of 128 columns, each handed to the MMA
    // thread as soon as it is done (SRDY0/SRDY1), and each refreshed for the
    // next chunk as soon as the MMAs of its half are done (SFULL0/SFULL1).
    const int nh = DK == 256 ? 2 : 1;
    const int gh = DK / 32 / nh;  // 32-column blocks per half (even)
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1;
      Scales sc;
      for (int hh = 0; hh < nh && ok; ++hh) {
        const int sf = nh == 1 ? SFULL1 : SFULL0 + hh;
        ok = grp_all(G, (hh > 0 || wait_bar(&bars[VRDY0 + s], (lc >> 1) & 1, abort_p, p.status)) &&
                            (lc == 0 || wait_bar(&bars[sf], (lc - 1) & 1, abort_p, p.status)));
        if (!ok) break;
        tc::tc_fence_after();
        if (hh == 0) sc = scs[s];
        // fp16 copy of S_c * 2^-ss for the cross term; S_acc <- gamma^L S_c *
        // 2^-sigma_next.  The loads of the next 32 columns overlap the work
        // on the current ones.
        const int g0 = hh * gh, g1 = g0 + gh;
        if (lc == 0 && !has_state) {
          uint32_t z32[32], z16[16];
#pragma unroll
          for (int i = 0; i < 32; ++i) z32[i] = 0u;
#pragma unroll
          for (int i = 0; i < 16; ++i) z16[i] = 0u;
#pragma unroll 1
          for (int g = g0; g < g1; ++g) {
            tc::tmem_st16(tb + lb + kTSh + g * 16, z16);
            tc::tmem_st32(tb + lb + kTS + g * 32, z32);
          }
        } else {
          const float2 fcp2 = make_float2(sc.f_cp, sc.f_cp), fpre2 = make_float2(sc.f_pre, sc.f_pre);
          uint32_t ra[32], rb[32];
          tc::tmem_ld32(tb + lb + kTS + g0 * 32, ra);
#pragma unroll 1
          for (int g = g0; g < g1; g += 2) {
            tc::tmem_ld_wait_on(ra);
            tc::tmem_ld32(tb + lb + kTS + (g + 1) * 32, rb);
            {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 x = make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
                const float2 y = tc::mul2(x, fcp2);
                pk[i] = tc::pack_f16(y.x, y.y);
                const float2 w = tc::mul2(x, fpre2);
                ra[2 * i] = __float_as_uint(w.x);
                ra[2 * i + 1] = __float_as_uint(w.y);
              }
              tc::tmem_st16(tb + lb + kTSh + g * 16, pk);
              tc::tmem_st32(tb + lb + kTS + g * 32, ra);
            }
            tc::tmem_ld_wait_on(rb);
            if (g + 2 < g1) tc::tmem_ld32(tb + lb + kTS + (g + 2) * 32, ra);
            {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 x = make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
                const float2 y = tc::mul2(x, fcp2);
                pk[i] = tc::pack_f16(y.x, y.y);
                const float2 w = tc::mul2(x, fpre2);
                rb[2 * i] = __float_as_uint(w.x);
                rb[2 * i + 1] = __float_as_uint(w.y);
              }
              tc::tmem_st16(tb + lb + kTSh + (g + 1) * 16, pk);
              tc::tmem_st32(tb + lb + kTS + (g + 1) * 32, rb);
            }
          }
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        grp_sync(G);
        if (et == 0) tc::mbar_arrive(&bars[SRDY0 + hh]);
      }
      sigma = sc.sigma_next;
    }
    if (ok && a.S_out && last_seg) {
      ok = grp_all(G, wait_bar(&bars[SFULL1], (ncl - 1) & 1, abort_p, p.status));
      if (ok) {
        tc::tc_fence_after();
        store_state(p, a.S_out, tb + lb + kTS, bh, vglob, exp2f((float)sigma));
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ output group
    const int G = 2;
    const int q = warp & 3;
    const int et = tid - 384;  // 0..127
    const int vrow = q * 32 + lane;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const bool gn = p.gn_eps >= 0.f;
    // Statistics: 4 threads per token, each reading eight 16-byte column
    // groups (conflict-free with a row pitch of 144 floats); 32 tokens per
    // pass, two passes.
    const int sq4 = et & 3, st0 = et >> 2;
    const float inv_nv = 1.f / (float)NV;
    if (a.S_in != nullptr || npc > 0) {  // the second half of the entry state's rows
      OT[et] = load_entry_state(p, a, tb + lb + kTS, bh, v0 + vrow, seg, c0, npc, lng, DK / 64,
                                DK / 32);
      tc::tc_fence_before();
      asm volatile("bar.sync 5, 256;" ::: "memory");
    }
    bool ok = true;
    for (int lc = 0; lc < ncl && ok; ++lc) {
      const int s = lc & 1, c = c0 + lc;
      const int L = min(kC, N - c * kC);
      ok = grp_all(G, wait_bar(&bars[OFULL0 + s], (lc >> 1) & 1, abort_p, p.status) &&
                          wait_bar(&bars[FRDY0 + s], (lc >> 1) & 1, abort_p, p.status));
      if (!ok) break;
      tc::tc_fence_after();
      // Per-chunk factors are read before OFREE: the R group rewrites them
      // for chunk lc+2 only after the scores of lc+2, which go to this O^T
      // buffer after OFREE.
      const float osc = oss[s];
      const float osc_inv = __frcp_rn(osc);  // osc is a power of two
      float fr[2];
      fr[0] = fsm[s * 64 + st0];
      fr[1] = fsm[s * 64 + st0 + 32];
      {
        uint32_t t0[32], t1[32];
        tc::tmem_ld32(tb + lb + tcol_o(lc), t0);
        tc::tmem_ld32(tb + lb + tcol_o(lc) + 32, t1);
        tc::tmem_ld_wait_on(t0);
        tc::tmem_ld_wait_on(t1);
        tc::tc_fence_before();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          OT[i * kOTPitch + vrow] = __uint_as_float(t0[i]);
          OT[(32 + i) * kOTPitch + vrow] = __uint_as_float(t1[i]);
        }
      }
      grp_sync(G);
      if (et == 0) tc::mbar_arrive(&bars[OFREE0 + s]);
      // Each thread reads its 2 x 32 values (tokens st0 and st0+32, column
      // groups 4(sq4 + 4m)) for the statistics, and again for the stores.
      float4 x[2][8];
      float mloc[2], M2loc[2];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const float4 *row =
            reinterpret_cast<const float4 *>(OT + (st0 + 32 * pass) * kOTPitch) + sq4;
#pragma unroll
        for (int m = 0; m < 8; ++m) x[pass][m] = row[4 * m];
      }
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        float2 sab = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 8; ++m)
          sab = tc::add2(sab, tc::add2(make_float2(x[pass][m].x, x[pass][m].y),
                                       make_float2(x[pass][m].z, x[pass][m].w)));
        float mu = sab.x + sab.y;
        mu += __shfl_xor_sync(0xffffffffu, mu, 1);
        mu += __shfl_xor_sync(0xffffffffu, mu, 2);
        mu *= (1.f / kW);
        const float2 nmu = make_float2(-mu, -mu);
        float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float2 d0 = tc::add2(make_float2(x[pass][m].x, x[pass][m].y), nmu);
          const float2 d1 = tc::add2(make_float2(x[pass][m].z, x[pass][m].w), nmu);
          q2 = tc::fma2(d0, d0, q2);
          q2 = tc::fma2(d1, d1, q2);
        }
        float M2 = q2.x + q2.y;
        M2 += __shfl_xor_sync(0xffffffffu, M2, 1);
        M2 += __shfl_xor_sync(0xffffffffu, M2, 2);
        mloc[pass] = mu * osc;  // O^T holds O * 2^-E; osc = 2^E
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
#pragma unroll 4
          for (int r2 = 0; r2 < NV; ++r2)
#pragma unroll
            for (int pass = 0; pass < 2; ++pass)
              tc::st_async_v2(gns + ((par * 8 + rank) * 64 + st0 + 32 * pass) * 2, &bars[GN0 + par],
                              r2, mloc[pass], M2loc[pass]);
        ok = grp_all(G, wait_bar_cluster(&bars[GN0 + par], (lc >> 1) & 1, abort_p, p.status));
        if (!ok) break;
        // Chan's merge of the NV partial (mean, M2) pairs of kW columns each.
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const float2 *sl = reinterpret_cast<const float2 *>(gns) + (par * 8) * 64 + st0 + 32 * pass;
          float msum = 0.f;
#pragma unroll 1
          for (int r2 = 0; r2 < NV; ++r2) msum += sl[r2 * 64].x;
          const float mu = msum * inv_nv;
          float M2t = 0.f;
#pragma unroll 1
          for (int r2 = 0; r2 < NV; ++r2) {
            const float2 pr = sl[r2 * 64];
            const float d = pr.x - mu;
            M2t += pr.y + (float)kW * d * d;
          }
          mean[pass] = mu;
          var[pass] = M2t * (inv_nv * (1.f / kW));
        }
      }
      // GroupNorm of x = f o: y = (o - mean) f / sqrt(f^2 var + eps); no
      // GroupNorm: y = f o.  Stored O^T is O * 2^-E: fold 2^E into the
      // per-token shift and scale.  Each thread stores its own values: for a
      // column group m, the 4 threads of a token write 16 consecutive
      // columns (32 bytes of bf16).
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        const int ti = st0 + 32 * pass;
        if (ti >= L) continue;
        const float4 *row = reinterpret_cast<const float4 *>(OT + ti * kOTPitch) + sq4;
        const float f = pass ? fr[1] : fr[0];
        const float mn = pass ? mean[1] : mean[0], vr = pass ? var[1] : var[0];
        const float shift = gn ? mn * osc_inv : 0.f;
        const float scale = (gn ? f * rsqrtf(f * f * vr + p.gn_eps) : f) * osc;
        const float2 sh2 = make_float2(-shift, -shift), sc2 = make_float2(scale, scale);
        const long long tok = (long long)c * kC + ti;
        const long long ob0 = b * p.so[0] + h * p.so[1] + tok * p.so[2] + v0 + 4 * sq4;
#pragma unroll 4  // loads and stores of four groups in flight (unrolled 1 or 8 is slower)
        for (int m = 0; m < 8; ++m) {
          const long long ob = ob0 + 16 * m;
          const float4 xm = row[4 * m];
          const float2 y0 = tc::mul2(tc::add2(make_float2(xm.x, xm.y), sh2), sc2);
          const float2 y1 = tc::mul2(tc::add2(make_float2(xm.z, xm.w), sh2), sc2);
          if (kStore != kStoreAny || (a.vec_out && p.out_bf16)) {
            *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(a.o) + ob) =
                make_uint2(tc::pack_bf16(y0.x, y0.y), tc::pack_bf16(y1.x, y1.y));
          } else if (a.vec_out) {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + ob) =
                make_float4(y0.x, y0.y, y1.x, y1.y);
          } else {
            st_elem(a.o, ob, y0.x, p.out_bf16);
            st_elem(a.o, ob + 1, y0.y, p.out_bf16);
            st_elem(a.o, ob + 2, y1.x, p.out_bf16);
            st_elem(a.o, ob + 3, y1.y, p.out_bf16);
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
                            const float *z_in, float *S_out, float *z_out, void *o,
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
  void (*kern)(KParams, CUtensorMap, CUtensorMap, CUtensorMap, TcArgs) =
      a.vec_out && p.out_bf16 ? chunk_tc_kernel<kStoreBf16> : chunk_tc_kernel<kStoreAny>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P * BH * a.NV));
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.NV;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p, tq, tk, tv, a);
}

}  // namespace ret
