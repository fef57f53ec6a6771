// One recurrent decode step (hwhale.com/article/285883, recurrent form
// S_n = gamma S_{n-1} + K_n^T V_n, Retention(X_n) = Q_n S_n, and the
// RecurrentRetention pseudocode: the output is read after the state update
// and summed over the key dimension; m0nads.wordpress.com, recurrent
// representation).  Followed by the per-head GroupNorm.
//
// Memory-bound: every step reads and writes the fp32 state S once
// (8 bytes per element).  Layout of work:
//   * a cluster of KS CTAs per (batch, head); CTA r owns rows
//     [r*dk/KS, (r+1)*dk/KS) of S (and of z) and output columns
//     [r*dv/KS, (r+1)*dv/KS);
//   * each thread holds a block of rows (8, or 32 when the grid is no larger
//     than the SM count) of one 16-byte column slice of S (float4 along d_v)
//     in registers.  The loads of the first such block are issued before the
//     inputs q, k, v are fetched and rotated, so the two latencies overlap;
//     the block is updated in registers, written back, and its share of q.S
//     accumulated;
//   * partial outputs are pushed into the owning CTA's shared memory
//     (asynchronous distributed shared memory stores that count their bytes
//     on the owner's mbarrier; no remote loads) and summed there in a fixed
//     order once the owner has seen all the bytes it expects: deterministic,
//     no atomics, and no cluster-wide barrier, whose release half would wait
//     for this step's state stores to drain (with the state in L2 and more
//     CTAs than SMs, plain stores and cluster barriers measured faster);
//   * GroupNorm: each CTA reduces its own columns to a (mean, M2) pair, the
//     pairs are pushed to every CTA of the cluster the same way and merged
//     there (Chan's pairwise update).  Every CTA waits for all the bytes
//     addressed to it, so none leaves while a peer may still write to it.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace ret {

namespace {
constexpr int NT = 128;   // threads per CTA
constexpr int KSMAX = 8;  // CTAs per cluster at most

// Sum `val` over the CTA; every thread gets the total (all threads must call).
__device__ __forceinline__ float block_sum(float val, float *wsum, int tid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
  if ((tid & 31) == 0) wsum[tid >> 5] = val;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += wsum[w];
  __syncthreads();  // wsum is reused by the next call
  return t;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Bounded wait (acquire at cluster scope) for phase 0 of an exchange
// barrier; each try suspends the thread for a while, so 2^20 tries are far
// beyond any legitimate wait.  A wait that runs out records the timeout
// and gives up.
__device__ __noinline__ void xwait(uint64_t *bar, unsigned *status) {
  for (unsigned i = 0; i < (1u << 20); ++i)
    if (tc::mbar_try_wait_cluster(bar, 0)) return;
  report(status, kDevTimeout);
}
}  // namespace

// RB = rows of S a thread holds in registers at once.  kAsyncX: the
// exchanges count their bytes on mbarriers (else: cluster barriers).
// kFullRow (with kAsyncX): every CTA receives the partials of all d_v
// columns and normalises the whole row itself, so the GroupNorm needs no
// second exchange (a few microseconds less at small batches, where the
// step is a chain of latencies).
// kGate: the MSR gate is applied to the output (a separate instantiation,
// so that the plain step keeps its register budget).
template <int RB, bool kAsyncX, bool kFullRow, bool kGate>
__global__ void __launch_bounds__(NT)
recurrent_step_kernel(KParams p, int KS, const void *__restrict__ q,
                      const void *__restrict__ k, const void *__restrict__ v,
                      float *__restrict__ S, float *__restrict__ z, void *__restrict__ o,
                      const __nv_bfloat16 *__restrict__ gate) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float wsum[NT / 32];
  __shared__ float qz_in[KSMAX];     // partial q.z pushed by each CTA
  __shared__ __align__(8) float2 st_in[KSMAX];  // (mean, M2) of each CTA's columns
  __shared__ __align__(8) uint64_t xbar[2];  // bytes of [0] partials and q.z, [1] statistics
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int bh = blockIdx.x / KS;
  const int b = bh / p.H, h = bh % p.H;
  const int dk = p.dk, dv = p.dv;
  const int R = dk / KS, k0 = rank * R, span = dv / KS;
  const int nvec = dv / 4;
  const int tid = threadIdx.x;
  float4 *Srow0 = reinterpret_cast<float4 *>(S + ((long long)bh * dk + k0) * dv);

  // Wait for the kernel before this one (the previous step's state stores)
  // before any global access.
  pdl_wait();
  // First block of S: rows 0..min(R,RB)-1 of column slice tid.  Nothing
  // these loads need depends on the inputs, so they go out first.
  float4 s[RB];
  if (tid < nvec) {
#pragma unroll
    for (int u = 0; u < RB; ++u)
      if (u < R) s[u] = Srow0[(long long)u * nvec + tid];
  }
  // The exchange barriers, each expecting the bytes its CTA will receive:
  // from every CTA of the cluster, its partial q.z and q.S for this CTA's
  // columns, and (GroupNorm) its column statistics.
  const bool gn = p.gn_eps >= 0.f;
  if (kAsyncX && tid == 0) {
    tc::mbar_init(&xbar[0], 1);
    tc::mbar_init(&xbar[1], 1);
    tc::fence_mbar_init();
    tc::mbar_arrive_expect_tx(&xbar[0], (uint32_t)(KS * ((kFullRow ? dv : span) + 1) * 4));
    if (gn && !kFullRow) tc::mbar_arrive_expect_tx(&xbar[1], (uint32_t)(KS * 8));
  }
  // Peers' shared memory may be written only once every CTA of the
  // cluster runs (and has set up its barriers): arrive now, wait just
  // before the first push.
  cluster_arrive_relaxed();

  const float g = p.gam[h];
  float *qr = sm;             // [R]
  float *kr = qr + R;         // [R]
  float *vs = kr + R;         // [dv]
  float *inbox = vs + dv;     // [KS][span] (kFullRow: [KS][dv]): partial q.S

  // Rotated q, k rows of this CTA (positions: the token sits at pos0).
  const long long qb = b * p.sq[0] + h * p.sq[1];
  const long long kb = b * p.sk[0] + h * p.sk[1];
  for (int t = tid; t < R / 2; t += NT) {
    const int j = k0 / 2 + t;
    float q0 = ld_elem(q, qb + 2 * j, p.in_bf16), q1 = ld_elem(q, qb + 2 * j + 1, p.in_bf16);
    float c0 = ld_elem(k, kb + 2 * j, p.in_bf16), c1 = ld_elem(k, kb + 2 * j + 1, p.in_bf16);
    if (p.rotate) {
      float cs, sn;
      rot_cs(p.pos0, p.th_hi[j], p.th_lo[j], cs, sn);
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
  cluster_wait();

  // z <- gamma z + k (rows of this CTA); the partial q.z of the row sum goes
  // to every CTA of the cluster.
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
    for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
    if (tid < KS) {
      if (kAsyncX)
        tc::st_async_f32(&qz_in[rank], &xbar[0], (uint32_t)tid, part);
      else
        cluster.map_shared_rank(qz_in, tid)[rank] = part;
    }
  }

  // Rows: S <- gamma S + k_a v ; acc += q_a S.  The first block is already
  // in registers; further column slices and row blocks (d_v > 512 or more
  // than 32 rows per CTA) are loaded here.
  for (int c = tid; c < nvec; c += NT) {
    const float4 vv = reinterpret_cast<const float4 *>(vs)[c];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int a0 = 0; a0 < R; a0 += RB) {
      if (c != tid || a0 != 0) {
#pragma unroll
        for (int u = 0; u < RB; ++u)
          if (a0 + u < R) s[u] = Srow0[(long long)(a0 + u) * nvec + c];
      }
#pragma unroll
      for (int u = 0; u < RB; ++u) {
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
    // Columns 4c..4c+3 belong to CTA e/span (span is a multiple of 4).
    const int e = 4 * c, dst = e / span;
    if (kFullRow) {
      for (int r = 0; r < KS; ++r)
        tc::st_async_v4(inbox + rank * dv + e, &xbar[0], (uint32_t)r, acc);
    } else if (kAsyncX)
      tc::st_async_v4(inbox + rank * span + (e - dst * span), &xbar[0], (uint32_t)dst, acc);
    else
      *reinterpret_cast<float4 *>(cluster.map_shared_rank(inbox, dst) + rank * span +
                                  (e - dst * span)) = acc;
  }
  // The state is written: the next kernel may be scheduled (it waits for
  // this one to complete in its own pdl_wait).
  pdl_launch_dependents();
  if (kAsyncX)
    xwait(&xbar[0], p.status);
  else
    cluster.sync();  // release the pushes above, acquire the peers'

  // Fixed-order sums of the KS partials for this CTA's columns
  // e0 + tid + NT*i (span = dv/KS <= 1024 columns, so i < 8).
  const int e0 = rank * span;
  float qz = 0.f;
  for (int r = 0; r < KS; ++r) qz += qz_in[r];
  const float sc = row_scale(p, h, p.pos0 + 1);
  const float f = sc * rsum_scale(p, sc * qz);
  if (kFullRow) {
    // The whole row: columns 4c..4c+3 for c = tid, tid + NT (d_v <= 1024).
    float4 xs[2];
    float lsum = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + NT * i;
      xs[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nvec) {
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < KS; ++r) {
          const float4 t4 = *reinterpret_cast<const float4 *>(inbox + r * dv + 4 * c);
          a4.x += t4.x; a4.y += t4.y; a4.z += t4.z; a4.w += t4.w;
        }
        xs[i] = make_float4(f * a4.x, f * a4.y, f * a4.z, f * a4.w);
        lsum += (xs[i].x + xs[i].y) + (xs[i].z + xs[i].w);
      }
    }
    float mu = 0.f, inv = 1.f;
    if (gn) {
      mu = block_sum(lsum, wsum, tid) / dv;
      float lm2 = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (tid + NT * i < nvec) {
          lm2 = fmaf(xs[i].x - mu, xs[i].x - mu, lm2);
          lm2 = fmaf(xs[i].y - mu, xs[i].y - mu, lm2);
          lm2 = fmaf(xs[i].z - mu, xs[i].z - mu, lm2);
          lm2 = fmaf(xs[i].w - mu, xs[i].w - mu, lm2);
        }
      inv = rsqrtf(block_sum(lm2, wsum, tid) / dv + p.gn_eps);
    }
    const long long ob = b * p.so[0] + h * p.so[1];
    const long long gb = ((long long)b * p.H + h) * dv;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + NT * i;
      if (c >= nvec || 4 * c < e0 || 4 * c >= e0 + span) continue;
      const float xv[4] = {xs[i].x, xs[i].y, xs[i].z, xs[i].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float y = (xv[u] - mu) * inv;
        if (kGate) {
          const float gi = __bfloat162float(gate[gb + 4 * c + u]);
          y = __bfloat162float(__float2bfloat16_rn(y)) * __fdividef(gi, 1.f + __expf(-gi));
        }
        st_elem(o, ob + 4 * c + u, y, p.out_bf16);
      }
    }
    return;
  }
  float x[8];
  float lsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = tid + NT * i;
    x[i] = 0.f;
    if (e < span) {
      float acc = 0.f;
      for (int r = 0; r < KS; ++r) acc += inbox[r * span + e];
      x[i] = f * acc;
      lsum += x[i];
    }
  }
  float mu = 0.f, inv = 1.f;
  if (p.gn_eps >= 0.f) {
    // This CTA's (mean, M2) over its span columns, then the merge of the
    // KS equal-sized groups: M2 = sum M2_r + span * sum (mean_r - mean)^2.
    const float mloc = block_sum(lsum, wsum, tid) / span;
    float lm2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (tid + NT * i < span) lm2 = fmaf(x[i] - mloc, x[i] - mloc, lm2);
    const float m2loc = block_sum(lm2, wsum, tid);
    if (kAsyncX) {
      if (tid < KS)
        tc::st_async_v2(reinterpret_cast<float *>(&st_in[rank]), &xbar[1], (uint32_t)tid, mloc,
                        m2loc);
      xwait(&xbar[1], p.status);
    } else {
      if (tid < KS) cluster.map_shared_rank(st_in, tid)[rank] = make_float2(mloc, m2loc);
      cluster.sync();
    }
    float msum = 0.f;
    for (int r = 0; r < KS; ++r) msum += st_in[r].x;
    mu = msum / KS;
    float m2 = 0.f, dm2 = 0.f;
    for (int r = 0; r < KS; ++r) {
      const float2 st = st_in[r];
      m2 += st.y;
      dm2 = fmaf(st.x - mu, st.x - mu, dm2);
    }
    m2 = fmaf((float)span, dm2, m2);
    inv = rsqrtf(m2 / dv + p.gn_eps);
  }
  const long long ob = b * p.so[0] + h * p.so[1] + e0;
  // The MSR layer's gate, when given (bf16 [B][H][d_v]): the GroupNorm
  // output rounded to bf16 as it would be stored, times swish(g) (fast
  // exponential and divide, as the separate gate pass computes it).
  const long long gb = ((long long)b * p.H + h) * dv + e0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (tid + NT * i < span) {
      float y = (x[i] - mu) * inv;
      if (kGate) {
        const float gi = __bfloat162float(gate[gb + tid + NT * i]);
        y = __bfloat162float(__float2bfloat16_rn(y)) * __fdividef(gi, 1.f + __expf(-gi));
      }
      st_elem(o, ob + tid + NT * i, y, p.out_bf16);
    }
}

cudaError_t launch_recurrent_step(const KParams &p, const void *q, const void *k,
                                  const void *v, float *S, float *z, void *o,
                                  cudaStream_t st, const void *gate) {
  if (p.B == 0 || p.H == 0) return cudaSuccess;
  // Cluster size: up to 8 CTAs per head, each keeping an even number of
  // rows and an equal share of the outputs, a multiple of 4 columns
  // (<= 8 * NT of them; d_v <= 1024).
  int KS = KSMAX;
  while (KS > 1 && (p.dk % KS || (p.dk / KS) % 2 || p.dv % KS || (p.dv / KS) % 4)) KS >>= 1;
  const int R = p.dk / KS;
  const size_t smem = sizeof(float) * (2 * R + 2 * p.dv);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.H * KS));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic serialization: the step's CTAs are placed while the kernel
  // before it (usually the previous step) finishes, and wait in pdl_wait.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // Row block: with at most one CTA per SM (small batches) the step is
  // latency-bound and every thread keeps all its rows (<= 32) in flight at
  // once; with more CTAs than SMs it is bandwidth-bound, and 8 rows a thread
  // (64 registers) let eight CTAs share an SM.  Measured at H=16, d_k=256,
  // d_v=512: 7.4 vs 7.9 us per step at B=1; 16.3 vs 26.2 us at B=8 and
  // 328 vs 400 us at B=128.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  //
  // Exchange: counted asynchronous pushes except where the state fits in
  // L2 with more CTAs than SMs (measured at B=1 / 8 / 32 / 128: 7.30 / 19.7
  // / 85.6 / 316.7 us with them, 7.44 / 16.9 / 90 / 329 with cluster
  // barriers, whose release half waits for the state stores to drain).
  const __nv_bfloat16 *g = reinterpret_cast<const __nv_bfloat16 *>(gate);
  const bool gated = g != nullptr;
  // Programmatic serialization only while the grid fits on the SMs (one CTA
  // each): with more CTAs, the next step's early CTAs share SMs with this
  // one's.  Measured at H=16, d_k=256, d_v=512: 6.40 vs 6.56 us per step at
  // B=1 with it, 17.3 vs 16.8 at B=8.
  if ((long long)p.B * p.H * KS > sms) cfg.numAttrs = 1;
  if ((long long)p.B * p.H * KS <= sms) {
    cfg.dynamicSmemBytes = sizeof(float) * (2 * R + p.dv + (size_t)KS * p.dv);
    return gated ? cudaLaunchKernelEx(&cfg, recurrent_step_kernel<32, true, true, true>, p, KS, q, k, v, S, z, o, g)
                 : cudaLaunchKernelEx(&cfg, recurrent_step_kernel<32, true, true, false>, p, KS, q, k, v, S, z, o, g);
  }
  const double state_bytes = (double)p.B * p.H * p.dk * p.dv * 4.0;
  if (state_bytes <= 96e6)
    return gated ? cudaLaunchKernelEx(&cfg, recurrent_step_kernel<8, false, false, true>, p, KS, q, k, v, S, z, o, g)
                 : cudaLaunchKernelEx(&cfg, recurrent_step_kernel<8, false, false, false>, p, KS, q, k, v, S, z, o, g);
  return gated ? cudaLaunchKernelEx(&cfg, recurrent_step_kernel<8, true, false, true>, p, KS, q, k, v, S, z, o, g)
               : cudaLaunchKernelEx(&cfg, recurrent_step_kernel<8, true, false, false>, p, KS, q, k, v, S, z, o, g);
}

}  // namespace ret
