// C ABI of the retention library: argument checks, per-head constants,
// workspace layout and dispatch to the kernels.  Nothing here allocates
// device memory or synchronises a stream (retention_poll_status excepted).
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#ifdef RET_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#include "common.cuh"
#include "ktimer.h"
#include "launch.h"

using namespace ret;

namespace {

thread_local int g_last_cuda_error = 0;

// Optional NVTX range per ABI call (build with RET_NVTX=1 in the environment):
// names the calls on a profiler's timeline.
#ifdef RET_NVTX
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define RET_RANGE(name) NvtxRange ret_range_(name)
#else
#define RET_RANGE(name) ((void)0)
#endif

// Tries of the prologue's reporting wait (retention_set_report_wait_budget).
std::atomic<unsigned> g_report_budget{1u << 24};

ret_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return RET_ECUDA;
}

#define RET_CUDA(call)                        \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool finite_pos(double x) { return isfinite(x) && x > 0.0; }

// Checks shared by every retention_* entry point.
bool desc_ok(const ret_desc *d) {
  if (!d) return false;
  if (d->B < 0 || d->H < 0 || d->N < 0) return false;
  if (d->H > RET_MAX_HEADS) return false;
  if ((long long)d->B * d->H > 65535) return false;
  if (d->d_k < 2 || d->d_k > 2 * kMaxPairs || (d->d_k % 2)) return false;
  if (d->d_v < 1 || d->d_v > 1024) return false;
  if (d->chunk < 1 || d->chunk > 256) return false;
  if (d->in_dtype != RET_F32 && d->in_dtype != RET_BF16) return false;
  if (d->out_dtype != RET_F32 && d->out_dtype != RET_BF16) return false;
  if (d->norm_flags & ~(RET_NORM_SCALE | RET_NORM_DROW | RET_NORM_RSUM)) return false;
  if (!(d->gn_eps == d->gn_eps)) return false;  // NaN
  if (d->pos0 < 0 || d->pos0 + (int64_t)d->N >= ((int64_t)1 << 24)) return false;
  if (d->rotate != 0 && d->rotate != 1) return false;
  if (d->rotate && !finite_pos(d->theta_base)) return false;
  if (d->H > 0 && !d->gamma) return false;
  for (int h = 0; h < d->H; ++h)
    if (!(d->gamma[h] >= 0.0 && d->gamma[h] <= 1.0)) return false;
  for (int i = 0; i < 3; ++i)
    if (d->sq[i] < 0 || d->sk[i] < 0 || d->sv[i] < 0 || d->so[i] < 0) return false;
  return true;
}

void make_params(const ret_desc *d, void *ws, KParams &p) {
  memset(&p, 0, sizeof(p));
  p.B = d->B; p.H = d->H; p.N = d->N; p.dk = d->d_k; p.dv = d->d_v; p.chunk = d->chunk;
  for (int i = 0; i < 3; ++i) {
    p.sq[i] = d->sq[i]; p.sk[i] = d->sk[i]; p.sv[i] = d->sv[i]; p.so[i] = d->so[i];
  }
  p.pos0 = d->pos0;
  p.norm_flags = d->norm_flags;
  p.rotate = d->rotate;
  p.in_bf16 = d->in_dtype == RET_BF16;
  p.out_bf16 = d->out_dtype == RET_BF16;
  p.gn_eps = d->gn_eps;
  p.inv_sqrt_dk = (float)(1.0 / sqrt((double)d->d_k));
  for (int h = 0; h < d->H; ++h) {
    const double g = d->gamma[h];
    p.gam[h] = (float)g;
    p.lng[h] = g == 0.0 ? -INFINITY : (float)log(g);
    p.omg[h] = (float)(1.0 - g);
  }
  for (int j = 0; j < d->d_k / 2; ++j) {
    const double th = d->rotate ? pow(d->theta_base, -2.0 * j / d->d_k) : 0.0;
    p.th_hi[j] = (float)th;
    p.th_lo[j] = (float)(th - (double)p.th_hi[j]);
  }
  p.status = reinterpret_cast<unsigned *>(ws);
  p.report_budget = g_report_budget.load(std::memory_order_relaxed);
}

// Workspace of the CUDA-core forms: status | Qr | Kr | Oraw | F | z copy.
struct SimtWs {
  size_t qr, kr, oraw, f, zc, total;
};

SimtWs simt_ws(const ret_desc *d) {
  SimtWs w;
  const size_t rows = (size_t)d->B * d->H * d->N;
  size_t off = kStatusBytes;
  w.qr = off; off = align256(off + rows * d->d_k * sizeof(float));
  w.kr = off; off = align256(off + rows * d->d_k * sizeof(float));
  w.oraw = off; off = align256(off + rows * d->d_v * sizeof(float));
  w.f = off; off = align256(off + rows * sizeof(float));
  w.zc = off; off = align256(off + (size_t)d->B * d->H * d->d_k * sizeof(float));
  w.total = off;
  return w;
}

// Workspace of the parallel form on the tensor cores: status | Q' | K'
// (fp16) | per-chunk records | raw rows (fp32) | row factors.
struct ParTcWs {
  size_t qp, kp, meta, oraw, f, total;
};

ParTcWs par_tc_ws(const ret_desc *d) {
  ParTcWs w;
  const size_t BH = (size_t)d->B * d->H, rows = BH * d->N;
  const size_t nch = ((size_t)d->N + 63) / 64;
  size_t off = kStatusBytes;
  w.qp = off; off = align256(off + rows * d->d_k * 2);
  w.kp = off; off = align256(off + rows * d->d_k * 2);
  w.meta = off; off = align256(off + BH * nch * sizeof(ChunkMeta));
  w.oraw = off; off = align256(off + rows * d->d_v * sizeof(float));
  w.f = off; off = align256(off + rows * sizeof(float));
  w.total = off;
  return w;
}

// Workspace of the backward: status | Q' | K' | dQ' | dK' (fp32 rows).
struct BwdWs {
  size_t qr, kr, dq, dk, total;
};

BwdWs bwd_ws(const ret_desc *d) {
  BwdWs w;
  const size_t bytes = (size_t)d->B * d->H * d->N * d->d_k * sizeof(float);
  size_t off = kStatusBytes;
  w.qr = off; off = align256(off + bytes);
  w.kr = off; off = align256(off + bytes);
  w.dq = off; off = align256(off + bytes);
  w.dk = off; off = align256(off + bytes);
  w.total = off;
  return w;
}

// Sequence segments of the tensor-core chunk kernel: at most kMaxSegments
// segments of at least kMinSegChunks chunks, and at most kMaxPieces pieces
// of partial state.
constexpr int kMaxSegments = 8, kMinSegChunks = 4, kMaxPieces = 8;

bool split_possible(const ret_desc *d) {
  const long long nch = ((long long)d->N + 63) / 64;
  return d->chunk == 64 && nch >= 2 * kMinSegChunks;
}

// Workspace of the tensor-core chunkwise path: status | Q' | K' | z copy |
// per-chunk records, key column sums | (segments) S copy, pieces.
// Q'/K' are fp16 with per-(head, chunk) exponents and magnitudes.
struct TcWs {
  size_t qp, kp, zc, meta, ks, sc, part, zpart, total;
};

TcWs tc_ws(const ret_desc *d) {
  TcWs w;
  const size_t BH = (size_t)d->B * d->H;
  const size_t rows = BH * d->N;
  const size_t nch = ((size_t)d->N + d->chunk - 1) / d->chunk;
  size_t off = kStatusBytes;
  w.qp = off; off = align256(off + rows * d->d_k * 2);
  w.kp = off; off = align256(off + rows * d->d_k * 2);
  w.zc = off; off = align256(off + BH * d->d_k * sizeof(float));
  w.meta = off; off = align256(off + BH * nch * sizeof(ChunkMeta));
  w.ks = off; off = align256(off + BH * nch * d->d_k * sizeof(float));
  const size_t sbytes = BH * d->d_k * d->d_v * sizeof(float);
  const bool split = split_possible(d);
  w.sc = off; off = align256(off + (split ? sbytes : 0));
  w.part = off; off = align256(off + (split ? kMaxPieces * sbytes : 0));
  w.zpart = off; off = align256(off + (split ? kMaxPieces * BH * d->d_k * sizeof(float) : 0));
  w.total = off;
  return w;
}

// How the tensor-core path splits the sequence: as many segments as keep
// every segment's CTAs (one per SM) resident together, and enough pieces to
// give the state kernel about two CTAs per SM.
SegPlan plan_segments(const ret_desc *d, int NV) {
  SegPlan pl;
  if (!split_possible(d)) return pl;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return pl;
  const int nch = (d->N + 63) / 64;
  const long long per_seg = (long long)d->B * d->H * NV;
  long long P = sms / per_seg;
  P = P < kMaxSegments ? P : kMaxSegments;
  P = P < nch / kMinSegChunks ? P : nch / kMinSegChunks;
  if (P < 2) return pl;
  const int seg_len = (int)((nch + P - 1) / P);
  P = (nch + seg_len - 1) / seg_len;
  if (P < 2) return pl;
  int split = 1;  // pieces per segment length: a divisor of seg_len
  for (int t = 1; t <= seg_len; ++t)
    if (seg_len % t == 0 && (P - 1) * t <= kMaxPieces && (P - 1) * t * per_seg <= 2LL * sms)
      split = t;
  // Equal segments: a later segment starts after loading its entry state
  // (split between two of the chunk kernel's groups, a few microseconds),
  // and giving the first segment four more chunks to make up for it
  // measured slower at B=1, H=16, N=8192 (304.9 against 303.0 us per step:
  // the state pass then also covers more chunks).
  pl.P = (int)P;
  pl.seg_len = seg_len;
  pl.piece_len = seg_len / split;
  pl.npieces = (int)(P - 1) * split;
  return pl;
}

// The tensor-core kernels work in 64-token chunks.  The chunkwise form is
// the same function for every chunk length (up to rounding), so a request
// for a chunk of 128 or 256 tokens runs there as 64-token chunks; other
// lengths keep the CUDA-core path and their own chunk.
ret_desc tc_desc(const ret_desc *d) {
  ret_desc t = *d;
  if (d->chunk % 64 == 0) t.chunk = 64;
  return t;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(reinterpret_cast<char *>(ws) + off);
}

// Do the byte ranges [a, a + na) and [b, b + nb) share a byte?
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

ret_status check_ws(void *ws, size_t have, size_t need) {
  if (need > 0 && (!ws || have < need)) return RET_EWORKSPACE;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255)) return RET_EWORKSPACE;
  return RET_OK;
}

// Chunkwise form: the tensor-core path where it applies, else CUDA cores.
ret_status chunkwise_impl(const ret_desc *d, const void *q, const void *k, const void *v,
                          const float *S_in, const float *z_in, float *S_out, float *z_out,
                          void *o, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (!desc_ok(d)) return RET_EINVAL;
  const bool empty = d->B == 0 || d->H == 0;
  if (!empty && d->N > 0 && (!q || !k || !v || !o)) return RET_EINVAL;
  KParams p, pt;
  make_params(d, ws, p);
  const ret_desc dt = tc_desc(d);
  make_params(&dt, ws, pt);
  const bool tc = !empty && d->N > 0 && chunk_tc_supported(pt, v, pt.sv);
  const SimtWs w = simt_ws(d);
  const TcWs tw = tc_ws(&dt);
  // The requirement is the one retention_workspace_size reports, whichever
  // kernel runs.
  ret_status rs = check_ws(ws, ws_bytes, w.total > tw.total ? w.total : tw.total);
  if (rs != RET_OK) return rs;
  if (empty) return RET_OK;
  const size_t sbytes = (size_t)d->B * d->H * d->d_k * d->d_v * sizeof(float);
  const size_t zbytes = (size_t)d->B * d->H * d->d_k * sizeof(float);
  if (d->N == 0) {  // no tokens: the state passes through unchanged
    if (S_out && S_out != S_in)
      RET_CUDA(S_in ? cudaMemcpyAsync(S_out, S_in, sbytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(S_out, 0, sbytes, st));
    if (z_out && z_out != z_in)
      RET_CUDA(z_in ? cudaMemcpyAsync(z_out, z_in, zbytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(z_out, 0, zbytes, st));
    return RET_OK;
  }
  if (tc) {
    // Tensor-core path: rotate-and-scale prologue (xi on queries, zeta on
    // keys, bf16), then the fused chunk kernel with the GroupNorm epilogue.
    __half *Qp = at<__half>(ws, tw.qp), *Kp = at<__half>(ws, tw.kp);
    ChunkMeta *meta = at<ChunkMeta>(ws, tw.meta);
    float *ks = at<float>(ws, tw.ks);
    const int need_z = (d->norm_flags & RET_NORM_RSUM) || z_out != nullptr;
    RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate_qk(pt, q, k, Qp, Kp, meta, need_z ? ks : nullptr, st)));
    if (z_in && z_out == z_in) {  // every CTA of a head reads z_in; one writes z_out
      RET_CUDA(cudaMemcpyAsync(at<float>(ws, tw.zc), z_in, zbytes, cudaMemcpyDeviceToDevice, st));
      z_in = at<float>(ws, tw.zc);
    }
    SegPlan seg = plan_segments(&dt, d->d_v / 128);
    if (seg.P > 1) {
      // Segments read S_in at their start while the last one writes S_out.
      if (S_in && S_out == S_in) {
        RET_CUDA(cudaMemcpyAsync(at<float>(ws, tw.sc), S_in, sbytes, cudaMemcpyDeviceToDevice, st));
        S_in = at<float>(ws, tw.sc);
      }
      seg.Part = at<float>(ws, tw.part);
      seg.zPart = at<float>(ws, tw.zpart);
      RET_CUDA(RET_TIMED_LAUNCH(kKStatePass, st, launch_state_tc(pt, Kp, v, meta, ks, seg.npieces, seg.piece_len, seg.Part, seg.zPart, need_z, st)));
    }
    RET_CUDA(RET_TIMED_LAUNCH(kKChunkTc, st, launch_chunk_tc(pt, Qp, Kp, v, meta, ks, S_in, z_in, S_out, z_out, o, need_z, seg, st)));
    return RET_OK;
  }
  float *Qr = at<float>(ws, w.qr), *Kr = at<float>(ws, w.kr);
  float *Oraw = at<float>(ws, w.oraw), *F = at<float>(ws, w.f);
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, q, p.sq, d->d_k, Qr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, k, p.sk, d->d_k, Kr, 0, nullptr, kScaleNone, st)));
  if (z_in && z_out == z_in) {  // every CTA of a head reads z_in; one writes z_out
    RET_CUDA(cudaMemcpyAsync(at<float>(ws, w.zc), z_in, zbytes, cudaMemcpyDeviceToDevice, st));
    z_in = at<float>(ws, w.zc);
  }
  RET_CUDA(RET_TIMED_LAUNCH(kKChunkSimt, st, launch_chunk_simt(p, Qr, Kr, v, S_in, z_in, S_out, z_out, Oraw, F, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKGroupNorm, st, launch_groupnorm(p, Oraw, F, o, st)));
  return RET_OK;
}

// Workspace of the state-only pass.  Tensor-core path: status | K' fp16 |
// per-chunk records | key column sums | pieces [P][B*H][d_k][d_v] and
// [P][B*H][d_k].  CUDA-core path: status | rotated keys fp32.
struct StateWs {
  size_t kp, meta, ks, part, zpart, kr, total;
};

constexpr int kStatePieces = 8;

StateWs state_ws(const ret_desc *d) {
  StateWs w;
  const size_t BH = (size_t)d->B * d->H, rows = BH * d->N;
  const size_t nch = ((size_t)d->N + 63) / 64;
  size_t off = kStatusBytes;
  w.kp = off; off = align256(off + rows * d->d_k * 2);
  w.meta = off; off = align256(off + BH * nch * sizeof(ChunkMeta));
  w.ks = off; off = align256(off + BH * nch * d->d_k * sizeof(float));
  w.part = off; off = align256(off + (size_t)kStatePieces * BH * d->d_k * d->d_v * sizeof(float));
  w.zpart = off; off = align256(off + (size_t)kStatePieces * BH * d->d_k * sizeof(float));
  const size_t tc_total = off;
  w.kr = kStatusBytes;
  const size_t simt_total = align256(kStatusBytes + rows * d->d_k * sizeof(float));
  w.total = tc_total > simt_total ? tc_total : simt_total;
  return w;
}

// The state after the call's tokens, S_out = gamma^N S_in + sum_m
// gamma^(N-1-m) K'_m^T V_m (z likewise), without outputs.  Tensor cores:
// keys-only prologue, the state kernel over pieces of whole chunks, then the
// decayed sum of S_in and the pieces.  CUDA cores otherwise.
ret_status state_impl(const ret_desc *d, const void *k, const void *v, const float *S_in,
                      const float *z_in, float *S_out, float *z_out, void *ws,
                      size_t ws_bytes, cudaStream_t st) {
  if (!desc_ok(d)) return RET_EINVAL;
  const StateWs w = state_ws(d);
  ret_status rs = check_ws(ws, ws_bytes, w.total);
  if (rs != RET_OK) return rs;
  if ((long long)d->B * d->H == 0 || (!S_out && !z_out)) return RET_OK;
  if (d->N > 0 && (!k || !v)) return RET_EINVAL;
  const size_t sbytes = (size_t)d->B * d->H * d->d_k * d->d_v * sizeof(float);
  const size_t zbytes = (size_t)d->B * d->H * d->d_k * sizeof(float);
  if (d->N == 0) {  // no tokens: the state passes through unchanged
    if (S_out && S_out != S_in)
      RET_CUDA(S_in ? cudaMemcpyAsync(S_out, S_in, sbytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(S_out, 0, sbytes, st));
    if (z_out && z_out != z_in)
      RET_CUDA(z_in ? cudaMemcpyAsync(z_out, z_in, zbytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(z_out, 0, zbytes, st));
    return RET_OK;
  }
  ret_desc dt = *d;
  dt.chunk = 64;
  KParams p;
  make_params(&dt, ws, p);
  if (chunk_tc_supported(p, v, p.sv)) {
    __half *Kp = at<__half>(ws, w.kp);
    ChunkMeta *meta = at<ChunkMeta>(ws, w.meta);
    float *ks = at<float>(ws, w.ks);
    const int need_z = z_out != nullptr;
    RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate_qk(p, nullptr, k, nullptr, Kp, meta, need_z ? ks : nullptr, st, true)));
    const int nch = (d->N + 63) / 64;
    const int piece_len = (nch + kStatePieces - 1) / kStatePieces;
    const int P = (nch + piece_len - 1) / piece_len;  // every piece holds a chunk
    float *Part = at<float>(ws, w.part), *zPart = at<float>(ws, w.zpart);
    RET_CUDA(RET_TIMED_LAUNCH(kKStatePass, st, launch_state_tc(p, Kp, v, meta, ks, P, piece_len, Part, zPart, need_z, st)));
    CombineParts parts;
    parts.S[0] = S_in;
    parts.z[0] = z_in;
    parts.t[0] = d->N;
    for (int i = 0; i < P; ++i) {
      const long long end = std::min((long long)(i + 1) * piece_len * 64, (long long)d->N);
      parts.S[1 + i] = Part + (size_t)i * d->B * d->H * d->d_k * d->d_v;
      parts.z[1 + i] = need_z ? zPart + (size_t)i * d->B * d->H * d->d_k : nullptr;
      parts.t[1 + i] = d->N - end;
    }
    parts.count = 1 + P;
    RET_CUDA(RET_TIMED_LAUNCH(kKStateCombine, st, launch_state_combine(p, parts, S_out, z_out, st)));
    return RET_OK;
  }
  float *Kr = at<float>(ws, w.kr);
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, k, p.sk, d->d_k, Kr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKStateSimt, st, launch_state_simt(p, Kr, v, S_in, z_in, S_out, z_out, st)));
  return RET_OK;
}

// ------------------------------------------------- tensor-core backward
// The gradients as five runs of the forward tensor-core path (see
// backward_tc.cu): dv and the state gradient from one run in reversed time,
// dq' and dk' from runs over pieces of d_v (at most 256 wide, the forward's
// score dimension).  bf16 inputs with d_k in {128, 256} and d_v a multiple
// of 128 (at most 1024); other shapes and fp32 take the CUDA-core kernels.
struct BwdTcWs {
  int w = 0, nvc = 0;
  size_t kr = 0, kr_rev = 0, qs_rev = 0, dos = 0, dos_rev = 0, v_rev = 0;
  size_t ts = 0, tds = 0, sdv = 0, dvr = 0, o[kBwdFinishMax] = {}, total = 0;
};

bool bwd_tc_shape(const ret_desc *d) {
  if (!(d->in_dtype == RET_BF16 && (d->d_k == 128 || d->d_k == 256) && d->d_v % 128 == 0 &&
        d->d_v <= 1024 && d->N > 0 && (long long)d->B * d->H > 0 &&
        (long long)d->B * d->H <= 65535))
    return false;
  // The forward's tensor-core range (gamma^64 >= 2^-16), which also keeps
  // the 1/gamma of the reversed runs' entry states small.
  for (int h = 0; h < d->H; ++h)
    if (!(d->gamma[h] > 0.0 && std::log(d->gamma[h]) * 64.0 >= -16.0 * std::log(2.0) * 0.999))
      return false;
  return true;
}

// A forward run inside the backward: bf16 in, fp32 out, no rotation, no
// normalisation, no GroupNorm, contiguous [B*H][N][d] operands unless the
// caller sets other strides.
void bwd_inner_desc(const ret_desc *d, int dk, int dv, ret_desc *r) {
  retention_desc_init(r, d->B, d->H, d->N, dk, dv, d->gamma);
  r->chunk = 64;
  r->in_dtype = RET_BF16;
  r->out_dtype = RET_F32;
  r->rotate = 0;
  r->norm_flags = 0;
  r->gn_eps = -1.f;
  r->pos0 = 0;
}

void contig(const ret_desc *d, int dim, int64_t s[3]) {
  s[0] = (int64_t)d->H * d->N * dim;
  s[1] = (int64_t)d->N * dim;
  s[2] = dim;
}

BwdTcWs bwd_tc_ws(const ret_desc *d) {
  BwdTcWs w;
  w.w = d->d_v % 256 == 0 ? 256 : 128;
  w.nvc = d->d_v / w.w;
  ret_desc a, b;
  bwd_inner_desc(d, d->d_k, d->d_v, &a);
  bwd_inner_desc(d, w.w, d->d_k, &b);
  const size_t ia = retention_workspace_size(&a), ib = retention_workspace_size(&b);
  const size_t BH = (size_t)d->B * d->H, rows = BH * d->N;
  const size_t sb = BH * d->d_k * d->d_v * sizeof(float);
  size_t off = align256(ia > ib ? ia : ib);  // the inner runs' workspace, status word first
  w.kr = off; off = align256(off + rows * d->d_k * 2);
  w.kr_rev = off; off = align256(off + rows * d->d_k * 2);
  w.qs_rev = off; off = align256(off + rows * d->d_k * 2);
  w.dos = off;
  if (d->out_dtype != RET_BF16) off = align256(off + rows * d->d_v * 2);
  w.dos_rev = off; off = align256(off + rows * d->d_v * 2);
  w.v_rev = off; off = align256(off + rows * d->d_v * 2);
  w.ts = off; off = align256(off + sb);
  w.tds = off; off = align256(off + sb);
  w.sdv = off; off = align256(off + sb);
  w.dvr = off; off = align256(off + rows * d->d_v * sizeof(float));
  for (int j = 0; j < w.nvc; ++j) {
    w.o[j] = off;
    off = align256(off + rows * d->d_k * sizeof(float));
  }
  w.total = off;
  return w;
}

ret_status bwd_tc_impl(const ret_desc *d, const KParams &p, const void *q, const void *k,
                       const void *v, const float *S_in, const void *dO, const float *dS_out,
                       void *dq, void *dk, void *dv, float *dS_in, void *ws, cudaStream_t st) {
  const BwdTcWs w = bwd_tc_ws(d);
  const int dkk = d->d_k, dvv = d->d_v, BH = d->B * d->H;
  const bool scale = (d->norm_flags & (RET_NORM_SCALE | RET_NORM_DROW)) != 0;
  const bool dO_bf16 = d->out_dtype == RET_BF16;
  __nv_bfloat16 *kr = at<__nv_bfloat16>(ws, w.kr), *kr_rev = at<__nv_bfloat16>(ws, w.kr_rev);
  __nv_bfloat16 *qs_rev = at<__nv_bfloat16>(ws, w.qs_rev), *dos = at<__nv_bfloat16>(ws, w.dos);
  __nv_bfloat16 *dos_rev = at<__nv_bfloat16>(ws, w.dos_rev);
  __nv_bfloat16 *v_rev = at<__nv_bfloat16>(ws, w.v_rev);
  float *ts = at<float>(ws, w.ts), *tds = at<float>(ws, w.tds), *dvr = at<float>(ws, w.dvr);
  const size_t inner_bytes = w.kr;
  // Operands: k' forward and reversed, s q' reversed, dO reversed (and a
  // bf16 copy when dO is fp32), v reversed.
  BwdPrepJobs jobs;
  jobs.count = 4;
  BwdPrepJob *J = jobs.job;
  J[0].src = k; J[0].d = dkk; J[0].rotate = p.rotate; J[0].fwd = kr; J[0].rev = kr_rev;
  J[1].src = q; J[1].d = dkk; J[1].rotate = p.rotate; J[1].rowscale = scale; J[1].rev = qs_rev;
  J[2].src = dO; J[2].d = dvv; J[2].bf16 = dO_bf16; J[2].fwd = dO_bf16 ? nullptr : dos;
  J[2].rev = dos_rev;
  J[3].src = v; J[3].d = dvv; J[3].rev = v_rev;
  for (int i = 0; i < 3; ++i) {
    J[0].s[i] = d->sk[i];
    J[1].s[i] = d->sq[i];
    J[2].s[i] = d->so[i];
    J[3].s[i] = d->sv[i];
  }
  RET_CUDA(RET_TIMED_LAUNCH(kKBwdPrep, st, launch_bwd_prep(p, jobs, st)));
  // Entry states, before dS_out (which dS_in may alias) is overwritten.
  float *sdv = nullptr;
  if (dS_out) {
    CombineParts parts;  // dS_out / gamma
    parts.count = 1;
    parts.S[0] = dS_out;
    parts.t[0] = -1;
    sdv = at<float>(ws, w.sdv);
    RET_CUDA(RET_TIMED_LAUNCH(kKStateCombine, st, launch_state_combine(p, parts, sdv, nullptr, st)));
    RET_CUDA(RET_TIMED_LAUNCH(kKBwdPrep, st, launch_bwd_transpose(sdv, BH, dkk, dvv, w.w, tds, st)));
  }
  if (S_in) RET_CUDA(RET_TIMED_LAUNCH(kKBwdPrep, st, launch_bwd_transpose(S_in, BH, dkk, dvv, w.w, ts, st)));
  // dv and U_0: the forward on (k', s q', dO) in reversed time.
  {
    ret_desc r;
    bwd_inner_desc(d, dkk, dvv, &r);
    ret_status rs = chunkwise_impl(&r, kr_rev, qs_rev, dos_rev, sdv, nullptr, dS_in, nullptr,
                                   dvr, ws, inner_bytes, st);
    if (rs != RET_OK) return rs;
  }
  BwdFinish F;
  F.x[0] = dvr;
  F.n_in = 1;
  F.d = dvv;
  F.reverse = 1;
  for (int i = 0; i < 3; ++i) F.s[i] = d->sv[i];
  F.out = dv;
  RET_CUDA(RET_TIMED_LAUNCH(kKBwdFinish, st, launch_bwd_finish(p, F, st)));
  if (dS_in) {  // dS_in = gamma U_0
    CombineParts parts;
    parts.count = 1;
    parts.S[0] = dS_in;
    parts.t[0] = 1;
    RET_CUDA(RET_TIMED_LAUNCH(kKStateCombine, st, launch_state_combine(p, parts, dS_in, nullptr, st)));
  }
  // dq' / s: per piece of d_v, the forward on (dO, v, k') from S_in^T;
  // dk': the forward on (v, dO, s q') in reversed time from (dS_out/gamma)^T.
  for (int pass = 0; pass < 2; ++pass) {
    BwdFinish G;
    for (int j = 0; j < w.nvc; ++j) {
      ret_desc r;
      bwd_inner_desc(d, w.w, dkk, &r);
      const void *Qp, *Kp, *Vp;
      const float *Sp;
      if (pass == 0) {
        if (dO_bf16) {
          for (int i = 0; i < 3; ++i) r.sq[i] = d->so[i];
          Qp = reinterpret_cast<const __nv_bfloat16 *>(dO) + (size_t)j * w.w;
        } else {
          contig(d, dvv, r.sq);
          Qp = dos + (size_t)j * w.w;
        }
        for (int i = 0; i < 3; ++i) r.sk[i] = d->sv[i];
        Kp = reinterpret_cast<const __nv_bfloat16 *>(v) + (size_t)j * w.w;
        Vp = kr;
        Sp = S_in ? ts + (size_t)j * BH * w.w * dkk : nullptr;
      } else {
        contig(d, dvv, r.sq);
        contig(d, dvv, r.sk);
        Qp = v_rev + (size_t)j * w.w;
        Kp = dos_rev + (size_t)j * w.w;
        Vp = qs_rev;
        Sp = dS_out ? tds + (size_t)j * BH * w.w * dkk : nullptr;
      }
      ret_status rs = chunkwise_impl(&r, Qp, Kp, Vp, Sp, nullptr, nullptr, nullptr,
                                     at<float>(ws, w.o[j]), ws, inner_bytes, st);
      if (rs != RET_OK) return rs;
      G.x[j] = at<float>(ws, w.o[j]);
    }
    G.n_in = w.nvc;
    G.d = dkk;
    G.unrotate = p.rotate;
    if (pass == 0) {
      G.rowscale = scale;
      for (int i = 0; i < 3; ++i) G.s[i] = d->sq[i];
      G.out = dq;
    } else {
      G.reverse = 1;
      for (int i = 0; i < 3; ++i) G.s[i] = d->sk[i];
      G.out = dk;
    }
    RET_CUDA(RET_TIMED_LAUNCH(kKBwdFinish, st, launch_bwd_finish(p, G, st)));
  }
  return RET_OK;
}

}  // namespace

extern "C" {

void retention_desc_init(ret_desc *d, int B, int H, int N, int d_k, int d_v,
                         const double *gamma) {
  if (!d) return;
  memset(d, 0, sizeof(*d));
  d->B = B; d->H = H; d->N = N; d->d_k = d_k; d->d_v = d_v;
  d->chunk = 64;
  d->in_dtype = RET_BF16;
  d->out_dtype = RET_BF16;
  d->gamma = gamma;
  d->theta_base = 10000.0;
  d->norm_flags = 0;
  d->gn_eps = 1e-6f;
  d->pos0 = 0;
  d->rotate = 1;
  d->sq[0] = d->sk[0] = (int64_t)H * N * d_k;
  d->sq[1] = d->sk[1] = (int64_t)N * d_k;
  d->sq[2] = d->sk[2] = d_k;
  d->sv[0] = d->so[0] = (int64_t)H * N * d_v;
  d->sv[1] = d->so[1] = (int64_t)N * d_v;
  d->sv[2] = d->so[2] = d_v;
}

size_t retention_workspace_size(const ret_desc *d) {
  if (!desc_ok(d)) return 0;
  const ret_desc dt = tc_desc(d);
  const size_t a = simt_ws(d).total, b = tc_ws(&dt).total, c = par_tc_ws(d).total;
  return std::max(a, std::max(b, c));
}

ret_status retention_rotate(const ret_desc *d, const void *x, const int64_t sx[3], int dim,
                            void *out, ret_dtype out_dtype, const float *scale,
                            ret_stream_t stream) {
  RET_RANGE("retention_rotate");
  if (!desc_ok(d) || !sx || dim != d->d_k) return RET_EINVAL;
  if (out_dtype != RET_F32 && out_dtype != RET_BF16) return RET_EINVAL;
  if ((long long)d->B * d->H * d->N == 0) return RET_OK;
  if (!x || !out) return RET_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (sx[i] < 0) return RET_EINVAL;
  KParams p;
  make_params(d, nullptr, p);
  const long long s[3] = {sx[0], sx[1], sx[2]};
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, (cudaStream_t)stream,
                            launch_rotate(p, x, s, dim, out, out_dtype == RET_BF16, scale,
                                          scale ? kScaleArray : kScaleNone,
                                          (cudaStream_t)stream)));
  return RET_OK;
}

ret_status retention_parallel_fwd(const ret_desc *d, const void *q, const void *k,
                                  const void *v, void *o, void *ws, size_t ws_bytes,
                                  ret_stream_t stream) {
  RET_RANGE("retention_parallel_fwd");
  if (!desc_ok(d)) return RET_EINVAL;
  const bool empty = (long long)d->B * d->H * d->N == 0;
  if (!empty && (!q || !k || !v || !o)) return RET_EINVAL;
  const SimtWs w = simt_ws(d);
  ret_status rs = check_ws(ws, ws_bytes, std::max(w.total, par_tc_ws(d).total));
  if (rs != RET_OK) return rs;
  if (empty) return RET_OK;
  cudaStream_t st = (cudaStream_t)stream;
  KParams p;
  make_params(d, ws, p);
  // Tensor cores for bf16 inputs in the chunk path's operand range (its
  // prologue writes the 64-token fp16 operands); CUDA cores otherwise.
  ret_desc d64 = *d;
  d64.chunk = 64;
  KParams pt;
  make_params(&d64, ws, pt);
  if (pt.dk % 64 == 0 && chunk_tc_supported(pt, v, pt.sv)) {
    const ParTcWs pw = par_tc_ws(d);
    __half *Qp = at<__half>(ws, pw.qp), *Kp = at<__half>(ws, pw.kp);
    ChunkMeta *meta = at<ChunkMeta>(ws, pw.meta);
    float *Oraw = at<float>(ws, pw.oraw), *F = at<float>(ws, pw.f);
    RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate_qk(pt, q, k, Qp, Kp, meta, nullptr, st)));
    bool fused = false;
    RET_CUDA(RET_TIMED_LAUNCH(kKParallelTc, st, launch_parallel_tc(pt, Qp, Kp, v, meta, Oraw, F, o, &fused, st)));
    if (!fused) RET_CUDA(RET_TIMED_LAUNCH(kKGroupNorm, st, launch_groupnorm(pt, Oraw, F, o, st)));
    return RET_OK;
  }
  float *Qr = at<float>(ws, w.qr), *Kr = at<float>(ws, w.kr);
  float *Oraw = at<float>(ws, w.oraw), *F = at<float>(ws, w.f);
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, q, p.sq, d->d_k, Qr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, k, p.sk, d->d_k, Kr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKParallelSimt, st, launch_parallel_simt(p, Qr, Kr, v, Oraw, F, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKGroupNorm, st, launch_groupnorm(p, Oraw, F, o, st)));
  return RET_OK;
}

ret_status retention_chunkwise_fwd(const ret_desc *d, const void *q, const void *k,
                                   const void *v, const float *S_in, const float *z_in,
                                   float *S_out, float *z_out, void *o, void *ws,
                                   size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("retention_chunkwise_fwd");
  return chunkwise_impl(d, q, k, v, S_in, z_in, S_out, z_out, o,
                        ws, ws_bytes, (cudaStream_t)stream);
}

size_t retention_state_workspace_size(const ret_desc *d) {
  if (!desc_ok(d)) return 0;
  return state_ws(d).total;
}

ret_status retention_chunkwise_state(const ret_desc *d, const void *k, const void *v,
                                     const float *S_in, const float *z_in, float *S_out,
                                     float *z_out, void *ws, size_t ws_bytes,
                                     ret_stream_t stream) {
  RET_RANGE("retention_chunkwise_state");
  return state_impl(d, k, v, S_in, z_in, S_out, z_out, ws, ws_bytes, (cudaStream_t)stream);
}

ret_status retention_state_combine(int B, int H, int d_k, int d_v, const double *gamma,
                                   int count, const float *const *S_parts,
                                   const float *const *z_parts, const int64_t *tokens,
                                   float *S_out, float *z_out, ret_stream_t stream) {
  RET_RANGE("retention_state_combine");
  if (B < 0 || H < 0 || H > RET_MAX_HEADS || d_k < 1 || d_v < 1 || count < 0 ||
      count > kMaxCombineParts)
    return RET_EINVAL;
  if ((long long)B * H == 0 || (!S_out && !z_out)) return RET_OK;
  if (!gamma || (count > 0 && !tokens)) return RET_EINVAL;
  for (int h = 0; h < H; ++h)
    if (!(gamma[h] >= 0.0 && gamma[h] <= 1.0)) return RET_EINVAL;
  CombineParts parts;
  parts.count = count;
  for (int i = 0; i < count; ++i) {
    if (tokens[i] < 0) return RET_EINVAL;
    parts.S[i] = S_parts ? S_parts[i] : nullptr;
    parts.z[i] = z_parts ? z_parts[i] : nullptr;
    parts.t[i] = tokens[i];
  }
  KParams p;
  memset(&p, 0, sizeof(p));
  p.B = B; p.H = H; p.dk = d_k; p.dv = d_v;
  for (int h = 0; h < H; ++h) {
    p.gam[h] = (float)gamma[h];
    p.lng[h] = gamma[h] == 0.0 ? -INFINITY : (float)log(gamma[h]);
  }
  RET_CUDA(RET_TIMED_LAUNCH(kKStateCombine, (cudaStream_t)stream, launch_state_combine(p, parts, S_out, z_out, (cudaStream_t)stream)));
  return RET_OK;
}

ret_status retention_recurrent_step(const ret_desc *d, const void *q, const void *k,
                                    const void *v, float *S, float *z, void *o, void *ws,
                                    size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("retention_recurrent_step");
  if (!desc_ok(d) || d->N != 1) return RET_EINVAL;
  if (d->d_v % 4) return RET_EINVAL;
  const bool empty = (long long)d->B * d->H == 0;
  if (!empty && (!q || !k || !v || !S || !o)) return RET_EINVAL;
  if (!empty && (d->norm_flags & RET_NORM_RSUM) && !z) return RET_EINVAL;
  if (reinterpret_cast<uintptr_t>(S) & 15) return RET_EINVAL;
  ret_status rs = check_ws(ws, ws_bytes, kStatusBytes);
  if (rs != RET_OK) return rs;
  if (empty) return RET_OK;
  KParams p;
  make_params(d, ws, p);
  RET_CUDA(RET_TIMED_LAUNCH(kKRecurrent, (cudaStream_t)stream, launch_recurrent_step(p, q, k, v, S, z, o, (cudaStream_t)stream)));
  return RET_OK;
}

size_t retention_backward_workspace_size(const ret_desc *d) {
  if (!desc_ok(d)) return 0;
  const size_t a = bwd_ws(d).total;
  if (!bwd_tc_shape(d)) return a;
  const size_t b = bwd_tc_ws(d).total;
  return a > b ? a : b;
}

ret_status retention_chunkwise_bwd(const ret_desc *d, const void *q, const void *k,
                                   const void *v, const float *S_in, const void *dO,
                                   const float *dS_out, void *dq, void *dk, void *dv,
                                   float *dS_in, void *ws, size_t ws_bytes,
                                   ret_stream_t stream) {
  RET_RANGE("retention_chunkwise_bwd");
  if (!desc_ok(d)) return RET_EINVAL;
  if ((d->norm_flags & RET_NORM_RSUM) || d->gn_eps >= 0.f) return RET_EUNSUPPORTED;
  const bool empty = d->B == 0 || d->H == 0;
  if (!empty && d->N > 0 && (!q || !k || !v || !dO || !dq || !dk || !dv)) return RET_EINVAL;
  const BwdWs w = bwd_ws(d);
  ret_status rs = check_ws(ws, ws_bytes, w.total);
  if (rs != RET_OK) return rs;
  if (empty) return RET_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (d->N == 0) {  // no tokens: the state gradient passes through
    const size_t sbytes = (size_t)d->B * d->H * d->d_k * d->d_v * sizeof(float);
    if (dS_in && dS_in != dS_out)
      RET_CUDA(dS_out ? cudaMemcpyAsync(dS_in, dS_out, sbytes, cudaMemcpyDeviceToDevice, st)
                      : cudaMemsetAsync(dS_in, 0, sbytes, st));
    return RET_OK;
  }
  KParams p;
  make_params(d, ws, p);
  if (bwd_tc_shape(d)) {
    rs = check_ws(ws, ws_bytes, bwd_tc_ws(d).total);
    if (rs != RET_OK) return rs;
    return bwd_tc_impl(d, p, q, k, v, S_in, dO, dS_out, dq, dk, dv, dS_in, ws, st);
  }
  float *Qr = at<float>(ws, w.qr), *Kr = at<float>(ws, w.kr);
  float *DQr = at<float>(ws, w.dq), *DKr = at<float>(ws, w.dk);
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, q, p.sq, d->d_k, Qr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKRotate, st, launch_rotate(p, k, p.sk, d->d_k, Kr, 0, nullptr, kScaleNone, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKBwdRows, st, launch_bwd_rows(p, false, Kr, v, dO, S_in, DQr, st)));
  // The reverse sweeps read dS_out before the value kernel writes dS_in, so
  // the two may be one buffer.
  RET_CUDA(RET_TIMED_LAUNCH(kKBwdRows, st, launch_bwd_rows(p, true, Qr, v, dO, dS_out, DKr, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKBwdValues, st, launch_bwd_values(p, Qr, Kr, dO, dS_out, dv, dS_in, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKUnrotate, st, launch_unrotate(p, DQr, p.sq, dq, p.in_bf16, st)));
  RET_CUDA(RET_TIMED_LAUNCH(kKUnrotate, st, launch_unrotate(p, DKr, p.sk, dk, p.in_bf16, st)));
  return RET_OK;
}

// bf16 GEMM used by the MSR layer: the tensor-core kernel where the shape
// allows, the CUDA-core kernel otherwise.
static cudaError_t gemm_any(const void *A, const void *Bm, void *C, int M, int N, int K,
                            unsigned *status, cudaStream_t st) {
  if (gemm_tc_supported(A, Bm, C, M, N, K))
    return RET_TIMED_LAUNCH(kKGemmTc, st, launch_gemm_tc(A, Bm, C, M, N, K, status, st));
  return RET_TIMED_LAUNCH(kKGemmSimt, st, launch_gemm_bf16(A, Bm, C, M, N, K, 1, st));
}

// ------------------------------------------------------------------ MSR
static bool msr_ok(const msr_desc *d) {
  if (!d) return false;
  if (d->B < 0 || d->N < 0 || d->d_model < 1 || d->H < 1 || d->H > RET_MAX_HEADS) return false;
  if (!d->gamma) return false;
  return true;
}

static void msr_inner_desc(const msr_desc *m, ret_desc *d) {
  retention_desc_init(d, m->B, m->H, m->N, m->d_k, m->d_v, m->gamma);
  d->chunk = m->chunk;
  d->theta_base = m->theta_base;
  d->norm_flags = m->norm_flags;
  d->gn_eps = m->gn_eps;
  d->pos0 = m->pos0;
  d->rotate = 1;
  const int64_t HK = (int64_t)m->H * m->d_k, HV = (int64_t)m->H * m->d_v;
  d->sq[0] = d->sk[0] = (int64_t)m->N * HK;
  d->sq[1] = d->sk[1] = m->d_k;
  d->sq[2] = d->sk[2] = HK;
  d->sv[0] = d->so[0] = (int64_t)m->N * HV;
  d->sv[1] = d->so[1] = m->d_v;
  d->sv[2] = d->so[2] = HV;
}

struct MsrWs {
  size_t q, k, v, g, y, inner, total;
};

static MsrWs msr_ws(const msr_desc *m, const ret_desc *inner) {
  MsrWs w;
  const size_t T = (size_t)m->B * m->N;
  const size_t HK = (size_t)m->H * m->d_k, HV = (size_t)m->H * m->d_v;
  size_t off = kStatusBytes;
  w.q = off; off = align256(off + T * HK * 2);
  w.k = off; off = align256(off + T * HK * 2);
  w.v = off; off = align256(off + T * HV * 2);
  w.g = off; off = align256(off + T * HV * 2);
  w.y = off; off = align256(off + T * HV * 2);
  w.inner = off; off = align256(off + retention_workspace_size(inner));
  w.total = off;
  return w;
}

size_t msr_workspace_size(const msr_desc *m) {
  if (!msr_ok(m)) return 0;
  ret_desc inner;
  msr_inner_desc(m, &inner);
  if (!desc_ok(&inner)) return 0;
  return msr_ws(m, &inner).total;
}

ret_status msr_layer_fwd(const msr_desc *m, const void *X, const void *WQ, const void *WK,
                         const void *WV, const void *WG, const void *WO, void *Y, void *ws,
                         size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("msr_layer_fwd");
  if (!msr_ok(m)) return RET_EINVAL;
  ret_desc inner;
  msr_inner_desc(m, &inner);
  if (!desc_ok(&inner)) return RET_EINVAL;
  const MsrWs w = msr_ws(m, &inner);
  ret_status rs = check_ws(ws, ws_bytes, w.total);
  if (rs != RET_OK) return rs;
  const int T = m->B * m->N;
  if (T == 0) return RET_OK;
  if (!X || !WQ || !WK || !WV || !WG || !WO || !Y) return RET_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const int HK = m->H * m->d_k, HV = m->H * m->d_v;
  void *Q = at<char>(ws, w.q), *K = at<char>(ws, w.k), *V = at<char>(ws, w.v);
  void *G = at<char>(ws, w.g), *Yg = at<char>(ws, w.y);
  unsigned *status = reinterpret_cast<unsigned *>(ws);
  RET_CUDA(gemm_any(X, WQ, Q, T, HK, m->d_model, status, st));
  RET_CUDA(gemm_any(X, WK, K, T, HK, m->d_model, status, st));
  RET_CUDA(gemm_any(X, WV, V, T, HV, m->d_model, status, st));
  // Retention (with GroupNorm) into Yg, then the gate: swish(X W_G) (.) Yg.
  // Fused into the chunk kernel's stores, the gate loads and exponentials
  // made that kernel 2.3 times slower at B=2, N=4096, H=8; here it is the
  // epilogue of the W_G product (which then never writes G), or, where the
  // tensor-core GEMM does not take the shape, a separate bandwidth pass.
  rs = chunkwise_impl(&inner, Q, K, V, nullptr, nullptr, nullptr, nullptr, Yg,
                      at<char>(ws, w.inner), ws_bytes - w.inner, st);
  if (rs != RET_OK) return rs;
  if (gemm_tc_supported(X, WG, Yg, T, HV, m->d_model)) {
    RET_CUDA(RET_TIMED_LAUNCH(kKGemmTc, st, launch_gemm_tc(X, WG, Yg, T, HV, m->d_model, status, st, true)));
  } else {
    RET_CUDA(gemm_any(X, WG, G, T, HV, m->d_model, status, st));
    RET_CUDA(RET_TIMED_LAUNCH(kKGate, st, launch_swish_gate(Yg, G, (long long)T * HV, st)));
  }
  RET_CUDA(gemm_any(Yg, WO, Y, T, m->d_model, HV, status, st));
  return RET_OK;
}

// ------------------------------------------------------------ RetNet block
static bool block_ok(const retnet_block_desc *d) {
  if (!d || !msr_ok(&d->msr)) return false;
  if (d->d_ffn < 1 || d->msr.d_model > 32768) return false;
  if (!(d->ln_eps >= 0.f)) return false;
  return msr_workspace_size(&d->msr) > 0;
}

struct BlockWs {
  size_t msr, xn, y, hf, total;
};

// The MSR layer's workspace comes first, so that its status word is the
// block's.
static BlockWs block_ws(const retnet_block_desc *d) {
  BlockWs w;
  const size_t T = (size_t)d->msr.B * d->msr.N;
  size_t off = 0;
  w.msr = off; off = align256(off + msr_workspace_size(&d->msr));
  w.xn = off; off = align256(off + T * d->msr.d_model * 2);
  w.y = off; off = align256(off + T * d->msr.d_model * 2);
  w.hf = off; off = align256(off + T * (size_t)d->d_ffn * 2);
  w.total = off;
  return w;
}

size_t retnet_block_workspace_size(const retnet_block_desc *d) {
  if (!block_ok(d)) return 0;
  return block_ws(d).total;
}

ret_status retnet_block_fwd(const retnet_block_desc *d, const void *X, const float *ln1_w,
                            const float *ln1_b, const void *WQ, const void *WK, const void *WV,
                            const void *WG, const void *WO, const float *ln2_w,
                            const float *ln2_b, const void *W1, const void *W2, void *Xout,
                            void *ws, size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("retnet_block_fwd");
  if (!block_ok(d)) return RET_EINVAL;
  const BlockWs w = block_ws(d);
  ret_status rs = check_ws(ws, ws_bytes, w.total);
  if (rs != RET_OK) return rs;
  const long long T = (long long)d->msr.B * d->msr.N;
  if (T == 0) return RET_OK;
  if (!X || !ln1_w || !ln1_b || !WQ || !WK || !WV || !WG || !WO || !ln2_w || !ln2_b || !W1 ||
      !W2 || !Xout)
    return RET_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const int dm = d->msr.d_model;
  void *Xn = at<char>(ws, w.xn), *Y = at<char>(ws, w.y), *Hf = at<char>(ws, w.hf);
  unsigned *status = reinterpret_cast<unsigned *>(ws);
  // Y = MSR(LN(X)) + X
  RET_CUDA(RET_TIMED_LAUNCH(kKLayerNorm, st, launch_layernorm(X, ln1_w, ln1_b, Xn, T, dm, d->ln_eps, st)));
  rs = msr_layer_fwd(&d->msr, Xn, WQ, WK, WV, WG, WO, Y, at<char>(ws, w.msr), w.xn - w.msr,
                     stream);
  if (rs != RET_OK) return rs;
  RET_CUDA(RET_TIMED_LAUNCH(kKResidual, st, launch_residual_add(Y, X, T * dm, st)));
  // X' = gelu(LN(Y) W1) W2 + Y   (X is not read again: Xout may alias it)
  RET_CUDA(RET_TIMED_LAUNCH(kKLayerNorm, st, launch_layernorm(Y, ln2_w, ln2_b, Xn, T, dm, d->ln_eps, st)));
  RET_CUDA(gemm_any(Xn, W1, Hf, (int)T, d->d_ffn, dm, status, st));
  RET_CUDA(RET_TIMED_LAUNCH(kKGelu, st, launch_gelu(Hf, T * d->d_ffn, st)));
  RET_CUDA(gemm_any(Hf, W2, Xout, (int)T, dm, d->d_ffn, status, st));
  RET_CUDA(RET_TIMED_LAUNCH(kKResidual, st, launch_residual_add(Xout, Y, T * dm, st)));
  return RET_OK;
}

// ------------------------------------------------- multi-layer decode step
struct DecWs {
  size_t xn, q, k, v, g, y, m, h1, part, total;
};

// Decode-batch GEMM jobs stream their weights on CUDA cores for up to
// kDecSkinnyRows rows; beyond, the tensor cores (128-row tiles, the missing
// rows read as zeros) split over K do the same stream with less work per
// weight byte, when the widths suit them.  Measured per layer of the
// 6.7B-scale stack: B=1 106 / 110 us (CUDA cores / tensor cores), B=2
// 113 / 117, B=4 138 / 122, B=8 185 / 139.
constexpr int kDecSkinnyRows = 2;

static bool dec_use_tc(int B, int Ntot, int K) {
  return B > kDecSkinnyRows && Ntot % 256 == 0 && K % 64 == 0;
}

// fp32 partials of one decode-batch GEMM job (either kernel's K slices).
static size_t dec_job_partial_bytes(int B, int Ntot, int K) {
  size_t tc = 0, sk = 0;
  if (dec_use_tc(B, Ntot, K)) tc = (size_t)gemm_tc_split(B, Ntot, K) * B * Ntot * sizeof(float);
  if (B <= 16) sk = gemm_skinny_partial_bytes(B, Ntot, K);
  return tc > sk ? tc : sk;
}

static size_t dec_partial_bytes(const retnet_stack_desc *d) {
  const msr_desc &m = d->block.msr;
  const int B = m.B, dm = m.d_model, HK = m.H * m.d_k, HV = m.H * m.d_v, F = d->block.d_ffn;
  // the four input projections as one job, W_O, W1, W2, and each alone
  const size_t c[6] = {dec_job_partial_bytes(B, 2 * HK + 2 * HV, dm),
                       dec_job_partial_bytes(B, HK, dm), dec_job_partial_bytes(B, HV, dm),
                       dec_job_partial_bytes(B, dm, HV), dec_job_partial_bytes(B, F, dm),
                       dec_job_partial_bytes(B, dm, F)};
  size_t mx = 0;
  for (size_t x : c) mx = x > mx ? x : mx;
  return mx;
}

static DecWs dec_ws(const retnet_stack_desc *d) {
  DecWs w;
  const msr_desc &m = d->block.msr;
  const size_t B = m.B, dm = m.d_model, HK = (size_t)m.H * m.d_k, HV = (size_t)m.H * m.d_v;
  size_t off = kStatusBytes;
  w.xn = off; off = align256(off + B * dm * 2);
  w.q = off; off = align256(off + B * HK * 2);
  w.k = off; off = align256(off + B * HK * 2);
  w.v = off; off = align256(off + B * HV * 2);
  w.g = off; off = align256(off + B * HV * 2);
  w.y = off; off = align256(off + B * HV * 2);
  w.m = off; off = align256(off + B * dm * 2);
  w.h1 = off; off = align256(off + B * (size_t)d->block.d_ffn * 2);
  w.part = off; off = align256(off + dec_partial_bytes(d));
  w.total = off;
  return w;
}

// The descriptor of one layer's decode step on the [B, H*d] projection rows.
static void dec_step_desc(const retnet_stack_desc *d, ret_desc *r) {
  const msr_desc &m = d->block.msr;
  retention_desc_init(r, m.B, m.H, 1, m.d_k, m.d_v, m.gamma);
  r->theta_base = m.theta_base;
  r->norm_flags = m.norm_flags;
  r->gn_eps = m.gn_eps;
  r->pos0 = m.pos0;
  r->rotate = 1;
  const int64_t HK = (int64_t)m.H * m.d_k, HV = (int64_t)m.H * m.d_v;
  r->sq[0] = r->sk[0] = HK;
  r->sq[1] = r->sk[1] = m.d_k;
  r->sq[2] = r->sk[2] = HK;
  r->sv[0] = r->so[0] = HV;
  r->sv[1] = r->so[1] = m.d_v;
  r->sv[2] = r->so[2] = HV;
}

static bool dec_ok(const retnet_stack_desc *d) {
  if (!d || d->n_layers < 0 || !block_ok(&d->block)) return false;
  ret_desc r;
  dec_step_desc(d, &r);
  return desc_ok(&r) && r.d_v % 4 == 0;
}

size_t retnet_decode_workspace_size(const retnet_stack_desc *d) {
  if (!dec_ok(d)) return 0;
  return dec_ws(d).total;
}

// Decode-batch GEMM: the weight-streaming kernel for up to 16 rows, else the
// general path.
static cudaError_t gemm_dec(const void *A, const void *Bm, void *C, int M, int N, int K,
                            float *part, unsigned *status, cudaStream_t st) {
  if (gemm_skinny_supported(A, Bm, C, M, N, K)) {
    cudaError_t e = RET_TIMED_LAUNCH(kKGemmSkinny, st, launch_gemm_skinny(A, Bm, M, N, K, part, st));
    if (e != cudaSuccess) return e;
    return RET_TIMED_LAUNCH(kKSkinnyReduce, st, launch_skinny_reduce(part, C, M, N, K, st));
  }
  return gemm_any(A, Bm, C, M, N, K, status, st);
}

// Several decode-batch GEMMs of one A (same K) as one job, with the
// reduce's epilogue (GELU, or a skip connection with R): the
// weight-streaming kernel for up to 16 rows, the tensor-core kernel split
// over K beyond; false when the job fits neither (the caller then runs the
// GEMMs apart).
static bool skinny_job_fits(int M, int count, const void *const *Bs, const int *Ns) {
  if (M < 1) return false;
  for (int i = 0; i < count; ++i)
    if (Ns[i] < 8 || Ns[i] % 8 || !Bs[i] || reinterpret_cast<uintptr_t>(Bs[i]) % 16) return false;
  return true;
}

static bool dec_job_tc(const void *A, int M, int count, const void *const *Bs, const int *Ns,
                       int K) {
  int Ntot = 0;
  for (int i = 0; i < count; ++i) {
    if (!gemm_tc_supported(A, Bs[i], Bs[i], M, Ns[i], K)) return false;
    Ntot += Ns[i];
  }
  return dec_use_tc(M, Ntot, K);
}

static bool dec_job_fits(const void *A, int M, int count, const void *const *Bs, const int *Ns,
                         int K) {
  if (!skinny_job_fits(M, count, Bs, Ns)) return false;
  return dec_job_tc(A, M, count, Bs, Ns, K) || M <= 16;
}

// early_b: no kernel that may still run when this job starts writes its
// weights (see launch_gemm_skinny_job).
static cudaError_t gemm_dec_job(const void *A, int count, const void *const *Bs, void *const *Cs,
                                const int *Ns, int M, int K, int epi, const void *R, float *part,
                                unsigned *status, cudaStream_t st, bool early_b = false) {
  SkinnyJob job;
  if (!skinny_job_init(job, count, Bs, Cs, Ns, epi, R)) return cudaErrorInvalidValue;
  if (!dec_job_tc(A, M, count, Bs, Ns, K)) {
    cudaError_t e = RET_TIMED_LAUNCH(kKGemmSkinny, st, launch_gemm_skinny_job(A, job, M, K, part, st, early_b));
    if (e != cudaSuccess) return e;
    return RET_TIMED_LAUNCH(kKSkinnyReduce, st, launch_skinny_reduce_job(part, job, M, K, st));
  }
  const int split = gemm_tc_split(M, job.Ntot, K);
  cudaError_t e = RET_TIMED_LAUNCH(kKGemmTc, st, launch_gemm_tc_partials(A, count, Bs, Ns, M, K, part, split, status, st, early_b));
  if (e != cudaSuccess) return e;
  return RET_TIMED_LAUNCH(kKSkinnyReduce, st, launch_skinny_reduce_split(part, job, M, split, st));
}

ret_status retnet_decode_step(const retnet_stack_desc *d, const retnet_layer_weights *layers,
                              float *const *S, float *const *z, void *X, void *ws,
                              size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("retnet_decode_step");
  if (!dec_ok(d)) return RET_EINVAL;
  const DecWs w = dec_ws(d);
  ret_status rs = check_ws(ws, ws_bytes, w.total);
  if (rs != RET_OK) return rs;
  const msr_desc &m = d->block.msr;
  if (m.B == 0 || d->n_layers == 0) return RET_OK;
  if (!X || !layers || !S) return RET_EINVAL;
  const bool rsum = (m.norm_flags & RET_NORM_RSUM) != 0;
  if (rsum && !z) return RET_EINVAL;
  for (int l = 0; l < d->n_layers; ++l) {
    const retnet_layer_weights &L = layers[l];
    if (!L.ln1_w || !L.ln1_b || !L.WQ || !L.WK || !L.WV || !L.WG || !L.WO || !L.ln2_w ||
        !L.ln2_b || !L.W1 || !L.W2 || !S[l] || (reinterpret_cast<uintptr_t>(S[l]) & 15))
      return RET_EINVAL;
    if (rsum && !z[l]) return RET_EINVAL;
  }
  // X is the only buffer updated in place besides the states; it must not
  // overlap the workspace, and no state may overlap X or the workspace.
  const size_t xbytes = (size_t)m.B * m.d_model * 2;
  const size_t sbytes = (size_t)m.B * m.H * m.d_k * m.d_v * sizeof(float);
  const size_t zbytes = (size_t)m.B * m.H * m.d_k * sizeof(float);
  if (overlaps(X, xbytes, ws, w.total)) return RET_EINVAL;
  for (int l = 0; l < d->n_layers; ++l) {
    if (overlaps(S[l], sbytes, X, xbytes) || overlaps(S[l], sbytes, ws, w.total))
      return RET_EINVAL;
    if (rsum && (overlaps(z[l], zbytes, X, xbytes) || overlaps(z[l], zbytes, ws, w.total) ||
                 overlaps(z[l], zbytes, S[l], sbytes)))
      return RET_EINVAL;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int B = m.B, dm = m.d_model, HK = m.H * m.d_k, HV = m.H * m.d_v, F = d->block.d_ffn;
  void *Xn = at<char>(ws, w.xn), *Q = at<char>(ws, w.q), *K = at<char>(ws, w.k);
  void *V = at<char>(ws, w.v), *G = at<char>(ws, w.g), *Y = at<char>(ws, w.y);
  void *Mo = at<char>(ws, w.m), *H1 = at<char>(ws, w.h1);
  float *part = at<float>(ws, w.part);
  unsigned *status = reinterpret_cast<unsigned *>(ws);
  ret_desc rd;
  dec_step_desc(d, &rd);
  KParams p;
  make_params(&rd, ws, p);
  for (int l = 0; l < d->n_layers; ++l) {
    const retnet_layer_weights &L = layers[l];
    // Y1 = MSR(LN1(X)) + X, the retention step on this layer's state.
    // The first kernel of the call starts once all earlier work is done, so
    // the GEMMs after it may copy weights before their wait (early_b).
    RET_CUDA(RET_TIMED_LAUNCH(kKLayerNorm, st, launch_layernorm(X, L.ln1_w, L.ln1_b, Xn, B, dm, d->block.ln_eps, st, l > 0)));
    // Few rows: the four projections of LN1(X) stream their weights in one
    // job, and the GELU and the skip connections ride on the reduces.
    const void *Win[4] = {L.WQ, L.WK, L.WV, L.WG};
    void *Cin[4] = {Q, K, V, G};
    const int Nin[4] = {HK, HK, HV, HV};
    const bool fused = dec_job_fits(Xn, B, 4, Win, Nin, dm) && dec_job_fits(Y, B, 1, &L.WO, &dm, HV) &&
                       dec_job_fits(Xn, B, 1, &L.W1, &F, dm) && dec_job_fits(H1, B, 1, &L.W2, &dm, F);
    if (fused) {
      RET_CUDA(gemm_dec_job(Xn, 4, Win, Cin, Nin, B, dm, kSkEpNone, nullptr, part, status, st, true));
    } else {
      RET_CUDA(gemm_dec(Xn, L.WQ, Q, B, HK, dm, part, status, st));
      RET_CUDA(gemm_dec(Xn, L.WK, K, B, HK, dm, part, status, st));
      RET_CUDA(gemm_dec(Xn, L.WV, V, B, HV, dm, part, status, st));
      RET_CUDA(gemm_dec(Xn, L.WG, G, B, HV, dm, part, status, st));
    }
    // The retention step with the gate applied to its output.
    RET_CUDA(RET_TIMED_LAUNCH(kKRecurrent, st, launch_recurrent_step(p, Q, K, V, S[l], rsum ? z[l] : nullptr, Y, st, G)));
    if (fused) {
      void *c = Mo;
      RET_CUDA(gemm_dec_job(Y, 1, &L.WO, &c, &dm, B, HV, kSkEpResidual, X, part, status, st, true));
    } else {
      RET_CUDA(gemm_dec(Y, L.WO, Mo, B, dm, HV, part, status, st));
      RET_CUDA(RET_TIMED_LAUNCH(kKResidual, st, launch_residual_add(Mo, X, (long long)B * dm, st)));
    }
    // X = gelu(LN2(Y1) W1) W2 + Y1.
    RET_CUDA(RET_TIMED_LAUNCH(kKLayerNorm, st, launch_layernorm(Mo, L.ln2_w, L.ln2_b, Xn, B, dm, d->block.ln_eps, st)));
    if (fused) {
      void *c = H1;
      RET_CUDA(gemm_dec_job(Xn, 1, &L.W1, &c, &F, B, dm, kSkEpGelu, nullptr, part, status, st, true));
      c = X;
      RET_CUDA(gemm_dec_job(H1, 1, &L.W2, &c, &dm, B, F, kSkEpResidual, Mo, part, status, st, true));
    } else {
      RET_CUDA(gemm_dec(Xn, L.W1, H1, B, F, dm, part, status, st));
      RET_CUDA(RET_TIMED_LAUNCH(kKGelu, st, launch_gelu(H1, (long long)B * F, st)));
      RET_CUDA(gemm_dec(H1, L.W2, X, B, dm, F, part, status, st));
      RET_CUDA(RET_TIMED_LAUNCH(kKResidual, st, launch_residual_add(X, Mo, (long long)B * dm, st)));
    }
  }
  return RET_OK;
}

// Few rows on the tensor cores: the K split only pays while the output
// tiles alone leave most SMs idle.
static bool gemm_wants_split(int M, int N, int K) {
  return M > 16 && M <= 256 && N % 256 == 0 && K % 64 == 0 && gemm_tc_split(M, N, K) > 1;
}

size_t retention_gemm_workspace_size(int M, int N, int K) {
  if (M < 0 || N < 0 || K < 1) return 0;
  size_t need = kStatusBytes;
  if (M >= 1 && M <= 16 && N >= 8 && N % 8 == 0)
    need += align256(gemm_skinny_partial_bytes(M, N, K));
  else if (gemm_wants_split(M, N, K))
    need += align256(dec_job_partial_bytes(M, N, K));
  return need;
}

ret_status retention_gemm_bf16(const void *A, const void *Bm, void *C, int M, int N, int K,
                               void *ws, size_t ws_bytes, ret_stream_t stream) {
  RET_RANGE("retention_gemm_bf16");
  if (M < 0 || N < 0 || K < 1) return RET_EINVAL;
  if ((long long)M * N == 0) return RET_OK;
  if (!A || !Bm || !C) return RET_EINVAL;
  ret_status rs = check_ws(ws, ws_bytes, kStatusBytes);
  if (rs != RET_OK) return rs;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned *status = reinterpret_cast<unsigned *>(ws);
  // Few rows with room for the split-K partials: the weight-streaming kernel
  // (up to 16 rows) or the tensor cores split over K (up to 256 rows).
  if (gemm_skinny_supported(A, Bm, C, M, N, K) &&
      ws_bytes >= retention_gemm_workspace_size(M, N, K)) {
    RET_CUDA(gemm_dec(A, Bm, C, M, N, K, at<float>(ws, kStatusBytes), status, st));
    return RET_OK;
  }
  if (gemm_wants_split(M, N, K) && gemm_tc_supported(A, Bm, C, M, N, K) &&
      ws_bytes >= retention_gemm_workspace_size(M, N, K)) {
    void *c = C;
    RET_CUDA(gemm_dec_job(A, 1, &Bm, &c, &N, M, K, kSkEpNone, nullptr, at<float>(ws, kStatusBytes),
                          status, st));
    return RET_OK;
  }
  RET_CUDA(gemm_any(A, Bm, C, M, N, K, status, st));
  return RET_OK;
}

const char *retention_status_string(ret_status s) {
  switch (s) {
    case RET_OK: return "ok";
    case RET_EINVAL: return "invalid argument";
    case RET_EUNSUPPORTED: return "unsupported configuration";
    case RET_EWORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case RET_ECUDA: return "CUDA error";
    case RET_ETIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int retention_last_cuda_error(void) { return g_last_cuda_error; }

void retention_set_report_wait_budget(unsigned tries) {
  g_report_budget.store(tries, std::memory_order_relaxed);
}

ret_status retention_poll_status(void *ws, ret_stream_t stream) {
  if (!ws) return RET_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned word = 0;
  RET_CUDA(cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st));
  RET_CUDA(cudaStreamSynchronize(st));
  if (word == kDevOk) return RET_OK;
  RET_CUDA(cudaMemsetAsync(ws, 0, sizeof(word), st));
  RET_CUDA(cudaStreamSynchronize(st));
  return word == kDevTimeout ? RET_ETIMEOUT : RET_EINVAL;
}

}  // extern "C"
