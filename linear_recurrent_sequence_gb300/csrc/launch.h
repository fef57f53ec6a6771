// Internal launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <utility>

#include "common.cuh"

namespace ret {

// Launch with programmatic stream serialization when pdl is set: the kernel
// may then start while the previous kernel on the stream still runs, so it
// must call pdl_wait() before it touches global memory that an earlier
// kernel may write or read (common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

enum ScaleMode { kScaleNone = 0, kScaleArray = 1, kScaleXi = 2, kScaleZeta = 3 };

// rotate.cu
cudaError_t launch_rotate(const KParams &p, const void *x, const long long s[3], int d,
                          void *out, int out_bf16, const float *scale, int mode,
                          cudaStream_t st);

// Per-(batch*head, chunk) record of the tensor-core path's fp16 operands,
// written by the prologue and copied into shared memory with each chunk.
struct ChunkMeta {
  int qexp, kexp;    // Q', K' are stored as fp16 * 2^-exp
  float qmax, kmax;  // largest pair norm of the rotated q / k rows before the decays
};

// Rotate-and-scale prologue of the tensor-core path (bf16 q, k; chunk 64):
// Q' = xi (.) rot(q), K' = zeta (.) rot(k) as contiguous fp16 [B*H][N][d_k]
// with per-chunk exponents, magnitudes and (if colsum) key column sums.
// keys_only: rotate k alone (q is not read; Q' and the query fields of meta
// are left as they are).
cudaError_t launch_rotate_qk(const KParams &p, const void *q, const void *k, __half *Qp,
                             __half *Kp, ChunkMeta *meta, float *colsum, cudaStream_t st,
                             bool keys_only = false);

// chunk_simt.cu: fp32 CUDA-core forms writing unnormalised rows + row factors.
// Qr, Kr: rotated contiguous fp32 [B,H,N,dk]; Oraw: fp32 [B,H,N,dv];
// F: fp32 [B,H,N] (row factor f = s(n) r(n)).
cudaError_t launch_chunk_simt(const KParams &p, const float *Qr, const float *Kr,
                              const void *v, const float *S_in, const float *z_in,
                              float *S_out, float *z_out, float *Oraw, float *F,
                              cudaStream_t st);
cudaError_t launch_parallel_simt(const KParams &p, const float *Qr, const float *Kr,
                                 const void *v, float *Oraw, float *F, cudaStream_t st);

// chunk_tc.cu: tensor-core chunkwise kernel (chunk 64, d_k in 64..256 step
// 64, d_v multiple of 128 up to 1024, bf16 inputs, gamma^64 >= 2^-16).
// Qp, Kp: contiguous fp16 [B,H,N,d_k] from the rotate-and-scale prologue
// (xi-scaled queries, zeta-scaled keys) with per-chunk records meta
// ([B*H][chunks]) and key column sums ksum ([B*H][chunks][d_k]).
bool chunk_tc_supported(const KParams &p, const void *v, const long long sv[3]);

// groupnorm.cu: o = GroupNorm(F * Oraw), written through so[]; and
// y <- y * swish(g) elementwise over n bf16 values (the MSR layer's gate).
cudaError_t launch_groupnorm(const KParams &p, const float *Oraw, const float *F,
                             void *o, cudaStream_t st);
cudaError_t launch_swish_gate(void *y, const void *g, long long n, cudaStream_t st);

// Sequence segments of the tensor-core chunk kernel.  P segments of seg_len
// chunks run as separate CTA groups; the entry state of segment k > 0 is
// assembled from the partial states of the npieces pieces (piece_len whole
// chunks each, covering chunks [0, (P-1) seg_len)) that state_tc writes.
struct SegPlan {
  int P = 1, seg_len = 0, npieces = 0, piece_len = 1;
  float *Part = nullptr, *zPart = nullptr;  // [piece][B*H][d_k][d_v], [piece][B*H][d_k]
};

cudaError_t launch_chunk_tc(const KParams &p, const void *Qp, const void *Kp, const void *v,
                            const ChunkMeta *meta, const float *ksum, const float *S_in,
                            const float *z_in, float *S_out, float *z_out, void *o,
                            int need_z, const SegPlan &seg, cudaStream_t st);

// state_tc.cu: partial states of the pieces of a SegPlan (tensor cores).
// Piece i covers chunks [i piece_len, min((i+1) piece_len, chunks)).
cudaError_t launch_state_tc(const KParams &p, const void *Kp, const void *v,
                            const ChunkMeta *meta, const float *ksum, int npieces,
                            int piece_len, float *Part, float *zPart, int need_z,
                            cudaStream_t st);

// state_combine.cu: S_out = sum_i gamma_h^(t_i) S_i over the parts (null
// entries skipped), z likewise; either output may be null and may alias a
// part.  States fp32 [B*H][d_k][d_v], z fp32 [B*H][d_k].
constexpr int kMaxCombineParts = 64;
struct CombineParts {
  int count = 0;
  const float *S[kMaxCombineParts] = {};
  const float *z[kMaxCombineParts] = {};
  long long t[kMaxCombineParts] = {};
};
cudaError_t launch_state_combine(const KParams &p, const CombineParts &parts, float *S_out,
                                 float *z_out, cudaStream_t st);
// The state after the call's tokens on CUDA cores: Kr rotated keys fp32
// [B*H][N][d_k], v through sv[]; S_out/z_out may alias S_in/z_in; either
// output may be null.
cudaError_t launch_state_simt(const KParams &p, const float *Kr, const void *v,
                              const float *S_in, const float *z_in, float *S_out, float *z_out,
                              cudaStream_t st);

// recurrent.cu: one decode step, state in place.  gate (optional, bf16
// [B][H][d_v]): the output is multiplied by swish(gate) after its bf16
// rounding, as the MSR layer's gate pass would.
cudaError_t launch_recurrent_step(const KParams &p, const void *q, const void *k,
                                  const void *v, float *S, float *z, void *o,
                                  cudaStream_t st, const void *gate = nullptr);

// gemm_tc.cu: tensor-core C[M,N] = A[M,K] B[K,N] (bf16 row-major, fp32
// accumulate); N % 256, K % 64 == 0 (any M >= 1) and 16-byte aligned pointers.
bool gemm_tc_supported(const void *A, const void *Bm, const void *C, int M, int N, int K);
// gate: C <- swish(A B) (.) C (bf16 C read and rewritten in the epilogue).
cudaError_t launch_gemm_tc(const void *A, const void *Bm, void *C, int M, int N, int K,
                           unsigned *status, cudaStream_t st, bool gate = false);
// Up to four B matrices of one A (same K), split over K: fp32 partials
// P[ks][M][sum N_i] (matrix i at its column offset), added by the skinny
// reduce (launch_skinny_reduce_split).  gemm_tc_split: the K split for a
// shape (about two work items per SM, partials at most 1/4 of B's bytes).
constexpr int kGemmJobMax = 4;
struct GemmJob {
  CUtensorMap tmB[kGemmJobMax];
  int count = 0, ldc = 0, ksplit = 1;
  int ntile0[kGemmJobMax + 1] = {}, col0[kGemmJobMax] = {};
  __nv_bfloat16 *C = nullptr;
  float *P = nullptr;
  int early_b = 0;  // B tiles of the first stages loaded before pdl_wait (as for the skinny job)
};
int gemm_tc_split(int M, int Ntot, int K);
cudaError_t launch_gemm_tc_partials(const void *A, int count, const void *const *Bs,
                                    const int *Ns, int M, int K, float *P, int ksplit,
                                    unsigned *status, cudaStream_t st, bool early_b = false);

// gemm_simt.cu: C[M,N] = A[M,K] B[K,N], bf16 in (row-major), fp32 accumulate.
cudaError_t launch_gemm_bf16(const void *A, const void *Bm, void *C, int M, int N,
                             int K, int out_bf16, cudaStream_t st);

// backward.cu: gradients on CUDA cores (fp32).  Z, Qr, Kr: rotated
// contiguous fp32 [B*H][N][d_k]; dO through so[] (out dtype); row outputs
// fp32 [B*H][N][d_k]; dv through sv[] (in dtype); states fp32 [B*H][d_k][d_v].
// rev = false: dQ' from S_in (T0) and K' (Z); rev = true: dK' from dS_out
// (T0) and Q' (Z).
cudaError_t launch_bwd_rows(const KParams &p, bool rev, const float *Z, const void *v,
                            const void *dO, const float *T0, float *out, cudaStream_t st);
cudaError_t launch_bwd_values(const KParams &p, const float *Qr, const float *Kr,
                              const void *dO, const float *dS_out, void *dv, float *dS_in,
                              cudaStream_t st);
// x (contiguous fp32 [B*H][N][d_k]) turned by e^{-i t theta} into out (strides s).
cudaError_t launch_unrotate(const KParams &p, const float *x, const long long s[3], void *out,
                            int out_bf16, cudaStream_t st);

// parallel_tc.cu: the parallel form on the tensor cores.  Qp, Kp and meta
// from launch_rotate_qk (64-token chunks).  d_v <= 256 (one CTA per row):
// writes o itself (*fused = true).  Wider: writes the raw rows Oraw [B*H][N]
// [d_v] and the row factors F [B*H][N] that launch_groupnorm turns into o.
// d_k a multiple of 64 up to 256, d_v a multiple of 128 up to 1024.
cudaError_t launch_parallel_tc(const KParams &p, const __half *Qp, const __half *Kp, const void *v,
                               const ChunkMeta *meta, float *Oraw, float *F, void *o,
                               bool *fused, cudaStream_t st);

// backward_tc.cu: operands of the tensor-core backward's forward runs.
// A prep job reads rows of src (strides s, bf16 or fp32, row width d, a
// multiple of 8), optionally rotates them (+t theta) and scales them by the
// first two normalisations' row factor, and writes bf16 rows to fwd[bh][t]
// and/or rev[bh][N-1-t] (contiguous [B*H][N][d], 16-byte aligned).
struct BwdPrepJob {
  const void *src = nullptr;
  long long s[3] = {};
  int bf16 = 1, d = 0, rotate = 0, rowscale = 0, vec = 0;
  __nv_bfloat16 *fwd = nullptr, *rev = nullptr;
};
constexpr int kBwdPrepMax = 4;
struct BwdPrepJobs {
  int count = 0;
  BwdPrepJob job[kBwdPrepMax];
};
cudaError_t launch_bwd_prep(const KParams &p, BwdPrepJobs jobs, cudaStream_t st);
// T_j[bh][e][a] = S[bh][a][j w + e]: the column blocks of width w transposed.
cudaError_t launch_bwd_transpose(const float *S, int BH, int dk, int dv, int w, float *T,
                                 cudaStream_t st);
// out (strides s, dtype) at t = the sum of n_in fp32 [B*H][N][d] inputs at
// row (reverse ? N-1-t : t), times the row factor when rowscale is set,
// turned back by -t theta when unrotate is set.
constexpr int kBwdFinishMax = 8;
struct BwdFinish {
  const float *x[kBwdFinishMax] = {};
  int n_in = 0, d = 0, reverse = 0, rowscale = 0, unrotate = 0, out_bf16 = 1, vec = 0;
  long long s[3] = {};
  void *out = nullptr;
};
cudaError_t launch_bwd_finish(const KParams &p, BwdFinish F, cudaStream_t st);

// block.cu: the RetNet block's LayerNorm (bf16 rows of d, fp32 gain and
// bias), skip connection y <- y + r and in-place GELU (bf16, n values).
// pdl = false: the kernel starts only once everything before it on the
// stream is complete (the first kernel of a chain whose later kernels read
// data before their pdl_wait, see launch_gemm_skinny_job).
cudaError_t launch_layernorm(const void *x, const float *w, const float *b, void *y, long long rows,
                             int d, float eps, cudaStream_t st, bool pdl = true);
cudaError_t launch_residual_add(void *y, const void *r, long long n, cudaStream_t st);
cudaError_t launch_gelu(void *y, long long n, cudaStream_t st);

// gemm_skinny.cu: C[M,N] = A[M,K] B[K,N] for M <= 16 rows (bf16 row-major,
// fp32 accumulation), split over K into fp32 partials [split][M][N] that
// launch_skinny_reduce adds in order into bf16 C.  Needs N % 8 == 0 and a
// 16-byte aligned B.
bool gemm_skinny_supported(const void *A, const void *Bm, const void *C, int M, int N, int K);
size_t gemm_skinny_partial_bytes(int M, int N, int K);
cudaError_t launch_gemm_skinny(const void *A, const void *Bm, int M, int N, int K,
                               float *partial, cudaStream_t st);
cudaError_t launch_skinny_reduce(const float *partial, void *C, int M, int N, int K,
                                 cudaStream_t st);
// Up to four weight matrices with the same K read in one launch (their
// columns side by side in the partials), and the reduce's epilogue: none,
// GELU, or a skip connection (one matrix; C = sum + R, R [M][N] bf16).
constexpr int kSkMaxMats = 4;
enum { kSkEpNone = 0, kSkEpGelu = 1, kSkEpResidual = 2 };
struct SkinnyJob {
  int count = 0, Ntot = 0, epi = kSkEpNone;
  const __nv_bfloat16 *B[kSkMaxMats] = {};
  __nv_bfloat16 *C[kSkMaxMats] = {};
  int N[kSkMaxMats] = {}, col0[kSkMaxMats] = {}, blk0[kSkMaxMats + 1] = {};
  const __nv_bfloat16 *R = nullptr;
};
bool skinny_job_init(SkinnyJob &job, int count, const void *const *Bs, void *const *Cs,
                     const int *Ns, int epi, const void *R);
// early_b: the first rows of the weights are copied before the kernel's
// pdl_wait, overlapping the kernel before it.  Only for callers that know
// no kernel that may still run writes the weights: every kernel launched
// since the last launch without programmatic serialization.
cudaError_t launch_gemm_skinny_job(const void *A, const SkinnyJob &job, int M, int K,
                                   float *partial, cudaStream_t st, bool early_b = false);
cudaError_t launch_skinny_reduce_job(const float *partial, const SkinnyJob &job, int M, int K,
                                     cudaStream_t st);
// The same reduce over `split` given slices (the tensor-core GEMM's partials).
cudaError_t launch_skinny_reduce_split(const float *partial, const SkinnyJob &job, int M,
                                       int split, cudaStream_t st);

}  // namespace ret
