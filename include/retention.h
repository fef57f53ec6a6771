/*
 * retention.h -- C ABI of the GB300 (sm_103a) multi-scale retention library.
 *
 * The operation is RetNet's retention ("Retentive Network: A Successor to
 * Transformer for Large Language Models", arXiv:2307.08621), as stated on
 * the pages this library follows:
 *   [hwhale]  hwhale.com/article/285883 -- RetNet explained: recurrence,
 *             diagonalised closed form, parallel / recurrent / chunkwise
 *             equations and pseudocode, the three normalisations, GroupNorm.
 *   [sdkjxy]  m.sdkjxy.cn RetNet architecture walkthrough: pairs as complex
 *             numbers (RoPE), zero initial state, gated MSR layer.
 *   [m0nads]  m0nads.wordpress.com "A dubious successor to Transformer":
 *             xPos rotation, recurrent pseudocode, chunkwise representation,
 *             gated multi-scale retention.
 *
 * Per head with decay gamma:
 *   Q = (X W_Q) (.) Theta,  K = (X W_K) (.) conj(Theta),  V = X W_V,
 *   Theta_t = e^{i t theta},  theta_j = theta_base^(-2j/d_k)   [hwhale, eq. of Q,K,V]
 *   D_nm = gamma^(n-m) (n >= m), else 0                          [hwhale, D]
 *   Retention(X) = (Q K^T (.) D) V                               [hwhale, parallel]
 *   S_n = gamma S_{n-1} + K_n^T V_n,  O_n = Q_n S_n              [hwhale, recurrent]
 *   chunk i: (Q_[i] K_[i]^T (.) D) V_[i] + (Q_[i] S_i) (.) xi,
 *            xi_row = gamma^(row+1)                              [hwhale, chunkwise]
 * then the optional normalisations (1/sqrt(d_k); D row-normalised by
 * sqrt(sum_{i<=n} D_ni); R row-normalised by max(|sum_i R_ni|, 1))
 * [hwhale, the three normalisations] and a GroupNorm per (token, head) over
 * d_v with no affine [hwhale, multi-head GroupNorm].
 *
 * Readings where the pages are silent or ambiguous:
 *   - the phase pairs element (2j, 2j+1) as x_2j + i x_2j+1 and multiplies
 *     by e^{+i t theta_j}; the key's conjugate is carried by the dot product,
 *     so score(t, m) = Re(q~_t conj(k~_m) e^{i (t-m) theta}) [hwhale closed form];
 *   - token index tau in [0, N) sits at absolute position t = pos0 + tau; the
 *     decay-row sum uses the 1-based n = t + 1;
 *   - the state S is unnormalised (sum gamma^(t-m) K'_m^T V_m); the
 *     normalisations touch outputs only.  The third normalisation's row sum
 *     covers the whole causal prefix, carried across calls by
 *     z = sum gamma^(t-m) K'_m (d_k floats per head);
 *   - the state entering a chunk of L tokens is carried by
 *     S <- gamma^L S + sum_j gamma^(L-1-j) K_j^T V_j.
 *
 * Conventions (every entry point):
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates device memory and never synchronises the
 *     stream (except retention_poll_status, which says so).
 *   - Calls are asynchronous on `stream` and return RET_OK once the work is
 *     enqueued.  Invalid descriptors, shapes, strides, pointers or workspace
 *     sizes return RET_EINVAL / RET_EWORKSPACE before anything is launched.
 *     A launch failure returns RET_ECUDA; the cudaError_t is kept per thread
 *     for retention_last_cuda_error().
 *   - Errors found on the device (a bounded wait that ran out) are written
 *     to a status word at the start of the workspace; read it with
 *     retention_poll_status().
 *   - Inputs are never modified, except S / z of retention_recurrent_step
 *     (documented in/out) and when the caller aliases S_out/z_out to S_in/z_in.
 */
#ifndef RETENTION_H
#define RETENTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *ret_stream_t;

typedef enum {
  RET_OK = 0,
  RET_EINVAL = 1,       /* bad shape, dtype, stride, pointer or option       */
  RET_EUNSUPPORTED = 2, /* valid request that this build cannot run          */
  RET_EWORKSPACE = 3,   /* ws NULL or ws_bytes < the size query's answer     */
  RET_ECUDA = 4,        /* a CUDA call failed; see retention_last_cuda_error */
  RET_ETIMEOUT = 5      /* a device-side bounded wait ran out                */
} ret_status;

typedef enum { RET_F32 = 0, RET_BF16 = 1 } ret_dtype;

/* Normalisation flags [hwhale, the three normalisations]. */
enum {
  RET_NORM_SCALE = 1, /* Q K^T / sqrt(d_k)                       */
  RET_NORM_DROW = 2,  /* D_nm / sqrt(sum_{i<=n} D_ni)             */
  RET_NORM_RSUM = 4   /* R_nm / max(|sum_{i<=n} R_ni|, 1)         */
};

/* Largest head count one call accepts (per-head constants travel in the
 * kernel parameters). */
#define RET_MAX_HEADS 256

typedef struct {
  int B, H, N;     /* batch, heads, tokens in this call (N >= 0)             */
  int d_k, d_v;    /* key/query and value widths per head                    */
  int chunk;       /* chunk length of the chunkwise form, 1..256             */
  ret_dtype in_dtype, out_dtype; /* q,k,v element type; o element type      */
  const double *gamma; /* HOST pointer, H decays, each in [0, 1]             */
  double theta_base;   /* theta_j = theta_base^(-2j/d_k); 10000 on the pages */
  int norm_flags;      /* RET_NORM_* bitmask; 0 = the plain equations         */
  float gn_eps;        /* GroupNorm epsilon (1e-6); negative = no GroupNorm  */
  int64_t pos0;        /* absolute position of token 0 (>= 0)                */
  int rotate;          /* 1 = apply Theta to q and k; 0 = inputs pre-rotated */
  /* Element strides of (b, h, n) for q, k, v, o.  The feature dimension is
   * contiguous (stride 1).  Contiguous [B,H,N,d] is {H*N*d, N*d, d}; a
   * [B,N,H,d] view is {N*H*d, d, H*d}. */
  int64_t sq[3], sk[3], sv[3], so[3];
} ret_desc;

/* Fill `d` with defaults for contiguous [B,H,N,d] bf16 in/out, chunk 64,
 * theta_base 10000, gn_eps 1e-6, rotate on, no normalisations, pos0 0. */
void retention_desc_init(ret_desc *d, int B, int H, int N, int d_k, int d_v,
                         const double *gamma);

/* Workspace bytes every retention_* call below needs for this descriptor
 * (the largest of the three forms).  0 for an invalid descriptor. */
size_t retention_workspace_size(const ret_desc *d);

/*
 * Rotate-and-scale prologue [hwhale, Q=(XW_Q)(.)Theta, K=(XW_K)(.)conj(Theta);
 * m0nads, xPos].  x: [B,H,N,d] through strides sx (d = d_k, even); out:
 * contiguous [B,H,N,d] of out_dtype.  Pair (2j, 2j+1) of token tau is turned
 * by (pos0 + tau) theta_j and multiplied by scale[tau] when `scale` (a
 * DEVICE array of N floats) is not NULL.
 */
ret_status retention_rotate(const ret_desc *d, const void *x, const int64_t sx[3],
                            int dim, void *out, ret_dtype out_dtype,
                            const float *scale, ret_stream_t stream);

/*
 * Parallel form [hwhale, Retention(X) = (Q K^T (.) D) V; ParallelRetention].
 * q,k: [B,H,N,d_k]; v, o: [B,H,N,d_v] via the descriptor's strides.
 * The call's tokens only (zero prior state); positions start at pos0.
 * bf16 inputs with d_k a multiple of 64 up to 256, d_v a multiple of 128 up
 * to 1024, v 16-byte aligned with strides a multiple of 8 elements and
 * every gamma^64 >= 2^-16 run on the tensor cores (rotated q, k rounded to
 * fp16 with power-of-two block scales, the decayed scores to bf16, fp32
 * accumulation); everything else on CUDA cores in fp32.  The chunk field
 * does not change the result.
 */
ret_status retention_parallel_fwd(const ret_desc *d, const void *q,
                                  const void *k, const void *v, void *o,
                                  void *ws, size_t ws_bytes, ret_stream_t stream);

/*
 * Chunkwise recurrent form [hwhale, chunkwise equation; ChunkwiseRetention;
 * m0nads, chunkwise representation].  Starts from S_in/z_in (NULL = zeros,
 * [sdkjxy] zero initial state) and writes the state after the last token to
 * S_out/z_out (NULL = not wanted).  S: fp32 [B,H,d_k,d_v] contiguous,
 * z: fp32 [B,H,d_k] contiguous.  S_out may alias S_in and z_out z_in.
 * The result is the same function for every chunk length (up to rounding).
 */
ret_status retention_chunkwise_fwd(const ret_desc *d, const void *q,
                                   const void *k, const void *v,
                                   const float *S_in, const float *z_in,
                                   float *S_out, float *z_out, void *o,
                                   void *ws, size_t ws_bytes, ret_stream_t stream);

/*
 * One recurrent decode step [hwhale, S_n = gamma S_{n-1} + K_n^T V_n,
 * O_n = Q_n S_n; RecurrentRetention: output read after the update, summed
 * over d_k].  Requires N == 1; the token sits at position pos0.  S (fp32
 * [B,H,d_k,d_v]) is read and overwritten in place; z (fp32 [B,H,d_k]) is
 * read and overwritten when RET_NORM_RSUM is set (may be NULL otherwise).
 */
ret_status retention_recurrent_step(const ret_desc *d, const void *q,
                                    const void *k, const void *v, float *S,
                                    float *z, void *o, void *ws, size_t ws_bytes,
                                    ret_stream_t stream);

/*
 * Backward of the chunkwise / recurrent form: reverse mode of
 * S_n = gamma S_{n-1} + K_n^T V_n, O_n = s_n Q_n S_n [hwhale, recurrent and
 * chunkwise equations], s_n the row factor of the first two normalisations.
 * Given dO (gradient of o: out_dtype through the `so` strides) and dS_out
 * (gradient of the final state, fp32 [B,H,d_k,d_v] contiguous; NULL = zero),
 * writes
 *   dq, dk, dv: gradients of q, k, v, with their layouts (sq, sk, sv strides)
 *               and element type (in_dtype); dq, dk are with respect to the
 *               unrotated inputs when `rotate` is set;
 *   dS_in:      gradient of the entry state (fp32 [B,H,d_k,d_v]; NULL = not
 *               wanted).  It may alias dS_out.
 * S_in: the entry state of the forward call (NULL = zeros).  The gradient of
 * the z row sums is not produced (z enters only the third normalisation).
 * Requires gn_eps < 0 (no GroupNorm) and norm_flags without RET_NORM_RSUM:
 * RET_EUNSUPPORTED otherwise.  No output may overlap an input, except dS_in
 * and dS_out.  The chunk field does not change the result.
 * bf16 inputs with d_k 128 or 256, d_v a multiple of 128 up to 1024 and
 * every gamma^64 >= 2^-16 run on the tensor cores, as runs of the forward
 * kernel on time-reversed operands (the adjoint of the recurrence is the
 * recurrence in reversed time); their operands are rounded to bf16 / fp16
 * as the forward rounds its own.  Everything else runs on CUDA cores in
 * fp32.  The workspace size covers whichever path the descriptor takes.
 */
size_t retention_backward_workspace_size(const ret_desc *d);
ret_status retention_chunkwise_bwd(const ret_desc *d, const void *q, const void *k,
                                   const void *v, const float *S_in, const void *dO,
                                   const float *dS_out, void *dq, void *dk, void *dv,
                                   float *dS_in, void *ws, size_t ws_bytes,
                                   ret_stream_t stream);

/* State-only pass [hwhale, recurrent form S_n = gamma S_{n-1} + K_n^T V_n
 * and its chunkwise carry S_{c+1} = gamma^L S_c + K_[c]^T (V_[c] (.) zeta)]:
 * the recurrent state after the call's N tokens, without any output,
 *   S_out = gamma^N S_in + sum_m gamma^(N-1-m) K'_m^T V_m,
 *   z_out = gamma^N z_in + sum_m gamma^(N-1-m) K'_m          (K'_m = Theta k_m)
 * with token m at absolute position pos0 + m.  q, o, chunk, norm_flags,
 * gn_eps and out_dtype of the descriptor are ignored; k, v as for
 * retention_chunkwise_fwd.  S_in/z_in may be NULL (zero state); S_out/z_out
 * may be NULL (not produced) or alias S_in/z_in.  This is the first pass of
 * a sequence split over several devices: each device runs its own segment
 * from a zero state, the segments' states are joined with
 * retention_state_combine, and each device then runs retention_chunkwise_fwd
 * on its segment from the state that enters it.  ws: at least
 * retention_state_workspace_size(d) bytes, 256-byte aligned. */
size_t retention_state_workspace_size(const ret_desc *d);
ret_status retention_chunkwise_state(const ret_desc *d, const void *k, const void *v,
                                     const float *S_in, const float *z_in, float *S_out,
                                     float *z_out, void *ws, size_t ws_bytes,
                                     ret_stream_t stream);

/* Decayed sum of recurrent states [hwhale, recurrent form: the recurrence is
 * linear, and a state carried over t tokens with no input becomes gamma^t S]:
 *   S_out[b,h] = sum_i gamma_h^(tokens[i]) S_parts[i][b,h]   (z likewise)
 * S_parts, z_parts: HOST arrays of `count` (<= 64) DEVICE pointers to fp32
 * [B, H, d_k, d_v] / [B, H, d_k] states; a NULL entry (or a NULL array)
 * counts as a zero state.  tokens: HOST array of `count` decay lengths (>= 0;
 * gamma^0 = 1 for every gamma).  gamma: HOST array of H decays in [0, 1].
 * S_out / z_out may be NULL (not produced) and may alias one of the parts.
 * No workspace; asynchronous on `stream`. */
ret_status retention_state_combine(int B, int H, int d_k, int d_v, const double *gamma,
                                   int count, const float *const *S_parts,
                                   const float *const *z_parts, const int64_t *tokens,
                                   float *S_out, float *z_out, ret_stream_t stream);

/*
 * Chunkwise forward without a caller-supplied workspace.  No counterpart on
 * the pages: it exists for callers that cannot allocate device memory, such
 * as a plugin that an inference runtime hands only its input and output
 * buffers, or a latency-critical loop where cudaMalloc (which can
 * synchronise the device) is forbidden after start-up.  Same arguments and
 * results as retention_chunkwise_fwd, minus ws/ws_bytes.
 *   - The workspace is a fixed array of RET_NOALLOC_SCRATCH_BYTES inside the
 *     library; every GPU that loads the library holds it until the process
 *     exits.  A problem whose workspace (retention_workspace_size) exceeds
 *     it returns RET_EUNSUPPORTED before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - All calls share the one array: calls that may overlap on the GPU (on
 *     different streams, or from several threads) race and must not be used.
 *   - No memory is allocated or freed.  The device status word at the start
 *     of the array is cleared at the start of each call and is not
 *     reported: if a bounded device-side wait ran out (possible only when
 *     the GPU stalls for seconds), that call's outputs are undefined and
 *     this entry point cannot tell the caller.  Callers that must detect
 *     it use retention_chunkwise_fwd with their own workspace and
 *     retention_poll_status.
 */
#define RET_NOALLOC_SCRATCH_BYTES (32u << 20)
ret_status retention_chunkwise_fwd_noalloc(const ret_desc *d, const void *q,
                                           const void *k, const void *v,
                                           const float *S_in, const float *z_in,
                                           float *S_out, float *z_out, void *o,
                                           ret_stream_t stream);

/* Gated multi-scale retention layer [m0nads, "Gated Multi-Scale Retention";
 * sdkjxy, MSR layer]: MSR(X) = (swish(X W_G) (.) GroupNorm_h(Retention_h)) W_O,
 * swish(x) = x sigmoid(x), heads with their own gamma. */
typedef struct {
  int B, N, d_model;   /* X: [B, N, d_model] bf16 contiguous                */
  int H, d_k, d_v;     /* W_Q,W_K: [d_model, H d_k]; W_V,W_G: [d_model, H d_v];
                          W_O: [H d_v, d_model]; all bf16 row-major (X W)    */
  int chunk;           /* chunk length of the retention step                 */
  const double *gamma; /* HOST pointer, H decays                             */
  double theta_base;
  int norm_flags;
  float gn_eps;
  int64_t pos0;
} msr_desc;

size_t msr_workspace_size(const msr_desc *d);

/* The layer's projections as a plain GEMM [m0nads, "Gated Multi-Scale
 * Retention": X W_Q, X W_K, X W_V, X W_G, Y W_O]: C[M,N] = A[M,K] B[K,N],
 * bf16 row-major device buffers, fp32 accumulation, bf16 result.  Runs on
 * the tensor cores when N % 256 == 0, K % 64 == 0 and the pointers are
 * 16-byte aligned (any M; 128-row tiles, the rows past M neither read nor
 * written).  With 1 <= M <= 16 rows (a decode batch),
 * N % 8 == 0, a 16-byte aligned B and a workspace of at least
 * retention_gemm_workspace_size(M, N, K) bytes it runs on the
 * weight-streaming kernel (split-K fp32 partials in the workspace, added in
 * a fixed order); every other shape runs on CUDA cores.  ws: at least 256
 * bytes (the device status word), 256-byte aligned. */
size_t retention_gemm_workspace_size(int M, int N, int K);
ret_status retention_gemm_bf16(const void *A, const void *B, void *C, int M, int N, int K,
                               void *ws, size_t ws_bytes, ret_stream_t stream);

/* Y: [B, N, d_model] bf16. */
ret_status msr_layer_fwd(const msr_desc *d, const void *X, const void *WQ,
                         const void *WK, const void *WV, const void *WG,
                         const void *WO, void *Y, void *ws, size_t ws_bytes,
                         ret_stream_t stream);

/* One RetNet block [m0nads, "Overall architecture": an MSR and an FFN, each
 * after a LayerNorm, each with a skip connection]:
 *   Y  = MSR(LN1(X)) + X,    X' = FFN(LN2(Y)) + Y,    FFN(x) = gelu(x W1) W2,
 * LN(x) = (x - mean) / sqrt(var + ln_eps) (.) w + b over d_model (biased
 * variance), gelu(x) = x Phi(x).  The pages name the FFN but not its
 * activation; GELU is the reading taken.
 * X, Xout: [B, N, d_model] bf16 contiguous (Xout may alias X); ln*_w, ln*_b:
 * fp32 [d_model] device arrays; W_Q..W_O as for msr_layer_fwd; W1:
 * [d_model, d_ffn], W2: [d_ffn, d_model] bf16 row-major.  Intermediates are
 * rounded to bf16 between the steps.  d_model <= 32768. */
typedef struct {
  msr_desc msr;  /* the MSR layer: shapes, decays, normalisations          */
  int d_ffn;     /* FFN hidden width                                       */
  float ln_eps;  /* LayerNorm epsilon (>= 0)                               */
} retnet_block_desc;

size_t retnet_block_workspace_size(const retnet_block_desc *d);

ret_status retnet_block_fwd(const retnet_block_desc *d, const void *X, const float *ln1_w,
                            const float *ln1_b, const void *WQ, const void *WK, const void *WV,
                            const void *WG, const void *WO, const float *ln2_w,
                            const float *ln2_b, const void *W1, const void *W2, void *Xout,
                            void *ws, size_t ws_bytes, ret_stream_t stream);

/* One decode step of a stack of RetNet blocks [m0nads, "Overall
 * architecture": L stacked blocks; hwhale, the recurrent form for
 * inference]: B sequences advance by one token through n_layers blocks, each
 * layer's retention on its own recurrent state.  `block` gives the shapes
 * shared by every layer (block.msr.N is ignored: one token, at absolute
 * position block.msr.pos0).  Per layer, as retnet_block_fwd with N = 1:
 *   Y1 = MSR(LN1(X)) + X with the decode step on S[l] (and z[l]),
 *   X  = gelu(LN2(Y1) W1) W2 + Y1.
 * X: [B, d_model] bf16, the token's input on entry and the stack's output on
 * return.  layers: HOST array of n_layers records of DEVICE pointers (layouts
 * as for retnet_block_fwd).  S: HOST array of n_layers DEVICE pointers to fp32
 * [B, H, d_k, d_v] states (16-byte aligned), read and updated in place;
 * z: HOST array of fp32 [B, H, d_k] row-sum states, needed only with
 * RET_NORM_RSUM (may be NULL otherwise).  Requires d_v % 4 == 0.
 * Aliasing: X is updated in place and must not overlap the workspace; each
 * S[l] and z[l] is updated in place and must not overlap X, the workspace
 * or each other (RET_EINVAL where a state overlaps X or the workspace).
 * Weights are only read and may be shared between layers.
 * Projections stream the weights with split-K partial sums added in a fixed
 * order: up to two rows on CUDA cores, more rows on the tensor cores where
 * the widths are multiples of 256 (else CUDA cores, up to 16 rows).  The
 * call's first kernel starts only once all earlier work on the stream is
 * complete; the projection kernels after it start reading their weights
 * before the kernel before them has finished, so weights written on the
 * stream before the call are seen, while weights written concurrently on
 * another stream are not allowed. */
typedef struct {
  retnet_block_desc block;
  int n_layers;
} retnet_stack_desc;

typedef struct {
  const float *ln1_w, *ln1_b;
  const void *WQ, *WK, *WV, *WG, *WO;
  const float *ln2_w, *ln2_b;
  const void *W1, *W2;
} retnet_layer_weights;

size_t retnet_decode_workspace_size(const retnet_stack_desc *d);

ret_status retnet_decode_step(const retnet_stack_desc *d, const retnet_layer_weights *layers,
                              float *const *S, float *const *z, void *X, void *ws,
                              size_t ws_bytes, ret_stream_t stream);

/* Human-readable text of a status code (static storage). */
const char *retention_status_string(ret_status s);

/* cudaError_t of the calling thread's last RET_ECUDA (0 if none). */
int retention_last_cuda_error(void);

/* Reads and clears the device status word at the start of `ws`.  This call
 * SYNCHRONISES `stream`.  Returns RET_OK or the first device-side error. */
ret_status retention_poll_status(void *ws, ret_stream_t stream);

/* ---- Instrumentation (no counterpart on the pages; a measuring aid). ----
 * The library counts every kernel it launches.  With the timer enabled it
 * also records a CUDA event pair on the launch stream around each launch,
 * so the device time of each kernel can be read back after the stream has
 * been synchronised.  Do not enable the timer while capturing a CUDA graph.
 * Kernel ids run from 0 to retention_kernel_count()-1. */
void retention_kernel_timer_enable(int on);
void retention_kernel_timer_reset(void);
int retention_kernel_count(void);
const char *retention_kernel_name(int id);
long long retention_launch_count(void);
/* Sum of the timed launches of kernel `id` (milliseconds), its launch count
 * since the last reset and how many of those were timed.  Returns a
 * ret_status value. */
int retention_kernel_timer_read(int id, double *total_ms, long long *launches, int *timed);

/* ---- Failure-path check (a test aid). ----
 * Sets the number of tries of the rotate-and-scale prologue's first,
 * reporting wait on each TMA copy (default 2^24; applies to launches made
 * after the call, process-wide).  A wait that runs out records RET_ETIMEOUT
 * in the status word; the prologue then waits (bounded, with the default
 * budget) for the copy before it reads it, so results stay valid.  With 0
 * every such wait reports at once, which lets a test see a device timeout
 * reach retention_poll_status without stalling or faulting the GPU. */
void retention_set_report_wait_budget(unsigned tries);

#ifdef __cplusplus
}
#endif
#endif /* RETENTION_H */
