/*
 * Retention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of RetNet retention, used to check the
 * CUDA library.  Only the test-suite, the package smoke check and the CPU
 * baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (pages about "Retentive Network: A Successor to Transformer for
 * Large Language Models", arXiv:2307.08621):
 *   [hwhale]  hwhale.com/article/285883 -- RetNet explained (Chinese): the
 *             recurrence, the diagonalised closed form, the parallel /
 *             recurrent / chunkwise equations and pseudocode, the three
 *             normalisations, multi-head gamma and GroupNorm.
 *   [sdkjxy]  m.sdkjxy.cn/emb/202307262193346.html -- RetNet architecture
 *             walkthrough (Chinese): pairs as complex numbers, RoPE link,
 *             initial state 0, gated MSR layer.
 *   [m0nads]  m0nads.wordpress.com "A dubious successor to Transformer"
 *             (Retentive Network notes): xPos rotation, recurrent pseudocode,
 *             chunkwise representation, gated multi-scale retention.
 *
 * Layouts (all contiguous, row-major, float64):
 *   q, k  [B][H][N][dk]      v, o  [B][H][N][dv]
 *   S     [B][H][dk][dv]     z     [B][H][dk]
 * Token index tau in [0, N) has absolute position t = pos0 + tau and the
 * 1-based position n = t + 1 used by the decay-row normalisation.
 *
 * Functions return 0 on success, -1 on invalid arguments.
 *
 * Parity pins: every function here is pinned by the CPU tests (identities
 * between the three forms, the complex closed form, textbook special cases,
 * hand-derived fixtures); see the tests' docstrings.
 */
#ifndef RETENTION_ORACLE_H
#define RETENTION_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORC_NORM_SCALE = 1, /* Q K^T / sqrt(d)                                    */
  ORC_NORM_DROW = 2,  /* D_nm / sqrt(sum_{i<=n} D_ni)                        */
  ORC_NORM_RSUM = 4   /* R_nm / max(|sum_{i<=n} R_ni|, 1)                   */
};

typedef struct {
  int B, H, N, dk, dv;
  const double *gamma; /* [H] decay per head, 0 <= gamma <= 1              */
  double theta_base;   /* theta_j = theta_base^(-2j/dk)                    */
  long long pos0;      /* absolute position of token 0                     */
  int rotate;          /* 1: apply the xPos/RoPE phase Theta to q and k    */
  int norm_flags;      /* ORC_NORM_* bitmask                               */
  double gn_eps;       /* GroupNorm epsilon; < 0 means no GroupNorm        */
  int threads;         /* OpenMP threads over (b,h); <= 0 means default    */
} orc_cfg;

/* Theta applied to x [B][H][N][d] (pairs (2j, 2j+1) as complex numbers). */
int orc_rotate(const orc_cfg *c, const double *x, int d, double *out);

/* Parallel form: (Q K^T (.) D) V with the normalisations, then GroupNorm. */
int orc_parallel(const orc_cfg *c, const double *q, const double *k,
                 const double *v, double *o);

/* Recurrent form, token by token.  S_in/z_in may be NULL (zero state);
 * S_out/z_out may be NULL.  Returns o for every token. */
int orc_recurrent(const orc_cfg *c, const double *q, const double *k,
                  const double *v, const double *S_in, const double *z_in,
                  double *S_out, double *z_out, double *o);

/* Chunkwise form with chunk size `chunk` (the last chunk may be short). */
int orc_chunkwise(const orc_cfg *c, int chunk, const double *q,
                  const double *k, const double *v, const double *S_in,
                  const double *z_in, double *S_out, double *z_out, double *o);

/* Closed form with complex arithmetic:
 * O_n = sum_m gamma^(n-m) (Q_n e^{i n theta}) (K_m e^{i m theta})^dagger V_m,
 * real part taken; same normalisations and GroupNorm as the other forms. */
int orc_closed_form(const orc_cfg *c, const double *q, const double *k,
                    const double *v, double *o);

/* Gradients of the recurrent form (reverse mode of the recurrence, token by
 * token): dO [B][H][N][dv] is the gradient of o, dS_out [B][H][dk][dv] that of
 * the final state (NULL = zero); S_in NULL = zero state.  Writes dq, dk (with
 * respect to the unrotated q, k), dv and, unless NULL, dS_in.  Covers the
 * first two normalisations (row factors that do not depend on the data);
 * returns -1 when ORC_NORM_RSUM is set or GroupNorm is on (gn_eps >= 0). */
int orc_recurrent_bwd(const orc_cfg *c, const double *q, const double *k,
                      const double *v, const double *S_in, const double *dO,
                      const double *dS_out, double *dq, double *dk, double *dv,
                      double *dS_in);

/* GroupNorm of `rows` groups of `dv` contiguous values; no affine. */
int orc_groupnorm(long long rows, int dv, double eps, const double *x,
                  double *y);

/* Decay-row sum sum_{i=1}^{n} gamma^(n-i) by its recurrence c_n = g c_{n-1} + 1. */
double orc_decay_row_sum(double gamma, long long n);

#ifdef __cplusplus
}
#endif
#endif
