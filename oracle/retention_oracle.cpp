// Retention oracle -- TEST INFRASTRUCTURE ONLY (see retention_oracle.h).
//
// Plain float64 loops, one (batch, head) pair at a time, written in the
// order and notation of the pages.  OpenMP is used only across independent
// (batch, head) pairs.  Nothing here is blocked, fused or reordered beyond
// what the equations themselves state.
#include "retention_oracle.h"

#include <cmath>
#include <complex>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" double orc_decay_row_sum(double gamma, long long n);

namespace {

bool cfg_ok(const orc_cfg *c) {
  if (!c || c->B < 0 || c->H < 0 || c->N < 0 || c->dk <= 0 || c->dv <= 0)
    return false;
  if (c->H > 0 && !c->gamma) return false;
  if (c->rotate && (c->dk % 2)) return false;
  for (int h = 0; h < c->H; ++h)
    if (!(c->gamma[h] >= 0.0 && c->gamma[h] <= 1.0)) return false;
  return true;
}

int nthreads(const orc_cfg *c) {
#ifdef _OPENMP
  return c->threads > 0 ? c->threads : omp_get_max_threads();
#else
  (void)c;
  return 1;
#endif
}

// theta_j = theta_base^(-2j/d): the per-pair frequency of the xPos/RoPE
// phase Theta_n = e^{i n theta} ([hwhale] "Q=(XW_Q)(.)Theta" equation;
// [sdkjxy] pairs of a d-vector as the real/imaginary parts of d/2 complex
// numbers, as in LLaMA's rotary embedding).
double theta_of(double base, int j, int d) {
  return std::pow(base, -2.0 * j / static_cast<double>(d));
}

// Multiply pair j = (x_2j, x_2j+1), read as x_2j + i x_2j+1, by e^{i t theta_j}.
void rotate_row(const double *x, int d, long long t, double base, double *y) {
  for (int j = 0; j < d / 2; ++j) {
    const double phi = static_cast<double>(t) * theta_of(base, j, d);
    const double cs = std::cos(phi), sn = std::sin(phi);
    const double a = x[2 * j], b = x[2 * j + 1];
    y[2 * j] = a * cs - b * sn;
    y[2 * j + 1] = a * sn + b * cs;
  }
}

// Multiply pair j by e^{-i t theta_j}: the inverse (and transpose) of rotate_row.
void unrotate_row(const double *x, int d, long long t, double base, double *y) {
  for (int j = 0; j < d / 2; ++j) {
    const double phi = static_cast<double>(t) * theta_of(base, j, d);
    const double cs = std::cos(phi), sn = std::sin(phi);
    const double a = x[2 * j], b = x[2 * j + 1];
    y[2 * j] = a * cs + b * sn;
    y[2 * j + 1] = b * cs - a * sn;
  }
}

double dot(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int i = 0; i < d; ++i) s += a[i] * b[i];
  return s;
}

// The per-row factor of the first two normalisations ([hwhale], the three
// normalisations): 1/sqrt(d) on Q K^T and 1/sqrt(sum_{i<=n} D_ni) on row n
// of D.  n is the 1-based absolute position.
// `cn` is sum_{i=1}^{n} gamma^(n-i) (see decay_row_sums).
double row_scale(const orc_cfg *c, double cn) {
  double s = 1.0;
  if (c->norm_flags & ORC_NORM_SCALE) s *= 1.0 / std::sqrt((double)c->dk);
  if (c->norm_flags & ORC_NORM_DROW) s *= 1.0 / std::sqrt(cn);
  return s;
}

// sum_{i=1}^{n} gamma^(n-i) for n = pos0+1 .. pos0+N, continuing the same
// recurrence as orc_decay_row_sum (so every value is bit-identical to it).
std::vector<double> decay_row_sums(double g, long long pos0, int N) {
  std::vector<double> out(N);
  double cn = orc_decay_row_sum(g, pos0);
  for (int tau = 0; tau < N; ++tau) {
    cn = g * cn + 1.0;
    out[tau] = cn;
  }
  return out;
}

// Third normalisation: R_nm / max(|sum_i R_ni|, 1).
double rsum_scale(const orc_cfg *c, double rowsum) {
  if (!(c->norm_flags & ORC_NORM_RSUM)) return 1.0;
  return 1.0 / std::fmax(std::fabs(rowsum), 1.0);
}

void rotated_copy(const orc_cfg *c, const double *x, int d, double *y) {
  for (int tau = 0; tau < c->N; ++tau) {
    if (c->rotate)
      rotate_row(x + (size_t)tau * d, d, c->pos0 + tau, c->theta_base,
                 y + (size_t)tau * d);
    else
      for (int i = 0; i < d; ++i) y[(size_t)tau * d + i] = x[(size_t)tau * d + i];
  }
}

void finish_groupnorm(const orc_cfg *c, double *o) {
  if (c->gn_eps >= 0.0)
    orc_groupnorm((long long)c->B * c->H * c->N, c->dv, c->gn_eps, o, o);
}

}  // namespace

extern "C" {

double orc_decay_row_sum(double gamma, long long n) {
  // sum_{i=1}^{n} D_ni with D_ni = gamma^(n-i): c_n = gamma * c_{n-1} + 1.
  double cn = 0.0;
  for (long long i = 1; i <= n; ++i) cn = gamma * cn + 1.0;
  return cn;
}

int orc_groupnorm(long long rows, int dv, double eps, const double *x,
                  double *y) {
  // GroupNorm with one group per (token, head) over its dv values, biased
  // variance, no affine ([hwhale] heads normalised independently).
  if (rows < 0 || dv <= 0 || eps < 0.0 || !x || !y) return -1;
  for (long long r = 0; r < rows; ++r) {
    const double *xr = x + (size_t)r * dv;
    double *yr = y + (size_t)r * dv;
    double mu = 0.0;
    for (int i = 0; i < dv; ++i) mu += xr[i];
    mu /= dv;
    double var = 0.0;
    for (int i = 0; i < dv; ++i) var += (xr[i] - mu) * (xr[i] - mu);
    var /= dv;
    const double inv = 1.0 / std::sqrt(var + eps);
    for (int i = 0; i < dv; ++i) yr[i] = (xr[i] - mu) * inv;
  }
  return 0;
}

int orc_rotate(const orc_cfg *c, const double *x, int d, double *out) {
  if (!c || !x || !out || d <= 0 || (d % 2)) return -1;
  const long long rows = (long long)c->B * c->H;
  for (long long bh = 0; bh < rows; ++bh)
    for (int tau = 0; tau < c->N; ++tau) {
      const size_t off = ((size_t)bh * c->N + tau) * d;
      rotate_row(x + off, d, c->pos0 + tau, c->theta_base, out + off);
    }
  return 0;
}

// Parallel representation ([hwhale] "Retention(X) = (Q K^T (.) D) V",
// ParallelRetention pseudocode; [m0nads] "Parallel representation").
// Row n of D is D_nm = gamma^(n-m) for n >= m, else 0.
int orc_parallel(const orc_cfg *c, const double *q, const double *k,
                 const double *v, double *o) {
  if (!cfg_ok(c) || !q || !k || !v || !o) return -1;
  const int N = c->N, dk = c->dk, dv = c->dv;
  const long long BH = (long long)c->B * c->H;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads(c))
  for (long long bh = 0; bh < BH; ++bh) {
    const double g = c->gamma[bh % c->H];
    std::vector<double> Q((size_t)N * dk), K((size_t)N * dk), Drow(N), Rrow(N);
    rotated_copy(c, q + (size_t)bh * N * dk, dk, Q.data());
    rotated_copy(c, k + (size_t)bh * N * dk, dk, K.data());
    const double *V = v + (size_t)bh * N * dv;
    double *O = o + (size_t)bh * N * dv;
    std::vector<double> acc(dv);
    const std::vector<double> crow = decay_row_sums(g, c->pos0, N);
    for (int n = 0; n < N; ++n) {
      for (int m = 0; m < N; ++m) Drow[m] = (n >= m) ? std::pow(g, n - m) : 0.0;
      const double s = row_scale(c, crow[n]);
      // Entries with D_nm = 0 (m > n) contribute exactly zero and are skipped.
      double rowsum = 0.0;
      for (int m = 0; m <= n; ++m) {
        Rrow[m] = dot(&Q[(size_t)n * dk], &K[(size_t)m * dk], dk) * Drow[m] * s;
        rowsum += Rrow[m];
      }
      const double r = rsum_scale(c, rowsum);
      for (int e = 0; e < dv; ++e) acc[e] = 0.0;
      for (int m = 0; m <= n; ++m)
        for (int e = 0; e < dv; ++e) acc[e] += Rrow[m] * V[(size_t)m * dv + e];
      for (int e = 0; e < dv; ++e) O[(size_t)n * dv + e] = r * acc[e];
    }
  }
  finish_groupnorm(c, o);
  return 0;
}

// Recurrent representation ([hwhale] "S_n = gamma S_{n-1} + K_n^T V_n",
// "Retention(X_n) = Q_n S_n", RecurrentRetention pseudocode: the output is
// read after the state update and summed over the key dimension).  The
// decayed key sum z_n = gamma z_{n-1} + K_n carries sum_{m<=n} R_nm across
// tokens for the third normalisation.
int orc_recurrent(const orc_cfg *c, const double *q, const double *k,
                  const double *v, const double *S_in, const double *z_in,
                  double *S_out, double *z_out, double *o) {
  if (!cfg_ok(c) || !q || !k || !v || !o) return -1;
  const int N = c->N, dk = c->dk, dv = c->dv;
  const long long BH = (long long)c->B * c->H;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads(c))
  for (long long bh = 0; bh < BH; ++bh) {
    const double g = c->gamma[bh % c->H];
    std::vector<double> S((size_t)dk * dv, 0.0), z(dk, 0.0), qr(dk), kr(dk), acc(dv);
    if (S_in) for (size_t i = 0; i < S.size(); ++i) S[i] = S_in[(size_t)bh * dk * dv + i];
    if (z_in) for (int i = 0; i < dk; ++i) z[i] = z_in[(size_t)bh * dk + i];
    const std::vector<double> crow = decay_row_sums(g, c->pos0, N);
    for (int tau = 0; tau < N; ++tau) {
      const long long t = c->pos0 + tau;
      const double *qt = q + ((size_t)bh * N + tau) * dk;
      const double *kt = k + ((size_t)bh * N + tau) * dk;
      const double *vt = v + ((size_t)bh * N + tau) * dv;
      if (c->rotate) {
        rotate_row(qt, dk, t, c->theta_base, qr.data());
        rotate_row(kt, dk, t, c->theta_base, kr.data());
      } else {
        for (int i = 0; i < dk; ++i) { qr[i] = qt[i]; kr[i] = kt[i]; }
      }
      for (int a = 0; a < dk; ++a) {
        for (int e = 0; e < dv; ++e)
          S[(size_t)a * dv + e] = g * S[(size_t)a * dv + e] + kr[a] * vt[e];
        z[a] = g * z[a] + kr[a];
      }
      const double s = row_scale(c, crow[tau]);
      const double r = rsum_scale(c, s * dot(qr.data(), z.data(), dk));
      double *ot = o + ((size_t)bh * N + tau) * dv;
      for (int e = 0; e < dv; ++e) acc[e] = 0.0;
      for (int a = 0; a < dk; ++a)
        for (int e = 0; e < dv; ++e) acc[e] += qr[a] * S[(size_t)a * dv + e];
      for (int e = 0; e < dv; ++e) ot[e] = r * s * acc[e];
    }
    if (S_out) for (size_t i = 0; i < S.size(); ++i) S_out[(size_t)bh * dk * dv + i] = S[i];
    if (z_out) for (int i = 0; i < dk; ++i) z_out[(size_t)bh * dk + i] = z[i];
  }
  finish_groupnorm(c, o);
  return 0;
}

// Chunkwise recurrent representation ([hwhale] chunkwise equation:
// Retention(X_[i]) = (Q_[i] K_[i]^T (.) D) V_[i] + (Q_[i] S_i) (.) xi with
// xi_ij = gamma^(i+1); ChunkwiseRetention pseudocode; [m0nads] "Chunkwise
// representation").  The state entering chunk i+1 is the recurrent state
// after the chunk's last token: S_{i+1} = gamma^L S_i + sum_j
// gamma^(L-1-j) K_j^T V_j for a chunk of L tokens (the recurrent form
// unrolled over L steps).
int orc_chunkwise(const orc_cfg *c, int chunk, const double *q,
                  const double *k, const double *v, const double *S_in,
                  const double *z_in, double *S_out, double *z_out, double *o) {
  if (!cfg_ok(c) || chunk <= 0 || !q || !k || !v || !o) return -1;
  const int N = c->N, dk = c->dk, dv = c->dv;
  const long long BH = (long long)c->B * c->H;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads(c))
  for (long long bh = 0; bh < BH; ++bh) {
    const double g = c->gamma[bh % c->H];
    std::vector<double> Q((size_t)N * dk), K((size_t)N * dk);
    rotated_copy(c, q + (size_t)bh * N * dk, dk, Q.data());
    rotated_copy(c, k + (size_t)bh * N * dk, dk, K.data());
    const double *V = v + (size_t)bh * N * dv;
    double *O = o + (size_t)bh * N * dv;
    std::vector<double> S((size_t)dk * dv, 0.0), z(dk, 0.0);
    if (S_in) for (size_t i = 0; i < S.size(); ++i) S[i] = S_in[(size_t)bh * dk * dv + i];
    if (z_in) for (int i = 0; i < dk; ++i) z[i] = z_in[(size_t)bh * dk + i];
    std::vector<double> Snext((size_t)dk * dv), znext(dk);
    std::vector<double> R(chunk), inner(dv), cross(dv), zeta(chunk);
    const std::vector<double> crow = decay_row_sums(g, c->pos0, N);
    for (int c0 = 0; c0 < N; c0 += chunk) {
      const int L = (N - c0 < chunk) ? (N - c0) : chunk;
      for (int i = 0; i < L; ++i) {
        const double *Qi = &Q[(size_t)(c0 + i) * dk];
        const double xi = std::pow(g, i + 1);
        // Intra-chunk scores (Q_[i] K_[i]^T (.) D) and their row sum.
        double rowsum = 0.0;
        for (int j = 0; j <= i; ++j) {
          R[j] = dot(Qi, &K[(size_t)(c0 + j) * dk], dk) * std::pow(g, i - j);
          rowsum += R[j];
        }
        rowsum += xi * dot(Qi, z.data(), dk);
        const double s = row_scale(c, crow[c0 + i]);
        const double r = rsum_scale(c, s * rowsum);
        for (int e = 0; e < dv; ++e) inner[e] = cross[e] = 0.0;
        for (int j = 0; j <= i; ++j)
          for (int e = 0; e < dv; ++e) inner[e] += R[j] * V[(size_t)(c0 + j) * dv + e];
        for (int a = 0; a < dk; ++a)
          for (int e = 0; e < dv; ++e) cross[e] += Qi[a] * S[(size_t)a * dv + e];
        for (int e = 0; e < dv; ++e)
          O[(size_t)(c0 + i) * dv + e] = r * s * (inner[e] + xi * cross[e]);
      }
      // State carried to the next chunk: zeta_j = gamma^(L-1-j).
      const double gL = std::pow(g, L);
      for (int j = 0; j < L; ++j) zeta[j] = std::pow(g, L - 1 - j);
      for (int a = 0; a < dk; ++a) {
        double *Sa = &Snext[(size_t)a * dv];
        for (int e = 0; e < dv; ++e) Sa[e] = gL * S[(size_t)a * dv + e];
        double za = gL * z[a];
        for (int j = 0; j < L; ++j) {
          const double kz = zeta[j] * K[(size_t)(c0 + j) * dk + a];
          const double *Vj = &V[(size_t)(c0 + j) * dv];
          for (int e = 0; e < dv; ++e) Sa[e] += kz * Vj[e];
          za += kz;
        }
        znext[a] = za;
      }
      S.swap(Snext);
      z.swap(znext);
    }
    if (S_out) for (size_t i = 0; i < S.size(); ++i) S_out[(size_t)bh * dk * dv + i] = S[i];
    if (z_out) for (int i = 0; i < dk; ++i) z_out[(size_t)bh * dk + i] = z[i];
  }
  finish_groupnorm(c, o);
  return 0;
}

// Diagonalised closed form ([hwhale] O_n = sum_m gamma^(n-m) (Q_n e^{in theta})
// (K_m e^{im theta})^dagger V_m, dagger = conjugate transpose; [sdkjxy] the
// conjugate of e^{in theta}).  Pairs of q and k are complex numbers; the
// real part of the complex score weights V.
int orc_closed_form(const orc_cfg *c, const double *q, const double *k,
                    const double *v, double *o) {
  if (!cfg_ok(c) || !q || !k || !v || !o) return -1;
  using cplx = std::complex<double>;
  const int N = c->N, dk = c->dk, dv = c->dv, P = dk / 2;
  if (dk % 2) return -1;
  const long long BH = (long long)c->B * c->H;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads(c))
  for (long long bh = 0; bh < BH; ++bh) {
    const double g = c->gamma[bh % c->H];
    std::vector<cplx> Qc((size_t)N * P), Kc((size_t)N * P);
    for (int tau = 0; tau < N; ++tau) {
      const double t = (double)(c->pos0 + tau);
      for (int j = 0; j < P; ++j) {
        const double th = c->rotate ? theta_of(c->theta_base, j, dk) : 0.0;
        const cplx phase = std::polar(1.0, t * th);  // e^{i t theta_j}
        const double *qt = q + ((size_t)bh * N + tau) * dk;
        const double *kt = k + ((size_t)bh * N + tau) * dk;
        Qc[(size_t)tau * P + j] = cplx(qt[2 * j], qt[2 * j + 1]) * phase;
        Kc[(size_t)tau * P + j] = cplx(kt[2 * j], kt[2 * j + 1]) * phase;
      }
    }
    const double *V = v + (size_t)bh * N * dv;
    double *O = o + (size_t)bh * N * dv;
    std::vector<double> w(N);
    const std::vector<double> crow = decay_row_sums(g, c->pos0, N);
    for (int n = 0; n < N; ++n) {
      double rowsum = 0.0;
      const double s = row_scale(c, crow[n]);
      for (int m = 0; m <= n; ++m) {
        cplx sc(0.0, 0.0);
        for (int j = 0; j < P; ++j)
          sc += Qc[(size_t)n * P + j] * std::conj(Kc[(size_t)m * P + j]);
        w[m] = std::pow(g, n - m) * sc.real() * s;
        rowsum += w[m];
      }
      const double r = rsum_scale(c, rowsum);
      for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int m = 0; m <= n; ++m) acc += w[m] * V[(size_t)m * dv + e];
        O[(size_t)n * dv + e] = r * acc;
      }
    }
  }
  finish_groupnorm(c, o);
  return 0;
}

// Gradients of the recurrent form by reverse mode, token by token.
// Forward ([hwhale] recurrent equations, as orc_recurrent): with q', k' the
// rotated rows and s_n the data-independent row factor of the first two
// normalisations, S_n = gamma S_{n-1} + k'_n^T v_n and o_n = s_n q'_n S_n.
// Reverse mode of that recurrence:
//   dq'_n = s_n S_n do_n                      (S_n: the state after token n)
//   G_n   = gradient of the loss w.r.t. S_n
//         = gamma G_{n+1} + s_n q'_n^T do_n,  G_{N} := dS_out (the last state)
//   dk'_n = G_n v_n,   dv_n = k'_n G_n,   dS_in = gamma G_0
// and dq, dk are dq', dk' turned back by e^{-i t theta_j} (the transpose of
// the rotation).  The third normalisation and GroupNorm are not covered.
int orc_recurrent_bwd(const orc_cfg *c, const double *q, const double *k,
                      const double *v, const double *S_in, const double *dO,
                      const double *dS_out, double *dq, double *dk, double *dv,
                      double *dS_in) {
  if (!cfg_ok(c) || !q || !k || !v || !dO || !dq || !dk || !dv) return -1;
  if ((c->norm_flags & ORC_NORM_RSUM) || c->gn_eps >= 0.0) return -1;
  const int N = c->N, dK = c->dk, dV = c->dv;
  const long long BH = (long long)c->B * c->H;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads(c))
  for (long long bh = 0; bh < BH; ++bh) {
    const double g = c->gamma[bh % c->H];
    const size_t qo = (size_t)bh * N * dK, vo = (size_t)bh * N * dV;
    const size_t so = (size_t)bh * dK * dV;
    std::vector<double> qr((size_t)N * dK), kr((size_t)N * dK);
    rotated_copy(c, q + qo, dK, qr.data());
    rotated_copy(c, k + qo, dK, kr.data());
    const std::vector<double> crow = decay_row_sums(g, c->pos0, N);
    std::vector<double> dqr((size_t)N * dK), dkr((size_t)N * dK);
    // Forward sweep: the state after each token, and dq'.
    std::vector<double> S((size_t)dK * dV, 0.0);
    if (S_in) for (size_t i = 0; i < S.size(); ++i) S[i] = S_in[so + i];
    for (int n = 0; n < N; ++n) {
      const double *kn = &kr[(size_t)n * dK];
      const double *vn = v + vo + (size_t)n * dV;
      const double *don = dO + vo + (size_t)n * dV;
      for (int a = 0; a < dK; ++a)
        for (int e = 0; e < dV; ++e)
          S[(size_t)a * dV + e] = g * S[(size_t)a * dV + e] + kn[a] * vn[e];
      const double sn = row_scale(c, crow[n]);
      for (int a = 0; a < dK; ++a)
        dqr[(size_t)n * dK + a] = sn * dot(&S[(size_t)a * dV], don, dV);
    }
    // Reverse sweep: G runs from the last token to the first.
    std::vector<double> G((size_t)dK * dV, 0.0);
    if (dS_out) for (size_t i = 0; i < G.size(); ++i) G[i] = dS_out[so + i];
    for (int n = N - 1; n >= 0; --n) {
      const double *qn = &qr[(size_t)n * dK];
      const double *kn = &kr[(size_t)n * dK];
      const double *vn = v + vo + (size_t)n * dV;
      const double *don = dO + vo + (size_t)n * dV;
      const double sn = row_scale(c, crow[n]);
      for (int a = 0; a < dK; ++a)
        for (int e = 0; e < dV; ++e) G[(size_t)a * dV + e] += sn * qn[a] * don[e];
      for (int a = 0; a < dK; ++a) dkr[(size_t)n * dK + a] = dot(&G[(size_t)a * dV], vn, dV);
      double *dvn = dv + vo + (size_t)n * dV;
      for (int e = 0; e < dV; ++e) {
        double acc = 0.0;
        for (int a = 0; a < dK; ++a) acc += kn[a] * G[(size_t)a * dV + e];
        dvn[e] = acc;
      }
      for (size_t i = 0; i < G.size(); ++i) G[i] *= g;  // now w.r.t. S_{n-1}
    }
    if (dS_in) for (size_t i = 0; i < G.size(); ++i) dS_in[so + i] = G[i];
    for (int n = 0; n < N; ++n) {
      if (c->rotate) {
        // The transpose of a turn by +t theta_j is a turn by -t theta_j.
        unrotate_row(&dqr[(size_t)n * dK], dK, c->pos0 + n, c->theta_base,
                     dq + qo + (size_t)n * dK);
        unrotate_row(&dkr[(size_t)n * dK], dK, c->pos0 + n, c->theta_base,
                     dk + qo + (size_t)n * dK);
      } else {
        for (int a = 0; a < dK; ++a) {
          dq[qo + (size_t)n * dK + a] = dqr[(size_t)n * dK + a];
          dk[qo + (size_t)n * dK + a] = dkr[(size_t)n * dK + a];
        }
      }
    }
  }
  return 0;
}

}  // extern "C"
