/*
 * ORACLE — plain fp64 CPU reference for the chunked TTT scan.
 *
 * This is test infrastructure. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the CUDA library never does, and
 * the two share no code.
 *
 * Sources (web pages, cited by title and section):
 *  [guide] "Test-Time Training (TTT) guide" (diosapp ai-tutorial), section 2
 *          (inner loop: one gradient step per token on a self-supervised
 *          reconstruction loss) and section 3 (TTT-Linear f(W,x)=Wx+b,
 *          TTT-MLP two layers, hidden 4x input, GELU; mini-batch TTT; dual form).
 *  [ch5]   "5 · TestingTime 训练与长上下文" (PaperTrace), section 1.1 (TTT layer =
 *          initial state, update rule, output rule; chunks of b = 16 whose
 *          gradients are all taken at the chunk-start weights; dual form),
 *          section 2.1 (write W_t = W_{t-1} - eta grad l(W_{t-1}; x_t), read
 *          y_t = f(q_t; W_t)), section 2.3 (f_W(k) = Wk, l = 1/2 ||W k - v||^2,
 *          gradient (W k - v) k^T), section 2.4 (read/write order, per-sequence
 *          reset), section 4 (inside a chunk the state writes without erasing,
 *          between chunks it overwrites).
 *
 * Readings where the pages are silent or garbled (listed in the design notes):
 *  - Row-vector convention: z = q W with W[i][j], i = input, j = output; the
 *    pages' W k equals k W^T, so results agree up to transposition.
 *  - Loss carries the factor 1/2 ([ch5] 2.3); chunk gradients are SUMMED
 *    (averaging equals eta / b).
 *  - Update-then-read: token t's output uses the state after its own
 *    gradient, so the intra-chunk mask includes the diagonal ([guide] 2's
 *    per-token loop updates, then outputs).
 *  - A final chunk shorter than b follows the same rule.
 *  - GELU is the tanh approximation of Hendrycks and Gimpel (2016).
 *  - No bias, no layer norm or residual inside f.
 *
 * Layouts (all row-major, contiguous): Q, K, V, Z [B][H][T][d];
 * TTT-Linear W0 [H][d][d] (shared by every batch row: each row restarts from
 * it), W_out [B][H][d][d]; TTT-MLP W1 [H][d][m], W2 [H][m][d] (m = hidden),
 * outputs [B][H][d][m] and [B][H][m][d]; eta [H].
 *
 * Parity pins: b = 1 equals the delta rule; W0 = 0 with one chunk equals
 * causal linear attention; primal equals dual; gradients equal finite
 * differences and autograd; eta = 0 is the plain forward; chaining two calls
 * equals one call; b = T equals the single closed form; the segment affine
 * maps, applied in turn from W0, give the primal scan's state at every
 * segment end, and a one-token chunk's map is I - eta k^T k, eta k^T v.
 * The tests hold them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * TTT-Linear, primal (per-token) form. For every chunk the weights at its
 * start, Wa, are fixed; each token t of the chunk in order:
 *   e_t = k_t Wa - v_t                 (gradient of 1/2||k W - v||^2 at Wa is k^T e)
 *   W   = W - eta k_t^T e_t            (one gradient step; within the chunk the
 *                                       steps add up, none erases another)
 *   z_t = q_t W                        (read-out after the update)
 * ------------------------------------------------------------------------- */
static void linear_primal_unit(const double* Q, const double* K, const double* V, double eta,
                               const double* W0, int64_t T, int64_t d, int64_t b, double* Z,
                               double* W, double* Wa, double* e) {
  memcpy(W, W0, sizeof(double) * d * d);
  for (int64_t c0 = 0; c0 < T; c0 += b) {
    const int64_t c1 = (c0 + b < T) ? c0 + b : T;
    memcpy(Wa, W, sizeof(double) * d * d);
    for (int64_t t = c0; t < c1; ++t) {
      const double* k = K + t * d;
      const double* v = V + t * d;
      const double* q = Q + t * d;
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += k[i] * Wa[i * d + j];
        e[j] = s - v[j];
      }
      for (int64_t i = 0; i < d; ++i)
        for (int64_t j = 0; j < d; ++j) W[i * d + j] -= eta * k[i] * e[j];
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += q[i] * W[i * d + j];
        Z[t * d + j] = s;
      }
    }
  }
}

int oracle_linear_primal(const double* Q, const double* K, const double* V, const double* eta,
                         const double* W0, int64_t B, int64_t H, int64_t T, int64_t d, int64_t b,
                         double* Z, double* W_out, int nthreads) {
  if (B < 0 || H < 1 || T < 0 || d < 1 || b < 1) return -1;
  set_threads(nthreads);
  int bad = 0;
#pragma omp parallel
  {
    double* Wa = (double*)malloc(sizeof(double) * d * d);
    double* e = (double*)malloc(sizeof(double) * d);
    if (!Wa || !e) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < B * H; ++u) {
      if (!Wa || !e) continue;
      const int64_t h = u % H;
      linear_primal_unit(Q + u * T * d, K + u * T * d, V + u * T * d, eta[h], W0 + h * d * d, T,
                         d, b, Z + u * T * d, W_out + u * d * d, Wa, e);
    }
    free(Wa);
    free(e);
  }
  return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * TTT-Linear, dual form of one chunk (rows t of Q_c, K_c, V_c; Wa = chunk start):
 *   E   = K_c Wa - V_c
 *   S   = tril(Q_c K_c^T), diagonal included
 *   Z_c = Q_c Wa - eta S E
 *   W   = Wa - eta K_c^T E
 * Kept apart from the primal loop; it exists to pin primal == dual.
 * ------------------------------------------------------------------------- */
static void linear_dual_unit(const double* Q, const double* K, const double* V, double eta,
                             const double* W0, int64_t T, int64_t d, int64_t b, double* Z,
                             double* W, double* E, double* S) {
  memcpy(W, W0, sizeof(double) * d * d);
  for (int64_t c0 = 0; c0 < T; c0 += b) {
    const int64_t n = ((c0 + b < T) ? c0 + b : T) - c0;
    const double* Kc = K + c0 * d;
    const double* Vc = V + c0 * d;
    const double* Qc = Q + c0 * d;
    for (int64_t t = 0; t < n; ++t)
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += Kc[t * d + i] * W[i * d + j];
        E[t * d + j] = s - Vc[t * d + j];
      }
    for (int64_t t = 0; t < n; ++t)
      for (int64_t u = 0; u < n; ++u) {
        double s = 0.0;
        if (u <= t)
          for (int64_t i = 0; i < d; ++i) s += Qc[t * d + i] * Kc[u * d + i];
        S[t * n + u] = s;
      }
    for (int64_t t = 0; t < n; ++t)
      for (int64_t j = 0; j < d; ++j) {
        double qw = 0.0, se = 0.0;
        for (int64_t i = 0; i < d; ++i) qw += Qc[t * d + i] * W[i * d + j];
        for (int64_t u = 0; u < n; ++u) se += S[t * n + u] * E[u * d + j];
        Z[(c0 + t) * d + j] = qw - eta * se;
      }
    for (int64_t i = 0; i < d; ++i)
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t t = 0; t < n; ++t) s += Kc[t * d + i] * E[t * d + j];
        W[i * d + j] -= eta * s;
      }
  }
}

int oracle_linear_dual(const double* Q, const double* K, const double* V, const double* eta,
                       const double* W0, int64_t B, int64_t H, int64_t T, int64_t d, int64_t b,
                       double* Z, double* W_out, int nthreads) {
  if (B < 0 || H < 1 || T < 0 || d < 1 || b < 1) return -1;
  set_threads(nthreads);
  const int64_t bb = (b < T) ? b : (T > 0 ? T : 1);
  int bad = 0;
#pragma omp parallel
  {
    double* E = (double*)malloc(sizeof(double) * bb * d);
    double* S = (double*)malloc(sizeof(double) * bb * bb);
    if (!E || !S) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < B * H; ++u) {
      if (!E || !S) continue;
      const int64_t h = u % H;
      linear_dual_unit(Q + u * T * d, K + u * T * d, V + u * T * d, eta[h], W0 + h * d * d, T, d,
                       bb, Z + u * T * d, W_out + u * d * d, E, S);
    }
    free(E);
    free(S);
  }
  return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * TTT-Linear, one decode token per (batch row, head).
 * The pair (W_anchor, W_run) carries the chunk-start weights and the running
 * weights; pos = tokens already seen, so this token is number pos and starts
 * a chunk when pos % b == 0 (then W_anchor == W_run on entry).
 *   e = k W_anchor - v;  W_run -= eta k^T e;  z = q W_run;
 *   if (pos + 1) % b == 0: W_anchor = W_run
 * q, k, v, z [B][H][d]; W_anchor, W_run [B][H][d][d].
 * ------------------------------------------------------------------------- */
int oracle_linear_decode_step(const double* q, const double* k, const double* v, const double* eta,
                              double* W_anchor, double* W_run, int64_t B, int64_t H, int64_t d,
                              int64_t pos, int64_t b, double* z) {
  if (B < 0 || H < 1 || d < 1 || b < 1 || pos < 0) return -1;
  double* e = (double*)malloc(sizeof(double) * d);
  if (!e) return -2;
  for (int64_t u = 0; u < B * H; ++u) {
    const int64_t h = u % H;
    const double* qu = q + u * d;
    const double* ku = k + u * d;
    const double* vu = v + u * d;
    double* Wa = W_anchor + u * d * d;
    double* Wr = W_run + u * d * d;
    for (int64_t j = 0; j < d; ++j) {
      double s = 0.0;
      for (int64_t i = 0; i < d; ++i) s += ku[i] * Wa[i * d + j];
      e[j] = s - vu[j];
    }
    for (int64_t i = 0; i < d; ++i)
      for (int64_t j = 0; j < d; ++j) Wr[i * d + j] -= eta[h] * ku[i] * e[j];
    for (int64_t j = 0; j < d; ++j) {
      double s = 0.0;
      for (int64_t i = 0; i < d; ++i) s += qu[i] * Wr[i * d + j];
      z[u * d + j] = s;
    }
    if ((pos + 1) % b == 0) memcpy(Wa, Wr, sizeof(double) * d * d);
  }
  free(e);
  return 0;
}

/* ---------------------------------------------------------------------------
 * TTT-Linear as a chain of affine maps (the segment-parallel form).
 * One chunk's gradient step, W <- W - eta K_c^T (K_c W - V_c), is affine in W:
 *   W <- A_c W + B_c,   A_c = I - eta K_c^T K_c,   B_c = eta K_c^T V_c.
 * Two maps applied in turn compose as (A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2).
 * For every segment of L tokens (the last may be shorter) this returns the
 * composition of its chunks' maps, so that the state at the segment's end is
 * A_s W_start + B_s. The pages write the chunk update ([ch5] section 4,
 * [guide] section 3) but not this rearrangement; it is exact algebra on it.
 * L must be a multiple of b, so that no chunk straddles two segments.
 * Outputs A_out, B_out [B][H][S][d][d], S = ceil(T / L).
 * ------------------------------------------------------------------------- */
static void linear_segment_maps_unit(const double* K, const double* V, double eta, int64_t T,
                                     int64_t d, int64_t b, int64_t L, double* A_out, double* B_out,
                                     double* Ac, double* Bc, double* tmp) {
  int64_t s = 0;
  for (int64_t s0 = 0; s0 < T; s0 += L, ++s) {
    const int64_t s1 = (s0 + L < T) ? s0 + L : T;
    double* A = A_out + s * d * d;
    double* Bm = B_out + s * d * d;
    for (int64_t i = 0; i < d; ++i)
      for (int64_t j = 0; j < d; ++j) {
        A[i * d + j] = (i == j) ? 1.0 : 0.0;
        Bm[i * d + j] = 0.0;
      }
    for (int64_t c0 = s0; c0 < s1; c0 += b) {
      const int64_t c1 = (c0 + b < s1) ? c0 + b : s1;
      /* the chunk's own map */
      for (int64_t i = 0; i < d; ++i)
        for (int64_t j = 0; j < d; ++j) {
          double kk = 0.0, kv = 0.0;
          for (int64_t t = c0; t < c1; ++t) {
            kk += K[t * d + i] * K[t * d + j];
            kv += K[t * d + i] * V[t * d + j];
          }
          Ac[i * d + j] = ((i == j) ? 1.0 : 0.0) - eta * kk;
          Bc[i * d + j] = eta * kv;
        }
      /* (A, B) <- (Ac A, Ac B + Bc) */
      for (int64_t i = 0; i < d; ++i)
        for (int64_t j = 0; j < d; ++j) {
          double sa = 0.0, sb = 0.0;
          for (int64_t k = 0; k < d; ++k) {
            sa += Ac[i * d + k] * A[k * d + j];
            sb += Ac[i * d + k] * Bm[k * d + j];
          }
          tmp[i * d + j] = sa;
          tmp[d * d + i * d + j] = sb + Bc[i * d + j];
        }
      memcpy(A, tmp, sizeof(double) * d * d);
      memcpy(Bm, tmp + d * d, sizeof(double) * d * d);
    }
  }
}

int oracle_linear_segment_maps(const double* K, const double* V, const double* eta, int64_t B,
                               int64_t H, int64_t T, int64_t d, int64_t b, int64_t L,
                               double* A_out, double* B_out, int nthreads) {
  if (B < 0 || H < 1 || T < 0 || d < 1 || b < 1 || L < 1 || L % b != 0) return -1;
  set_threads(nthreads);
  const int64_t S = (T + L - 1) / L;
  int bad = 0;
#pragma omp parallel
  {
    double* Ac = (double*)malloc(sizeof(double) * d * d);
    double* Bc = (double*)malloc(sizeof(double) * d * d);
    double* tmp = (double*)malloc(sizeof(double) * 2 * d * d);
    if (!Ac || !Bc || !tmp) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < B * H; ++u) {
      if (!Ac || !Bc || !tmp) continue;
      const int64_t h = u % H;
      linear_segment_maps_unit(K + u * T * d, V + u * T * d, eta[h], T, d, b, L,
                               A_out + u * S * d * d, B_out + u * S * d * d, Ac, Bc, tmp);
    }
    free(Ac);
    free(Bc);
    free(tmp);
  }
  return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * tanh-GELU (Hendrycks and Gimpel 2016) and its derivative:
 *   sigma(u)  = 1/2 u (1 + th),  th = tanh(c (u + a u^3)), c = sqrt(2/pi), a = 0.044715
 *   sigma'(u) = 1/2 (1 + th) + 1/2 u (1 - th^2) c (1 + 3 a u^2)
 * ------------------------------------------------------------------------- */
static const double GELU_C = 0.79788456080286535587989211986876; /* sqrt(2/pi) */
static const double GELU_A = 0.044715;

double oracle_gelu(double u) {
  const double th = tanh(GELU_C * (u + GELU_A * u * u * u));
  return 0.5 * u * (1.0 + th);
}

double oracle_gelu_prime(double u) {
  const double th = tanh(GELU_C * (u + GELU_A * u * u * u));
  return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * GELU_C * (1.0 + 3.0 * GELU_A * u * u);
}

/* ---------------------------------------------------------------------------
 * TTT-MLP, primal (per-token) form. f(x) = sigma(x W1) W2, W1 [d][m], W2 [m][d].
 * Per chunk the weights W1a, W2a at its start are fixed; each token t:
 *   u = k W1a, a = sigma(u), g = a W2a - v             (forward, residual)
 *   delta = (g W2a^T) .* sigma'(u)                     (backprop to the hidden layer)
 *   W1 -= eta k^T delta;  W2 -= eta a^T g              (gradient of 1/2||f(k)-v||^2 at W1a, W2a)
 *   z_t = sigma(q W1) W2                               (read-out after the update)
 * ------------------------------------------------------------------------- */
static void mlp_primal_unit(const double* Q, const double* K, const double* V, double eta,
                            const double* W10, const double* W20, int64_t T, int64_t d, int64_t m,
                            int64_t b, double* Z, double* W1, double* W2, double* W1a, double* W2a,
                            double* uu, double* a, double* g, double* dl, double* hq) {
  memcpy(W1, W10, sizeof(double) * d * m);
  memcpy(W2, W20, sizeof(double) * m * d);
  for (int64_t c0 = 0; c0 < T; c0 += b) {
    const int64_t c1 = (c0 + b < T) ? c0 + b : T;
    memcpy(W1a, W1, sizeof(double) * d * m);
    memcpy(W2a, W2, sizeof(double) * m * d);
    for (int64_t t = c0; t < c1; ++t) {
      const double* k = K + t * d;
      const double* v = V + t * d;
      const double* q = Q + t * d;
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += k[i] * W1a[i * m + p];
        uu[p] = s;
        a[p] = oracle_gelu(s);
      }
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t p = 0; p < m; ++p) s += a[p] * W2a[p * d + j];
        g[j] = s - v[j];
      }
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t j = 0; j < d; ++j) s += g[j] * W2a[p * d + j];
        dl[p] = s * oracle_gelu_prime(uu[p]);
      }
      for (int64_t i = 0; i < d; ++i)
        for (int64_t p = 0; p < m; ++p) W1[i * m + p] -= eta * k[i] * dl[p];
      for (int64_t p = 0; p < m; ++p)
        for (int64_t j = 0; j < d; ++j) W2[p * d + j] -= eta * a[p] * g[j];
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += q[i] * W1[i * m + p];
        hq[p] = oracle_gelu(s);
      }
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t p = 0; p < m; ++p) s += hq[p] * W2[p * d + j];
        Z[t * d + j] = s;
      }
    }
  }
}

int oracle_mlp_primal(const double* Q, const double* K, const double* V, const double* eta,
                      const double* W1_0, const double* W2_0, int64_t B, int64_t H, int64_t T,
                      int64_t d, int64_t m, int64_t b, double* Z, double* W1_out, double* W2_out,
                      int nthreads) {
  if (B < 0 || H < 1 || T < 0 || d < 1 || m < 1 || b < 1) return -1;
  set_threads(nthreads);
  int bad = 0;
#pragma omp parallel
  {
    double* W1a = (double*)malloc(sizeof(double) * d * m);
    double* W2a = (double*)malloc(sizeof(double) * m * d);
    double* buf = (double*)malloc(sizeof(double) * (4 * m + d));
    if (!W1a || !W2a || !buf) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < B * H; ++u) {
      if (!W1a || !W2a || !buf) continue;
      const int64_t h = u % H;
      mlp_primal_unit(Q + u * T * d, K + u * T * d, V + u * T * d, eta[h], W1_0 + h * d * m,
                      W2_0 + h * m * d, T, d, m, b, Z + u * T * d, W1_out + u * d * m,
                      W2_out + u * m * d, W1a, W2a, buf, buf + m, buf + 2 * m, buf + 2 * m + d,
                      buf + 3 * m + d);
    }
    free(W1a);
    free(W2a);
    free(buf);
  }
  return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * TTT-MLP, dual form of one chunk (W1a, W2a = chunk start; n rows):
 *   U = K W1a;  A = sigma(U);  G = A W2a - V;  D = (G W2a^T) .* sigma'(U)
 *   Hq = Q W1a - eta tril(Q K^T) D;  Aq = sigma(Hq)
 *   Z  = Aq W2a - eta tril(Aq A^T) G
 *   W1 = W1a - eta K^T D;  W2 = W2a - eta A^T G
 * (q W1_t = q W1a - eta sum_{s<=t} (q.k_s) delta_s, and likewise for W2.)
 * Kept apart from the primal loop; it exists to pin primal == dual.
 * ------------------------------------------------------------------------- */
static void mlp_dual_unit(const double* Q, const double* K, const double* V, double eta,
                          const double* W10, const double* W20, int64_t T, int64_t d, int64_t m,
                          int64_t b, double* Z, double* W1, double* W2, double* U, double* A,
                          double* G, double* D, double* Aq) {
  memcpy(W1, W10, sizeof(double) * d * m);
  memcpy(W2, W20, sizeof(double) * m * d);
  for (int64_t c0 = 0; c0 < T; c0 += b) {
    const int64_t n = ((c0 + b < T) ? c0 + b : T) - c0;
    const double* Kc = K + c0 * d;
    const double* Vc = V + c0 * d;
    const double* Qc = Q + c0 * d;
    for (int64_t t = 0; t < n; ++t)
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += Kc[t * d + i] * W1[i * m + p];
        U[t * m + p] = s;
        A[t * m + p] = oracle_gelu(s);
      }
    for (int64_t t = 0; t < n; ++t)
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t p = 0; p < m; ++p) s += A[t * m + p] * W2[p * d + j];
        G[t * d + j] = s - Vc[t * d + j];
      }
    for (int64_t t = 0; t < n; ++t)
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t j = 0; j < d; ++j) s += G[t * d + j] * W2[p * d + j];
        D[t * m + p] = s * oracle_gelu_prime(U[t * m + p]);
      }
    for (int64_t t = 0; t < n; ++t) {
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += Qc[t * d + i] * W1[i * m + p];
        double r = 0.0;
        for (int64_t u = 0; u <= t; ++u) {
          double qk = 0.0;
          for (int64_t i = 0; i < d; ++i) qk += Qc[t * d + i] * Kc[u * d + i];
          r += qk * D[u * m + p];
        }
        Aq[t * m + p] = oracle_gelu(s - eta * r);
      }
    }
    for (int64_t t = 0; t < n; ++t)
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t p = 0; p < m; ++p) s += Aq[t * m + p] * W2[p * d + j];
        double r = 0.0;
        for (int64_t u = 0; u <= t; ++u) {
          double aa = 0.0;
          for (int64_t p = 0; p < m; ++p) aa += Aq[t * m + p] * A[u * m + p];
          r += aa * G[u * d + j];
        }
        Z[(c0 + t) * d + j] = s - eta * r;
      }
    for (int64_t i = 0; i < d; ++i)
      for (int64_t p = 0; p < m; ++p) {
        double s = 0.0;
        for (int64_t t = 0; t < n; ++t) s += Kc[t * d + i] * D[t * m + p];
        W1[i * m + p] -= eta * s;
      }
    for (int64_t p = 0; p < m; ++p)
      for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        for (int64_t t = 0; t < n; ++t) s += A[t * m + p] * G[t * d + j];
        W2[p * d + j] -= eta * s;
      }
  }
}

int oracle_mlp_dual(const double* Q, const double* K, const double* V, const double* eta,
                    const double* W1_0, const double* W2_0, int64_t B, int64_t H, int64_t T,
                    int64_t d, int64_t m, int64_t b, double* Z, double* W1_out, double* W2_out,
                    int nthreads) {
  if (B < 0 || H < 1 || T < 0 || d < 1 || m < 1 || b < 1) return -1;
  set_threads(nthreads);
  const int64_t bb = (b < T) ? b : (T > 0 ? T : 1);
  int bad = 0;
#pragma omp parallel
  {
    double* buf = (double*)malloc(sizeof(double) * bb * (4 * m + d));
    if (!buf) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < B * H; ++u) {
      if (!buf) continue;
      const int64_t h = u % H;
      mlp_dual_unit(Q + u * T * d, K + u * T * d, V + u * T * d, eta[h], W1_0 + h * d * m,
                    W2_0 + h * m * d, T, d, m, bb, Z + u * T * d, W1_out + u * d * m,
                    W2_out + u * m * d, buf, buf + bb * m, buf + 2 * bb * m, buf + 2 * bb * m + bb * d,
                    buf + 3 * bb * m + bb * d);
    }
    free(buf);
  }
  return bad ? -2 : 0;
}

/* Elementwise sigma and sigma' over an array (for the tests' pins). */
void oracle_gelu_array(const double* x, int64_t n, double* y, double* yp) {
  for (int64_t i = 0; i < n; ++i) {
    if (y) y[i] = oracle_gelu(x[i]);
    if (yp) yp[i] = oracle_gelu_prime(x[i]);
  }
}
