/*
 * sffn_oracle.c -- plain fp64 CPU oracle of the gated FFN forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library: it is written straight from the
 * formulas of "Model casting: compute the gate, then skip most of the FFN"
 * (ai.thesatyajit.com), sections "What an FFN actually computes",
 * "The 3x ceiling, and why W1 is always on", "Model casting: make sparsity a
 * target" (R-S+ definition) and "LoPA Gating: moving the ceiling".
 *
 * Definitions followed (one token x in R^D, hidden width H):
 *   z = W1 x                     standard gate,  W1 in R^{H x D}
 *   z = U (V x)                  low-rank gate,  U in R^{H x r}, V in R^{r x D}
 *                                (the UV part of W1 = G + UV)
 *
 * and, by flag (the "_ex" entry points), the pages' full low-rank form:
 *   OR_FLAG_TILED_G    z_i += x_{i mod D}          G = the tiled identity T,
 *                                                  (Tx)_i = x_{i mod D} (appendix,
 *                                                  Figure 6 (c))
 *   OR_FLAG_RMSNORM    V x -> RMSNorm(V x) = t / sqrt(mean_k t_k^2 + eps), no
 *                      gain ("W1(x) = Gx + U RMSNorm(Vx)")
 *   OR_FLAG_DOUBLE_ACT u = A(W3 x) instead of W3 x ("they apply the activation
 *                      to the outputs of both W1 and W3"); either gate
 * and a live threshold thr >= 0 (the "_ex" entry points): unit i is live iff
 * |A(z_i)| > thr, and a dead unit contributes exactly nothing ("treating
 * anything below epsilon as zero").  With thr = 0 the ReLU and R-S+ live sets
 * are {i : z_i > 0} as before; SiLU keeps every unit with z_i != 0.
 *   a = A(z)                     A = ReLU, or R-S+ (x*sigmoid(x) for x >= 0,
 *                                0 for x < 0), or SiLU (x*sigmoid(x) for every
 *                                x: the smooth gate, "Model casting: compute the
 *                                gate, then skip most of the FFN", sections on
 *                                SiLU and on thresholding small values)
 *   u = W3 x                     W3 in R^{H x D}
 *   y = W2 (a .* u)              W2 in R^{D x H}
 *
 * Everything is accumulated in double precision, each sum in ascending index
 * order, with no blocking, fusion or reordering.  Inputs are the values the
 * device sees: fp32 arrays, or bf16 bit patterns (uint16, the upper half of an
 * IEEE binary32), widened exactly to double.
 *
 * Two evaluations are provided:
 *   oracle_ffn_dense      -- the formula above over all H units (the definition)
 *   oracle_ffn_gate_first -- the gate-first order the pages describe: compute
 *                            the gate, keep the live set S = {i : z_i > 0}
 *                            (|A(z_i)| > thr in the "_ex" forms),
 *                            evaluate W3 rows and W2 columns only for i in S.
 * The pages' claim (skipping dead units leaves y unchanged) says the two agree
 * exactly; the tests check that.
 *
 * Weight-only int8 (the "_q8" entry points): "Model Casting and Low-Parameter
 * Gating", appendix Table 17, quantises the cast models weight-only to int8 and
 * int4 and gives no scale convention.  Reading taken: symmetric, one fp32
 * scale per output channel -- per row of W1 and of W3 (per unit i), per row of
 * W2 (per output element y_m) -- s = max_j |w_j| / 127, code =
 * round-half-to-even(w / s) clamped to [-127, 127], both decided in binary32
 * (the precision of the weights being quantised); an all-zero row has s = 0
 * and codes 0.  The forward is the definition above with every weight replaced
 * by its dequantised value q * s (exact in double); x is bf16.  Weight-only
 * int4 takes 7 in place of 127 (codes in [-7, 7]), and for W1 and W3 one scale
 * per group of 64 consecutive columns of a row instead of one per row: with a
 * single int4 scale per row, one large entry (a gate bias carried as a weight
 * column, say) sets a step that rounds every ordinary entry of the row to 0.
 * W2 keeps one scale per output element.  The "_qg" entry points take the
 * group; the "_q8" ones are group = D.
 *
 * Portable C99 + OpenMP; no SIMD intrinsics, no -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_BF16 1
#define OR_RELU 0
#define OR_RSP 1
#define OR_SILU 2
#define OR_FLAG_TILED_G 1
#define OR_FLAG_RMSNORM 2
#define OR_FLAG_DOUBLE_ACT 4

/* exact widening of one stored element to double */
static double elem(const void* p, int dtype, size_t i) {
  if (dtype == OR_F32) return (double)((const float*)p)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* widen n consecutive elements starting at element offset off */
static void widen_row(const void* p, int dtype, size_t off, int n, double* out) {
  for (int j = 0; j < n; ++j) out[j] = elem(p, dtype, off + (size_t)j);
}

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int j = 0; j < n; ++j) s += a[j] * b[j];
  return s;
}

/* The activation A.  ReLU and R-S+ vanish for z <= 0; SiLU is z * sigmoid(z)
   everywhere. */
static double activation(int act, double z) {
  if (act == OR_SILU) return z / (1.0 + exp(-z));
  if (!(z > 0.0)) return 0.0;
  if (act == OR_RELU) return z;
  return z / (1.0 + exp(-z)); /* R-S+ on the positive side: z * sigmoid(z) */
}

/* the thresholded gate: A(z) when |A(z)| > thr (the unit is live), else 0 */
static double gate_value(int act, double thr, double z) {
  const double a = activation(act, z);
  return fabs(a) > thr ? a : 0.0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int check_args(int D, int H, int r, int act, int dtype, int B, int flags, double eps, double thr) {
  if (D <= 0 || H <= 0 || r < 0 || B < 0) return -1;
  if (act != OR_RELU && act != OR_RSP && act != OR_SILU) return -1;
  if (!(thr >= 0.0) || thr > 1e300) return -1;
  if (dtype != OR_F32 && dtype != OR_BF16) return -1;
  if (flags & ~(OR_FLAG_TILED_G | OR_FLAG_RMSNORM | OR_FLAG_DOUBLE_ACT)) return -1;
  if ((flags & (OR_FLAG_TILED_G | OR_FLAG_RMSNORM)) && r == 0) return -1; /* low-rank gate only */
  if (!(eps >= 0.0)) return -1;
  return 0;
}

/* the up value of one unit: W3 x, or A(W3 x) with the double activation */
static double up_value(int act, int flags, double u) {
  return (flags & OR_FLAG_DOUBLE_ACT) ? activation(act, u) : u;
}

/* Gate pre-activations z[H] for one token xd[D] (already widened). */
static int gate(int D, int H, int r, int dtype, int flags, double eps, const void* W1,
                const void* U, const void* V, const double* xd, double* z) {
  if (r == 0) {
    int bad = 0;
#pragma omp parallel
    {
      double* row = (double*)malloc(sizeof(double) * (size_t)D);
      if (!row) {
#pragma omp atomic write
        bad = 1;
      }
#pragma omp for schedule(static)
      for (int i = 0; i < H; ++i) {
        if (!row) continue;
        widen_row(W1, dtype, (size_t)i * D, D, row);
        z[i] = dot(row, xd, D);
      }
      free(row);
    }
    return bad ? -2 : 0;
  }
  /* low-rank gate: t = V x (kept in double, not rounded), optionally
     t <- t / sqrt(mean(t^2) + eps); z = U t, optionally + x_{i mod D} */
  double* t = (double*)malloc(sizeof(double) * (size_t)r);
  if (!t) return -2;
  int bad = 0;
#pragma omp parallel
  {
    double* row = (double*)malloc(sizeof(double) * (size_t)(D > r ? D : r));
    if (!row) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(static)
    for (int k = 0; k < r; ++k) {
      if (!row) continue;
      widen_row(V, dtype, (size_t)k * D, D, row);
      t[k] = dot(row, xd, D);
    }
#pragma omp single
    {
      if (flags & OR_FLAG_RMSNORM) {
        double ss = 0.0;
        for (int k = 0; k < r; ++k) ss += t[k] * t[k];
        const double scale = 1.0 / sqrt(ss / (double)r + eps);
        for (int k = 0; k < r; ++k) t[k] *= scale;
      }
    }
#pragma omp for schedule(static)
    for (int i = 0; i < H; ++i) {
      if (!row) continue;
      widen_row(U, dtype, (size_t)i * r, r, row);
      z[i] = dot(row, t, r);
      if (flags & OR_FLAG_TILED_G) z[i] += xd[i % D];
    }
    free(row);
  }
  free(t);
  return bad ? -2 : 0;
}

/*
 * Dense definition.  Per token b (x[b] is row b of x[B,D]):
 *   y[b] = W2 (A(gate) .* (W3 x[b])), summing over all H units.
 * Outputs: y[B*D] (double), z[B*H] (double pre-activations, may be NULL),
 * n_live[B] (= |{i : z_i > 0}|, may be NULL).  Returns 0, or <0 on bad
 * arguments / allocation failure.
 */
int oracle_ffn_dense_ex(int D, int H, int r, int act, int dtype, int B, int flags, double eps, double thr,
                        const void* W1, const void* U, const void* V,
                        const void* W3, const void* W2, const void* x,
                        double* y, double* z, int* n_live) {
  if (check_args(D, H, r, act, dtype, B, flags, eps, thr)) return -1;
  double* xd = (double*)malloc(sizeof(double) * (size_t)D);
  double* zb = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)H);
  if (!xd || !zb || !g) {
    free(xd); free(zb); free(g);
    return -2;
  }
  int rc = 0;
  for (int b = 0; b < B && rc == 0; ++b) {
    widen_row(x, dtype, (size_t)b * D, D, xd);
    rc = gate(D, H, r, dtype, flags, eps, W1, U, V, xd, zb);
    if (rc) break;
    int bad = 0;
#pragma omp parallel
    {
      double* row = (double*)malloc(sizeof(double) * (size_t)(D > H ? D : H));
      if (!row) {
#pragma omp atomic write
        bad = 1;
      }
      /* up projection and gate product over every unit */
#pragma omp for schedule(static)
      for (int i = 0; i < H; ++i) {
        if (!row) continue;
        widen_row(W3, dtype, (size_t)i * D, D, row);
        double u = dot(row, xd, D);
        g[i] = gate_value(act, thr, zb[i]) * up_value(act, flags, u);
      }
      /* down projection: y_m = sum_i W2[m,i] g_i, i ascending */
#pragma omp for schedule(static)
      for (int m = 0; m < D; ++m) {
        if (!row) continue;
        widen_row(W2, dtype, (size_t)m * H, H, row);
        y[(size_t)b * D + m] = dot(row, g, H);
      }
      free(row);
    }
    if (bad) { rc = -2; break; }
    int cnt = 0;
    for (int i = 0; i < H; ++i) cnt += (fabs(activation(act, zb[i])) > thr);
    if (n_live) n_live[b] = cnt;
    if (z) memcpy(z + (size_t)b * H, zb, sizeof(double) * (size_t)H);
  }
  free(xd); free(zb); free(g);
  return rc;
}

int oracle_ffn_dense(int D, int H, int r, int act, int dtype, int B,
                     const void* W1, const void* U, const void* V,
                     const void* W3, const void* W2, const void* x,
                     double* y, double* z, int* n_live) {
  return oracle_ffn_dense_ex(D, H, r, act, dtype, B, 0, 0.0, 0.0, W1, U, V, W3, W2, x, y, z, n_live);
}

/*
 * Gate-first evaluation: the gate over all units, then only the live set.
 *   S = {i : z_i > 0} in ascending order ({i : |A(z_i)| > thr} in the _ex form)
 *   h_i = A(z_i) * (W3[i,:] . x)          for i in S
 *   y_m = sum_{i in S} W2[m,i] h_i       (i ascending)
 * Same outputs and return codes as oracle_ffn_dense; idx[B*H] (may be NULL)
 * receives S for each token, padded with -1.
 */
int oracle_ffn_gate_first_ex(int D, int H, int r, int act, int dtype, int B, int flags, double eps, double thr,
                             const void* W1, const void* U, const void* V,
                             const void* W3, const void* W2, const void* x,
                             double* y, int* idx, int* n_live) {
  if (check_args(D, H, r, act, dtype, B, flags, eps, thr)) return -1;
  double* xd = (double*)malloc(sizeof(double) * (size_t)D);
  double* zb = (double*)malloc(sizeof(double) * (size_t)H);
  double* h = (double*)malloc(sizeof(double) * (size_t)H);
  int* S = (int*)malloc(sizeof(int) * (size_t)H);
  if (!xd || !zb || !h || !S) {
    free(xd); free(zb); free(h); free(S);
    return -2;
  }
  int rc = 0;
  for (int b = 0; b < B && rc == 0; ++b) {
    widen_row(x, dtype, (size_t)b * D, D, xd);
    rc = gate(D, H, r, dtype, flags, eps, W1, U, V, xd, zb);
    if (rc) break;
    int k = 0;
    for (int i = 0; i < H; ++i)
      if (fabs(activation(act, zb[i])) > thr) S[k++] = i;
    int bad = 0;
#pragma omp parallel
    {
      double* row = (double*)malloc(sizeof(double) * (size_t)D);
      if (!row) {
#pragma omp atomic write
        bad = 1;
      }
#pragma omp for schedule(static)
      for (int q = 0; q < k; ++q) {
        if (!row) continue;
        int i = S[q];
        widen_row(W3, dtype, (size_t)i * D, D, row);
        h[q] = activation(act, zb[i]) * up_value(act, flags, dot(row, xd, D));
      }
#pragma omp for schedule(static)
      for (int m = 0; m < D; ++m) {
        double s = 0.0;
        for (int q = 0; q < k; ++q)
          s += elem(W2, dtype, (size_t)m * H + (size_t)S[q]) * h[q];
        y[(size_t)b * D + m] = s;
      }
      free(row);
    }
    if (bad) { rc = -2; break; }
    if (n_live) n_live[b] = k;
    if (idx) {
      for (int q = 0; q < H; ++q) idx[(size_t)b * H + q] = (q < k) ? S[q] : -1;
    }
  }
  free(xd); free(zb); free(h); free(S);
  return rc;
}

int oracle_ffn_gate_first(int D, int H, int r, int act, int dtype, int B,
                          const void* W1, const void* U, const void* V,
                          const void* W3, const void* W2, const void* x,
                          double* y, int* idx, int* n_live) {
  return oracle_ffn_gate_first_ex(D, H, r, act, dtype, B, 0, 0.0, 0.0, W1, U, V, W3, W2, x, y, idx, n_live);
}

/* ------------------------------------------------------------------------ int8 */

/* Symmetric quantisation of W[rows, cols] to codes in [-qmax, qmax] with one
 * scale per group of `group` consecutive columns of a row (group = cols: one
 * per row), s[i * (cols / group) + g]; binary32 decisions.  qmax = 127 for int8
 * weights, 7 for int4. */
int oracle_quantize_rows_g(int rows, int cols, int qmax, int group, const float* W, int8_t* q, float* s) {
  if (rows < 0 || cols <= 0 || qmax < 1 || qmax > 127 || group < 1 || cols % group) return -1;
  const float qm = (float)qmax;
  const int ng = cols / group;
  for (int i = 0; i < rows; ++i) {
    for (int g = 0; g < ng; ++g) {
      const float* w = W + (size_t)i * cols + (size_t)g * group;
      float amax = 0.0f;
      for (int j = 0; j < group; ++j) {
        const float a = fabsf(w[j]);
        if (a > amax) amax = a;
      }
      const float sc = amax / qm;
      s[(size_t)i * ng + g] = sc;
      for (int j = 0; j < group; ++j) {
        float v = 0.0f;
        if (sc > 0.0f) {
          v = rintf(w[j] / sc); /* default rounding mode: to nearest, ties to even */
          if (v > qm) v = qm;
          if (v < -qm) v = -qm;
        }
        q[(size_t)i * cols + (size_t)g * group + j] = (int8_t)v;
      }
    }
  }
  return 0;
}

/* Per-row symmetric quantisation to codes in [-qmax, qmax] (one scale per row). */
int oracle_quantize_rows_q(int rows, int cols, int qmax, const float* W, int8_t* q, float* s) {
  return oracle_quantize_rows_g(rows, cols, qmax, cols, W, q, s);
}

/* Per-row symmetric int8 quantisation of W[rows, cols] (binary32 decisions). */
int oracle_quantize_rows(int rows, int cols, const float* W, int8_t* q, float* s) {
  return oracle_quantize_rows_q(rows, cols, 127, W, q, s);
}

/* row i of a quantised matrix, dequantised: q[i, j] * s[i, j / group] (exact in double) */
static void dequant_row_g(const int8_t* q, const float* s, size_t i, int n, int group, double* out) {
  const size_t ng = (size_t)(n / group);
  for (int j = 0; j < n; ++j) out[j] = (double)q[i * (size_t)n + j] * (double)s[i * ng + (size_t)(j / group)];
}
static void dequant_row(const int8_t* q, const float* s, size_t i, int n, double* out) {
  dequant_row_g(q, s, i, n, n, out);
}

/*
 * Dense definition with weight-only quantised weights: q1, q3 [H, D] with one
 * scale per group of `group` columns, s1, s3 [H, D / group] (group = D: one per
 * row, the int8 form); q2 [D, H] with scales s2 [D]; x [B, D] bf16 bits.  flags
 * may only hold OR_FLAG_DOUBLE_ACT (the standard gate).  Outputs as
 * oracle_ffn_dense_ex.  oracle_ffn_dense_q8 is the form with group = D.
 */
int oracle_ffn_dense_qg(int D, int H, int act, int B, int flags, double thr, int group,
                        const int8_t* q1, const float* s1, const int8_t* q3, const float* s3,
                        const int8_t* q2, const float* s2, const void* x,
                        double* y, double* z, int* n_live) {
  if (check_args(D, H, 0, act, OR_BF16, B, flags, 0.0, thr)) return -1;
  if (flags & ~OR_FLAG_DOUBLE_ACT) return -1;
  if (group < 1 || D % group) return -1;
  double* xd = (double*)malloc(sizeof(double) * (size_t)D);
  double* zb = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)H);
  if (!xd || !zb || !g) {
    free(xd); free(zb); free(g);
    return -2;
  }
  int rc = 0;
  for (int b = 0; b < B && rc == 0; ++b) {
    widen_row(x, OR_BF16, (size_t)b * D, D, xd);
    int bad = 0;
#pragma omp parallel
    {
      double* row = (double*)malloc(sizeof(double) * (size_t)(D > H ? D : H));
      if (!row) {
#pragma omp atomic write
        bad = 1;
      }
      /* gate and up projection of every unit */
#pragma omp for schedule(static)
      for (int i = 0; i < H; ++i) {
        if (!row) continue;
        dequant_row_g(q1, s1, (size_t)i, D, group, row);
        zb[i] = dot(row, xd, D);
        dequant_row_g(q3, s3, (size_t)i, D, group, row);
        const double u = dot(row, xd, D);
        g[i] = gate_value(act, thr, zb[i]) * up_value(act, flags, u);
      }
      /* down projection: y_m = sum_i (q2[m, i] s2[m]) g_i, i ascending */
#pragma omp for schedule(static)
      for (int m = 0; m < D; ++m) {
        if (!row) continue;
        dequant_row(q2, s2, (size_t)m, H, row);
        y[(size_t)b * D + m] = dot(row, g, H);
      }
      free(row);
    }
    if (bad) { rc = -2; break; }
    int cnt = 0;
    for (int i = 0; i < H; ++i) cnt += (fabs(activation(act, zb[i])) > thr);
    if (n_live) n_live[b] = cnt;
    if (z) memcpy(z + (size_t)b * H, zb, sizeof(double) * (size_t)H);
  }
  free(xd); free(zb); free(g);
  return rc;
}

int oracle_ffn_dense_q8(int D, int H, int act, int B, int flags, double thr,
                        const int8_t* q1, const float* s1, const int8_t* q3, const float* s3,
                        const int8_t* q2, const float* s2, const void* x,
                        double* y, double* z, int* n_live) {
  return oracle_ffn_dense_qg(D, H, act, B, flags, thr, D, q1, s1, q3, s3, q2, s2, x, y, z, n_live);
}

/*
 * The low-rank gate ("LoPA Gating: moving the ceiling", the plain form
 * z = U (V x)) with weight-only int8 weights, one scale per row of every
 * matrix: qU [H, r] with sU [H], qV [r, D] with sV [r], q3 [H, D] with s3 [H],
 * q2 [D, H] with s2 [D]; x [B, D] bf16 bits.
 *     t = dequant(V) x,  z_i = dequant(U)[i, :] . t,  then as oracle_ffn_dense_q8.
 * flags may only hold OR_FLAG_DOUBLE_ACT.  Outputs as oracle_ffn_dense_ex.
 */
int oracle_ffn_lopa_q8(int D, int H, int r, int act, int B, int flags, double thr,
                       const int8_t* qU, const float* sU, const int8_t* qV, const float* sV,
                       const int8_t* q3, const float* s3, const int8_t* q2, const float* s2, const void* x,
                       double* y, double* z, int* n_live) {
  if (check_args(D, H, r, act, OR_BF16, B, flags, 0.0, thr) || r <= 0) return -1;
  if (flags & ~OR_FLAG_DOUBLE_ACT) return -1;
  double* xd = (double*)malloc(sizeof(double) * (size_t)D);
  double* t = (double*)malloc(sizeof(double) * (size_t)r);
  double* zb = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)H);
  double* row = (double*)malloc(sizeof(double) * (size_t)(D > H ? D : H));
  if (!xd || !t || !zb || !g || !row) {
    free(xd); free(t); free(zb); free(g); free(row);
    return -2;
  }
  for (int b = 0; b < B; ++b) {
    widen_row(x, OR_BF16, (size_t)b * D, D, xd);
    for (int k = 0; k < r; ++k) {  /* t = V x */
      dequant_row(qV, sV, (size_t)k, D, row);
      t[k] = dot(row, xd, D);
    }
    for (int i = 0; i < H; ++i) {  /* z = U t, u = W3 x, g = A(z) u */
      dequant_row(qU, sU, (size_t)i, r, row);
      zb[i] = dot(row, t, r);
      dequant_row(q3, s3, (size_t)i, D, row);
      const double u = dot(row, xd, D);
      g[i] = gate_value(act, thr, zb[i]) * up_value(act, flags, u);
    }
    for (int m = 0; m < D; ++m) {  /* y_m = sum_i (q2[m, i] s2[m]) g_i, i ascending (one group per row) */
      dequant_row_g(q2, s2, (size_t)m, H, H, row);
      y[(size_t)b * D + m] = dot(row, g, H);
    }
    int cnt = 0;
    for (int i = 0; i < H; ++i) cnt += (fabs(activation(act, zb[i])) > thr);
    if (n_live) n_live[b] = cnt;
    if (z) memcpy(z + (size_t)b * H, zb, sizeof(double) * (size_t)H);
  }
  free(xd); free(t); free(zb); free(g); free(row);
  return 0;
}
