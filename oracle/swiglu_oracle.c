/*
 * Reference oracle for the fused SwiGLU MLP, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through
 * the seeded synthetic inputs.
 *
 * Everything is plain, slow, obviously-correct fp64 loops.  There is no
 * blocking, fusion or reordering beyond the definitions below.  Where a sum
 * runs over the first index of a row-major matrix, the matrix is first
 * copied transposed (values only) so that the loop reads consecutive memory;
 * every sum still adds its terms in the order of its definition.
 *
 * What it computes (sources):
 *   "[RFC] Full-pipeline SwiGLU MLP with forward/backward co-optimization"
 *   (Liger-Kernel issue #1347), section "Summary": the MLP is
 *       G = X Wg^T,  U = X Wu^T,  A = SiLU(G) * U,  Y = A Wd^T
 *   with G, U and A kept for backward, and the four gradients dI (= dX),
 *   dWg, dWu, dWd of section "Correctness".
 *   "Scope one-round FP32 SwiGLU to the exact Qwen3.5 contract" (xorl PR #51),
 *   review section: the one-round program computes SiLU and the product in
 *   fp32 and rounds once to the storage type; the historical two-round
 *   program rounds SiLU(gate) to the storage type before the product.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - rounding is round-to-nearest-even, applied once, straight from fp64;
 *   - A is formed from the unrounded G and U accumulators;
 *   - backward uses the stored (rounded) G, U, A; dA is never rounded;
 *   - gradients are rounded once to the storage type.
 *
 *   Gate/down multipliers (the Falcon-H1 variant the maintainer thread of
 *   the RFC defers to a follow-up, "[RFC] Full-pipeline SwiGLU MLP ...",
 *   maintainer thread; the pages do not define it, the plain reading is
 *   taken):  A = SiLU(mg G) * U,  Y = md (A Wd^T), G = X Wg^T, U = X Wu^T;
 *   the stored gate pre-activation is mg G.  By the chain rule
 *       dA = md (dY Wd),  dU = dA SiLU(mg G),  dG = dA U SiLU'(mg G) mg,
 *       dWd = md (dY^T A),  dWg = dG^T X,  dWu = dU^T X,  dX = dG Wg + dU Wu.
 *   mg = md = 1 is the standard MLP.  Gradient accumulation (beta = 1):
 *   dW = rnd(dW_before + the new sum), one rounding.
 *
 * Modes:
 *   ORACLE_EXACT     fp64 throughout, nothing rounded (finite differences);
 *   ORACLE_ONE_ROUND rounds at the same points as the GPU path (parity);
 *   ORACLE_TWO_ROUND negative control: A = rnd(rnd(SiLU(Gs)) * Us).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ODT_BF16 = 0, ODT_F16 = 1, ODT_F32 = 2, ODT_F64 = 3 };
enum { ORACLE_EXACT = 0, ORACLE_ONE_ROUND = 1, ORACLE_TWO_ROUND = 2 };

/* ---------------------------------------------------------------------- */
/* Storage types: decoding and round-to-nearest-even                       */
/* ---------------------------------------------------------------------- */

static double decode_bf16(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;   /* bf16 is the top half of fp32 */
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)frac, -24);                 /* subnormal */
  } else if (e == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), e - 25);     /* (1.frac) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static double load_elem(const void* p, int64_t i, int dt) {
  switch (dt) {
    case ODT_BF16: return decode_bf16(((const uint16_t*)p)[i]);
    case ODT_F16: return decode_f16(((const uint16_t*)p)[i]);
    case ODT_F32: return (double)((const float*)p)[i];
    default: return ((const double*)p)[i];
  }
}

/* Round x (fp64) to the nearest value of the storage type, ties to even,
 * keeping subnormals and sending overflow to +-inf.  The type has a p-bit
 * significand, minimum normal exponent emin, and overflows at 2^ovf. */
double oracle_round(double x, int dt) {
  int p, emin, ovf;
  switch (dt) {
    case ODT_BF16: p = 8; emin = -126; ovf = 128; break;
    case ODT_F16: p = 11; emin = -14; ovf = 16; break;
    case ODT_F32: p = 24; emin = -126; ovf = 128; break;
    default: return x;
  }
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int e;
  frexp(x, &e);                   /* |x| in [2^(e-1), 2^e) */
  int q = e - p;                  /* exponent of one unit in the last place */
  if (q < emin - (p - 1)) q = emin - (p - 1);   /* subnormal spacing */
  double r = ldexp(nearbyint(ldexp(x, -q)), q);  /* default mode: ties-to-even */
  if (fabs(r) >= ldexp(1.0, ovf)) r = copysign(INFINITY, x);
  return r;
}

static double rnd(double x, int mode, int dt) {
  return mode == ORACLE_EXACT ? x : oracle_round(x, dt);
}

/* Decode n storage elements into fp64 (a convenience for the tests). */
void oracle_decode(const void* src, int dt, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = load_elem(src, i, dt);
}

void oracle_round_array(const double* src, int dt, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round(src[i], dt);
}

/* ---------------------------------------------------------------------- */
/* SiLU and its derivative                                                 */
/* ---------------------------------------------------------------------- */

/* sigma(g) = 1 / (1 + e^-g);  SiLU(g) = g * sigma(g). */
double oracle_sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

double oracle_silu(double g) { return g * oracle_sigmoid(g); }

/* d/dg [g * sigma(g)] = sigma + g * sigma * (1 - sigma) = sigma * (1 + g (1 - sigma)). */
double oracle_dsilu(double g) {
  double s = oracle_sigmoid(g);
  return s * (1.0 + g * (1.0 - s));
}

/* ---------------------------------------------------------------------- */
/* The elementwise SwiGLU stage (every form of the oracle goes through    */
/* these two functions)                                                    */
/* ---------------------------------------------------------------------- */

/* Forward: A from the gate and up sums g, u (gate multiplier applied) and
 * their stored values gs, us.  One-round: SiLU(g) * u in fp64 from the
 * unrounded sums, rounded once; two-round (negative control): SiLU of the
 * stored gate rounded first, then the product with the stored up value. */
static double swiglu_a(double g, double u, double gs, double us, int mode, int dt) {
  if (mode == ORACLE_TWO_ROUND) return oracle_round(oracle_round(oracle_silu(gs), dt) * us, dt);
  return rnd(oracle_silu(g) * u, mode, dt);
}

/* Backward: from dA (never rounded) and the stored g, u,
 *   dU = dA SiLU(g),  dG = dA u SiLU'(g) mg, each rounded once. */
static void dswiglu(double da, double g, double u, double mg, int mode, int dt, double* dg,
                    double* du) {
  *du = rnd(da * oracle_silu(g), mode, dt);
  *dg = rnd(da * u * oracle_dsilu(g) * mg, mode, dt);
}

/* The elementwise stage alone, over n elements (for checking the GPU's
 * epilogue arithmetic on chosen values).  Forward, when A is not NULL:
 * A[i] from g[i], u[i] (the sums, gate multiplier applied) and gs[i], us[i]
 * (their stored values; used by the two-round program only).  Backward,
 * when dG and dU are not NULL: dG[i], dU[i] from da[i] and the stored
 * gs[i], us[i], with gate multiplier mg. */
void oracle_elementwise(int64_t n, const double* g, const double* u, const double* gs,
                        const double* us, const double* da, int mode, int dt, double mg,
                        double* A, double* dG, double* dU) {
  for (int64_t i = 0; i < n; ++i) {
    if (A) A[i] = swiglu_a(g[i], u[i], gs[i], us[i], mode, dt);
    if (dG && dU) dswiglu(da[i], gs[i], us[i], mg, mode, dt, dG + i, dU + i);
  }
}

/* ---------------------------------------------------------------------- */
/* Memory layout helpers.  They move values only: every sum below adds    */
/* its terms in the order its definition gives, whatever the layout.      */
/* ---------------------------------------------------------------------- */

/* Storage matrix [rows, cols] -> fp64 copy of its transpose [cols, rows], so
 * that a sum over the row index reads consecutive memory. */
static double* decode_transposed(const void* src, int dt, int64_t rows, int64_t cols) {
  double* t = (double*)malloc((size_t)rows * (size_t)cols * sizeof(double));
  if (!t) abort();
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < cols; ++c)
    for (int64_t r = 0; r < rows; ++r) t[c * rows + r] = load_elem(src, r * cols + c, dt);
  return t;
}

/* ---------------------------------------------------------------------- */
/* Full forward                                                            */
/* ---------------------------------------------------------------------- */

/* One row of the gate/up stage: for hidden unit j,
 *   g = mg * sum_k X[m,k] Wg[j,k],  u = sum_k X[m,k] Wu[j,k]. */
static void gate_up_row(const void* X, const void* Wg, const void* Wu, int in_dt,
                        int64_t m, int64_t D, int64_t H, int mode, int dt, double mg,
                        double* Grow, double* Urow, double* Arow) {
  for (int64_t j = 0; j < H; ++j) {
    double g = 0.0, u = 0.0;
    for (int64_t k = 0; k < D; ++k) {
      double x = load_elem(X, m * D + k, in_dt);
      g += x * load_elem(Wg, j * D + k, in_dt);
      u += x * load_elem(Wu, j * D + k, in_dt);
    }
    g = mg * g;
    double gs = rnd(g, mode, dt), us = rnd(u, mode, dt);
    if (Grow) Grow[j] = gs;
    if (Urow) Urow[j] = us;
    Arow[j] = swiglu_a(g, u, gs, us, mode, dt);
  }
}

/* Y[m,d] = md * sum_j A[m,j] Wd[d,j]. */
static void down_row(const double* Arow, const void* Wd, int in_dt, int64_t D, int64_t H,
                     int mode, int dt, double md, double* Yrow) {
  for (int64_t d = 0; d < D; ++d) {
    double y = 0.0;
    for (int64_t j = 0; j < H; ++j) y += Arow[j] * load_elem(Wd, d * H + j, in_dt);
    Yrow[d] = rnd(md * y, mode, dt);
  }
}

/* X [M,D], Wg/Wu [H,D], Wd [D,H] in storage type in_dt (row-major); gate and
 * down multipliers mg, md.  Outputs (fp64, row-major): G (the stored gate
 * pre-activation mg X Wg^T), U, A [M,H] (G/U may be NULL), Y [M,D]. */
void oracle_fwd_ex(const void* X, const void* Wg, const void* Wu, const void* Wd, int in_dt,
                   int64_t M, int64_t D, int64_t H, int mode, int dt, double mg, double md,
                   double* G, double* U, double* A, double* Y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    gate_up_row(X, Wg, Wu, in_dt, m, D, H, mode, dt, mg,
                G ? G + m * H : NULL, U ? U + m * H : NULL, A + m * H);
    down_row(A + m * H, Wd, in_dt, D, H, mode, dt, md, Y + m * D);
  }
}

/* The standard MLP: mg = md = 1. */
void oracle_fwd(const void* X, const void* Wg, const void* Wu, const void* Wd, int in_dt,
                int64_t M, int64_t D, int64_t H, int mode, int dt,
                double* G, double* U, double* A, double* Y) {
  oracle_fwd_ex(X, Wg, Wu, Wd, in_dt, M, D, H, mode, dt, 1.0, 1.0, G, U, A, Y);
}

/* ---------------------------------------------------------------------- */
/* Full backward                                                           */
/* ---------------------------------------------------------------------- */

/* dA[m,j] = md * sum_d dY[m,d] Wd[d,j] (kept in fp64, never rounded), then
 *   dU = dA * SiLU(G),  dG = dA * U * SiLU'(G) * mg
 * with G (= mg X Wg^T), U the stored values.  WdT is Wd transposed (fp64
 * [H, D]): WdT[j*D + d] = Wd[d, j]. */
static void dgu_row(const void* dY, const double* WdT, int in_dt, const double* Grow,
                    const double* Urow, int64_t m, int64_t D, int64_t H, int mode, int dt,
                    double mg, double md, double* dGrow, double* dUrow) {
  for (int64_t j = 0; j < H; ++j) {
    double da = 0.0;
    for (int64_t d = 0; d < D; ++d) da += load_elem(dY, m * D + d, in_dt) * WdT[j * D + d];
    da = md * da;
    dswiglu(da, Grow[j], Urow[j], mg, mode, dt, dGrow + j, dUrow + j);
  }
}

/* dX[m,k] = sum_j dG[m,j] Wg[j,k] + sum_j dU[m,j] Wu[j,k] for one row m, the
 * two sums each over j in order; WgT, WuT: Wg, Wu transposed (fp64 [D, H]). */
static void dx_row(const double* dGrow, const double* dUrow, const double* WgT,
                   const double* WuT, int64_t D, int64_t H, int mode, int dt, double* dXrow) {
  for (int64_t k = 0; k < D; ++k) {
    double pg = 0.0, pu = 0.0;
    for (int64_t j = 0; j < H; ++j) {
      pg += dGrow[j] * WgT[k * H + j];
      pu += dUrow[j] * WuT[k * H + j];
    }
    dXrow[k] = rnd(pg + pu, mode, dt);
  }
}

/* Inputs: dY [M,D]; X, Wg, Wu, Wd as in oracle_fwd; G, U, A [M,H] the stored
 * forward values (fp64 arrays holding storage-type values); multipliers mg,
 * md as in oracle_fwd_ex; dWg0, dWu0, dWd0: the gradients already held, to
 * which the new ones are added (beta = 1), or NULL (overwrite).
 * Outputs (fp64): dG, dU [M,H]; dX [M,D]; dWg, dWu [H,D]; dWd [D,H].
 * Separate form: dWg = dG^T X, dWu = dU^T X, dX = dG Wg + dU Wu. */
void oracle_bwd_ex(const void* dY, const void* X, const void* Wg, const void* Wu,
                   const void* Wd, int in_dt, const double* G, const double* U,
                   const double* A, int64_t M, int64_t D, int64_t H, int mode, int dt,
                   double mg, double md, const double* dWg0, const double* dWu0,
                   const double* dWd0, double* dG, double* dU, double* dX, double* dWg,
                   double* dWu, double* dWd) {
  double* WdT = decode_transposed(Wd, in_dt, D, H);   /* [H, D] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m)
    dgu_row(dY, WdT, in_dt, G + m * H, U + m * H, m, D, H, mode, dt, mg, md, dG + m * H,
            dU + m * H);
  free(WdT);

  /* dWd[d,j] = md * sum_m dY[m,d] A[m,j]  (dYT[d*M + m] = dY[m,d], AT[j*M + m] = A[m,j]) */
  double* dYT = decode_transposed(dY, in_dt, M, D);   /* [D, M] */
  double* AT = decode_transposed(A, ODT_F64, M, H);   /* [H, M] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t d = 0; d < D; ++d)
    for (int64_t j = 0; j < H; ++j) {
      double s = 0.0;
      for (int64_t m = 0; m < M; ++m) s += dYT[d * M + m] * AT[j * M + m];
      s = md * s;
      if (dWd0) s += dWd0[d * H + j];
      dWd[d * H + j] = rnd(s, mode, dt);
    }
  free(dYT);
  free(AT);

  /* dWg[j,k] = sum_m dG[m,j] X[m,k];  dWu[j,k] = sum_m dU[m,j] X[m,k] */
  double* XT = decode_transposed(X, in_dt, M, D);     /* [D, M] */
  double* dGT = decode_transposed(dG, ODT_F64, M, H); /* [H, M] */
  double* dUT = decode_transposed(dU, ODT_F64, M, H);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t j = 0; j < H; ++j)
    for (int64_t k = 0; k < D; ++k) {
      double sg = 0.0, su = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        double x = XT[k * M + m];
        sg += dGT[j * M + m] * x;
        su += dUT[j * M + m] * x;
      }
      if (dWg0) sg += dWg0[j * D + k];
      if (dWu0) su += dWu0[j * D + k];
      dWg[j * D + k] = rnd(sg, mode, dt);
      dWu[j * D + k] = rnd(su, mode, dt);
    }
  free(XT);
  free(dGT);
  free(dUT);

  /* dX[m,k] = sum_j dG[m,j] Wg[j,k] + sum_j dU[m,j] Wu[j,k] */
  double* WgT = decode_transposed(Wg, in_dt, H, D);   /* [D, H] */
  double* WuT = decode_transposed(Wu, in_dt, H, D);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m)
    dx_row(dG + m * H, dU + m * H, WgT, WuT, D, H, mode, dt, dX + m * D);
  free(WgT);
  free(WuT);
}

/* The standard MLP, gradients overwritten. */
void oracle_bwd(const void* dY, const void* X, const void* Wg, const void* Wu,
                const void* Wd, int in_dt, const double* G, const double* U,
                const double* A, int64_t M, int64_t D, int64_t H, int mode, int dt,
                double* dG, double* dU, double* dX, double* dWg, double* dWu, double* dWd) {
  oracle_bwd_ex(dY, X, Wg, Wu, Wd, in_dt, G, U, A, M, D, H, mode, dt, 1.0, 1.0, NULL, NULL,
                NULL, dG, dU, dX, dWg, dWu, dWd);
}

/* ---------------------------------------------------------------------- */
/* Sampled forms for full-size shapes                                      */
/* ---------------------------------------------------------------------- */

/* For the token rows listed in rows[0..R): the stored G, U, A rows, the Y row,
 * and the dX row (through that row's dG, dU).  Outputs are packed per sampled
 * row: G_s, U_s, A_s, dG_s, dU_s [R,H]; Y_s, dX_s [R,D].  Cost ~7 D H per row. */
void oracle_rows(const void* X, const void* Wg, const void* Wu, const void* Wd,
                 const void* dY, int in_dt, int64_t M, int64_t D, int64_t H,
                 const int64_t* rows, int64_t R, int mode, int dt,
                 double* G_s, double* U_s, double* A_s, double* Y_s,
                 double* dG_s, double* dU_s, double* dX_s) {
  (void)M;
  double* WdT = decode_transposed(Wd, in_dt, D, H);   /* [H, D] */
  double* WgT = decode_transposed(Wg, in_dt, H, D);   /* [D, H] */
  double* WuT = decode_transposed(Wu, in_dt, H, D);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < R; ++r) {
    int64_t m = rows[r];
    gate_up_row(X, Wg, Wu, in_dt, m, D, H, mode, dt, 1.0, G_s + r * H, U_s + r * H,
                A_s + r * H);
    down_row(A_s + r * H, Wd, in_dt, D, H, mode, dt, 1.0, Y_s + r * D);
    dgu_row(dY, WdT, in_dt, G_s + r * H, U_s + r * H, m, D, H, mode, dt, 1.0, 1.0,
            dG_s + r * H, dU_s + r * H);
    dx_row(dG_s + r * H, dU_s + r * H, WgT, WuT, D, H, mode, dt, dX_s + r * D);
  }
  free(WdT);
  free(WgT);
  free(WuT);
}

/* For the hidden units listed in cols[0..C): row j of dWg and dWu and column j
 * of dWd, each a full reduction over all M token rows.  Outputs packed per
 * sampled unit: dWg_s, dWu_s [C,D]; dWd_s [C,D] (dWd_s[c,d] = dWd[d, cols[c]]).
 * Cost ~6 M D per unit. */
void oracle_cols(const void* X, const void* Wg, const void* Wu, const void* Wd,
                 const void* dY, int in_dt, int64_t M, int64_t D, int64_t H,
                 const int64_t* cols, int64_t C, int mode, int dt,
                 double* dWg_s, double* dWu_s, double* dWd_s) {
  for (int64_t c = 0; c < C; ++c) {
    int64_t j = cols[c];
    double* dg = (double*)malloc((size_t)M * sizeof(double));
    double* du = (double*)malloc((size_t)M * sizeof(double));
    double* a = (double*)malloc((size_t)M * sizeof(double));
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
      double g = 0.0, u = 0.0, da = 0.0;
      for (int64_t k = 0; k < D; ++k) {
        double x = load_elem(X, m * D + k, in_dt);
        g += x * load_elem(Wg, j * D + k, in_dt);
        u += x * load_elem(Wu, j * D + k, in_dt);
      }
      for (int64_t d = 0; d < D; ++d)
        da += load_elem(dY, m * D + d, in_dt) * load_elem(Wd, d * H + j, in_dt);
      double gs = rnd(g, mode, dt), us = rnd(u, mode, dt);
      a[m] = swiglu_a(g, u, gs, us, mode, dt);
      dswiglu(da, gs, us, 1.0, mode, dt, dg + m, du + m);
    }
#pragma omp parallel for schedule(static)
    for (int64_t d = 0; d < D; ++d) {
      double sg = 0.0, su = 0.0, sd = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        double x = load_elem(X, m * D + d, in_dt);
        sg += dg[m] * x;
        su += du[m] * x;
        sd += load_elem(dY, m * D + d, in_dt) * a[m];
      }
      dWg_s[c * D + d] = rnd(sg, mode, dt);
      dWu_s[c * D + d] = rnd(su, mode, dt);
      dWd_s[c * D + d] = rnd(sd, mode, dt);
    }
    free(dg);
    free(du);
    free(a);
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
