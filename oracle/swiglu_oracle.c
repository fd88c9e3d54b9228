/*
 * Reference oracle for the fused SwiGLU MLP, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through
 * the seeded synthetic inputs.
 *
 * Everything is plain, slow, obviously-correct fp64 loops.  There is no
 * blocking, fusion or reordering beyond the definitions below.
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
    double a;
    if (mode == ORACLE_TWO_ROUND)
      a = oracle_round(oracle_round(oracle_silu(gs), dt) * us, dt);
    else
      a = rnd(oracle_silu(g) * u, mode, dt);    /* one rounding, from unrounded g, u */
    if (Grow) Grow[j] = gs;
    if (Urow) Urow[j] = us;
    Arow[j] = a;
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
 * with G (= mg X Wg^T), U the stored values. */
static void dgu_row(const void* dY, const void* Wd, int in_dt, const double* Grow,
                    const double* Urow, int64_t m, int64_t D, int64_t H, int mode, int dt,
                    double mg, double md, double* dGrow, double* dUrow) {
  for (int64_t j = 0; j < H; ++j) {
    double da = 0.0;
    for (int64_t d = 0; d < D; ++d)
      da += load_elem(dY, m * D + d, in_dt) * load_elem(Wd, d * H + j, in_dt);
    da = md * da;
    double g = Grow[j], u = Urow[j];
    dUrow[j] = rnd(da * oracle_silu(g), mode, dt);
    dGrow[j] = rnd(da * u * oracle_dsilu(g) * mg, mode, dt);
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
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m)
    dgu_row(dY, Wd, in_dt, G + m * H, U + m * H, m, D, H, mode, dt, mg, md, dG + m * H,
            dU + m * H);

  /* dWd[d,j] = md * sum_m dY[m,d] A[m,j] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t d = 0; d < D; ++d)
    for (int64_t j = 0; j < H; ++j) {
      double s = 0.0;
      for (int64_t m = 0; m < M; ++m) s += load_elem(dY, m * D + d, in_dt) * A[m * H + j];
      s = md * s;
      if (dWd0) s += dWd0[d * H + j];
      dWd[d * H + j] = rnd(s, mode, dt);
    }

  /* dWg[j,k] = sum_m dG[m,j] X[m,k];  dWu[j,k] = sum_m dU[m,j] X[m,k] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t j = 0; j < H; ++j)
    for (int64_t k = 0; k < D; ++k) {
      double sg = 0.0, su = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        double x = load_elem(X, m * D + k, in_dt);
        sg += dG[m * H + j] * x;
        su += dU[m * H + j] * x;
      }
      if (dWg0) sg += dWg0[j * D + k];
      if (dWu0) su += dWu0[j * D + k];
      dWg[j * D + k] = rnd(sg, mode, dt);
      dWu[j * D + k] = rnd(su, mode, dt);
    }

  /* dX[m,k] = sum_j dG[m,j] Wg[j,k] + sum_j dU[m,j] Wu[j,k] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < D; ++k) {
      double pg = 0.0, pu = 0.0;
      for (int64_t j = 0; j < H; ++j) {
        pg += dG[m * H + j] * load_elem(Wg, j * D + k, in_dt);
        pu += dU[m * H + j] * load_elem(Wu, j * D + k, in_dt);
      }
      dX[m * D + k] = rnd(pg + pu, mode, dt);
    }
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
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < R; ++r) {
    int64_t m = rows[r];
    gate_up_row(X, Wg, Wu, in_dt, m, D, H, mode, dt, 1.0, G_s + r * H, U_s + r * H,
                A_s + r * H);
    down_row(A_s + r * H, Wd, in_dt, D, H, mode, dt, 1.0, Y_s + r * D);
    dgu_row(dY, Wd, in_dt, G_s + r * H, U_s + r * H, m, D, H, mode, dt, 1.0, 1.0,
            dG_s + r * H, dU_s + r * H);
    for (int64_t k = 0; k < D; ++k) {
      double pg = 0.0, pu = 0.0;
      for (int64_t j = 0; j < H; ++j) {
        pg += dG_s[r * H + j] * load_elem(Wg, j * D + k, in_dt);
        pu += dU_s[r * H + j] * load_elem(Wu, j * D + k, in_dt);
      }
      dX_s[r * D + k] = rnd(pg + pu, mode, dt);
    }
  }
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
      if (mode == ORACLE_TWO_ROUND)
        a[m] = oracle_round(oracle_round(oracle_silu(gs), dt) * us, dt);
      else
        a[m] = rnd(oracle_silu(g) * u, mode, dt);
      du[m] = rnd(da * oracle_silu(gs), mode, dt);
      dg[m] = rnd(da * us * oracle_dsilu(gs), mode, dt);
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
