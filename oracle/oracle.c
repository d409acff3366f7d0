/*
 * oracle.c -- float64 CPU reference for the row-wise normalization layers
 * (DyT, LayerNorm, Llama-style RMSNorm), forward and backward, including
 * the per-feature parameter-gradient column sums.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; it exists so that tests, the smoke check and the CPU
 * baseline timing can compare the CUDA kernels against an independent,
 * plainly written definition.  It shares no code, header or constant with
 * the CUDA library.
 *
 * Every computation is the textbook definition written out in float64,
 * row by row, with serial sums in index order and no blocking or
 * reordering.  Inputs arrive as raw float32, bfloat16 or float16 (raw
 * 16-bit patterns) or float64 arrays and are widened exactly to float64.
 *
 * Two modes:
 *   ORC_MATH   -- pure float64, no intermediate rounding (closed-form,
 *                 finite-difference and invariant checks);
 *   ORC_PARITY -- float64 plus round-to-nearest-even to the activation
 *                 dtype at the intermediate rounding points that the
 *                 fused-RMSNorm page (DeepSpeed PR 8645, quoted in PR
 *                 8664, section "Semantics") fixes: the normalized value,
 *                 grad_out * weight, and grad_out * normalized when the
 *                 weight has the activation dtype.  DyT and LayerNorm have
 *                 no intermediate rounding point; their only rounding is
 *                 the final store, which the caller applies.
 *
 * Outputs are float64 values BEFORE the final rounding to the output
 * dtype, plus a "scale" companion that the tests use to judge
 * cancellation: the first-order bound on the rounding error of evaluating
 * the output in a lower precision, divided by the unit roundoff.  A sum's
 * error is bounded by the sum of its terms' magnitudes, so inner
 * reductions (means) enter the scale as means of magnitudes; column sums
 * come with the sum of their squared terms instead.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2, ORC_F16 = 3 };
enum { ORC_MATH = 0, ORC_PARITY = 1 };

/* Largest finite bfloat16: significand 0xFF (8 bits) times 2^(127-7). */
#define BF16_MAX_FINITE (255.0 * 1329227995784915872903807060280344576.0 /* 2^120 */)
/* Largest finite IEEE binary16: significand 0x7FF (11 bits) times 2^(15-10). */
#define F16_MAX_FINITE 65504.0

/* Relative distance to a bfloat16 rounding midpoint below which a value
 * computed in float32 elsewhere may legitimately round the other way. */
#define NEAR_TIE_REL (1.0 / 131072.0) /* 2^-17 */

/* ---------------------------------------------------------------- inputs */

/* IEEE binary16 bit pattern to its exact value: 1 sign bit, 5 exponent
 * bits (bias 15), 10 fraction bits; exponent 0 holds zero and the
 * subnormals (fraction * 2^-24), exponent 31 infinity and NaN. */
static double f16_value(uint16_t h)
{
    int e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);
    return (h & 0x8000) ? -v : v;
}

static double widen(const void* p, int dt, int64_t i)
{
    if (dt == ORC_F64) return ((const double*)p)[i];
    if (dt == ORC_F32) return (double)((const float*)p)[i];
    if (dt == ORC_F16) return f16_value(((const uint16_t*)p)[i]);
    /* bfloat16 is the upper half of a float32 bit pattern. */
    uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------- rounding */

/*
 * Round a float64 to the nearest bfloat16, ties to even, directly (never
 * through float32).  bfloat16 keeps 8 significant bits and float32's
 * exponent range, so a normal value a in [2^(k-1), 2^k) is a multiple of
 * 2^(k-8); below the normal range (2^-126) the spacing stays 2^-133.
 * nearbyint() rounds half to even in the default rounding mode.
 * *near_tie is set when the value lies within NEAR_TIE_REL (relative) of a
 * rounding midpoint.
 */
static double round_bf16(double v, int* near_tie)
{
    if (near_tie) *near_tie = 0;
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int k;
    (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
    int qe = k - 8;
    if (qe < -133) qe = -133;
    double m = ldexp(a, -qe); /* exact: scaling by a power of two */
    double mr = nearbyint(m);
    if (near_tie) {
        double frac = m - floor(m);
        if (fabs(frac - 0.5) < NEAR_TIE_REL * m) *near_tie = 1;
    }
    double r = ldexp(mr, qe);
    if (r > BF16_MAX_FINITE) r = INFINITY;
    return copysign(r, v);
}

/*
 * Round a float64 to the nearest IEEE binary16, ties to even, directly.
 * binary16 keeps 11 significant bits; a normal value a in [2^(k-1), 2^k)
 * is a multiple of 2^(k-11), and below the normal range (2^-14) the
 * spacing stays 2^-24.  Results above the largest finite value (65504,
 * i.e. inputs from 65520 up) become infinity.  *near_tie as for bfloat16.
 */
static double round_f16(double v, int* near_tie)
{
    if (near_tie) *near_tie = 0;
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int k;
    (void)frexp(a, &k);
    int qe = k - 11;
    if (qe < -24) qe = -24;
    double m = ldexp(a, -qe);
    double mr = nearbyint(m);
    if (near_tie) {
        double frac = m - floor(m);
        if (fabs(frac - 0.5) < NEAR_TIE_REL * m) *near_tie = 1;
    }
    double r = ldexp(mr, qe);
    if (r > F16_MAX_FINITE) r = INFINITY;
    return copysign(r, v);
}

/* Round to the activation dtype: bfloat16 and binary16 as above, float32 by
 * the C conversion (round to nearest even), float64 unchanged. */
static double round_to(double v, int dt, int* near_tie)
{
    if (dt == ORC_BF16) return round_bf16(v, near_tie);
    if (dt == ORC_F16) return round_f16(v, near_tie);
    if (near_tie) *near_tie = 0;
    if (dt == ORC_F32) return (double)(float)v;
    return v;
}

/* Spacing of the activation dtype at |v|: the gap between the two
 * neighbours that a near-tie rounding of v chooses between (bfloat16: 8
 * significant bits down to 2^-133; binary16: 11 bits down to 2^-24;
 * float32: 24 bits down to 2^-149). */
static double spacing(double v, int dt)
{
    int bits = dt == ORC_BF16 ? 8 : dt == ORC_F16 ? 11 : 24;
    int lo = dt == ORC_BF16 ? -133 : dt == ORC_F16 ? -24 : -149;
    double a = fabs(v);
    if (a == 0.0 || isnan(a) || isinf(a)) return ldexp(1.0, lo);
    int k;
    (void)frexp(a, &k);
    int qe = k - bits;
    if (qe < lo) qe = lo;
    return ldexp(1.0, qe);
}

double orc_round_bf16(double v) { return round_bf16(v, NULL); }
void orc_round_bf16_array(const double* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = round_bf16(in[i], NULL);
}

int orc_bf16_near_tie(double v)
{
    int t;
    (void)round_bf16(v, &t);
    return t;
}

double orc_round_f16(double v) { return round_f16(v, NULL); }
void orc_round_f16_array(const double* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = round_f16(in[i], NULL);
}

static int64_t row_of(const int64_t* rows, int64_t r) { return rows ? rows[r] : r; }

/* ================================================================== DyT
 * Dynamic Tanh: y = gamma_j * tanh(alpha * x_ij) + beta_j with a scalar
 * alpha and per-channel gamma, beta (the fused DyT kernels of Liger-Kernel
 * PR 1617, "fix(dyt): use a 1D grid and tile small-width rows").
 * The backward uses the exact derivatives with sech^2 = 1 / cosh^2:
 *   dx_ij   = dy_ij * gamma_j * alpha * sech^2(alpha x_ij)
 *   dgamma_j = sum_i dy_ij * tanh(alpha x_ij)
 *   dbeta_j  = sum_i dy_ij
 *   dalpha   = sum_ij dy_ij * gamma_j * x_ij * sech^2(alpha x_ij)
 * IEEE evaluation throughout: with alpha = +inf every real element gives
 * tanh = +-1 and sech^2 = 0, so dx = (inf * 0) = NaN while the parameter
 * gradients stay finite, as that page's Summary requires of real rows.
 */

static double sech2(double z)
{
    double c = cosh(z);
    return 1.0 / (c * c);
}

int orc_dyt_fwd_rows(const void* x, int xt, int64_t M, int64_t N, double alpha,
                     const double* gamma, const double* beta, const int64_t* rows,
                     int64_t nrows, double* y, double* y_scale)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        for (int64_t j = 0; j < N; ++j) {
            double t = tanh(alpha * widen(x, xt, i * N + j));
            double gt = gamma[j] * t;
            y[r * N + j] = gt + beta[j];
            if (y_scale) y_scale[r * N + j] = fabs(gt) + fabs(beta[j]);
        }
    }
    return 0;
}

int orc_dyt_bwd_rows(const void* x, const void* dy, int xt, int64_t M, int64_t N,
                     double alpha, const double* gamma, const int64_t* rows,
                     int64_t nrows, double* dx)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        for (int64_t j = 0; j < N; ++j) {
            double xv = widen(x, xt, i * N + j);
            double g = widen(dy, xt, i * N + j);
            dx[r * N + j] = g * gamma[j] * alpha * sech2(alpha * xv);
        }
    }
    return 0;
}

/* Column sums over all M rows, serial in row order.  *_ss receive the sum
 * of the squared terms (the natural magnitude of a sum of random terms). */
int orc_dyt_bwd_cols(const void* x, const void* dy, int xt, int64_t M, int64_t N,
                     double alpha, const double* gamma, double* dgamma, double* dgamma_ss,
                     double* dbeta, double* dbeta_ss, double* dalpha, double* dalpha_ss)
{
    double da = 0.0, da_ss = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        dgamma[j] = dgamma_ss[j] = dbeta[j] = dbeta_ss[j] = 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double xv = widen(x, xt, i * N + j);
            double g = widen(dy, xt, i * N + j);
            double z = alpha * xv;
            double tg = g * tanh(z);
            double ta = g * gamma[j] * xv * sech2(z);
            dgamma[j] += tg;
            dgamma_ss[j] += tg * tg;
            dbeta[j] += g;
            dbeta_ss[j] += g * g;
            da += ta;
            da_ss += ta * ta;
        }
    }
    *dalpha = da;
    *dalpha_ss = da_ss;
    return 0;
}

/* ============================================================ LayerNorm
 * Standard LayerNorm over the last dimension with the biased variance and
 * eps inside the square root:
 *   mu_i = (1/N) sum_j x_ij,  var_i = (1/N) sum_j (x_ij - mu_i)^2,
 *   r_i = 1 / sqrt(var_i + eps),  xhat = (x - mu) r,
 *   y = xhat * gamma_j + beta_j  (gamma absent = 1, beta absent = 0).
 * The backward takes the saved per-row mean and rstd as inputs (the
 * torch-xpu-ops page "Layernorm bwd OPT #1880" describes a backward fed
 * with the forward's statistics):
 *   g = dy * gamma,  dx = r (g - mean_j g - xhat mean_j(g xhat)),
 *   dgamma_j = sum_i dy xhat,  dbeta_j = sum_i dy.
 */

int orc_ln_fwd_rows(const void* x, int xt, int64_t M, int64_t N, double eps,
                    const double* gamma, const double* beta, const int64_t* rows,
                    int64_t nrows, double* y, double* y_scale, double* mean, double* rstd)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        double s = 0.0, sa = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            s += widen(x, xt, i * N + j);
            sa += fabs(widen(x, xt, i * N + j));
        }
        double mu = s / (double)N;
        double mabs = sa / (double)N; /* scale of the mean's rounding error */
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double d = widen(x, xt, i * N + j) - mu;
            ss += d * d;
        }
        double var = ss / (double)N;
        double rs = 1.0 / sqrt(var + eps);
        if (mean) mean[r] = mu;
        if (rstd) rstd[r] = rs;
        for (int64_t j = 0; j < N; ++j) {
            double xh = (widen(x, xt, i * N + j) - mu) * rs;
            double g = gamma ? gamma[j] : 1.0;
            double b = beta ? beta[j] : 0.0;
            y[r * N + j] = xh * g + b;
            if (y_scale)
                y_scale[r * N + j] =
                    (fabs(widen(x, xt, i * N + j)) + mabs) * rs * fabs(g) + fabs(b);
        }
    }
    return 0;
}

int orc_ln_bwd_rows(const void* x, const void* dy, int xt, int64_t M, int64_t N,
                    const double* mean, const double* rstd, const double* gamma,
                    const int64_t* rows, int64_t nrows, double* dx, double* dx_scale)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        double mu = mean[i], rs = rstd[i];
        double sg = 0.0, sgx = 0.0, sga = 0.0, sgxa = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double xh = (widen(x, xt, i * N + j) - mu) * rs;
            double g = widen(dy, xt, i * N + j) * (gamma ? gamma[j] : 1.0);
            sg += g;
            sgx += g * xh;
            sga += fabs(g);
            sgxa += fabs(g * xh);
        }
        double a = sg / (double)N;
        double b = sgx / (double)N;
        double aa = sga / (double)N, ba = sgxa / (double)N; /* error scales of a, b */
        for (int64_t j = 0; j < N; ++j) {
            double xh = (widen(x, xt, i * N + j) - mu) * rs;
            double g = widen(dy, xt, i * N + j) * (gamma ? gamma[j] : 1.0);
            dx[r * N + j] = rs * (g - a - xh * b);
            if (dx_scale) dx_scale[r * N + j] = fabs(rs) * (fabs(g) + aa + fabs(xh) * ba);
        }
    }
    return 0;
}

int orc_ln_bwd_cols(const void* x, const void* dy, int xt, int64_t M, int64_t N,
                    const double* mean, const double* rstd, double* dgamma,
                    double* dgamma_ss, double* dbeta, double* dbeta_ss)
{
    for (int64_t j = 0; j < N; ++j) dgamma[j] = dgamma_ss[j] = dbeta[j] = dbeta_ss[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double xh = (widen(x, xt, i * N + j) - mean[i]) * rstd[i];
            double g = widen(dy, xt, i * N + j);
            dgamma[j] += g * xh;
            dgamma_ss[j] += (g * xh) * (g * xh);
            dbeta[j] += g;
            dbeta_ss[j] += g * g;
        }
    }
    return 0;
}

/* ============================================================== RMSNorm
 * Llama-style RMSNorm, weight * (x.float() * rsqrt(mean(x.float()^2) + eps))
 * .to(x.dtype), with the rounding points of the fused-RMSNorm page
 * (DeepSpeed PR 8645 quoted in PR 8664, section "Semantics"):
 *   r = 1 / sqrt(mean_j x^2 + eps)           (float64 here)
 *   n = round_x(x r)                          (one rounding of the normalized value)
 *   y = w * n                                 (final rounding by the caller)
 * Backward, rounding where eager autograd rounds:
 *   xhat = x r (unrounded),  dn = round_x(dy w),
 *   dx   = r (dn - xhat mean_j(dn xhat))      (final rounding by the caller)
 *   dw_j = sum_i term,  term = round_x(dy n) when the weight has the
 *          activation dtype, and dy n unrounded when the weight is float32.
 * r is always recomputed from x: the saved rstd is an optional cache of the
 * GPU path, not part of the definition.  At width one the input derivative
 * is dn eps / (x^2 + eps)^(3/2) (the PR 8664 page, "Numerics").
 *
 * Expression variants (the same page, "Which modules are replaced" and "Not
 * covered": classes that multiply by the weight before the cast, and the
 * Gemma family's (1 + weight)), selected by `variant`:
 *   ORC_RMS_CAST_FIRST  (0)  the expression above;
 *   ORC_RMS_WEIGHT_FIRST (1) y = w * (x r), one rounding at the output: the
 *                         weight multiplies the float32 normalized value;
 *   ORC_RMS_GEMMA       (2)  y = (x r) * (1 + w), with 1 + w formed in
 *                         float32 (a rounding point in parity mode).
 * Their backward, by the same autograd reading, has no intermediate
 * rounding: dn = dy * w' (w' = w or 1 + w), dx = r (dn - xhat mean_j(dn xhat)),
 * dw_j = sum_i dy xhat (d w'/d w = 1).
 *
 * Near-tie allowances (parity mode, 16-bit activations): where a value
 * reaches a bfloat16 or binary16 rounding point within NEAR_TIE_REL of a midpoint, an
 * implementation that computes it in float32 may round it to the other
 * neighbour.  The *_allow outputs give, per output, the largest change such
 * a flip can cause (zero where no rounding is near a tie).  dy*w is exact
 * in float32 when both are 16-bit (8 or 11 significant bits each), so it
 * is only flagged for a float32 weight.
 */

enum { ORC_RMS_CAST_FIRST = 0, ORC_RMS_WEIGHT_FIRST = 1, ORC_RMS_GEMMA = 2 };

/* The weight the variant multiplies by: w, or 1 + w (rounded to float32 in
 * parity mode, where eager forms it as a float32 sum). */
static double rms_weight(double w, int variant, int mode)
{
    if (variant != ORC_RMS_GEMMA) return w;
    return mode == ORC_PARITY ? (double)(float)(1.0 + w) : 1.0 + w;
}

static double rms_r(const void* x, int xt, int64_t i, int64_t N, double eps)
{
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        double v = widen(x, xt, i * N + j);
        s += v * v;
    }
    return 1.0 / sqrt(s / (double)N + eps);
}

int orc_rms_fwd_rows(const void* x, int xt, int64_t M, int64_t N, double eps,
                     const double* w, int mode, int variant, const int64_t* rows,
                     int64_t nrows, double* y, double* y_scale, double* rstd, double* y_allow)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        double rs = rms_r(x, xt, i, N, eps);
        if (rstd) rstd[r] = rs;
        for (int64_t j = 0; j < N; ++j) {
            double v = widen(x, xt, i * N + j) * rs;
            double wj = rms_weight(w[j], variant, mode);
            int tie = 0;
            if (mode == ORC_PARITY && variant == ORC_RMS_CAST_FIRST) v = round_to(v, xt, &tie);
            y[r * N + j] = wj * v;
            if (y_scale) y_scale[r * N + j] = fabs(wj * v);
            if (y_allow) y_allow[r * N + j] = tie ? fabs(wj) * spacing(v, xt) : 0.0;
        }
    }
    return 0;
}

int orc_rms_bwd_rows(const void* x, const void* dy, int xt, int wt, int64_t M, int64_t N,
                     double eps, const double* w, int mode, int variant, const int64_t* rows,
                     int64_t nrows, double* dx, double* dx_scale, double* dx_allow)
{
    (void)M;
    const int round_dn = mode == ORC_PARITY && variant == ORC_RMS_CAST_FIRST;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row_of(rows, r);
        double rs = rms_r(x, xt, i, N, eps);
        double s = 0.0, sa = 0.0, flip = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double xh = widen(x, xt, i * N + j) * rs;
            double dn = widen(dy, xt, i * N + j) * rms_weight(w[j], variant, mode);
            int tie = 0;
            if (round_dn) dn = round_to(dn, xt, &tie);
            if (tie && wt == ORC_F32) flip += spacing(dn, xt) * fabs(xh);
            s += dn * xh;
            sa += fabs(dn * xh);
        }
        double b = s / (double)N;
        double ba = sa / (double)N; /* error scale of b */
        flip /= (double)N; /* largest change of b from flipped dn roundings */
        for (int64_t j = 0; j < N; ++j) {
            double xh = widen(x, xt, i * N + j) * rs;
            double dn = widen(dy, xt, i * N + j) * rms_weight(w[j], variant, mode);
            int tie = 0;
            if (round_dn) dn = round_to(dn, xt, &tie);
            dx[r * N + j] = rs * (dn - xh * b);
            if (dx_scale) dx_scale[r * N + j] = fabs(rs) * (fabs(dn) + fabs(xh) * ba);
            if (dx_allow) {
                double own = (tie && wt == ORC_F32) ? spacing(dn, xt) : 0.0;
                dx_allow[r * N + j] = fabs(rs) * (own + fabs(xh) * flip);
            }
        }
    }
    return 0;
}

/* wt: dtype of the weight (ORC_F32, or a 16-bit code equal to xt); it
 * selects whether each dw term is rounded to the activation dtype before
 * the sum. */
int orc_rms_bwd_cols(const void* x, const void* dy, int xt, int wt, int64_t M, int64_t N,
                     double eps, int mode, int variant, double* dw, double* dw_ss,
                     double* dw_allow)
{
    const int cast_first = variant == ORC_RMS_CAST_FIRST;
    for (int64_t j = 0; j < N; ++j) {
        dw[j] = dw_ss[j] = 0.0;
        if (dw_allow) dw_allow[j] = 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        double rs = rms_r(x, xt, i, N, eps);
        for (int64_t j = 0; j < N; ++j) {
            double n = widen(x, xt, i * N + j) * rs;
            int tie = 0;
            if (mode == ORC_PARITY && cast_first) n = round_to(n, xt, &tie);
            double g = widen(dy, xt, i * N + j);
            double term = g * n;
            int round_term = (mode == ORC_PARITY && cast_first && wt != ORC_F32);
            if (round_term) term = round_to(term, xt, NULL);
            dw[j] += term;
            dw_ss[j] += term * term;
            if (dw_allow && tie)
                dw_allow[j] += fabs(g) * spacing(n, xt) + (round_term ? spacing(term, xt) : 0.0);
        }
    }
    return 0;
}
