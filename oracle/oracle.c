/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the row-wise
 * reduce-then-normalize path (LayerNorm, RMSNorm, residual-add + RMSNorm,
 * BatchNorm2d training forward, inference forward and training backward,
 * row softmax).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or table with the
 * CUDA sources.
 *
 * Rules followed here:
 *   - every statistic and every output is computed in IEEE double;
 *   - each output is rounded exactly once, to its storage type, with
 *     round-to-nearest-even (helpers below, written from the IEEE-754
 *     definition of a binary format with subnormals and overflow to inf);
 *   - the only place the path itself fixes a lower precision is the residual
 *     add of the fused pre-norm path: an fp32 add, then rounding to the I/O
 *     type (CUDA fused RMSNorm kernel page, diycv.top, section 3.2);
 *   - no blocking, fusion or reordering beyond the formulas: loops go over
 *     rows (or channels) and then over elements, in index order.
 *
 * Storage types (dtype codes): 0 = binary32, 1 = binary16, 2 = bfloat16.
 * Half-width types are passed as raw uint16 bit patterns.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (ISO mode, no
 * contraction, so every double operation is rounded as written).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the fp32 residual add needs FLT_EVAL_METHOD == 0 (float ops rounded to float)"
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };
enum { ORC_OK = 0, ORC_BAD_ARGS = -1 };

/* ------------------------------------------------------------------------ */
/* IEEE-754 helpers                                                          */
/* ------------------------------------------------------------------------ */

/* Value of a binary16 bit pattern: 1 sign, 5 exponent (bias 15), 10 fraction. */
double orc_f16_bits_to_double(uint16_t h)
{
    const int s = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f + 1024), e - 25);  /* (1 + f/2^10) * 2^(e-15) */
    return s ? -mag : mag;
}

/* Value of a bfloat16 bit pattern: 1 sign, 8 exponent (bias 127), 7 fraction. */
double orc_bf16_bits_to_double(uint16_t b)
{
    const int s = b >> 15, e = (b >> 7) & 0xff, f = b & 0x7f;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);             /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f + 128), e - 134);  /* (1 + f/2^7) * 2^(e-127) */
    return s ? -mag : mag;
}

/*
 * Round a double to the nearest value of a binary format with `ebits`
 * exponent bits and `mbits` fraction bits (ties to even), and encode it.
 * Subnormals are kept; magnitudes that round past the largest finite value
 * become infinity; NaN becomes the quiet NaN with the input's sign.
 */
static uint16_t orc_encode(double v, int ebits, int mbits)
{
    const int bias = (1 << (ebits - 1)) - 1;
    const unsigned all_ones = (1u << ebits) - 1u;
    const unsigned sign = signbit(v) ? (1u << (ebits + mbits)) : 0u;
    if (isnan(v))
        return (uint16_t)(sign | (all_ones << mbits) | (1u << (mbits - 1)));
    const double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | (all_ones << mbits));
    if (a == 0.0)
        return (uint16_t)sign;

    int e2;
    (void)frexp(a, &e2);           /* a lies in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                /* unbiased exponent of a */
    const int emin = 1 - bias;     /* exponent of the smallest normal */
    if (E < emin)
        E = emin;                  /* subnormal range: the quantum stops shrinking */
    const int q = E - mbits;       /* weight 2^q of the last kept bit */

    const double s = ldexp(a, -q); /* a / 2^q, exact */
    double n = floor(s);
    const double r = s - n;        /* exact */
    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) == 1.0))
        n += 1.0;                  /* round half to even */

    unsigned N = (unsigned)n;      /* rounded value is N * 2^q, N <= 2^(mbits+1) */
    if (N >= (1u << (mbits + 1))) {
        N >>= 1;                   /* carry out of the significand */
        E += 1;
    }
    unsigned biased, frac;
    if (N >= (1u << mbits)) {      /* normal */
        biased = (unsigned)(E + bias);
        frac = N - (1u << mbits);
    } else {                       /* subnormal (E == emin) */
        biased = 0;
        frac = N;
    }
    if (biased >= all_ones)        /* overflow */
        return (uint16_t)(sign | (all_ones << mbits));
    return (uint16_t)(sign | (biased << mbits) | frac);
}

uint16_t orc_double_to_f16_bits(double v) { return orc_encode(v, 5, 10); }
uint16_t orc_double_to_bf16_bits(double v) { return orc_encode(v, 8, 7); }

/* binary32: the C conversion is IEEE round-to-nearest-even (default mode). */
float orc_double_to_f32(double v) { return (float)v; }

static double orc_get(int dt, const void *p, int64_t i)
{
    switch (dt) {
    case ORC_F32:  return (double)((const float *)p)[i];
    case ORC_F16:  return orc_f16_bits_to_double(((const uint16_t *)p)[i]);
    default:       return orc_bf16_bits_to_double(((const uint16_t *)p)[i]);
    }
}

/* The one rounding of an output to its storage type. */
static void orc_put(int dt, void *p, int64_t i, double v)
{
    switch (dt) {
    case ORC_F32:  ((float *)p)[i] = orc_double_to_f32(v); break;
    case ORC_F16:  ((uint16_t *)p)[i] = orc_double_to_f16_bits(v); break;
    default:       ((uint16_t *)p)[i] = orc_double_to_bf16_bits(v); break;
    }
}

static int orc_dtype_ok(int dt) { return dt == ORC_F32 || dt == ORC_F16 || dt == ORC_BF16; }

/* Compensated (Neumaier) running sum in double. */
typedef struct { double s, c; } orc_sum;

static void orc_sum_add(orc_sum *a, double x)
{
    const double t = a->s + x;
    if (fabs(a->s) >= fabs(x))
        a->c += (a->s - t) + x;
    else
        a->c += (x - t) + a->s;
    a->s = t;
}

static double orc_sum_get(const orc_sum *a) { return a->s + a->c; }

/* ------------------------------------------------------------------------ */
/* LayerNorm                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * LayerNorm over each row of a row-major [rows, N] tensor.
 *   mean = (1/N) sum_i x_i
 *   var  = (1/N) sum_i (x_i - mean)^2        (biased; a true second pass)
 *   y_i  = (x_i - mean) / sqrt(var + eps) * gamma_i + beta_i
 * Follows the definition in the CUDA handbook LayerNorm walkthrough
 * (lpnh.cn/news/2756757), section 1; gamma/beta are optional as in its
 * section 2 apply kernel (absent gamma = 1, absent beta = 0).
 * eps arrives as a binary32 and is widened exactly.
 * Outputs: y (storage type, may be NULL), y_wide (double, may be NULL),
 * mean and rstd = 1/sqrt(var+eps) per row (double, may be NULL).
 */
int orc_layernorm(int dt, const void *x, const void *gamma, const void *beta,
                  void *y, double *y_wide, double *mean_out, double *rstd_out,
                  int64_t rows, int64_t N, float eps)
{
    if (!orc_dtype_ok(dt) || !x || rows < 0 || N < 1)
        return ORC_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t base = r * N;
        orc_sum s = {0.0, 0.0};
        for (int64_t i = 0; i < N; ++i)
            orc_sum_add(&s, orc_get(dt, x, base + i));
        const double mean = orc_sum_get(&s) / (double)N;

        orc_sum q = {0.0, 0.0};
        for (int64_t i = 0; i < N; ++i) {
            const double d = orc_get(dt, x, base + i) - mean;
            orc_sum_add(&q, d * d);
        }
        const double var = orc_sum_get(&q) / (double)N;
        const double rstd = 1.0 / sqrt(var + (double)eps);

        for (int64_t i = 0; i < N; ++i) {
            const double g = gamma ? orc_get(dt, gamma, i) : 1.0;
            const double b = beta ? orc_get(dt, beta, i) : 0.0;
            const double out = (orc_get(dt, x, base + i) - mean) * rstd * g + b;
            if (y)
                orc_put(dt, y, base + i, out);
            if (y_wide)
                y_wide[base + i] = out;
        }
        if (mean_out)
            mean_out[r] = mean;
        if (rstd_out)
            rstd_out[r] = rstd;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm and residual-add + RMSNorm                                        */
/* ------------------------------------------------------------------------ */

/*
 * RMSNorm over each row:  y_i = x_i / sqrt((1/N) sum_j x_j^2 + eps) * w_i.
 * Formula of the CUDA fused RMSNorm kernel page (diycv.top), sections 0.3
 * and 2 (normalize, then scale by the weight); absent w = 1.
 * rstd_out receives 1/sqrt(mean(x^2)+eps) per row (may be NULL).
 */
int orc_rmsnorm(int dt, const void *x, const void *w, void *y, double *y_wide,
                double *rstd_out, int64_t rows, int64_t N, float eps)
{
    if (!orc_dtype_ok(dt) || !x || rows < 0 || N < 1)
        return ORC_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t base = r * N;
        orc_sum s = {0.0, 0.0};
        for (int64_t i = 0; i < N; ++i) {
            const double v = orc_get(dt, x, base + i);
            orc_sum_add(&s, v * v);
        }
        const double ms = orc_sum_get(&s) / (double)N;
        const double rstd = 1.0 / sqrt(ms + (double)eps);
        for (int64_t i = 0; i < N; ++i) {
            const double wi = w ? orc_get(dt, w, i) : 1.0;
            const double out = orc_get(dt, x, base + i) * rstd * wi;
            if (y)
                orc_put(dt, y, base + i, out);
            if (y_wide)
                y_wide[base + i] = out;
        }
        if (rstd_out)
            rstd_out[r] = rstd;
    }
    return ORC_OK;
}

/*
 * Fused pre-norm path (CUDA fused RMSNorm kernel page, diycv.top, sections
 * 0.3, 2 and 3.2):
 *   residual_out_i = round_to_storage( fp32(x_i) + fp32(residual_i) )
 *   y = RMSNorm(residual_out, w)
 * The add is done in binary32 and rounded to the storage type first; the
 * statistics then use that rounded value, the one written to the residual
 * stream.  residual_out is required.
 */
int orc_add_rmsnorm(int dt, const void *x, const void *residual, const void *w,
                    void *residual_out, void *y, double *y_wide, double *rstd_out,
                    int64_t rows, int64_t N, float eps)
{
    if (!orc_dtype_ok(dt) || !x || !residual || !residual_out || rows < 0 || N < 1)
        return ORC_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t base = r * N;
        orc_sum s = {0.0, 0.0};
        for (int64_t i = 0; i < N; ++i) {
            const float a = (float)orc_get(dt, x, base + i);        /* exact */
            const float b = (float)orc_get(dt, residual, base + i); /* exact */
            const float sum = a + b;                                /* binary32 add */
            orc_put(dt, residual_out, base + i, (double)sum);
            const double v = orc_get(dt, residual_out, base + i);
            orc_sum_add(&s, v * v);
        }
        const double ms = orc_sum_get(&s) / (double)N;
        const double rstd = 1.0 / sqrt(ms + (double)eps);
        for (int64_t i = 0; i < N; ++i) {
            const double wi = w ? orc_get(dt, w, i) : 1.0;
            const double out = orc_get(dt, residual_out, base + i) * rstd * wi;
            if (y)
                orc_put(dt, y, base + i, out);
            if (y_wide)
                y_wide[base + i] = out;
        }
        if (rstd_out)
            rstd_out[r] = rstd;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* BatchNorm2d training forward (NCHW)                                       */
/* ------------------------------------------------------------------------ */

/*
 * Training-mode BatchNorm over an NCHW tensor x[batch][C][HW]: element
 * (n, c, k) sits at ((n*C + c)*HW + k).  Per channel c, over all n and k:
 *   mean_c = (1/cnt) sum x,  var_c = (1/cnt) sum (x - mean_c)^2  (biased),
 *   cnt = batch*HW,
 *   y = (x - mean_c) / sqrt(var_c + eps) * gamma_c + beta_c.
 * save_mean[c] = mean_c, save_rstd[c] = 1/sqrt(var_c + eps).
 * Running statistics (updated in place when the pointers are non-NULL):
 *   running_mean = (1 - m) * running_mean + m * mean_c
 *   running_var  = (1 - m) * running_var  + m * var_c * cnt / (cnt - 1)
 * Forward definition and running-mean rule: BatchNorm CUDA implementation
 * walkthrough (jianying88.com/news/30214), sections 2.1 and 2.4.  That page
 * does not print the running-variance rule; the unbiased form above is the
 * convention of the torch.nn.BatchNorm2d operator the page replaces.
 * gamma/beta are optional (absent = 1 / 0).  Requires cnt > 1.
 */
int orc_batchnorm_train(int dt, const void *x, const void *gamma, const void *beta,
                        void *y, double *y_wide, double *save_mean, double *save_rstd,
                        double *running_mean, double *running_var,
                        int64_t batch, int64_t C, int64_t HW, float eps, float momentum)
{
    if (!orc_dtype_ok(dt) || !x || batch < 0 || C < 1 || HW < 1)
        return ORC_BAD_ARGS;
    const int64_t cnt = batch * HW;
    if (cnt < 2)
        return ORC_BAD_ARGS;
    const double m = (double)momentum;
    for (int64_t c = 0; c < C; ++c) {
        orc_sum s = {0.0, 0.0};
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k)
                orc_sum_add(&s, orc_get(dt, x, (n * C + c) * HW + k));
        const double mean = orc_sum_get(&s) / (double)cnt;

        orc_sum q = {0.0, 0.0};
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k) {
                const double d = orc_get(dt, x, (n * C + c) * HW + k) - mean;
                orc_sum_add(&q, d * d);
            }
        const double var = orc_sum_get(&q) / (double)cnt;
        const double rstd = 1.0 / sqrt(var + (double)eps);

        const double g = gamma ? orc_get(dt, gamma, c) : 1.0;
        const double b = beta ? orc_get(dt, beta, c) : 0.0;
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k) {
                const int64_t i = (n * C + c) * HW + k;
                const double out = (orc_get(dt, x, i) - mean) * rstd * g + b;
                if (y)
                    orc_put(dt, y, i, out);
                if (y_wide)
                    y_wide[i] = out;
            }
        if (save_mean)
            save_mean[c] = mean;
        if (save_rstd)
            save_rstd[c] = rstd;
        if (running_mean)
            running_mean[c] = (1.0 - m) * running_mean[c] + m * mean;
        if (running_var)
            running_var[c] = (1.0 - m) * running_var[c]
                             + m * var * (double)cnt / (double)(cnt - 1);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* BatchNorm2d inference forward (BatchNorm CUDA implementation walkthrough, */
/* jianying88.com/news/30214, section 2.4: inference normalizes with the     */
/* running statistics kept during training instead of the batch's):        */
/*   y = (x - running_mean_c) / sqrt(running_var_c + eps) * gamma_c + beta_c */
/* NCHW: x[n][c][k] at (n*C + c)*HW + k.  running_* are binary32 inputs.    */
/* ------------------------------------------------------------------------ */
int orc_batchnorm_infer(int dt, const void *x, const void *gamma, const void *beta,
                        void *y, double *y_wide, const float *running_mean,
                        const float *running_var, int64_t batch, int64_t C, int64_t HW,
                        float eps)
{
    if (!orc_dtype_ok(dt) || !x || !running_mean || !running_var || batch < 0 || C < 1
        || HW < 1)
        return ORC_BAD_ARGS;
    for (int64_t c = 0; c < C; ++c) {
        const double mean = (double)running_mean[c];
        const double rstd = 1.0 / sqrt((double)running_var[c] + (double)eps);
        const double g = gamma ? orc_get(dt, gamma, c) : 1.0;
        const double b = beta ? orc_get(dt, beta, c) : 0.0;
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k) {
                const int64_t i = (n * C + c) * HW + k;
                const double out = (orc_get(dt, x, i) - mean) * rstd * g + b;
                if (y)
                    orc_put(dt, y, i, out);
                if (y_wide)
                    y_wide[i] = out;
            }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* BatchNorm2d training backward (BatchNorm CUDA implementation walkthrough, */
/* section 3.1).  With xhat = (x - mean_c) * rstd_c over the channel's       */
/* count = batch*HW elements:                                               */
/*   dbeta_c  = sum dy                                                       */
/*   dgamma_c = sum dy * xhat                                                */
/*   dx       = gamma_c * rstd_c * (dy - dbeta_c/count - xhat * dgamma_c/count) */
/* mean_c and rstd_c are the statistics the training forward saved; they    */
/* are inputs here (xhat is recomputed from x, not stored).  The section's  */
/* first statement of dx leaves out the factor gamma_c; its restatement in  */
/* terms of the two sums has it, and only that form is the derivative of    */
/* y = xhat * gamma + beta, so that form is the one followed.               */
/* dgamma/dbeta may be NULL (not written); gamma NULL means 1.              */
/* ------------------------------------------------------------------------ */
int orc_batchnorm_backward(int dt, const void *dy, const void *x, const void *gamma,
                           const double *mean, const double *rstd, void *dx,
                           double *dx_wide, double *dgamma, double *dbeta,
                           int64_t batch, int64_t C, int64_t HW)
{
    if (!orc_dtype_ok(dt) || !dy || !x || !mean || !rstd || batch < 1 || C < 1 || HW < 1)
        return ORC_BAD_ARGS;
    const double cnt = (double)(batch * HW);
    for (int64_t c = 0; c < C; ++c) {
        orc_sum s1 = {0.0, 0.0}, s2 = {0.0, 0.0};
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k) {
                const int64_t i = (n * C + c) * HW + k;
                const double g_out = orc_get(dt, dy, i);
                const double xhat = (orc_get(dt, x, i) - mean[c]) * rstd[c];
                orc_sum_add(&s1, g_out);
                orc_sum_add(&s2, g_out * xhat);
            }
        const double db = orc_sum_get(&s1), dg = orc_sum_get(&s2);
        const double g = gamma ? orc_get(dt, gamma, c) : 1.0;
        for (int64_t n = 0; n < batch; ++n)
            for (int64_t k = 0; k < HW; ++k) {
                const int64_t i = (n * C + c) * HW + k;
                const double xhat = (orc_get(dt, x, i) - mean[c]) * rstd[c];
                const double out =
                    g * rstd[c] * (orc_get(dt, dy, i) - db / cnt - xhat * dg / cnt);
                if (dx)
                    orc_put(dt, dx, i, out);
                if (dx_wide)
                    dx_wide[i] = out;
            }
        if (dgamma)
            dgamma[c] = dg;
        if (dbeta)
            dbeta[c] = db;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Row softmax (LLM-ops page, smarter.xin, section 1, "Softmax"):           */
/*   m = max_j x_j,  d = sum_j exp(x_j - m),  y_i = exp(x_i - m) / d        */
/* The online single-pass form on that page reaches the same m and d; this  */
/* is the plain definition.  row_max/row_sum (m and d) may be NULL.         */
/* ------------------------------------------------------------------------ */
int orc_softmax(int dt, const void *x, void *y, double *y_wide, double *row_max,
                double *row_sum, int64_t rows, int64_t N)
{
    if (!orc_dtype_ok(dt) || !x || rows < 0 || N < 1)
        return ORC_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            const double v = orc_get(dt, x, r * N + j);
            if (v > m)
                m = v;
        }
        orc_sum s = {0.0, 0.0};
        for (int64_t j = 0; j < N; ++j)
            orc_sum_add(&s, exp(orc_get(dt, x, r * N + j) - m));
        const double d = orc_sum_get(&s);
        for (int64_t j = 0; j < N; ++j) {
            const double out = exp(orc_get(dt, x, r * N + j) - m) / d;
            if (y)
                orc_put(dt, y, r * N + j, out);
            if (y_wide)
                y_wide[r * N + j] = out;
        }
        if (row_max)
            row_max[r] = m;
        if (row_sum)
            row_sum[r] = d;
    }
    return ORC_OK;
}
