/*
 * rmsmod oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the fused adaLN
 * row operations compute.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library; the product
 * (librmsmod.so and its Python binding) never calls into it, and the two
 * share no source, header, table or helper.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (-ffp-contract=off is essential: GNU C contracts a*b+c into an FMA by
 * default, which would erase the separate roundings written below.)
 *
 * Notation used in the comments:
 *   R(v)  round an fp32 value to bf16, round-to-nearest-even (no FTZ)
 *   f(h)  the exact widening of a bf16 value to fp32
 *   every "+", "-", "*", "/" on float operands below is one IEEE fp32
 *   operation in round-to-nearest.
 *
 * Sources (web pages describing the method):
 *   [GLM]   sglang PR #34008 "GLM-Image bit-exact fused aten LayerNorm+modulate / qk-LN"
 *   [ERNIE] sglang PR #33854 "ERNIE-Image bit-exact fused RMSNorm+scale/shift"
 *   [FLUX]  sglang PR #34004 "FLUX.1 fused adaLN modulate (bit-exact) + RoPE cache hoist"
 *   [QWEN]  RL-Kernel PR #538 "[Qwen-Image][CUDA] Final AdaLN output (final_adaln_out)"
 *   [WAN]   sglang PR #38650 "Fuse the Wan VAE conv bias epilogue and tile the RMSNorm+SiLU kernel"
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes):
 *   - Row statistics are "fp32 statistics": the exact mean / biased variance /
 *     mean square of the bf16 row, rounded once to fp32.  They are accumulated
 *     here in double with Neumaier compensation, which equals the correctly
 *     rounded value except when the exact statistic lies within about 2^-50
 *     (relative) of an fp32 rounding midpoint.
 *   - rstd = 1 / sqrt(stat + eps) as three IEEE fp32 operations (add, sqrt,
 *     divide), all correctly rounded.
 *   - RMSNorm's "x * rstd * w" is evaluated left to right, one final rounding.
 *   - qk-LayerNorm's affine is "* w" then "+ b", two fp32 operations, one
 *     final rounding.
 *   - Wan RMSNorm is x * rsqrt(mean(x^2) + eps) * gamma, gamma applied before
 *     SiLU with no intermediate rounding; SiLU is evaluated in double on the
 *     fp32 pre-activation, rounded to fp32, then to bf16.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

typedef uint16_t bf16_t;

/* ---------------------------------------------------------------------- */
/* bf16 <-> fp32                                                           */
/* ---------------------------------------------------------------------- */

/* f(h): bf16 is the upper half of an fp32 bit pattern, so widening is exact. */
static float widen(bf16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float v;
    memcpy(&v, &u, sizeof v);
    return v;
}

/*
 * R(v): fp32 -> bf16, round to nearest, ties to even, by integer arithmetic
 * (the "bitcast round-to-nearest-even helper" of [ERNIE] §What
 * "rounding-faithful" means here, also used by [GLM] for its modulate chain).
 * Adding 0x7FFF plus the lowest kept bit and truncating rounds the 16
 * dropped bits to nearest with ties to even; a carry out of the mantissa
 * correctly bumps the exponent, and the largest finite values round to Inf.
 * Subnormals are rounded like any other value (no flush to zero).  NaN maps
 * to a quiet NaN with the input's sign.
 */
static bf16_t round_bf16(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (bf16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (bf16_t)(u >> 16);
}

ORACLE_API bf16_t oracle_round_bf16(float v) { return round_bf16(v); }

ORACLE_API float oracle_widen_bf16(bf16_t h) { return widen(h); }

/* Round every fp32 value of `in` (n of them). */
ORACLE_API void oracle_round_bf16_array(const float* in, bf16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = round_bf16(in[i]);
}

/* Round the fp32 values whose bit patterns are start, start+1, ..., start+count-1. */
ORACLE_API void oracle_round_bf16_sweep(uint32_t start, int64_t count, bf16_t* out)
{
    for (int64_t i = 0; i < count; ++i) {
        uint32_t u = start + (uint32_t)i;
        float v;
        memcpy(&v, &u, sizeof v);
        out[i] = round_bf16(v);
    }
}

/* ---------------------------------------------------------------------- */
/* Elementwise chains: each eager op is one fp32 op followed by R.         */
/* [FLUX] §Modifications, commit 2: matching the per-op rounding of the    */
/* eager chain is all that bit-exactness of an elementwise chain needs.    */
/* ---------------------------------------------------------------------- */

/* out = R(f(R(f(y) * f(R(1 + f(scale))))) + f(shift))
 * The three bf16 boundaries of norm(x) * (1 + scale) + shift: [GLM] §What
 * "rounding-faithful" means here (last bullet), [ERNIE] same section,
 * [FLUX] §Modifications commit 2. */
static bf16_t modulate_one(bf16_t y, bf16_t scale, bf16_t shift)
{
    bf16_t one_plus = round_bf16(1.0f + widen(scale));
    bf16_t t = round_bf16(widen(y) * widen(one_plus));
    return round_bf16(widen(t) + widen(shift));
}

/* The same chain with fp16 storage ([FLUX] §Accuracy Tests: the modulate
 * kernel's unit tests cover bf16 and fp16).  R16 is the C language's
 * fp32 -> _Float16 conversion (IEEE round-to-nearest-even, subnormals kept,
 * overflow to Inf); widening fp16 -> fp32 is exact. */
typedef uint16_t f16_t;

static f16_t round_f16(float v)
{
    _Float16 h = (_Float16)v;
    f16_t bits;
    memcpy(&bits, &h, sizeof bits);
    return bits;
}

static float widen_f16(f16_t bits)
{
    _Float16 h;
    memcpy(&h, &bits, sizeof h);
    return (float)h;
}

ORACLE_API f16_t oracle_round_f16(float v) { return round_f16(v); }

ORACLE_API float oracle_widen_f16(f16_t h) { return widen_f16(h); }

/* Round the fp32 values whose bit patterns are start, ..., start+count-1 to fp16. */
ORACLE_API void oracle_round_f16_sweep(uint32_t start, int64_t count, f16_t* out)
{
    for (int64_t i = 0; i < count; ++i) {
        uint32_t u = start + (uint32_t)i;
        float v;
        memcpy(&v, &u, sizeof v);
        out[i] = round_f16(v);
    }
}

/* out = R16(f(R16(f(y) * f(R16(1 + f(scale))))) + f(shift)) over [B, S, D]. */
ORACLE_API void oracle_modulate_f16(const f16_t* y, const f16_t* scale, const f16_t* shift,
                                    f16_t* out, int64_t B, int64_t S, int64_t D,
                                    int64_t mod_bstride)
{
    for (int64_t b = 0; b < B; ++b) {
        const f16_t* sc = scale + b * mod_bstride;
        const f16_t* sh = shift + b * mod_bstride;
        for (int64_t s = 0; s < S; ++s) {
            int64_t row = (b * S + s) * D;
            for (int64_t d = 0; d < D; ++d) {
                f16_t one_plus = round_f16(1.0f + widen_f16(sc[d]));
                f16_t t = round_f16(widen_f16(y[row + d]) * widen_f16(one_plus));
                out[row + d] = round_f16(widen_f16(t) + widen_f16(sh[d]));
            }
        }
    }
}

/* res = R(f(residual) + f(R(f(gate) * f(update))))
 * The eager pair round(gate*update), round(residual + ...): [ERNIE] §What
 * "rounding-faithful" means here (residual variant); [GLM] §Motivation (ff gate). */
static bf16_t gate_add_one(bf16_t residual, bf16_t gate, bf16_t update)
{
    bf16_t g = round_bf16(widen(gate) * widen(update));
    return round_bf16(widen(residual) + widen(g));
}

/* x + bias the way aten's add_ does it on a bf16 tensor: the fp32 bias is
 * first cast to bf16, then one fp32 add and one rounding.  [WAN] §New kernel,
 * lossless (conv_bias_epilogue: "x.dtype(float(x) + float(bias))", bias cast
 * to x.dtype first). */
static bf16_t bias_as_bf16(const void* bias, int bias_is_fp32, int64_t c)
{
    if (bias_is_fp32)
        return round_bf16(((const float*)bias)[c]);
    return ((const bf16_t*)bias)[c];
}

/* Standalone modulate over [B, S, D]; scale/shift row b lives at
 * base + b * mod_bstride elements (0 = one row shared by every batch). */
ORACLE_API void oracle_modulate(const bf16_t* y, const bf16_t* scale, const bf16_t* shift,
                                bf16_t* out, int64_t B, int64_t S, int64_t D,
                                int64_t mod_bstride)
{
    for (int64_t b = 0; b < B; ++b) {
        const bf16_t* sc = scale + b * mod_bstride;
        const bf16_t* sh = shift + b * mod_bstride;
        for (int64_t s = 0; s < S; ++s) {
            int64_t row = (b * S + s) * D;
            for (int64_t d = 0; d < D; ++d)
                out[row + d] = modulate_one(y[row + d], sc[d], sh[d]);
        }
    }
}

/* Standalone gated residual over [B, S, D]; gate row b at gate + b * gate_bstride. */
ORACLE_API void oracle_residual_gate_add(const bf16_t* residual, const bf16_t* gate,
                                         const bf16_t* update, bf16_t* res_out, int64_t B,
                                         int64_t S, int64_t D, int64_t gate_bstride)
{
    for (int64_t b = 0; b < B; ++b) {
        const bf16_t* g = gate + b * gate_bstride;
        for (int64_t s = 0; s < S; ++s) {
            int64_t row = (b * S + s) * D;
            for (int64_t d = 0; d < D; ++d)
                res_out[row + d] = gate_add_one(residual[row + d], g[d], update[row + d]);
        }
    }
}

/* Standalone conv-bias epilogue over `pixels` channels-last rows of C:
 * out = R(f(x) + f(b16)), and with a residual h: out = R(f(R(f(x) + f(b16))) + f(h)).
 * [WAN] §New kernel, lossless. */
ORACLE_API void oracle_conv_bias_epilogue(const bf16_t* x, const void* bias, int bias_is_fp32,
                                          const bf16_t* h, bf16_t* out, int64_t pixels,
                                          int64_t C)
{
    for (int64_t p = 0; p < pixels; ++p) {
        for (int64_t c = 0; c < C; ++c) {
            bf16_t v = round_bf16(widen(x[p * C + c]) + widen(bias_as_bf16(bias, bias_is_fp32, c)));
            if (h)
                v = round_bf16(widen(v) + widen(h[p * C + c]));
            out[p * C + c] = v;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Row statistics                                                          */
/* ---------------------------------------------------------------------- */

/* Neumaier-compensated running sum in double (the compensated sequential
 * sums of the CPU reference in [QWEN] §What). */
typedef struct {
    double s, c;
} csum_t;

static void csum_add(csum_t* a, double v)
{
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v))
        a->c += (a->s - t) + v;
    else
        a->c += (v - t) + a->s;
    a->s = t;
}

/* The compensated total; a non-finite running sum (Inf/NaN in the row) is
 * returned as is, so IEEE propagation matches a plain sum. */
static double csum_value(const csum_t* a)
{
    if (!isfinite(a->s))
        return a->s;
    return a->s + a->c;
}

/* LayerNorm statistics of one row of n bf16 values ([GLM] §What
 * "rounding-faithful" means here: mean and the biased variance sigma2 / N in
 * fp32).  mean_f = fp32(sum x / n); var_f = fp32(sum (x - mu)^2 / n) with mu
 * the double mean. */
static void ln_stats(const bf16_t* x, int64_t n, float* mean_f, float* var_f)
{
    csum_t s1 = {0.0, 0.0};
    for (int64_t i = 0; i < n; ++i)
        csum_add(&s1, (double)widen(x[i]));
    double mu = csum_value(&s1) / (double)n;

    csum_t s2 = {0.0, 0.0};
    for (int64_t i = 0; i < n; ++i) {
        double d = (double)widen(x[i]) - mu;
        csum_add(&s2, d * d);
    }
    *mean_f = (float)mu;
    *var_f = (float)(csum_value(&s2) / (double)n);
}

/* RMSNorm mean square fp32(sum x^2 / n) ([ERNIE] §What "rounding-faithful"
 * means here: rstd from sum_sq / H + eps). */
static float rms_stat(const bf16_t* x, int64_t n)
{
    csum_t s = {0.0, 0.0};
    for (int64_t i = 0; i < n; ++i) {
        double v = (double)widen(x[i]);
        csum_add(&s, v * v);
    }
    return (float)(csum_value(&s) / (double)n);
}

/* rstd = 1 / sqrt(stat + eps): fp32 add, correctly rounded sqrt, correctly
 * rounded divide. */
static float rstd_of(float stat, float eps)
{
    float t = stat + eps;
    float r = sqrtf(t);
    return 1.0f / r;
}

/* Exposed for the statistics pins: mean, biased variance and mean square of
 * each of `rows` rows of n bf16 values. */
ORACLE_API void oracle_row_stats(const bf16_t* x, int64_t rows, int64_t n, float* mean,
                                 float* var, float* meansq)
{
    for (int64_t r = 0; r < rows; ++r) {
        float m, v;
        ln_stats(x + r * n, n, &m, &v);
        if (mean)
            mean[r] = m;
        if (var)
            var[r] = v;
        if (meansq)
            meansq[r] = rms_stat(x + r * n, n);
    }
}

/* ---------------------------------------------------------------------- */
/* Normalisation steps (y before the modulate epilogue)                    */
/* ---------------------------------------------------------------------- */

/* LayerNorm without affine: y = R((f(x) - mean) * rstd), a subtract and a
 * multiply with no FMA ([GLM] §What "rounding-faithful" means here: the output
 * is cvt.rn.bf16 of FMUL(rstd, FADD(x, -mean))). */
ORACLE_API void oracle_ln_normalize(const bf16_t* x, bf16_t* y, int64_t rows, int64_t D,
                                    float eps, float* mean_out, float* rstd_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const bf16_t* xr = x + r * D;
        float mean, var;
        ln_stats(xr, D, &mean, &var);
        float rstd = rstd_of(var, eps);
        for (int64_t d = 0; d < D; ++d) {
            float centred = widen(xr[d]) - mean;
            y[r * D + d] = round_bf16(centred * rstd);
        }
        if (mean_out)
            mean_out[r] = mean;
        if (rstd_out)
            rstd_out[r] = rstd;
    }
}

/* RMSNorm with optional weight (NULL = 1): y = R((f(x) * rstd) * f(w)), one
 * final rounding ([ERNIE] §What "rounding-faithful" means here). */
ORACLE_API void oracle_rms_normalize(const bf16_t* x, const bf16_t* w, bf16_t* y, int64_t rows,
                                     int64_t D, float eps, float* rstd_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const bf16_t* xr = x + r * D;
        float rstd = rstd_of(rms_stat(xr, D), eps);
        for (int64_t d = 0; d < D; ++d) {
            float v = widen(xr[d]) * rstd;
            if (w)
                v = v * widen(w[d]);
            y[r * D + d] = round_bf16(v);
        }
        if (rstd_out)
            rstd_out[r] = rstd;
    }
}

/* ---------------------------------------------------------------------- */
/* The fused operations                                                     */
/* ---------------------------------------------------------------------- */

/* LayerNorm (no affine) + modulate over x [B, S, D]
 * ([GLM] §Motivation and §What "rounding-faithful" means here; [QWEN] §What). */
ORACLE_API void oracle_ln_modulate(const bf16_t* x, const bf16_t* scale, const bf16_t* shift,
                                   bf16_t* out, int64_t B, int64_t S, int64_t D,
                                   int64_t mod_bstride, float eps, float* mean_out,
                                   float* rstd_out)
{
    /* y is staged in `out` (same shape), then modulated in place. */
    oracle_ln_normalize(x, out, B * S, D, eps, mean_out, rstd_out);
    oracle_modulate(out, scale, shift, out, B, S, D, mod_bstride);
}

/* Single-rounding tier of LN + modulate ([FLUX] §Modifications commit 3,
 * quality="high"): the modulate folds into the LayerNorm's elementwise
 * affine, layer_norm(x, weight = R(1 + scale), bias = shift).  Only the
 * [1, D] row 1 + scale keeps its eager rounding; the normalised value is not
 * rounded before the affine, which runs in fp32 (a multiply, then an add, no
 * FMA), and the result is rounded once:
 *   w = R(1 + f(scale_b)),  out = R(((f(x) - mean) * rstd) * f(w) + f(shift_b)).
 * Rows of batch b use scale_b = scale + b * mod_bstride, as ln_modulate. */
ORACLE_API void oracle_ln_modulate_folded(const bf16_t* x, const bf16_t* scale,
                                          const bf16_t* shift, bf16_t* out, int64_t B,
                                          int64_t S, int64_t D, int64_t mod_bstride, float eps,
                                          float* mean_out, float* rstd_out)
{
    for (int64_t b = 0; b < B; ++b) {
        const bf16_t* sc = scale + b * mod_bstride;
        const bf16_t* sh = shift + b * mod_bstride;
        for (int64_t s = 0; s < S; ++s) {
            const int64_t r = b * S + s;
            const bf16_t* xr = x + r * D;
            float mean, var;
            ln_stats(xr, D, &mean, &var);
            float rstd = rstd_of(var, eps);
            for (int64_t d = 0; d < D; ++d) {
                float w = widen(round_bf16(1.0f + widen(sc[d])));
                float centred = widen(xr[d]) - mean;
                float normed = centred * rstd;
                float scaled = normed * w;
                out[r * D + d] = round_bf16(scaled + widen(sh[d]));
            }
            if (mean_out)
                mean_out[r] = mean;
            if (rstd_out)
                rstd_out[r] = rstd;
        }
    }
}

/* RMSNorm (optional weight) + modulate over x [B, S, D] ([ERNIE] first site). */
ORACLE_API void oracle_rmsnorm_modulate(const bf16_t* x, const bf16_t* weight,
                                        const bf16_t* scale, const bf16_t* shift, bf16_t* out,
                                        int64_t B, int64_t S, int64_t D, int64_t mod_bstride,
                                        float eps, float* rstd_out)
{
    oracle_rms_normalize(x, weight, out, B * S, D, eps, rstd_out);
    oracle_modulate(out, scale, shift, out, B, S, D, mod_bstride);
}

/* Gated residual + RMSNorm + modulate ([ERNIE] second site): the residual
 * stream res = R(residual + R(gate * update)) is returned in res_out and is
 * what the statistics are taken over. */
ORACLE_API void oracle_gated_rmsnorm_modulate(const bf16_t* residual, const bf16_t* update,
                                              const bf16_t* gate, int64_t gate_bstride,
                                              const bf16_t* weight, const bf16_t* scale,
                                              const bf16_t* shift, int64_t mod_bstride,
                                              bf16_t* res_out, bf16_t* out, int64_t B,
                                              int64_t S, int64_t D, float eps, float* rstd_out)
{
    oracle_residual_gate_add(residual, gate, update, res_out, B, S, D, gate_bstride);
    oracle_rms_normalize(res_out, weight, out, B * S, D, eps, rstd_out);
    oracle_modulate(out, scale, shift, out, B, S, D, mod_bstride);
}

/* Per-head LayerNorm with affine over rows of head_dim values, q rows and k
 * rows with their own (w, b) ([GLM] §Motivation, qk-norm nn.LayerNorm(128);
 * §What "rounding-faithful" means here, qk bullet).
 * z = R(((f(x) - mean) * rstd) * f(w) + f(b)). */
static void qk_rows(const bf16_t* x, const bf16_t* w, const bf16_t* b, bf16_t* out,
                    int64_t rows, int64_t hd, float eps, float* mean_out, float* rstd_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const bf16_t* xr = x + r * hd;
        float mean, var;
        ln_stats(xr, hd, &mean, &var);
        float rstd = rstd_of(var, eps);
        for (int64_t d = 0; d < hd; ++d) {
            float centred = widen(xr[d]) - mean;
            float normed = centred * rstd;
            float scaled = normed * widen(w[d]);
            out[r * hd + d] = round_bf16(scaled + widen(b[d]));
        }
        if (mean_out)
            mean_out[r] = mean;
        if (rstd_out)
            rstd_out[r] = rstd;
    }
}

/* mean_out / rstd_out (nullable) hold rows_q + rows_k values, q rows first. */
ORACLE_API void oracle_qk_layernorm(const bf16_t* q, const bf16_t* k, const bf16_t* wq,
                                    const bf16_t* bq, const bf16_t* wk, const bf16_t* bk,
                                    bf16_t* q_out, bf16_t* k_out, int64_t rows_q,
                                    int64_t rows_k, int64_t head_dim, float eps,
                                    float* mean_out, float* rstd_out)
{
    qk_rows(q, wq, bq, q_out, rows_q, head_dim, eps, mean_out, rstd_out);
    qk_rows(k, wk, bk, k_out, rows_k, head_dim, eps, mean_out ? mean_out + rows_q : NULL,
            rstd_out ? rstd_out + rows_q : NULL);
}

/* Channels-last RMSNorm + SiLU with the deferred conv bias folded in
 * ([WAN] §Quality-gated and §Modifications): per pixel row of C channels,
 *   xb = R(f(x) + f(b16))            (bias applied first, aten add_ arithmetic)
 *   rstd = 1 / sqrt(fp32(mean(xb^2)) + eps)
 *   z = (f(xb) * rstd) * f(gamma)    (fp32, not rounded)
 *   out = R(fp32(z / (1 + exp(-z))))  (SiLU evaluated in double)
 * bias may be NULL (no fold). */
ORACLE_API void oracle_rmsnorm_silu_cl(const bf16_t* x, const void* bias, int bias_is_fp32,
                                       const bf16_t* gamma, bf16_t* out, int64_t pixels,
                                       int64_t C, float eps, float* rstd_out)
{
    bf16_t* xb = out; /* the biased row is staged in the output row */
    for (int64_t p = 0; p < pixels; ++p) {
        const bf16_t* xr = x + p * C;
        bf16_t* orow = out + p * C;
        for (int64_t c = 0; c < C; ++c)
            xb[p * C + c] =
                bias ? round_bf16(widen(xr[c]) + widen(bias_as_bf16(bias, bias_is_fp32, c))) : xr[c];
        float rstd = rstd_of(rms_stat(orow, C), eps);
        for (int64_t c = 0; c < C; ++c) {
            float z = (widen(orow[c]) * rstd) * widen(gamma[c]);
            double zd = (double)z;
            double silu = zd / (1.0 + exp(-zd));
            orow[c] = round_bf16((float)silu);
        }
        if (rstd_out)
            rstd_out[p] = rstd;
    }
}

/* ---------------------------------------------------------------------- */
/* Backward of LayerNorm (no affine) + modulate ([QWEN] §What: forward and */
/* backward of out = LayerNorm(x) * (1 + scale) + shift; d_scale and      */
/* d_shift are token sums reduced by fixed 32-way balanced trees in fp32,  */
/* applied recursively until one value remains, so the result depends     */
/* only on the sequence length, not on the batch or the position in it).  */
/* ---------------------------------------------------------------------- */

/* One 32-way balanced tree: the complete binary tree over 32 slots of fp32
 * adds, slot i holding v[i] for i < n and +0 beyond. */
static float tree32(const float* v, int n)
{
    float level[32];
    for (int i = 0; i < 32; ++i)
        level[i] = i < n ? v[i] : 0.0f;
    for (int width = 32; width > 1; width /= 2)
        for (int i = 0; i < width / 2; ++i)
            level[i] = level[2 * i] + level[2 * i + 1];
    return level[0];
}

/* The token sum of n values v[0], v[stride], ...: while more than one value
 * remains, replace each run of 32 consecutive values (the last run may be
 * shorter) by its 32-way tree.  scratch holds n floats. */
static float token_tree_sum(const float* v, int64_t n, int64_t stride, float* scratch)
{
    if (n <= 0)
        return 0.0f;
    for (int64_t i = 0; i < n; ++i)
        scratch[i] = v[i * stride];
    while (n > 1) {
        int64_t m = (n + 31) / 32;
        for (int64_t j = 0; j < m; ++j) {
            int64_t len = n - 32 * j < 32 ? n - 32 * j : 32;
            scratch[j] = tree32(scratch + 32 * j, (int)len);
        }
        n = m;
    }
    return scratch[0];
}

ORACLE_API float oracle_token_tree_sum(const float* v, int64_t n, float* scratch)
{
    return token_tree_sum(v, n, 1, scratch);
}

/* Gradients of out = R(R(y * s1) + shift), y = R(yhat), yhat = (f(x) - mean) * rstd,
 * s1 = R(1 + f(scale_b)), with the roundings passed straight through:
 *   dyhat[d]   = f(g[d]) * f(s1[d])                       (exact in fp32)
 *   c1         = fp32(sum_d dyhat / D),  c2 = fp32(sum_d dyhat * yhat / D)
 *                (exact sums in double, rounded once)
 *   grad_x[d]  = R(rstd * ((dyhat - c1) - yhat * c2))     (fp32 ops, no FMA)
 *   grad_shift[b, d] = T_s(f(g[b, s, d]))
 *   grad_scale[b, d] = T_s(f(g[b, s, d]) * f(y[b, s, d])) (the products are exact)
 * with T_s the token tree sum over the S rows of batch b.  mean / rstd are
 * the forward's per-row statistics.  Any output may be NULL; c1_out / c2_out
 * (nullable, [B*S]) expose the row reductions for the pins. */
ORACLE_API void oracle_ln_modulate_backward(const bf16_t* x, const bf16_t* scale,
                                            const bf16_t* grad_out, const float* mean,
                                            const float* rstd, int64_t B, int64_t S,
                                            int64_t D, int64_t mod_bstride, bf16_t* grad_x,
                                            float* grad_scale, float* grad_shift,
                                            float* c1_out, float* c2_out, float* work)
{
    /* work: 2 * S floats (the token values of one column) + S floats scratch */
    float* colg = work;
    float* colgy = work + S;
    float* scratch = work + 2 * S;
    for (int64_t b = 0; b < B; ++b) {
        const bf16_t* sc = scale + b * mod_bstride;
        for (int64_t s = 0; s < S; ++s) {
            const int64_t r = b * S + s;
            const bf16_t* xr = x + r * D;
            const bf16_t* gr = grad_out + r * D;
            csum_t a1 = {0.0, 0.0}, a2 = {0.0, 0.0};
            for (int64_t d = 0; d < D; ++d) {
                float s1 = widen(round_bf16(1.0f + widen(sc[d])));
                float yhat = (widen(xr[d]) - mean[r]) * rstd[r];
                float dy = widen(gr[d]) * s1;
                csum_add(&a1, (double)dy);
                csum_add(&a2, (double)dy * (double)yhat);
            }
            float c1 = (float)(csum_value(&a1) / (double)D);
            float c2 = (float)(csum_value(&a2) / (double)D);
            if (c1_out)
                c1_out[r] = c1;
            if (c2_out)
                c2_out[r] = c2;
            if (grad_x) {
                for (int64_t d = 0; d < D; ++d) {
                    float s1 = widen(round_bf16(1.0f + widen(sc[d])));
                    float yhat = (widen(xr[d]) - mean[r]) * rstd[r];
                    float dy = widen(gr[d]) * s1;
                    float t = (dy - c1) - yhat * c2;
                    grad_x[r * D + d] = round_bf16(rstd[r] * t);
                }
            }
        }
        for (int64_t d = 0; d < D; ++d) {
            for (int64_t s = 0; s < S; ++s) {
                const int64_t r = b * S + s;
                float g = widen(grad_out[r * D + d]);
                float y = widen(round_bf16((widen(x[r * D + d]) - mean[r]) * rstd[r]));
                colg[s] = g;
                colgy[s] = g * y;
            }
            if (grad_shift)
                grad_shift[b * D + d] = token_tree_sum(colg, S, 1, scratch);
            if (grad_scale)
                grad_scale[b * D + d] = token_tree_sum(colgy, S, 1, scratch);
        }
    }
}
