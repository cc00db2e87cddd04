/*
 * Oracle for the fused, weight-quantized SwiGLU expansion
 *
 *     hidden = silu(x . Wg^T) * (x . Wu^T)
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct CPU
 * definition that the CUDA path is checked against.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product library
 * never links or calls it, and it shares no code, header, table or helper with
 * the CUDA sources.
 *
 * Sources (mlx-bun source-diff pages; cited by page title and section):
 *  - "mlx-bun 0.0.7 -> 0.0.9, page 42", file src/model/fused-swiglu-kernel.ts:
 *      header comment "PRECISION (two variants)" defines MATCH and F32;
 *      the SOURCE kernel body defines the operand tiles (dequantised weights are
 *      staged in the activation dtype before the block MMA), the gate/up tiles
 *      stored in the activation dtype out of the float accumulator, and the
 *      MATCH epilogue sigma -> silu -> product, each rounded to the activation dtype;
 *      fusedSwiglu() defines the shapes: x [M,H], packed W [I, H*bits/32],
 *      scales/biases [I, H/groupSize], hidden [M,I] in x's dtype.
 *  - same page, src/model/steel-linear-kernel.ts: y = x . W^T with the float
 *      accumulator cast to the activation dtype at the store.
 *  - "mlx-bun 0.0.7 -> 0.0.9, page 43", src/model/qwen3.ts, Qwen3MLP.forward:
 *      the unfused composition gate=qmm, up=qmm, sig=sigmoid(gate),
 *      silu=gate*sig, hidden=silu*up, each op producing a bf16 array.
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *  - codes are packed little-endian: code k of a row sits at bits
 *    (k mod pf)*bits of word k/pf, pf = 32/bits;
 *  - w = scale*q + bias, rounded ONCE to the activation dtype T (round to
 *    nearest, ties to even);
 *  - accumulation is exact-product / f64-sum (the float accumulator's order is
 *    free, so the oracle takes the most accurate one);
 *  - F32 keeps gate and up unrounded: hidden = T(g * u / (1 + exp(-g))).
 *
 * T is bf16 or f16 (fusedSwigluSupported() accepts both activation dtypes);
 * x, scales, biases and results share it.  Everything is computed in f64 with
 * explicit rounding to T at each point where the method rounds.  T values
 * travel as their raw uint16 bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_MATCH = 0, ORC_F32 = 1, ORC_DEBUG_GATE = 2, ORC_DEBUG_UP = 3 };

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 bit pattern -> exact double.  bf16 is the top half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round an integer-valued double to nearest, ties to even. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double frac = q - fl;               /* exact: q and fl share an exponent range */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/*
 * double -> bf16 with ONE rounding (nearest, ties to even), straight from the
 * exact double value (no detour through binary32, which would round twice).
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits, so a
 * normal number carries 8 significant bits; subnormals have spacing 2^-133.
 */
uint16_t orc_f64_to_bf16(double v)
{
    if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);

    int e2;                      /* a = m * 2^e2, m in [0.5, 1) */
    frexp(a, &e2);
    int e = e2 - 1;              /* 2^e <= a < 2^(e+1) */
    int ulp_exp = e - 7;         /* spacing of 8-significant-bit numbers at 2^e */
    if (ulp_exp < -133) ulp_exp = -133;   /* subnormal spacing */
    double q = ldexp(a, -ulp_exp);        /* exact: power-of-two scaling */
    double r = ldexp(round_half_even(q), ulp_exp);
    /* largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds past it is inf */
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;          /* exact: r has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | ((bits >> 16) & 0x7FFFu));
}

/* ---------------------------------------------------------------- f16 ----- */

/* IEEE binary16 bit pattern -> exact double: 1 sign bit, 5 exponent bits
 * (bias 15), 10 stored fraction bits; exponent field 0 holds the subnormals
 * (spacing 2^-24), 31 the infinities and NaNs. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1, ex = (h >> 10) & 0x1F, fr = h & 0x3FF;
    double a;
    if (ex == 0) a = ldexp((double)fr, -24);
    else if (ex == 31) a = fr ? NAN : INFINITY;
    else a = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -a : a;
}

/*
 * double -> binary16 with ONE rounding (nearest, ties to even) from the exact
 * double value.  A normal number carries 11 significant bits; below 2^-14 the
 * spacing is fixed at 2^-24.  Values that round to 2^16 or beyond are inf
 * (the largest finite binary16 is (2 - 2^-10) * 2^15 = 65504).
 */
uint16_t orc_f64_to_f16(double v)
{
    if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFE00u : 0x7E00u);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);

    int e2;
    frexp(a, &e2);
    int e = e2 - 1;              /* 2^e <= a < 2^(e+1) */
    int ulp_exp = e - 10;
    if (ulp_exp < -24) ulp_exp = -24;
    double r = ldexp(round_half_even(ldexp(a, -ulp_exp)), ulp_exp);
    if (r >= 65536.0) return (uint16_t)(sign | 0x7C00u);
    if (r < ldexp(1.0, -14))     /* subnormal (or the smallest normal, same encoding) */
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    frexp(r, &e2);
    e = e2 - 1;                  /* rounding may have carried into the next binade */
    int fr = (int)(ldexp(r, 10 - e) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)fr);
}

/* ------------------------------------------------------- activation dtype -- */

/* The activation dtype T of the pages' kernels: bf16 (ORC_BF16) or f16
 * (ORC_F16).  x, the scales and biases, the dequantised weights, the stored
 * projections and hidden are all T; every rounding point rounds to T. */
enum { ORC_BF16 = 0, ORC_F16 = 1 };

static double act_to_f64(uint16_t h, int dt) { return dt == ORC_F16 ? orc_f16_to_f64(h) : orc_bf16_to_f64(h); }
static uint16_t f64_to_act(double v, int dt) { return dt == ORC_F16 ? orc_f64_to_f16(v) : orc_f64_to_bf16(v); }

/* ------------------------------------------------------------ codes ------- */

/* Code k of a packed row: word k/pf, bit offset (k mod pf)*bits, LSB first. */
static unsigned code_at(const uint32_t *row_words, int64_t k, int bits)
{
    int64_t pf = 32 / bits;
    uint32_t word = row_words[k / pf];
    unsigned shift = (unsigned)((k % pf) * bits);
    return (word >> shift) & ((1u << bits) - 1u);
}

void orc_unpack(const uint32_t *words, int64_t n_codes, int bits, uint8_t *codes)
{
    for (int64_t k = 0; k < n_codes; ++k) codes[k] = (uint8_t)code_at(words, k, bits);
}

/*
 * Dequantise rows [0, rows) of a [rows, K] affine-quantised matrix into the
 * operand the block MMA consumes (dtype T, see above), returned as exact doubles:
 *     w[r,k] = T( scale[r, k/gs] * q[r,k] + bias[r, k/gs] ).
 * scale*q has at most 16 significant bits; the sum with the bias is exact in
 * double whenever the exponents of scale and bias differ by less than ~36,
 * which holds for every input the generators produce.
 */
void orc_dequant(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                 int64_t rows, int64_t K, int gs, int bits, int dt, double *out)
{
    int64_t words_per_row = K * bits / 32;
    int64_t groups_per_row = K / gs;
    for (int64_t r = 0; r < rows; ++r) {
        const uint32_t *wr = w + r * words_per_row;
        for (int64_t k = 0; k < K; ++k) {
            double sc = act_to_f64(s[r * groups_per_row + k / gs], dt);
            double bi = act_to_f64(b[r * groups_per_row + k / gs], dt);
            double q = (double)code_at(wr, k, bits);
            out[r * K + k] = act_to_f64(f64_to_act(sc * q + bi, dt), dt);
        }
    }
}

/* ----------------------------------------------------------- epilogues ---- */

static double ract(double v, int dt) { return act_to_f64(f64_to_act(v, dt), dt); }

/* MATCH: gate/up arrive as T (the stored projection); sigmoid, silu and the
 * product are each rounded to T, op for op with sigmoid -> mul -> mul. */
static double match_epilogue(double gb, double ub, int dt)
{
    double sig = ract(1.0 / (1.0 + exp(-gb)), dt);
    double silu = ract(gb * sig, dt);
    return ract(silu * ub, dt);
}

/* F32: no intermediate rounding; silu(g)*u = g*u/(1+exp(-g)) rounded once. */
static double f32_epilogue(double g, double u, int dt)
{
    return ract(g * u / (1.0 + exp(-g)), dt);
}

static uint16_t epilogue(int variant, double g, double u, int dt)
{
    switch (variant) {
    case ORC_MATCH:      return f64_to_act(match_epilogue(ract(g, dt), ract(u, dt), dt), dt);
    case ORC_F32:        return f64_to_act(f32_epilogue(g, u, dt), dt);
    case ORC_DEBUG_GATE: return f64_to_act(g, dt);
    case ORC_DEBUG_UP:   return f64_to_act(u, dt);
    default:             return dt == ORC_F16 ? 0x7E00u : 0x7FC0u;
    }
}

/* --------------------------------------------------------------- matmul --- */

static double dot_f64(const double *xr, const double *wr, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += xr[k] * wr[k];   /* products exact */
    return acc;
}

static double *act_rows_to_f64(const uint16_t *x, int64_t rows, int64_t K, int dt)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)(rows * K > 0 ? rows * K : 1));
    if (!xd) return NULL;
    for (int64_t i = 0; i < rows * K; ++i) xd[i] = act_to_f64(x[i], dt);
    return xd;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Full fused expansion for rows of x listed in `rows` (NULL = all M rows) and
 * all I outputs.  out is [n_rows, I] bf16.  g_acc/u_acc (optional, [n_rows, I])
 * receive the f64 projections before any rounding.  Returns 0, or -1 on
 * allocation failure.
 */
int orc_qswiglu_rows(const uint16_t *x, int64_t M, int64_t H, int64_t I,
                     const uint32_t *wg, const uint16_t *sg, const uint16_t *bg, int gs_g, int bits_g,
                     const uint32_t *wu, const uint16_t *su, const uint16_t *bu, int gs_u, int bits_u,
                     int variant, int dt, const int64_t *rows, int64_t n_rows,
                     uint16_t *out, double *g_acc, double *u_acc)
{
    if (rows == NULL) n_rows = M;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(n_rows * H > 0 ? n_rows * H : 1));
    if (!xd) return -1;
    for (int64_t j = 0; j < n_rows; ++j) {
        int64_t m = rows ? rows[j] : j;
        for (int64_t k = 0; k < H; ++k) xd[j * H + k] = act_to_f64(x[m * H + k], dt);
    }
    int64_t wpr_g = H * bits_g / 32, wpr_u = H * bits_u / 32;
    int64_t gpr_g = H / gs_g, gpr_u = H / gs_u;
    int failed = 0;
#pragma omp parallel
    {
        double *wgr = (double *)malloc(sizeof(double) * (size_t)H);
        double *wur = (double *)malloc(sizeof(double) * (size_t)H);
        if (!wgr || !wur) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t i = 0; i < I; ++i) {
                orc_dequant(wg + i * wpr_g, sg + i * gpr_g, bg + i * gpr_g, 1, H, gs_g, bits_g, dt, wgr);
                orc_dequant(wu + i * wpr_u, su + i * gpr_u, bu + i * gpr_u, 1, H, gs_u, bits_u, dt, wur);
                for (int64_t j = 0; j < n_rows; ++j) {
                    double g = dot_f64(xd + j * H, wgr, H);
                    double u = dot_f64(xd + j * H, wur, H);
                    out[j * I + i] = epilogue(variant, g, u, dt);
                    if (g_acc) g_acc[j * I + i] = g;
                    if (u_acc) u_acc[j * I + i] = u;
                }
            }
        }
        free(wgr);
        free(wur);
    }
    free(xd);
    return failed ? -1 : 0;
}

int orc_qswiglu(const uint16_t *x, int64_t M, int64_t H, int64_t I,
                const uint32_t *wg, const uint16_t *sg, const uint16_t *bg, int gs_g, int bits_g,
                const uint32_t *wu, const uint16_t *su, const uint16_t *bu, int gs_u, int bits_u,
                int variant, int dt, uint16_t *out)
{
    return orc_qswiglu_rows(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u,
                            variant, dt, NULL, M, out, NULL, NULL);
}

/*
 * Individual outputs hidden[m, i] for a list of (m, i) pairs (sampled checks at
 * sizes where the full product is too slow).  pairs is [n, 2] row-major.
 */
int orc_qswiglu_pairs(const uint16_t *x, int64_t M, int64_t H, int64_t I,
                      const uint32_t *wg, const uint16_t *sg, const uint16_t *bg, int gs_g, int bits_g,
                      const uint32_t *wu, const uint16_t *su, const uint16_t *bu, int gs_u, int bits_u,
                      int variant, int dt, const int64_t *pairs, int64_t n, uint16_t *out)
{
    (void)M; (void)I;
    int64_t wpr_g = H * bits_g / 32, wpr_u = H * bits_u / 32;
    int64_t gpr_g = H / gs_g, gpr_u = H / gs_u;
    int failed = 0;
#pragma omp parallel
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(3 * H));
        if (!buf) {
#pragma omp atomic write
            failed = 1;
        } else {
            double *xr = buf, *wgr = buf + H, *wur = buf + 2 * H;
#pragma omp for schedule(dynamic, 8)
            for (int64_t p = 0; p < n; ++p) {
                int64_t m = pairs[2 * p], i = pairs[2 * p + 1];
                for (int64_t k = 0; k < H; ++k) xr[k] = act_to_f64(x[m * H + k], dt);
                orc_dequant(wg + i * wpr_g, sg + i * gpr_g, bg + i * gpr_g, 1, H, gs_g, bits_g, dt, wgr);
                orc_dequant(wu + i * wpr_u, su + i * gpr_u, bu + i * gpr_u, 1, H, gs_u, bits_u, dt, wur);
                out[p] = epilogue(variant, dot_f64(xr, wgr, H), dot_f64(xr, wur, H), dt);
            }
        }
        free(buf);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------ unfused composition ----- */

/*
 * Quantised linear y = T(x . W^T + r): the float accumulator cast to the
 * activation dtype at the store.  x [M,K], W packed [N, K*bits/32], y [M,N];
 * r [M,N] (optional, NULL = 0) is a residual added before that one rounding,
 * as the whole-MLP kernel of fused-mlp-kernel.ts adds h to its accumulator.
 */
int orc_qmm(const uint16_t *x, int64_t M, int64_t K, int64_t N,
            const uint32_t *w, const uint16_t *s, const uint16_t *b, int gs, int bits, int dt,
            const uint16_t *r, uint16_t *y)
{
    double *xd = act_rows_to_f64(x, M, K, dt);
    if (!xd) return -1;
    int64_t wpr = K * bits / 32, gpr = K / gs;
    int failed = 0;
#pragma omp parallel
    {
        double *wr = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!wr) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t n = 0; n < N; ++n) {
                orc_dequant(w + n * wpr, s + n * gpr, b + n * gpr, 1, K, gs, bits, dt, wr);
                for (int64_t m = 0; m < M; ++m) {
                    double acc = dot_f64(xd + m * K, wr, K);
                    if (r) acc += act_to_f64(r[m * N + n], dt);
                    y[m * N + n] = f64_to_act(acc, dt);
                }
            }
        }
        free(wr);
    }
    free(xd);
    return failed ? -1 : 0;
}

/*
 * The whole MLP block (fused-mlp-kernel.ts, "the kernel outputs h + mlp(x)"):
 * hidden = the fused expansion of x in T (variant MATCH or F32), then
 * y = T(h + hidden . Wd^T) with the sum over I in f64 and one rounding.
 * hidden [M, I] and y [M, Ho] are outputs; h [M, Ho] may be NULL (no residual).
 */
int orc_mlp(const uint16_t *x, const uint16_t *h, int64_t M, int64_t H, int64_t I, int64_t Ho,
            const uint32_t *wg, const uint16_t *sg, const uint16_t *bg, int gs_g, int bits_g,
            const uint32_t *wu, const uint16_t *su, const uint16_t *bu, int gs_u, int bits_u,
            const uint32_t *wd, const uint16_t *sd, const uint16_t *bd, int gs_d, int bits_d,
            int variant, int dt, uint16_t *hidden, uint16_t *y)
{
    int rc = orc_qswiglu(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, dt, hidden);
    if (rc != 0) return rc;
    return orc_qmm(hidden, M, I, Ho, wd, sd, bd, gs_d, bits_d, dt, h, y);
}

/*
 * Elementwise silu(g)*u over T arrays, as the unfused path applies it to the
 * two stored projections.  MATCH rounds sigmoid, silu and the product to T;
 * F32 rounds once at the store.
 */
void orc_silu_mul(const uint16_t *g, const uint16_t *u, int64_t n, int variant, int dt, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double gv = act_to_f64(g[i], dt), uv = act_to_f64(u[i], dt);
        double h = (variant == ORC_F32) ? f32_epilogue(gv, uv, dt) : match_epilogue(gv, uv, dt);
        out[i] = f64_to_act(h, dt);
    }
}
