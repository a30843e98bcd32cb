/*
 * gsa_oracle.c -- plain, slow CPU oracle for the grouped scaled activation
 * fused with block-scaled (MXFP8 / NVFP4) quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path; the two meet only through
 * the seeded input generator.
 *
 * Sources (the web pages this method is described on):
 *   [P1] "[PyTorch] Enable fused activation recompute for ScaledTanhSReLU"
 *        (NVIDIA/TransformerEngine PR #3473), Description and the
 *        regeneration-error table; the "bounding the activation at s**2"
 *        remark in the review thread.
 *   [P2] "Activation + GroupedLinear Fusion for MOE" (PR #3238),
 *        Greptile Summary (fused per-row scale x activation x grouped
 *        quantization; SwiGLU, clamped SwiGLU, SReLU; backward returns
 *        (grouped_dy, dense_dy, grad_scales)), sequence diagram.
 *   [P3] "[PyTorch] Preserve FP8 recompute state for inner autocast"
 *        (PR #3284), the E4M3 cast+descale error table.
 * The pages print no formulas.  Where they are silent the oracle takes the
 * plainest reading; each reading is labelled R1..R17 where it is used.
 *
 * Arithmetic: scalar IEEE binary32, round-to-nearest-even, compiled with
 * -ffp-contract=off so that no multiply-add is fused.  Format encoders are
 * written from the format definitions as nearest-value searches over the
 * table of representable magnitudes (ties to the even code).
 *
 * GeLU, sigmoid and identity (R16) are the further unary activations the
 * review thread of [P1] names as fitting the same fused kernel.
 * Parity unpinned (conventions the pages do not fix): R2 (GLU half order),
 * R3 (clamped-SwiGLU form and constants), R5 (dprobs summation order),
 * R9 (per-expert tensor scale), R11 (RHT sign convention and op order).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ACT_SRELU = 0, ACT_TANH_SRELU = 1, ACT_SWIGLU = 2, ACT_CLAMPED_SWIGLU = 3,
       ACT_GELU = 4, ACT_SIGMOID = 5, ACT_IDENTITY = 6 };

/* act_params layout shared with the Python wrapper: {s, limit, alpha, offset} */
typedef struct { float s, limit, alpha, off; } act_params;

/* ------------------------------------------------------------------ BF16 */

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round binary32 to bfloat16, nearest-even (NaN is out of contract, R13). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------- format tables */

/* OCP FP8 E4M3 (FN): 4 exponent bits (bias 7), 3 mantissa bits, no inf,
 * magnitude code 0x7F is NaN.  Magnitude codes 0..126, 126 = 448. */
static double e4m3_mag(int code)
{
    int e = (code >> 3) & 15, m = code & 7;
    if (e == 0) return ldexp((double)m / 8.0, -6);
    return ldexp(1.0 + (double)m / 8.0, e - 7);
}

/* FP4 E2M1: 2 exponent bits (bias 1), 1 mantissa bit, magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6} for codes 0..7. */
static double e2m1_mag(int code)
{
    int e = (code >> 1) & 3, m = code & 1;
    if (e == 0) return (double)m * 0.5;
    return ldexp(1.0 + (double)m / 2.0, e - 1);
}

static double g_e4m3[127];
static double g_e2m1[8];
static int g_tables_ready = 0;

static void tables_init(void)
{
    if (g_tables_ready) return;
    for (int c = 0; c < 127; ++c) g_e4m3[c] = e4m3_mag(c);
    for (int c = 0; c < 8; ++c) g_e2m1[c] = e2m1_mag(c);
    g_tables_ready = 1;
}

/* Nearest representable magnitude, ties to the even code, saturating at
 * the largest finite magnitude.  vals[] ascending, vals[0] == 0.  Adjacent
 * codes differ in the mantissa LSB, so "even code" is round-half-even. */
static int nearest_code(double a, const double *vals, int n)
{
    if (a >= vals[n - 1]) return n - 1;
    int lo = 0, hi = n - 1; /* invariant: vals[lo] <= a < vals[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (vals[mid] <= a) lo = mid; else hi = mid;
    }
    double dlo = a - vals[lo], dhi = vals[hi] - a;
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

/* E4M3, round-to-nearest-even, saturating to +-448 (satfinite). */
uint8_t oracle_e4m3_encode(float v)
{
    tables_init();
    int neg = signbit(v) ? 1 : 0;
    int c = nearest_code(fabs((double)v), g_e4m3, 127);
    return (uint8_t)((neg << 7) | c);
}

float oracle_e4m3_decode(uint8_t code)
{
    if ((code & 0x7F) == 0x7F) return NAN;
    double m = e4m3_mag(code & 0x7F);
    return (float)((code & 0x80) ? -m : m);
}

/* E2M1, round-to-nearest-even, saturating to +-6. Returns a 4-bit code. */
uint8_t oracle_e2m1_encode(float v)
{
    tables_init();
    int neg = signbit(v) ? 1 : 0;
    int c = nearest_code(fabs((double)v), g_e2m1, 8);
    return (uint8_t)((neg << 3) | c);
}

float oracle_e2m1_decode(uint8_t code)
{
    double m = e2m1_mag(code & 7);
    return (float)((code & 8) ? -m : m);
}

/* ------------------------------------------------- MXFP8 block (R7) */

/* Smallest integer e in [-127, 127] with amax <= 448 * 2^e (exact compare).
 * amax == 0 gives -127.  The E8M0 scale code is e + 127. */
int oracle_mx_scale_exp(float amax)
{
    for (int e = -127; e < 127; ++e)
        if ((double)amax <= 448.0 * ldexp(1.0, e)) return e;
    return 127;
}

/* Quantize n values (n <= 32) as one MXFP8 block. */
void oracle_mxfp8_block(const float *v, int n, uint8_t *codes, uint8_t *scale_code)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));
    int e = oracle_mx_scale_exp(amax);
    *scale_code = (uint8_t)(e + 127);
    float s = ldexpf(1.0f, -e);
    for (int i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(v[i] * s);
}

/* --------------------------------------------------- NVFP4 (R8, R9) */

/* Per-expert encode scale S_enc = (448 * 6) / amax, 1 for amax == 0,
 * capped at FLT_MAX. */
float oracle_nvfp4_tensor_scale(float amax)
{
    if (amax == 0.0f) return 1.0f;
    float s = 2688.0f / amax;
    if (!(s <= FLT_MAX)) s = FLT_MAX;
    return s;
}

/* Quantize n values (n <= 16) as one NVFP4 block under S_enc.
 * codes[] receives one 4-bit code per value (unpacked). */
void oracle_nvfp4_block(const float *v, int n, float S_enc, uint8_t *codes, uint8_t *scale_code)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float t = amax / 6.0f;
    uint8_t sb = oracle_e4m3_encode(t * S_enc);
    float sbf = oracle_e4m3_decode(sb);
    float r = (sbf == 0.0f) ? 0.0f : S_enc / sbf;
    /* The quotient overflows when S_enc / E4M3(sb) exceeds FLT_MAX (an expert
     * amax below about 2^-116); like S_enc it is capped at FLT_MAX (reading
     * R17), so that every product v * r is finite (0 * inf has no value). */
    if (r > FLT_MAX) r = FLT_MAX;
    *scale_code = sb;
    for (int i = 0; i < n; ++i) codes[i] = oracle_e2m1_encode(v[i] * r);
}

/* ------------------------------------------------------------ RHT (R11) */

/* w = (1/4) * H16 * diag(d) * v, d_i = -1 where bit i of mask is set,
 * H16 the Sylvester Hadamard matrix; evaluated as: sign flips, four
 * butterfly stages (stride 1, 2, 4, 8), then the exact 1/4 scale. */
void oracle_rht16(const float *v, uint16_t mask, float *w)
{
    float x[16];
    for (int i = 0; i < 16; ++i) x[i] = ((mask >> i) & 1u) ? -v[i] : v[i];
    for (int h = 1; h < 16; h <<= 1) {
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            float a = x[i], b = x[i + h];
            x[i] = a + b;
            x[i + h] = a - b;
        }
    }
    for (int i = 0; i < 16; ++i) w[i] = x[i] * 0.25f;
}

/* ------------------------------------------------------ activations */

/* 1/sqrt(2) and 1/sqrt(2 pi), rounded to binary32 from their decimal expansions. */
#define O_RSQRT2 0.70710678118654752440f
#define O_RSQRT2PI 0.39894228040143267794f

/* Forward activation value (FP32).  For the GLU forms a is the gate half
 * X[:, j] and b the linear half X[:, H + j] (R2). */
float oracle_act(int act, float a, float b, const act_params *P)
{
    switch (act) {
    case ACT_SRELU: {
        float r = (a > 0.0f) ? a : 0.0f;
        return r * r;
    }
    case ACT_TANH_SRELU: { /* s^2 * tanh^2(relu(x)/s), bounded by s^2 (R1) */
        float r = (a > 0.0f) ? a : 0.0f;
        float u = r / P->s;
        float t = tanhf(u);
        return (P->s * P->s) * (t * t);
    }
    case ACT_SWIGLU: {
        float sg = 1.0f / (1.0f + expf(-a));
        float si = a * sg;
        return si * b;
    }
    case ACT_CLAMPED_SWIGLU: { /* R3 */
        float L = P->limit;
        float ac = fminf(a, L);
        float bc = fminf(fmaxf(b, -L), L);
        float sg = 1.0f / (1.0f + expf(-(P->alpha * ac)));
        float gl = ac * sg;
        return gl * (bc + P->off);
    }
    case ACT_GELU: { /* x * Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2 (R16) */
        float c = erfcf(-(a * O_RSQRT2));
        return (0.5f * a) * c;
    }
    case ACT_SIGMOID:
        return 1.0f / (1.0f + expf(-a));
    case ACT_IDENTITY:
        return a;
    }
    return NAN;
}

/* Activation value and its partial derivatives (FP32). */
void oracle_act_grad(int act, float a, float b, const act_params *P,
                     float *val, float *da, float *db)
{
    *db = 0.0f;
    switch (act) {
    case ACT_SRELU: {
        float r = (a > 0.0f) ? a : 0.0f;
        *val = r * r;
        *da = (a > 0.0f) ? r + r : 0.0f;
        return;
    }
    case ACT_TANH_SRELU: {
        float r = (a > 0.0f) ? a : 0.0f;
        float u = r / P->s;
        float t = tanhf(u);
        float tt = t * t;
        *val = (P->s * P->s) * tt;
        *da = (a > 0.0f) ? ((2.0f * P->s) * t) * (1.0f - tt) : 0.0f;
        return;
    }
    case ACT_SWIGLU: {
        float sg = 1.0f / (1.0f + expf(-a));
        float si = a * sg;
        *val = si * b;
        *da = b * (sg + si * (1.0f - sg));
        *db = si;
        return;
    }
    case ACT_CLAMPED_SWIGLU: {
        float L = P->limit;
        float ac = fminf(a, L);
        float bc = fminf(fmaxf(b, -L), L);
        float z = P->alpha * ac;
        float sg = 1.0f / (1.0f + expf(-z));
        float gl = ac * sg;
        float lin = bc + P->off;
        *val = gl * lin;
        *da = (a <= L) ? lin * (sg + (z * sg) * (1.0f - sg)) : 0.0f;
        *db = (b >= -L && b <= L) ? gl : 0.0f;
        return;
    }
    case ACT_GELU: { /* d/dx x Phi(x) = Phi(x) + x phi(x), phi(x) = exp(-x^2/2) / sqrt(2 pi) */
        float c = erfcf(-(a * O_RSQRT2));
        *val = (0.5f * a) * c;
        float phi = expf(-((0.5f * a) * a)) * O_RSQRT2PI;
        *da = 0.5f * c + a * phi;
        return;
    }
    case ACT_SIGMOID: { /* s' = s (1 - s) */
        float sg = 1.0f / (1.0f + expf(-a));
        *val = sg;
        *da = sg * (1.0f - sg);
        return;
    }
    case ACT_IDENTITY:
        *val = a;
        *da = 1.0f;
        return;
    }
    *val = *da = NAN;
}

static int is_glu(int act) { return act == ACT_SWIGLU || act == ACT_CLAMPED_SWIGLU; }

/* Y = p * act(X) for nrows rows, rounded to BF16.  x: [nrows, W_in] bf16,
 * y: [nrows, W] bf16 with W = W_in (unary) or W_in / 2 (GLU). */
void oracle_act_fwd_rows(const uint16_t *x, const float *p, int64_t nrows, int64_t W_in,
                         int act, const float *prm, uint16_t *y)
{
    const act_params *P = (const act_params *)prm;
    int64_t W = is_glu(act) ? W_in / 2 : W_in;
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *xr = x + r * W_in;
        for (int64_t j = 0; j < W; ++j) {
            float a = oracle_bf16_to_f32(xr[j]);
            float b = is_glu(act) ? oracle_bf16_to_f32(xr[W + j]) : 0.0f;
            float v = oracle_act(act, a, b, P);
            y[r * W + j] = oracle_f32_to_bf16(v * p[r]);
        }
    }
}

/* Y = p * act(X) from the FP32 FC1 accumulator itself (no BF16 round trip of
 * X), rounded to BF16: the forward that the ScaledTanhSReLU recompute page
 * contrasts with the regeneration from the saved BF16 copy (its suggested
 * test comment: the forward applies the activation to its FP32 accumulator,
 * the backward to the saved BF16 FC1 output).  x: [nrows, W_in] float. */
void oracle_act_fwd_rows_f32(const float *x, const float *p, int64_t nrows, int64_t W_in,
                             int act, const float *prm, uint16_t *y)
{
    const act_params *P = (const act_params *)prm;
    int64_t W = is_glu(act) ? W_in / 2 : W_in;
    for (int64_t r = 0; r < nrows; ++r) {
        const float *xr = x + r * W_in;
        for (int64_t j = 0; j < W; ++j) {
            float a = xr[j];
            float b = is_glu(act) ? xr[W + j] : 0.0f;
            float v = oracle_act(act, a, b, P);
            y[r * W + j] = oracle_f32_to_bf16(v * p[r]);
        }
    }
}

/* dprobs reduction order (R5): serial left-to-right sums of consecutive
 * 32-term blocks starting from 0, then a pairwise tree over the block sums:
 * each level adds neighbours (2j, 2j+1); an unpaired last node moves up. */
float oracle_dprobs_sum(const float *t, int64_t n)
{
    int64_t nb = (n + 31) / 32;
    if (nb == 0) return 0.0f;
    float *s = (float *)malloc(sizeof(float) * (size_t)nb);
    for (int64_t b = 0; b < nb; ++b) {
        float acc = 0.0f;
        for (int64_t k = b * 32; k < n && k < b * 32 + 32; ++k) acc = acc + t[k];
        s[b] = acc;
    }
    int64_t m = nb;
    while (m > 1) {
        int64_t half = m / 2;
        for (int64_t j = 0; j < half; ++j) s[j] = s[2 * j] + s[2 * j + 1];
        if (m & 1) s[half] = s[m - 1];
        m = half + (m & 1);
    }
    float out = s[0];
    free(s);
    return out;
}

/* Backward for nrows rows: g = dY * p; dX = bf16(g * act'(X)) (GLU: both
 * halves); dprobs[r] = sum_j dY[r, j] * act(X)[r, j] with FP32, unscaled,
 * unrounded act (R4) in the R5 order.  dx / dprobs may be NULL. */
void oracle_act_bwd_rows(const uint16_t *dy, const uint16_t *x, const float *p, int64_t nrows,
                         int64_t W_in, int act, const float *prm, uint16_t *dx, float *dprobs)
{
    const act_params *P = (const act_params *)prm;
    int glu = is_glu(act);
    int64_t W = glu ? W_in / 2 : W_in;
    float *terms = (float *)malloc(sizeof(float) * (size_t)(W > 0 ? W : 1));
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *xr = x + r * W_in;
        const uint16_t *dyr = dy + r * W;
        for (int64_t j = 0; j < W; ++j) {
            float a = oracle_bf16_to_f32(xr[j]);
            float b = glu ? oracle_bf16_to_f32(xr[W + j]) : 0.0f;
            float val, da, db;
            oracle_act_grad(act, a, b, P, &val, &da, &db);
            float d = oracle_bf16_to_f32(dyr[j]);
            float g = d * p[r];
            if (dx) {
                dx[r * W_in + j] = oracle_f32_to_bf16(g * da);
                if (glu) dx[r * W_in + W + j] = oracle_f32_to_bf16(g * db);
            }
            terms[j] = d * val;
        }
        if (dprobs) dprobs[r] = oracle_dprobs_sum(terms, W);
    }
    free(terms);
}

/* ------------------------------------------------- rowwise quantization */

/* MXFP8 rowwise: v [nrows, W] bf16 -> data [nrows, W] E4M3,
 * scale [nrows, ceil(W/32)] E8M0. */
void oracle_mxfp8_rows(const uint16_t *v, int64_t nrows, int64_t W, uint8_t *data, uint8_t *scale)
{
    int64_t nb = (W + 31) / 32;
    float buf[32];
    uint8_t codes[32];
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int n = (int)((W - b * 32) < 32 ? (W - b * 32) : 32);
            for (int i = 0; i < n; ++i) buf[i] = oracle_bf16_to_f32(v[r * W + b * 32 + i]);
            oracle_mxfp8_block(buf, n, codes, &scale[r * nb + b]);
            memcpy(&data[r * W + b * 32], codes, (size_t)n);
        }
    }
}

/* NVFP4 rowwise under one S_enc: data [nrows, W/2] (value 2k in the low
 * nibble, 2k+1 in the high nibble), scale [nrows, W/16] E4M3. W % 16 == 0. */
void oracle_nvfp4_rows(const uint16_t *v, int64_t nrows, int64_t W, float S_enc,
                       uint8_t *data, uint8_t *scale)
{
    int64_t nb = W / 16;
    float buf[16];
    uint8_t codes[16];
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 16; ++i) buf[i] = oracle_bf16_to_f32(v[r * W + b * 16 + i]);
            oracle_nvfp4_block(buf, 16, S_enc, codes, &scale[r * nb + b]);
            for (int i = 0; i < 8; ++i)
                data[r * (W / 2) + b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    }
}

/* max |v| over a bf16 array (NVFP4 rowwise tensor amax of one expert). */
float oracle_amax_bf16(const uint16_t *v, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) m = fmaxf(m, fabsf(oracle_bf16_to_f32(v[i])));
    return m;
}

/* ---------------------------------------------- columnwise quantization */

/* Gather the 'blk'-row chunk i of column j of one expert's [Me, W] values,
 * zero-padded past row Me (R10). */
static void gather_col(const uint16_t *v, int64_t Me, int64_t W, int64_t j, int64_t i,
                       int blk, float *out)
{
    for (int k = 0; k < blk; ++k) {
        int64_t row = i * blk + k;
        out[k] = (row < Me) ? oracle_bf16_to_f32(v[row * W + j]) : 0.0f;
    }
}

/* MXFP8 columnwise copy of one expert: the rowwise quantization of the
 * zero-padded transpose.  data [W, Mp] E4M3, scale [W, Mp/32], Mp =
 * ceil(Me/32)*32; padding rows are stored (as code 0). */
void oracle_mxfp8_cols(const uint16_t *v, int64_t Me, int64_t W, uint8_t *data, uint8_t *scale)
{
    int64_t nblk = (Me + 31) / 32, Mp = nblk * 32;
    float buf[32];
    for (int64_t j = 0; j < W; ++j)
        for (int64_t i = 0; i < nblk; ++i) {
            gather_col(v, Me, W, j, i, 32, buf);
            oracle_mxfp8_block(buf, 32, &data[j * Mp + i * 32], &scale[j * nblk + i]);
        }
}

/* NVFP4 columnwise chunk values: the gathered 16-chunk, through the RHT
 * when rht != 0. */
static void nvfp4_col_chunk(const uint16_t *v, int64_t Me, int64_t W, int64_t j, int64_t i,
                            int rht, uint16_t mask, float *out)
{
    float g[16];
    gather_col(v, Me, W, j, i, 16, g);
    if (rht) oracle_rht16(g, mask, out);
    else memcpy(out, g, sizeof g);
}

/* Columnwise tensor amax of one expert: max |chunk value| over every
 * (optionally transformed) 16-chunk of the zero-padded transpose. */
float oracle_amax_cols(const uint16_t *v, int64_t Me, int64_t W, int rht, uint16_t mask)
{
    int64_t nblk = (Me + 15) / 16;
    float w[16], m = 0.0f;
    for (int64_t j = 0; j < W; ++j)
        for (int64_t i = 0; i < nblk; ++i) {
            nvfp4_col_chunk(v, Me, W, j, i, rht, mask, w);
            for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(w[k]));
        }
    return m;
}

/* NVFP4 columnwise copy of one expert: data [W, Mp/2], scale [W, Mp/16],
 * Mp = ceil(Me/16)*16. */
void oracle_nvfp4_cols(const uint16_t *v, int64_t Me, int64_t W, int rht, uint16_t mask,
                       float S_enc, uint8_t *data, uint8_t *scale)
{
    int64_t nblk = (Me + 15) / 16, Mp = nblk * 16;
    float w[16];
    uint8_t codes[16];
    for (int64_t j = 0; j < W; ++j)
        for (int64_t i = 0; i < nblk; ++i) {
            nvfp4_col_chunk(v, Me, W, j, i, rht, mask, w);
            oracle_nvfp4_block(w, 16, S_enc, codes, &scale[j * nblk + i]);
            for (int k = 0; k < 8; ++k)
                data[j * (Mp / 2) + i * 8 + k] = (uint8_t)(codes[2 * k] | (codes[2 * k + 1] << 4));
        }
}

/* ---------------------------------------------- bulk encoders (for pins) */

void oracle_e4m3_encode_n(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e2m1_encode_n(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_f32_to_bf16_n(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(v[i]);
}

void oracle_act_grad_n(int act, const float *a, const float *b, int64_t n, const float *prm,
                       float *val, float *da, float *db)
{
    for (int64_t i = 0; i < n; ++i)
        oracle_act_grad(act, a[i], b ? b[i] : 0.0f, (const act_params *)prm, &val[i], &da[i], &db[i]);
}
