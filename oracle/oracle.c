/*
 * CPU oracle for the memory-bound decoder-layer fusions -- TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Every value is carried in double. The steps follow the source pages' order:
 *   residual add -> mean of squares -> add epsilon -> reciprocal square root -> multiply by the
 *   weight [P1, "Fusing operations, measured"]; silu(gate) * up over the stacked projection [P1];
 *   quantisation of the activation to FP8 E4M3 with a per-tensor or per-token scale [P2 Part V, P5 s.3].
 * Readings where the pages are silent:
 *   - the norm is taken of the bf16-rounded sum, which is what the unfused model normalises;
 *   - the product w * s * inv and silu(g) * up are not rounded before they are quantised or written;
 *   - the quantised value is the unrounded product divided by the fp32 scale;
 *   - magnitudes above 448 saturate to 448; an all-zero row has scale 0 and codes 0.
 * Build: plain C11 with -ffp-contract=off so that x86 and Arm hosts give identical bits.
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 */

double orc_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

uint16_t orc_bf16_round(double v) {
    /* bf16 has 8 significant bits and the fp32 exponent range: the spacing of representable values
     * in [2^(e-1), 2^e) is 2^(e-8), and never below 2^-133 (the subnormal spacing). */
    if (isnan(v)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;
    if (q < -133) q = -133;
    double units = ldexp(a, -q);         /* exact: a scaling by a power of two */
    double rounded = nearbyint(units);   /* default rounding mode: nearest, ties to even */
    double res = ldexp(rounded, q);
    const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (res > max_bf16) return (uint16_t)(sign | 0x7F80);
    float f = (float)res; /* exact: res lies on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* ---------------------------------------------------------------- FP8 E4M3 */

/* magnitude of the non-negative code c in [0, 126]: exponent field E = c >> 3, mantissa M = c & 7;
 * E == 0 is subnormal (M / 8 * 2^-6), otherwise (1 + M / 8) * 2^(E - 7). */
static double e4m3_magnitude(int c) {
    int E = c >> 3, M = c & 7;
    if (E == 0) return (double)M / 512.0;
    return (double)(8 + M) * (double)(1u << E) / 1024.0; /* exact: small integers and powers of two */
}

double orc_e4m3_decode(uint8_t code) {
    int c = code & 0x7F;
    if (c == 0x7F) return NAN;
    double m = e4m3_magnitude(c);
    return (code & 0x80) ? -m : m;
}

uint8_t orc_e4m3_encode(double v) {
    if (isnan(v)) return (uint8_t)0x7F;
    uint8_t sign = signbit(v) ? (uint8_t)0x80 : (uint8_t)0;
    double a = fabs(v);
    int best = 126;
    if (a < 448.0) {
        double best_d = INFINITY;
        for (int c = 0; c <= 126; ++c) {
            double d = fabs(a - e4m3_magnitude(c));
            if (d < best_d || (d == best_d && (c & 1) == 0)) {
                best = c;
                best_d = d;
            }
        }
    }
    return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------- E2M1 (NVFP4 element) */

/* magnitude of code c in [0, 7]: exponent field E = c >> 1, mantissa M = c & 1; E == 0 is subnormal
 * (M / 2), otherwise (1 + M / 2) * 2^(E - 1). */
static double e2m1_magnitude(int c) {
    int E = c >> 1, M = c & 1;
    if (E == 0) return 0.5 * (double)M;
    return (1.0 + 0.5 * (double)M) * (double)(1 << (E - 1));
}

double orc_e2m1_decode(uint8_t code) {
    double m = e2m1_magnitude(code & 7);
    return (code & 8) ? -m : m;
}

uint8_t orc_e2m1_encode(double v) {
    if (isnan(v)) return 7;   /* no NaN in E2M1; not generated */
    uint8_t sign = signbit(v) ? (uint8_t)8 : (uint8_t)0;
    double a = fabs(v);
    int best = 7;
    if (a < 6.0) {
        double best_d = INFINITY;
        for (int c = 0; c <= 7; ++c) {
            double d = fabs(a - e2m1_magnitude(c));
            if (d < best_d || (d == best_d && (c & 1) == 0)) {
                best = c;
                best_d = d;
            }
        }
    }
    return (uint8_t)(sign | best);
}

/* NVFP4 of one row of exact values: block scales sf[n/16], codes packed two per byte. */
static void nvfp4_row(const double* v, int64_t n, float S, uint8_t* q, uint8_t* sf) {
    for (int64_t b = 0; b < n / 16; ++b) {
        double amax = 0.0;
        for (int j = 0; j < 16; ++j) {
            double a = fabs(v[b * 16 + j]);
            if (a > amax) amax = a;
        }
        uint8_t code = orc_e4m3_encode(amax / (6.0 * (double)S));
        sf[b] = code;
        double scale = orc_e4m3_decode(code) * (double)S;
        for (int j = 0; j < 16; j += 2) {
            uint8_t lo = scale == 0.0 ? (uint8_t)0 : orc_e2m1_encode(v[b * 16 + j] / scale);
            uint8_t hi = scale == 0.0 ? (uint8_t)0 : orc_e2m1_encode(v[b * 16 + j + 1] / scale);
            q[(b * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* ---------------------------------------------------------------- SiLU */

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* ---------------------------------------------------------------- add + RMSNorm */

/* One row: writes the residual and returns inv = 1 / sqrt(mean(s^2) + eps). */
static double add_and_inv_rms(const uint16_t* x, const uint16_t* r, int64_t H, float eps,
                              uint16_t* residual_out) {
    double sum_sq = 0.0;
    for (int64_t j = 0; j < H; ++j) {
        uint16_t s = orc_bf16_round(orc_bf16_to_double(x[j]) + orc_bf16_to_double(r[j]));
        residual_out[j] = s;
        double sd = orc_bf16_to_double(s);
        sum_sq += sd * sd;
    }
    double mean_sq = sum_sq / (double)H;
    return 1.0 / sqrt(mean_sq + (double)eps);
}

static double normed(const uint16_t* residual_row, const uint16_t* w, int64_t j, double inv) {
    return orc_bf16_to_double(w[j]) * orc_bf16_to_double(residual_row[j]) * inv;
}

int orc_add_rmsnorm(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T, int64_t H,
                    float eps, uint16_t* residual_out, double* v_out, uint16_t* out) {
    if (T < 0 || H <= 0) return -1;
    if (T > 0 && (!x || !r || !w || !residual_out)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* xr = x + t * H;
        const uint16_t* rr = r + t * H;
        uint16_t* sr = residual_out + t * H;
        double inv = add_and_inv_rms(xr, rr, H, eps, sr);
        for (int64_t j = 0; j < H; ++j) {
            double v = normed(sr, w, j, inv);
            if (v_out) v_out[t * H + j] = v;
            if (out) out[t * H + j] = orc_bf16_round(v);
        }
    }
    return 0;
}

/* quantise one row of exact values with the given fp32 scale (0 gives code 0). */
static void quantise_row(const double* v, int64_t n, float scale, uint8_t* q) {
    for (int64_t j = 0; j < n; ++j) q[j] = scale == 0.0f ? (uint8_t)0 : orc_e4m3_encode(v[j] / (double)scale);
}

static float dynamic_scale(const double* v, int64_t n) {
    double amax = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double a = fabs(v[j]);
        if (a > amax) amax = a;
    }
    return (float)(amax / 448.0);
}

int orc_add_rmsnorm_quant_fp8(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T,
                              int64_t H, float eps, int mode, float* scale, uint16_t* residual_out,
                              uint8_t* q_out, double* v_out) {
    if (T < 0 || H <= 0 || (mode != 0 && mode != 1)) return -1;
    if (T > 0 && (!x || !r || !w || !scale || !residual_out || !q_out)) return -1;
    double* row = (double*)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
    if (T > 0 && !row) return -1;
    for (int64_t t = 0; t < T; ++t) {
        uint16_t* sr = residual_out + t * H;
        double inv = add_and_inv_rms(x + t * H, r + t * H, H, eps, sr);
        for (int64_t j = 0; j < H; ++j) row[j] = normed(sr, w, j, inv);
        float sc = mode == 0 ? scale[0] : dynamic_scale(row, H);
        if (mode == 1) scale[t] = sc;
        quantise_row(row, H, sc, q_out + t * H);
        if (v_out) memcpy(v_out + t * H, row, (size_t)H * sizeof(double));
    }
    free(row);
    return 0;
}

int orc_add_rmsnorm_quant_nvfp4(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T, int64_t H,
                                float eps, float tensor_scale, uint16_t* residual_out, uint8_t* q_out,
                                uint8_t* sf_out, double* v_out) {
    if (T < 0 || H <= 0 || H % 16 != 0 || !(tensor_scale > 0.0f) || isinf(tensor_scale)) return -1;
    if (T > 0 && (!x || !r || !w || !residual_out || !q_out || !sf_out)) return -1;
    double* row = (double*)malloc((size_t)H * sizeof(double));
    if (!row) return -1;
    for (int64_t t = 0; t < T; ++t) {
        uint16_t* sr = residual_out + t * H;
        double inv = add_and_inv_rms(x + t * H, r + t * H, H, eps, sr);
        for (int64_t j = 0; j < H; ++j) row[j] = normed(sr, w, j, inv);
        nvfp4_row(row, H, tensor_scale, q_out + t * (H / 2), sf_out + t * (H / 16));
        if (v_out) memcpy(v_out + t * H, row, (size_t)H * sizeof(double));
    }
    free(row);
    return 0;
}

/* ---------------------------------------------------------------- AllReduce half + add + RMSNorm */

/* Exact sum of bf16 values, rounded once to bf16.
 * Every finite bf16 value is an integer multiple of 2^-133 (the subnormal step): with exponent field e and
 * mantissa m, v = +-M * 2^sh * 2^-133 where M = m, sh = 0 for e == 0 and M = 128 + m, sh = e - 1 otherwise.
 * A double does not hold such a sum exactly when the addends' exponents span more than about 42 bits (a
 * subnormal beside a value near 1), so the sum is kept as an integer: the positive and the negative addends
 * accumulate separately in 320-bit unsigned integers (five 64-bit limbs; 8 addends below 2^(8 + 253) fit),
 * the smaller total is subtracted from the larger, and the difference N (sum = +-N * 2^-133) is rounded to 8
 * significant bits, ties to even. A zero sum is +0 (an empty sum plus zero terms). */
#define ORC_LIMBS 5
typedef struct {
    uint64_t w[ORC_LIMBS]; /* little-endian limbs */
} orc_u320;

static void u320_add_shifted(orc_u320* a, uint64_t m, int sh) { /* a += m * 2^sh, m < 2^8, 0 <= sh < 255 */
    int limb = sh / 64, off = sh % 64;
    uint64_t lo = m << off;
    uint64_t hi = off ? (m >> (64 - off)) : 0;
    uint64_t carry = 0;
    for (int i = limb; i < ORC_LIMBS; ++i) {
        uint64_t add = (i == limb) ? lo : ((i == limb + 1) ? hi : 0);
        uint64_t s1 = a->w[i] + add;
        uint64_t c1 = s1 < add ? 1 : 0;
        uint64_t s2 = s1 + carry;
        uint64_t c2 = s2 < carry ? 1 : 0;
        a->w[i] = s2;
        carry = c1 | c2;
    }
}

static int u320_cmp(const orc_u320* a, const orc_u320* b) {
    for (int i = ORC_LIMBS - 1; i >= 0; --i)
        if (a->w[i] != b->w[i]) return a->w[i] < b->w[i] ? -1 : 1;
    return 0;
}

static orc_u320 u320_sub(const orc_u320* a, const orc_u320* b) { /* a - b, a >= b */
    orc_u320 r;
    uint64_t borrow = 0;
    for (int i = 0; i < ORC_LIMBS; ++i) {
        uint64_t d1 = a->w[i] - b->w[i];
        uint64_t b1 = a->w[i] < b->w[i] ? 1 : 0;
        uint64_t d2 = d1 - borrow;
        uint64_t b2 = d1 < borrow ? 1 : 0;
        r.w[i] = d2;
        borrow = b1 | b2;
    }
    return r;
}

static int u320_bit(const orc_u320* a, int i) { return (int)((a->w[i / 64] >> (i % 64)) & 1u); }

uint16_t orc_bf16_sum(const uint16_t* v, int n) {
    orc_u320 pos, neg;
    memset(&pos, 0, sizeof pos);
    memset(&neg, 0, sizeof neg);
    for (int k = 0; k < n; ++k) {
        int e = (v[k] >> 7) & 0xFF, m = v[k] & 0x7F;
        uint64_t M = (uint64_t)(e == 0 ? m : 128 + m);
        int sh = e == 0 ? 0 : e - 1;
        u320_add_shifted((v[k] & 0x8000) ? &neg : &pos, M, sh);
    }
    int c = u320_cmp(&pos, &neg);
    if (c == 0) return 0; /* +0 */
    uint16_t sign = c < 0 ? (uint16_t)0x8000 : (uint16_t)0;
    orc_u320 N = c < 0 ? u320_sub(&neg, &pos) : u320_sub(&pos, &neg);
    int p = ORC_LIMBS * 64 - 1;
    while (!u320_bit(&N, p)) --p; /* highest set bit */
    if (p < 8) return (uint16_t)(sign | (uint16_t)N.w[0]); /* N < 256: exactly a bf16 (subnormal or field 1) */
    uint32_t q = 0;
    for (int i = p; i > p - 8; --i) q = (q << 1) | (uint32_t)u320_bit(&N, i);   /* 8 significant bits */
    int round = u320_bit(&N, p - 8), sticky = 0;
    for (int i = p - 9; i >= 0 && !sticky; --i) sticky = u320_bit(&N, i);
    if (round && (sticky || (q & 1u))) ++q;
    if (q == 256) {
        q = 128;
        ++p;
    }
    int field = p - 6; /* value = q / 128 * 2^(p - 133) */
    if (field >= 255) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (uint16_t)(field << 7) | (uint16_t)(q - 128));
}

/* x row t = bf16 of the exact sum of the partials' row t. */
static void reduce_partials(const uint16_t* const* partials, int n, int64_t t, int64_t H, uint16_t* x_row) {
    uint16_t v[8];
    for (int64_t j = 0; j < H; ++j) {
        for (int k = 0; k < n; ++k) v[k] = partials[k][t * H + j];
        x_row[j] = orc_bf16_sum(v, n);
    }
}

static int check_partials(const uint16_t* const* partials, int n, int64_t T) {
    if (n < 1 || n > 8) return -1;
    if (T > 0 && !partials) return -1;
    for (int k = 0; T > 0 && k < n; ++k)
        if (!partials[k]) return -1;
    return 0;
}

int orc_allreduce_add_rmsnorm(const uint16_t* const* partials, int n, const uint16_t* r, const uint16_t* w,
                              int64_t T, int64_t H, float eps, uint16_t* residual_out, double* v_out,
                              uint16_t* out) {
    if (T < 0 || H <= 0 || check_partials(partials, n, T) != 0) return -1;
    uint16_t* x_row = (uint16_t*)malloc((size_t)H * sizeof(uint16_t));
    if (!x_row) return -1;
    int rc = 0;
    for (int64_t t = 0; t < T && rc == 0; ++t) {
        reduce_partials(partials, n, t, H, x_row);
        rc = orc_add_rmsnorm(x_row, r + t * H, w, 1, H, eps, residual_out + t * H, v_out ? v_out + t * H : NULL,
                             out ? out + t * H : NULL);
    }
    free(x_row);
    return rc;
}

int orc_allreduce_add_rmsnorm_quant_fp8(const uint16_t* const* partials, int n, const uint16_t* r,
                                        const uint16_t* w, int64_t T, int64_t H, float eps, int mode,
                                        float* scale, uint16_t* residual_out, uint8_t* q_out, double* v_out) {
    if (T < 0 || H <= 0 || check_partials(partials, n, T) != 0 || (mode != 0 && mode != 1)) return -1;
    uint16_t* x_row = (uint16_t*)malloc((size_t)H * sizeof(uint16_t));
    if (!x_row) return -1;
    int rc = 0;
    for (int64_t t = 0; t < T && rc == 0; ++t) {
        reduce_partials(partials, n, t, H, x_row);
        rc = orc_add_rmsnorm_quant_fp8(x_row, r + t * H, w, 1, H, eps, mode, mode == 0 ? scale : scale + t,
                                       residual_out + t * H, q_out + t * H, v_out ? v_out + t * H : NULL);
    }
    free(x_row);
    return rc;
}

/* ---------------------------------------------------------------- SwiGLU */

int orc_swiglu(const uint16_t* gate_up, int64_t T, int64_t I, double* h_out, uint16_t* out) {
    if (T < 0 || I <= 0) return -1;
    if (T > 0 && !gate_up) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* g = gate_up + t * 2 * I;
        const uint16_t* u = g + I;
        for (int64_t j = 0; j < I; ++j) {
            double h = orc_silu(orc_bf16_to_double(g[j])) * orc_bf16_to_double(u[j]);
            if (h_out) h_out[t * I + j] = h;
            if (out) out[t * I + j] = orc_bf16_round(h);
        }
    }
    return 0;
}

int orc_swiglu_quant_nvfp4(const uint16_t* gate_up, int64_t T, int64_t I, float tensor_scale, uint8_t* q_out,
                           uint8_t* sf_out, double* h_out) {
    if (T < 0 || I <= 0 || I % 16 != 0 || !(tensor_scale > 0.0f) || isinf(tensor_scale)) return -1;
    if (T > 0 && (!gate_up || !q_out || !sf_out)) return -1;
    double* row = (double*)malloc((size_t)I * sizeof(double));
    if (!row) return -1;
    for (int64_t t = 0; t < T; ++t) {
        orc_swiglu(gate_up + t * 2 * I, 1, I, row, NULL);
        nvfp4_row(row, I, tensor_scale, q_out + t * (I / 2), sf_out + t * (I / 16));
        if (h_out) memcpy(h_out + t * I, row, (size_t)I * sizeof(double));
    }
    free(row);
    return 0;
}

int orc_swiglu_quant_fp8(const uint16_t* gate_up, int64_t T, int64_t I, int mode, float* scale,
                         uint8_t* q_out, double* h_out) {
    if (T < 0 || I <= 0 || (mode != 0 && mode != 1)) return -1;
    if (T > 0 && (!gate_up || !scale || !q_out)) return -1;
    double* row = (double*)malloc((size_t)(I > 0 ? I : 1) * sizeof(double));
    if (T > 0 && !row) return -1;
    for (int64_t t = 0; t < T; ++t) {
        orc_swiglu(gate_up + t * 2 * I, 1, I, row, NULL);
        float sc = mode == 0 ? scale[0] : dynamic_scale(row, I);
        if (mode == 1) scale[t] = sc;
        quantise_row(row, I, sc, q_out + t * I);
        if (h_out) memcpy(h_out + t * I, row, (size_t)I * sizeof(double));
    }
    free(row);
    return 0;
}
