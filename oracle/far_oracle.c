/*
 * CPU oracle for fused residual-add + RMSNorm under the mixed-precision
 * rounding contract.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench may load it; the library itself never does, and
 * it shares no code with the CUDA sources.
 *
 * What it computes, per row t of a [tokens, hidden] row-major matrix, follows
 * the case study "Aligning fused RMSNorm rounding across vLLM backends":
 *   section "Finding the rounding boundary" (the stage table) and
 *   section "Implementation and tradeoffs":
 *
 *   s_i   = fl32(x_i + r_i)                  add in binary32, kept unrounded
 *                                            (no-residual variant: s_i = x_i)
 *   residual_out_i = RNE_act(s_i)            rounded only when stored
 *   S     = RN32( sum_i fl32(s_i * s_i) )    squares in binary32; the sum is the
 *                                            correctly rounded binary32 value of
 *                                            the exact sum of those squares
 *   var   = fl32(S / hidden)                 mean of the squares
 *   rstd  = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   a_i   = fl32(s_i * rstd)                 normalised from the binary32 sum
 *   n_i   = RNE_wd(a_i)                      cast to the weight dtype first ...
 *   out_i = RNE_od(fl32(n_i * w_i))          ... then multiplied by the weight
 *
 * The dtype policy follows the LyCORIS page "Precision", section "Dtype
 * policy": fp16, bf16 and fp32 may be combined freely except fp16 with bf16,
 * which is rejected; the output dtype od is the promotion of the operands'
 * dtypes (fp32 if either is fp32).
 *
 * Readings taken where the pages leave a step open:
 *  - The sum of squares: the pages fix binary32 accumulation but let the
 *    reduction order vary ("Testing the contract").  The oracle takes the one
 *    order-free binary32 value, the correct rounding of the exact sum of the
 *    binary32 squares, computed with an exact fixed-point accumulator.
 *  - rstd is 1/sqrt with IEEE square root and IEEE division (eps inside the
 *    root, as the "Mixed-Precision Kernels" page's layer-norm sketch places it).
 *  - Rounding is to nearest, ties to even, everywhere; no flush to zero;
 *    overflow of a 16-bit format gives infinity; NaN propagates.
 *
 * Quantised output (the variants with a per-token scale), following the
 * "Mixed-Precision Kernels" page, section "Quantised Kernels: INT8 and FP8
 * Inference" (symmetric scale = max_abs / 127), applied per row to the
 * contract's out values, so the fused result equals normalising and then
 * quantising separately:
 *   amax  = max_i |out_i|                      (a NaN in the row makes it NaN)
 *   scale = fl32(amax / QMAX)                  QMAX = 127 (int8) or 448 (FP8 E4M3)
 *   inv   = fl32(QMAX / amax), 0 when amax = 0
 *   q_i   = Q(fl32(out_i * inv))               int8: nearest integer, ties to even,
 *                                              clamped to [-127, 127], NaN -> 0;
 *                                              E4M3: nearest, ties to even, finite
 *                                              values saturated to +-448, NaN stays NaN
 *
 * LayerNorm under the same contract (the "Mixed-Precision Kernels" page, section
 * "Kernel-Level Mechanics: Cast Placement and Fusion": widen on load, mean and
 * variance in binary32, narrow on store), taken in two passes over the row
 * rather than the sketch's E[s^2] - mean^2:
 *   mean  = fl32(RN32(sum_i s_i) / hidden)     correctly rounded exact signed sum
 *   d_i   = fl32(s_i - mean)
 *   var   = fl32(RN32(sum_i fl32(d_i * d_i)) / hidden)
 *   rstd  = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   n_i   = RNE_wd(fl32(d_i * rstd))           cast to the weight dtype first
 *   out_i = RNE_od(fl32(fl32(n_i * gamma_i) + beta_i))   gamma, beta in the weight dtype
 *
 * GEMM with fp16 storage and fp32 compute (the Luminal page "Luminal FP16 Backend
 * Repair and H100 Evidence", section "What Was Fixed"): the exact sum of the exact
 * fp16 products, rounded once to fp16 (the projection cast), then the fp16 bias
 * added with one more fp16 rounding; see oracle_gemm_f16.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (binary32
 * arithmetic must not be fused or reassociated).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ------------------------------------------------------------------ */
/* binary32 bits                                                       */
/* ------------------------------------------------------------------ */

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float float_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/*
 * Round a binary32 value to the nearest value of a narrower binary format
 * (p significand bits including the leading one, normal exponents emin..emax,
 * subnormals below), ties to even, overflow to infinity.  Every value of
 * fp16 and bf16 is also a binary32 value, so the result is returned as one.
 */
static float round_to_format(float v, int p, int emin, int emax) {
    if (isnan(v)) return v;
    if (isinf(v) || v == 0.0f) return v;
    uint32_t b = bits_of(v);
    int negative = (int)(b >> 31);
    int field = (int)((b >> 23) & 0xffu);
    uint64_t m;   /* integer significand */
    int e;        /* value = m * 2^e     */
    if (field == 0) { m = b & 0x7fffffu; e = -149; }
    else { m = (b & 0x7fffffu) | 0x800000u; e = field - 150; }
    int lead = 63 - __builtin_clzll(m) + e;         /* exponent of the leading bit */
    int q = (lead > emin ? lead : emin) - (p - 1);  /* exponent of the target's last place */
    int drop = q - e;                                /* low bits that do not fit */
    if (drop > 0) {
        if (drop > 40) {
            m = 0;                                   /* below half the smallest subnormal */
        } else {
            uint64_t keep = m >> drop;
            uint64_t rest = m & ((1ull << drop) - 1);
            uint64_t half = 1ull << (drop - 1);
            if (rest > half || (rest == half && (keep & 1u))) keep += 1;
            m = keep;
        }
        e = q;
    }
    double mag = ldexp((double)m, e);
    if (mag >= ldexp(1.0, emax + 1)) mag = INFINITY;
    float r = (float)mag;   /* exact: mag is a value of the target format, or infinity */
    return negative ? -r : r;
}

static float round_f16(float v) { return round_to_format(v, 11, -14, 15); }
static float round_bf16(float v) { return round_to_format(v, 8, -126, 127); }

static float round_to(int dtype, float v) {
    if (dtype == OR_F16) return round_f16(v);
    if (dtype == OR_BF16) return round_bf16(v);
    return v;
}

/* bits of a binary32 value that is exactly an fp16 value (or inf / NaN) */
static uint16_t encode_f16(float v) {
    uint32_t b = bits_of(v);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    if (isinf(v)) return (uint16_t)(sign | 0x7c00u);
    if (v == 0.0f) return sign;
    int e = (int)((b >> 23) & 0xffu) - 127;   /* fp16 values are normal binary32 values */
    uint32_t m = (b & 0x7fffffu) | 0x800000u;
    if (e >= -14) return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((m >> 13) & 0x3ffu));
    return (uint16_t)(sign | (uint16_t)(m >> (-e - 1)));  /* subnormal: v / 2^-24 */
}

static float decode_f16(uint16_t h) {
    int negative = h >> 15;
    int field = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    float v;
    if (field == 31) v = man ? NAN : INFINITY;
    else if (field == 0) v = ldexpf((float)man, -24);
    else v = ldexpf((float)(1024 + man), field - 25);
    return negative ? -v : v;
}

/* bits of a binary32 value that is exactly a bf16 value (or inf / NaN) */
static uint16_t encode_bf16(float v) {
    uint32_t b = bits_of(v);
    if (isnan(v)) return (uint16_t)(((b >> 16) & 0x8000u) | 0x7fc0u);
    return (uint16_t)(b >> 16);
}

static float decode_bf16(uint16_t h) { return float_of((uint32_t)h << 16); }

/* ---- FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no
   infinities; S.1111.111 is NaN, so the largest finite value is 1.75 * 2^8 = 448) */

/* nearest E4M3 value (ties to even), finite values saturated to +-448 */
static float round_e4m3_satfinite(float v) {
    if (isnan(v)) return v;
    float r = isinf(v) ? v : round_to_format(v, 4, -6, 8);  /* 480 = 1.111b * 2^8 is NaN, not a value */
    if (r > 448.0f) r = 448.0f;
    if (r < -448.0f) r = -448.0f;
    return r;
}

static uint8_t encode_e4m3(float v) {  /* v is an E4M3 value or NaN */
    uint32_t b = bits_of(v);
    uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
    if (isnan(v)) return (uint8_t)(sign | 0x7fu);
    if (v == 0.0f) return sign;
    int e = (int)((b >> 23) & 0xffu) - 127;
    uint32_t m = (b & 0x7fffffu) | 0x800000u;
    if (e >= -6) return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((m >> 20) & 0x7u));
    return (uint8_t)(sign | (uint8_t)(m >> (-e + 14)));  /* subnormal: v / 2^-9 */
}

static float decode_e4m3(uint8_t c) {
    int negative = c >> 7, field = (c >> 3) & 0xf, man = c & 7;
    float v;
    if (field == 15 && man == 7) v = NAN;
    else if (field == 0) v = ldexpf((float)man, -9);
    else v = ldexpf((float)(8 + man), field - 10);
    return negative ? -v : v;
}

/* nearest integer (ties to even), clamped to [-127, 127]; NaN -> 0 */
static int8_t quant_int8(float v) {
    if (isnan(v)) return 0;
    if (v >= 127.0f) return 127;
    if (v <= -127.0f) return -127;
    float f = floorf(v);
    float d = v - f;                      /* exact: |v| < 2^23 */
    float n = f;
    if (d > 0.5f || (d == 0.5f && fmodf(f, 2.0f) != 0.0f)) n = f + 1.0f;
    return (int8_t)n;
}

static float load(const void* base, int dtype, int64_t i) {
    if (dtype == OR_F16) return decode_f16(((const uint16_t*)base)[i]);
    if (dtype == OR_BF16) return decode_bf16(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

/* store a value that is already a value of `dtype` */
static void store(void* base, int dtype, int64_t i, float v) {
    if (dtype == OR_F16) ((uint16_t*)base)[i] = encode_f16(v);
    else if (dtype == OR_BF16) ((uint16_t*)base)[i] = encode_bf16(v);
    else ((float*)base)[i] = v;
}

/* ------------------------------------------------------------------ */
/* exact sum of binary32 values                                        */
/* ------------------------------------------------------------------ */

/*
 * Fixed-point accumulator: bit k of the integer has weight 2^(k-149), the
 * last place of the smallest binary32 subnormal, so every finite binary32
 * value is an integer here.  The largest finite value needs bit 277; ten
 * 32-bit limbs (320 bits) leave room for more than 2^40 terms.
 */
#define ACC_LIMBS 10

typedef struct {
    uint32_t limb[ACC_LIMBS];
    int has_nan, has_pinf, has_ninf;
} exact_acc;

static void acc_init(exact_acc* a) { memset(a, 0, sizeof *a); }

/* add a non-negative binary32 value (the squares are never negative) */
static void acc_add(exact_acc* a, float v) {
    if (isnan(v)) { a->has_nan = 1; return; }
    if (isinf(v)) { if (v > 0) a->has_pinf = 1; else a->has_ninf = 1; return; }
    uint32_t b = bits_of(v) & 0x7fffffffu;
    int field = (int)(b >> 23);
    uint64_t m = b & 0x7fffffu;
    int pos = 0;                             /* value = m * 2^(pos - 149) */
    if (field != 0) { m |= 0x800000u; pos = field - 1; }
    int k = pos / 32;
    uint64_t chunk = m << (pos % 32);        /* at most 55 bits */
    uint64_t carry = 0;
    for (int j = k; j < ACC_LIMBS; ++j) {
        uint64_t add = (j == k) ? (chunk & 0xffffffffu) : (j == k + 1) ? (chunk >> 32) : 0;
        if (j > k + 1 && carry == 0) break;
        uint64_t t = (uint64_t)a->limb[j] + add + carry;
        a->limb[j] = (uint32_t)t;
        carry = t >> 32;
    }
}

static int acc_bit(const exact_acc* a, int k) { return (int)((a->limb[k / 32] >> (k % 32)) & 1u); }

/* the accumulated exact sum, rounded to nearest binary32 (ties to even) */
static float acc_round(const exact_acc* a) {
    if (a->has_nan || (a->has_pinf && a->has_ninf)) return NAN;
    if (a->has_pinf) return INFINITY;
    if (a->has_ninf) return -INFINITY;
    int top = -1;
    for (int k = ACC_LIMBS * 32 - 1; k >= 0; --k)
        if (acc_bit(a, k)) { top = k; break; }
    if (top < 0) return 0.0f;
    if (top < 24) {                           /* fewer than 24 bits: exact */
        uint64_t n = 0;
        for (int k = top; k >= 0; --k) n = (n << 1) | (uint64_t)acc_bit(a, k);
        return (float)ldexp((double)n, -149);
    }
    uint64_t keep = 0;                        /* the 24 leading bits */
    for (int k = top; k > top - 24; --k) keep = (keep << 1) | (uint64_t)acc_bit(a, k);
    int guard = acc_bit(a, top - 24);
    int sticky = 0;
    for (int k = top - 25; k >= 0 && !sticky; --k) sticky = acc_bit(a, k);
    if (guard && (sticky || (keep & 1u))) keep += 1;
    double mag = ldexp((double)keep, top - 23 - 149);  /* exact in binary64 */
    return (float)mag;  /* exact, or infinity when the rounded sum reaches 2^128 */
}

/* exact signed sum: the magnitudes of positive and negative terms in two
   accumulators, their difference taken exactly, then rounded once */
typedef struct { exact_acc pos, neg; } signed_acc;

static void sacc_init(signed_acc* a) { acc_init(&a->pos); acc_init(&a->neg); }

static void sacc_add(signed_acc* a, float v) {
    if (isnan(v)) { a->pos.has_nan = 1; return; }
    if (isinf(v)) { if (v > 0) a->pos.has_pinf = 1; else a->neg.has_pinf = 1; return; }
    if (v > 0) acc_add(&a->pos, v);
    else if (v < 0) acc_add(&a->neg, -v);
}

/* -1, 0, +1 as the magnitude in A is below, equal to, above the one in B */
static int acc_compare(const exact_acc* A, const exact_acc* B) {
    for (int k = ACC_LIMBS - 1; k >= 0; --k) {
        if (A->limb[k] != B->limb[k]) return A->limb[k] > B->limb[k] ? 1 : -1;
    }
    return 0;
}

static float sacc_round(const signed_acc* a) {
    if (a->pos.has_nan || (a->pos.has_pinf && a->neg.has_pinf)) return NAN;
    if (a->pos.has_pinf) return INFINITY;
    if (a->neg.has_pinf) return -INFINITY;
    int c = acc_compare(&a->pos, &a->neg);
    if (c == 0) return 0.0f;  /* x + (-x) is +0 under round to nearest */
    const exact_acc* big = c > 0 ? &a->pos : &a->neg;
    const exact_acc* small = c > 0 ? &a->neg : &a->pos;
    exact_acc diff;
    acc_init(&diff);
    uint64_t borrow = 0;
    for (int k = 0; k < ACC_LIMBS; ++k) {
        uint64_t t = (uint64_t)big->limb[k] - (uint64_t)small->limb[k] - borrow;
        diff.limb[k] = (uint32_t)t;
        borrow = (t >> 63) & 1u;  /* wrapped below zero */
    }
    float m = acc_round(&diff);
    return c > 0 ? m : -m;
}

/* ------------------------------------------------------------------ */
/* dtype policy                                                        */
/* ------------------------------------------------------------------ */

static int valid_dtype(int d) { return d == OR_F32 || d == OR_F16 || d == OR_BF16; }

/* output dtype = promotion of act and wd; -1 for fp16 with bf16 or an unknown code */
int oracle_output_dtype(int act, int wd) {
    if (!valid_dtype(act) || !valid_dtype(wd)) return -1;
    if ((act == OR_F16 && wd == OR_BF16) || (act == OR_BF16 && wd == OR_F16)) return -1;
    if (act == OR_F32 || wd == OR_F32) return OR_F32;
    return act;
}

/* ------------------------------------------------------------------ */
/* the row                                                             */
/* ------------------------------------------------------------------ */

/* rstd of one row of binary32 sums s[0..hidden); also returns S and var */
static float row_rstd(const float* s, int64_t hidden, float eps, float* S_out, float* var_out) {
    exact_acc acc;
    acc_init(&acc);
    for (int64_t i = 0; i < hidden; ++i) {
        float sq = s[i] * s[i];
        acc_add(&acc, sq);
    }
    float S = acc_round(&acc);
    float var = S / (float)hidden;
    float tv = var + eps;
    float root = sqrtf(tv);
    float rstd = 1.0f / root;
    if (S_out) *S_out = S;
    if (var_out) *var_out = var;
    return rstd;
}

static int run(const void* x, const void* residual, const void* weight, float eps,
               void* out, void* residual_out, int64_t tokens, int64_t hidden,
               int act, int wd, int has_residual) {
    int od = oracle_output_dtype(act, wd);
    if (od < 0) return -1;
    if (tokens < 0 || hidden <= 0) return -2;
    size_t sa = act == OR_F32 ? 4 : 2, so = od == OR_F32 ? 4 : 2;
    float* s = (float*)malloc((size_t)hidden * sizeof(float));
    if (!s) return -3;
    for (int64_t t = 0; t < tokens; ++t) {
        const char* xr = (const char*)x + (size_t)t * (size_t)hidden * sa;
        const char* rr = has_residual ? (const char*)residual + (size_t)t * (size_t)hidden * sa : NULL;
        char* orow = (char*)out + (size_t)t * (size_t)hidden * so;
        char* rorow = has_residual ? (char*)residual_out + (size_t)t * (size_t)hidden * sa : NULL;
        for (int64_t i = 0; i < hidden; ++i) {
            float xf = load(xr, act, i);             /* widening is exact */
            if (has_residual) {
                float rf = load(rr, act, i);
                s[i] = xf + rf;                      /* binary32 add, kept unrounded */
                store(rorow, act, i, round_to(act, s[i]));
            } else {
                s[i] = xf;
            }
        }
        float rstd = row_rstd(s, hidden, eps, NULL, NULL);
        for (int64_t i = 0; i < hidden; ++i) {
            float a = s[i] * rstd;                   /* from the binary32 sum */
            float n = round_to(wd, a);               /* weight dtype first */
            float prod = n * load(weight, wd, i);    /* then the weight */
            store(orow, od, i, round_to(od, prod));
        }
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------ */
/* exported entry points (host pointers; same argument order as the    */
/* library's, with the two dtypes passed separately)                   */
/* ------------------------------------------------------------------ */

int oracle_fused_add_rmsnorm(const void* x, const void* residual, const void* weight, float eps,
                             void* out, void* residual_out, int64_t tokens, int64_t hidden,
                             int act, int wd) {
    return run(x, residual, weight, eps, out, residual_out, tokens, hidden, act, wd, 1);
}

int oracle_rmsnorm(const void* x, const void* weight, float eps, void* out,
                   int64_t tokens, int64_t hidden, int act, int wd) {
    return run(x, NULL, weight, eps, out, NULL, tokens, hidden, act, wd, 0);
}

/* per-row intermediates of the fused op: S, var and rstd (for pins) */
int oracle_row_stats(const void* x, const void* residual, float eps, int64_t tokens, int64_t hidden,
                     int act, float* S, float* var, float* rstd) {
    size_t sa = act == OR_F32 ? 4 : 2;
    float* s = (float*)malloc((size_t)hidden * sizeof(float));
    if (!s) return -3;
    for (int64_t t = 0; t < tokens; ++t) {
        const char* xr = (const char*)x + (size_t)t * (size_t)hidden * sa;
        const char* rr = residual ? (const char*)residual + (size_t)t * (size_t)hidden * sa : NULL;
        for (int64_t i = 0; i < hidden; ++i)
            s[i] = rr ? load(xr, act, i) + load(rr, act, i) : load(xr, act, i);
        rstd[t] = row_rstd(s, hidden, eps, &S[t], &var[t]);
    }
    free(s);
    return 0;
}

/* correctly rounded binary32 sum of n non-negative binary32 values */
float oracle_exact_sum(const float* v, int64_t n) {
    exact_acc acc;
    acc_init(&acc);
    for (int64_t i = 0; i < n; ++i) acc_add(&acc, v[i]);
    return acc_round(&acc);
}

/* ------------------------------------------------------------------ */
/* LayerNorm                                                           */
/* ------------------------------------------------------------------ */

/* mean and rstd of one row of binary32 sums s[0..hidden); d[] receives s - mean */
static float ln_row_stats(const float* s, float* d, int64_t hidden, float eps, float* mean_out) {
    signed_acc sa;
    sacc_init(&sa);
    for (int64_t i = 0; i < hidden; ++i) sacc_add(&sa, s[i]);
    float S1 = sacc_round(&sa);
    float mean = S1 / (float)hidden;
    exact_acc acc;
    acc_init(&acc);
    for (int64_t i = 0; i < hidden; ++i) {
        d[i] = s[i] - mean;
        float sq = d[i] * d[i];
        acc_add(&acc, sq);
    }
    float S2 = acc_round(&acc);
    float var = S2 / (float)hidden;
    float tv = var + eps;
    float root = sqrtf(tv);
    if (mean_out) *mean_out = mean;
    return 1.0f / root;
}

static int run_ln(const void* x, const void* residual, const void* gamma, const void* beta, float eps,
                  void* out, void* residual_out, int64_t tokens, int64_t hidden, int act, int wd,
                  int has_residual) {
    int od = oracle_output_dtype(act, wd);
    if (od < 0) return -1;
    if (tokens < 0 || hidden <= 0) return -2;
    size_t sa = act == OR_F32 ? 4 : 2, so = od == OR_F32 ? 4 : 2;
    float* s = (float*)malloc((size_t)hidden * sizeof(float));
    float* d = (float*)malloc((size_t)hidden * sizeof(float));
    if (!s || !d) { free(s); free(d); return -3; }
    for (int64_t t = 0; t < tokens; ++t) {
        const char* xr = (const char*)x + (size_t)t * (size_t)hidden * sa;
        const char* rr = has_residual ? (const char*)residual + (size_t)t * (size_t)hidden * sa : NULL;
        char* orow = (char*)out + (size_t)t * (size_t)hidden * so;
        char* rorow = has_residual ? (char*)residual_out + (size_t)t * (size_t)hidden * sa : NULL;
        for (int64_t i = 0; i < hidden; ++i) {
            float xf = load(xr, act, i);
            if (has_residual) {
                s[i] = xf + load(rr, act, i);
                store(rorow, act, i, round_to(act, s[i]));
            } else {
                s[i] = xf;
            }
        }
        float rstd = ln_row_stats(s, d, hidden, eps, NULL);
        for (int64_t i = 0; i < hidden; ++i) {
            float a = d[i] * rstd;
            float n = round_to(wd, a);                  /* weight dtype first */
            float t1 = n * load(gamma, wd, i);          /* then the scale ... */
            float u = t1 + load(beta, wd, i);           /* ... and the shift */
            store(orow, od, i, round_to(od, u));
        }
    }
    free(s);
    free(d);
    return 0;
}

int oracle_fused_add_layernorm(const void* x, const void* residual, const void* gamma, const void* beta,
                               float eps, void* out, void* residual_out, int64_t tokens, int64_t hidden,
                               int act, int wd) {
    return run_ln(x, residual, gamma, beta, eps, out, residual_out, tokens, hidden, act, wd, 1);
}

int oracle_layernorm(const void* x, const void* gamma, const void* beta, float eps, void* out,
                     int64_t tokens, int64_t hidden, int act, int wd) {
    return run_ln(x, NULL, gamma, beta, eps, out, NULL, tokens, hidden, act, wd, 0);
}

/* per-row mean and rstd of the fused LayerNorm (for pins) */
int oracle_ln_row_stats(const void* x, const void* residual, float eps, int64_t tokens, int64_t hidden,
                        int act, float* mean, float* rstd) {
    size_t sa = act == OR_F32 ? 4 : 2;
    float* s = (float*)malloc((size_t)hidden * sizeof(float));
    float* d = (float*)malloc((size_t)hidden * sizeof(float));
    if (!s || !d) { free(s); free(d); return -3; }
    for (int64_t t = 0; t < tokens; ++t) {
        const char* xr = (const char*)x + (size_t)t * (size_t)hidden * sa;
        const char* rr = residual ? (const char*)residual + (size_t)t * (size_t)hidden * sa : NULL;
        for (int64_t i = 0; i < hidden; ++i)
            s[i] = rr ? load(xr, act, i) + load(rr, act, i) : load(xr, act, i);
        rstd[t] = ln_row_stats(s, d, hidden, eps, &mean[t]);
    }
    free(s);
    free(d);
    return 0;
}

/* correctly rounded binary32 sum of n binary32 values of any sign */
float oracle_exact_signed_sum(const float* v, int64_t n) {
    signed_acc a;
    sacc_init(&a);
    for (int64_t i = 0; i < n; ++i) sacc_add(&a, v[i]);
    return sacc_round(&a);
}

/* ------------------------------------------------------------------ */
/* quantised output                                                    */
/* ------------------------------------------------------------------ */

enum { OR_Q_INT8 = 1, OR_Q_FP8_E4M3 = 2 };

/* quantise one row of out values (already values of od) into q, return its scale */
static float quantise_row(const float* o, int64_t hidden, int qtype, void* qrow) {
    const float qmax = qtype == OR_Q_INT8 ? 127.0f : 448.0f;
    float amax = 0.0f;
    for (int64_t i = 0; i < hidden; ++i) {
        float a = fabsf(o[i]);
        if (isnan(a) || a > amax) amax = isnan(amax) ? amax : a;
    }
    float scale = amax / qmax;
    float inv = amax == 0.0f ? 0.0f : qmax / amax;
    for (int64_t i = 0; i < hidden; ++i) {
        float v = o[i] * inv;
        if (qtype == OR_Q_INT8) ((int8_t*)qrow)[i] = quant_int8(v);
        else ((uint8_t*)qrow)[i] = encode_e4m3(round_e4m3_satfinite(v));
    }
    return scale;
}

static int run_quant(const void* x, const void* residual, const void* weight, float eps, void* q,
                     float* scale, void* residual_out, int64_t tokens, int64_t hidden, int act, int wd,
                     int qtype, int has_residual) {
    int od = oracle_output_dtype(act, wd);
    if (od < 0) return -1;
    if (tokens < 0 || hidden <= 0 || (qtype != OR_Q_INT8 && qtype != OR_Q_FP8_E4M3)) return -2;
    size_t sa = act == OR_F32 ? 4 : 2, so = od == OR_F32 ? 4 : 2;
    void* orow = malloc((size_t)hidden * so);
    float* of = (float*)malloc((size_t)hidden * sizeof(float));
    if (!orow || !of) { free(orow); free(of); return -3; }
    for (int64_t t = 0; t < tokens; ++t) {
        const char* xr = (const char*)x + (size_t)t * (size_t)hidden * sa;
        const char* rr = has_residual ? (const char*)residual + (size_t)t * (size_t)hidden * sa : NULL;
        char* ror = has_residual ? (char*)residual_out + (size_t)t * (size_t)hidden * sa : NULL;
        /* the unquantised row first, exactly as the plain op computes it */
        int rc = run(xr, rr, weight, eps, orow, ror, 1, hidden, act, wd, has_residual);
        if (rc != 0) { free(orow); free(of); return rc; }
        for (int64_t i = 0; i < hidden; ++i) of[i] = load(orow, od, i);
        scale[t] = quantise_row(of, hidden, qtype, (char*)q + (size_t)t * (size_t)hidden);
    }
    free(orow);
    free(of);
    return 0;
}

int oracle_fused_add_rmsnorm_quant(const void* x, const void* residual, const void* weight, float eps,
                                   void* q, float* scale, void* residual_out, int64_t tokens,
                                   int64_t hidden, int act, int wd, int qtype) {
    return run_quant(x, residual, weight, eps, q, scale, residual_out, tokens, hidden, act, wd, qtype, 1);
}

int oracle_rmsnorm_quant(const void* x, const void* weight, float eps, void* q, float* scale,
                         int64_t tokens, int64_t hidden, int act, int wd, int qtype) {
    return run_quant(x, NULL, weight, eps, q, scale, NULL, tokens, hidden, act, wd, qtype, 0);
}

uint8_t oracle_f32_to_e4m3(float v) { return encode_e4m3(round_e4m3_satfinite(v)); }
float oracle_e4m3_to_f32(uint8_t c) { return decode_e4m3(c); }
int oracle_f32_to_int8(float v) { return quant_int8(v); }

/* format conversions, exposed so they can be pinned on their own */
uint16_t oracle_f32_to_f16(float v) { return encode_f16(round_f16(v)); }
uint16_t oracle_f32_to_bf16(float v) { return encode_bf16(round_bf16(v)); }
float oracle_f16_to_f32(uint16_t h) { return decode_f16(h); }
float oracle_bf16_to_f32(uint16_t h) { return decode_bf16(h); }

/* ------------------------------------------------------------------ */
/* GEMM with fp16 storage and fp32 compute                             */
/* ------------------------------------------------------------------ */
/*
 * The consumer projection of the Luminal page "Luminal FP16 Backend Repair and
 * H100 Evidence" (section "What Was Fixed", the corrected adapter): the fp16
 * operands are widened exactly, multiplied and summed in fp32, the result is
 * cast to fp16 (the projection's rounding boundary), then the fp16 bias is added
 * in fp16.  With x [M, K] and the transposed weight wt [N, K], both row-major:
 *
 *   p[m,n] = RNE_f16( sum_k x[m,k] * wt[n,k] )        (out_dtype fp16)
 *   y[m,n] = RNE_f16( p[m,n] + bias[n] )              (bias optional)
 *   out[m,n] = RN32( sum_k x[m,k] * wt[n,k] )         (out_dtype fp32, no bias)
 *
 * The sum is the exact sum, rounded once: "fp32 arithmetic" fixes no order of
 * the additions, and the exact sum is the value every order approximates (the
 * page's own reference evaluates it in fp64).  Each product of two fp16 values
 * is exactly a binary32 value (22 significant bits, magnitudes from 2^-48 to
 * below 2^32), so the products enter the exact accumulator unrounded.
 */

/* the exact non-negative sum in `a`, rounded to nearest (ties to even) in the binary
   format with p significand bits and normal exponents emin..emax; infinity above it */
static double acc_round_format(const exact_acc* a, int p, int emin, int emax) {
    if (a->has_nan || (a->has_pinf && a->has_ninf)) return NAN;
    if (a->has_pinf) return INFINITY;
    if (a->has_ninf) return -INFINITY;
    int top = -1;
    for (int k = ACC_LIMBS * 32 - 1; k >= 0; --k)
        if (acc_bit(a, k)) { top = k; break; }
    if (top < 0) return 0.0;
    int lead = top - 149;                            /* exponent of the leading bit */
    int q = (lead > emin ? lead : emin) - (p - 1);   /* exponent of the last place kept */
    int kq = q + 149;                                /* its bit index */
    uint64_t keep = 0;
    int guard = 0, sticky = 0;
    for (int k = top; k >= 0; --k) {
        int bit = acc_bit(a, k);
        if (k >= kq) keep = (keep << 1) | (uint64_t)bit;
        else if (k == kq - 1) guard = bit;
        else if (bit) { sticky = 1; break; }
    }
    if (kq > 0 && guard && (sticky || (keep & 1u))) keep += 1;
    double mag = kq > 0 ? ldexp((double)keep, q) : ldexp((double)keep, -149);
    if (mag >= ldexp(1.0, emax + 1)) mag = INFINITY;
    return mag;
}

/* the same for a signed sum */
static double sacc_round_format(const signed_acc* a, int p, int emin, int emax) {
    if (a->pos.has_nan || (a->pos.has_pinf && a->neg.has_pinf)) return NAN;
    if (a->pos.has_pinf) return INFINITY;
    if (a->neg.has_pinf) return -INFINITY;
    int c = acc_compare(&a->pos, &a->neg);
    if (c == 0) return 0.0;
    const exact_acc* big = c > 0 ? &a->pos : &a->neg;
    const exact_acc* small = c > 0 ? &a->neg : &a->pos;
    exact_acc diff;
    acc_init(&diff);
    uint64_t borrow = 0;
    for (int k = 0; k < ACC_LIMBS; ++k) {
        uint64_t t = (uint64_t)big->limb[k] - (uint64_t)small->limb[k] - borrow;
        diff.limb[k] = (uint32_t)t;
        borrow = (t >> 63) & 1u;
    }
    double m = acc_round_format(&diff, p, emin, emax);
    return c > 0 ? m : -m;
}

/* a binary64 value rounded to nearest (ties to even) in the fp16 format */
static double round_double_f16(double v) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    const int p = 11, emin = -14, emax = 15;
    int lead = ilogb(v);
    int q = (lead > emin ? lead : emin) - (p - 1);
    double scaled = ldexp(fabs(v), -q);   /* exact: a power-of-two scaling */
    double keep = floor(scaled);
    double rest = scaled - keep;          /* exact */
    if (rest > 0.5 || (rest == 0.5 && fmod(keep, 2.0) != 0.0)) keep += 1.0;
    double mag = ldexp(keep, q);
    if (mag >= ldexp(1.0, emax + 1)) mag = INFINITY;
    return v < 0 ? -mag : mag;
}

/* x [M, K], wt [N, K], bias [N] (or NULL): fp16 bit patterns; out [M, N] fp16 bits
   (out_dtype OR_F16) or binary32 (OR_F32, bias must be NULL) */
int oracle_gemm_f16(const uint16_t* x, const uint16_t* wt, const uint16_t* bias, void* out, int64_t M,
                    int64_t N, int64_t K, int out_dtype) {
    if (M < 0 || N < 0 || K < 0) return 4;
    if (out_dtype != OR_F16 && out_dtype != OR_F32) return 2;
    if (out_dtype == OR_F32 && bias) return 2;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            signed_acc acc;
            sacc_init(&acc);
            for (int64_t k = 0; k < K; ++k) {
                float a = decode_f16(x[m * K + k]);
                float b = decode_f16(wt[n * K + k]);
                sacc_add(&acc, a * b);   /* exact: see above */
            }
            if (out_dtype == OR_F32) {
                ((float*)out)[m * N + n] = (float)sacc_round_format(&acc, 24, -126, 127);
                continue;
            }
            double p16 = sacc_round_format(&acc, 11, -14, 15);   /* the projection cast */
            double y = bias ? round_double_f16(p16 + (double)decode_f16(bias[n])) : p16;
            ((uint16_t*)out)[m * N + n] = encode_f16((float)y);   /* y is an fp16 value */
        }
    }
    return 0;
}
