/*
 * fme_oracle.c -- the plain CPU oracle for the low-precision MoE expert path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA library: every table below is built
 * here from the format definitions, one scalar at a time.
 *
 * What it computes, and where each step comes from:
 *
 *   - "Composer 2 Technical Report" (papercache.org summary), section 6.1,
 *     paragraph on the NVFP4 variant of the MoE forward: bf16 values become
 *     FP4 E2M1 codes with an FP8 E4M3 scale per block of 16 along K and an
 *     FP32 scale per token.  Same page, paragraph on hardware-level math
 *     precision: the NVFP4 quantizer must use IEEE-compliant (correctly
 *     rounded) division.  "Cursor Composer 2 report deep dive"
 *     (machinelearningatscale.substack.com), section 1 "The kernel section",
 *     restates both points.
 *   - Same report, section 6.1, paragraph on MXFP8 in the MoE backward: the
 *     standard MXFP8 format, FP8 E4M3 values with an FP8 E8M0 scale per block
 *     of 32 elements.
 *   - "Scaling and Optimizing Frontier Model Training" (Fireworks summary),
 *     "MXFP8 expert kernels": block-scaled grouped GEMMs in which the tensor
 *     core dequantizes inside the multiply.  The oracle computes that result
 *     from its plain definition: dequantize both operands exactly, multiply
 *     and sum in fp64.
 *   - Same page, same section: the experts are DeepSeek-V3-class (hidden 7168,
 *     intermediate 2048; the gate/up projection is twice the intermediate
 *     width).  The activation between the two projections is read as SwiGLU,
 *     h = silu(g) * u with silu(v) = v / (1 + e^-v), g and u the two halves of
 *     the gate/up output; the oracle evaluates it in fp64, and its gradient
 *     (the backward of the gate/up side, d(gate/up) from dh) in fp64 too.
 *   - "Cursor Composer 2 report deep dive", section 2, and the report's
 *     section 6.1: tokens are quantized before dispatch to their experts and
 *     the experts' outputs are combined per token in BF16; section 6.2: the
 *     per-token expert choices are replayed.  The oracle groups assignment
 *     a = t * top_k + k (token t's k-th expert) by expert keeping the order of
 *     a (a stable counting sort), and combines out[t] = sum over k in order of
 *     weight * y[row], each product and sum one fp32 operation, rounded once to
 *     bf16 at the end.
 *
 * Readings taken where the pages are silent (the plainest reading the rest of
 * the pages supports, each named here):
 *   - per-token decode scale S_t = amax_t / (6 * 448), fp32, IEEE division;
 *   - block scale sb = RNE-satfinite-E4M3(amax_b / fl32(6 * S_t));
 *   - element code q = RNE-satfinite-E2M1(fl32(x / fl32(dec(sb) * S_t)));
 *   - a row with amax 0, or a block whose scale code is 0, gets codes 0x0;
 *   - codes keep the sign of their input, so a negative value that rounds
 *     to zero becomes -0 (E2M1 0x8, E4M3 0x80);
 *   - MXFP8 scale X = 2^(floor(log2 amax) - 8), E8M0 code clamped to
 *     [0, 254], code 0 for an all-zero block; q = RNE-satfinite-E4M3(x / X)
 *     computed exactly (X is a power of two);
 *   - column-wise MXFP8 restarts its 32-blocks at each group offset and pads
 *     each group to a multiple of 128 positions with zeros.
 *
 * Arithmetic rules: every fp32 operation is one IEEE binary32 operation
 * rounded to nearest even.  Build with -ffp-contract=off and without
 * -ffast-math so that no multiply-add is fused and no operation reordered.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- inputs -- */

/* bf16 is the upper half of a binary32. */
static float bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ----------------------------------------------------------- code tables -- */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent 0 is subnormal: 0.M * 2^0.  No Inf, no NaN. */
double fme_orc_e2m1_value(uint8_t code) {
    int sign = (code >> 3) & 1;
    int exp = (code >> 1) & 3;
    int man = code & 1;
    double mag;
    if (exp == 0)
        mag = 0.5 * man;
    else
        mag = ldexp(1.0 + 0.5 * man, exp - 1);
    return sign ? -mag : mag;
}

/* E4M3 ("fn" flavour of the OCP 8-bit formats): sign bit 7, exponent bits
 * 6..3 (bias 7), mantissa bits 2..0.  Exponent 0 is subnormal:
 * 0.MMM * 2^-6.  S.1111.111 is NaN; there is no Inf, so the largest finite
 * magnitude is 1.110b * 2^8 = 448. */
double fme_orc_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exp = (code >> 3) & 15;
    int man = code & 7;
    double mag;
    if (exp == 15 && man == 7)
        return NAN;
    if (exp == 0)
        mag = ldexp(man / 8.0, -6);
    else
        mag = ldexp(1.0 + man / 8.0, exp - 7);
    return sign ? -mag : mag;
}

/* E8M0: an unsigned power of two, 2^(code - 127); 0xFF is NaN. */
double fme_orc_e8m0_value(uint8_t code) {
    if (code == 0xFF)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Round |v| to the nearest entry of an increasing table of non-negative
 * magnitudes (index = code without its sign bit).  Ties go to the entry whose
 * index is even, i.e. whose mantissa LSB is 0.  Anything at or above the last
 * entry saturates to it ("satfinite").  The sign of v, including the sign of
 * -0.0, is put back as the sign bit. */
static uint8_t round_to_table(double v, const double *mag, int n, int sign_shift) {
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    int idx;
    if (a >= mag[n - 1]) {
        idx = n - 1;
    } else {
        int lo = 0, hi = n - 1; /* invariant: mag[lo] <= a < mag[hi] */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (mag[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        double midpoint = 0.5 * (mag[lo] + mag[hi]); /* exact: few-bit values */
        if (a < midpoint)
            idx = lo;
        else if (a > midpoint)
            idx = hi;
        else
            idx = (lo % 2 == 0) ? lo : hi;
    }
    return (uint8_t)((neg << sign_shift) | idx);
}

static double e2m1_mag[8];
static double e4m3_mag[127]; /* codes 0x00 .. 0x7E; 0x7F is NaN */
static int tables_ready = 0;

static void build_tables(void) {
    if (tables_ready)
        return;
    for (int c = 0; c < 8; ++c)
        e2m1_mag[c] = fme_orc_e2m1_value((uint8_t)c);
    for (int c = 0; c < 127; ++c)
        e4m3_mag[c] = fme_orc_e4m3_value((uint8_t)c);
    tables_ready = 1;
}

uint8_t fme_orc_e2m1_encode(double v) {
    build_tables();
    return round_to_table(v, e2m1_mag, 8, 3);
}

uint8_t fme_orc_e4m3_encode(double v) {
    build_tables();
    return round_to_table(v, e4m3_mag, 127, 7);
}

/* ----------------------------------------------- NVFP4, per-token scale -- */

/*
 * NVFP4 variant of the MoE forward (report section 6.1; deep-dive section 1):
 * for every row t of x [rows x k] (k a multiple of 16):
 *   amax_t = max_k |x_tk|                       (exact)
 *   S_t    = fl32(amax_t / 2688)                (IEEE division, 2688 = 6*448)
 *   d      = fl32(6 * S_t)
 *   per block b of 16 consecutive k:
 *     sb_b = E4M3(fl32(amax_b / d))             (IEEE division)
 *     e_b  = fl32(dec(sb_b) * S_t)
 *     q_k  = E2M1(fl32(x_k / e_b))              (IEEE division)
 * Outputs, logical (not swizzled) layouts:
 *   codes [rows x k/2], two codes per byte, the even k in the low nibble;
 *   sf    [rows x k/16] E4M3 codes;
 *   scale [rows]        S_t.
 * Nothing crosses rows: a row's outputs depend on that row alone.
 */
static void quant_nvfp4_rows(const uint16_t *x, int64_t rows, int64_t k, int per_tensor,
                             uint8_t *codes, uint8_t *sf, float *scale) {
    const int64_t nblk = k / 16;
    if (rows <= 0 || k <= 0)
        return;
    float tensor_amax = 0.0f;
    if (per_tensor) {
        for (int64_t i = 0; i < rows * k; ++i) {
            float a = fabsf(bf16_value(x[i]));
            if (a > tensor_amax)
                tensor_amax = a;
        }
    }
    for (int64_t t = 0; t < rows; ++t) {
        const uint16_t *xr = x + t * k;
        uint8_t *cr = codes + t * (k / 2);
        uint8_t *sr = sf + t * nblk;

        float amax = 0.0f;
        for (int64_t j = 0; j < k; ++j) {
            float a = fabsf(bf16_value(xr[j]));
            if (a > amax)
                amax = a;
        }
        if (per_tensor)
            amax = tensor_amax;
        memset(cr, 0, (size_t)(k / 2));
        if (amax == 0.0f) {
            scale[t] = 0.0f;
            memset(sr, 0, (size_t)nblk);
            continue;
        }
        float s_t = amax / 2688.0f;
        float d = 6.0f * s_t;
        scale[t] = s_t;

        for (int64_t b = 0; b < nblk; ++b) {
            const uint16_t *xb = xr + b * 16;
            float amax_b = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(bf16_value(xb[j]));
                if (a > amax_b)
                    amax_b = a;
            }
            float ratio = amax_b / d;
            uint8_t sb = fme_orc_e4m3_encode(ratio);
            sr[b] = sb;
            double sb_val = fme_orc_e4m3_value(sb);
            if (sb_val == 0.0)
                continue; /* block codes stay 0x0 */
            float e = (float)sb_val * s_t;
            for (int j = 0; j < 16; ++j) {
                float q = bf16_value(xb[j]) / e;
                uint8_t c = fme_orc_e2m1_encode(q);
                int64_t kk = b * 16 + j;
                if (kk % 2 == 0)
                    cr[kk / 2] |= c;
                else
                    cr[kk / 2] |= (uint8_t)(c << 4);
            }
        }
    }
}

void fme_orc_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t k,
                         uint8_t *codes, uint8_t *sf, float *scale) {
    quant_nvfp4_rows(x, rows, k, 0, codes, sf, scale);
}

/*
 * Standard NVFP4, the comparator ("Cursor Composer 2 report deep dive", section
 * 1; report section 6.1: standard NVFP4 has a per-tensor FP32 scale): the steps
 * above with amax_t replaced by the amax of the whole tensor, so S (scale[t]) is
 * the same for every row and a row's codes depend on every other row.
 */
void fme_orc_quant_nvfp4_pertensor(const uint16_t *x, int64_t rows, int64_t k,
                                   uint8_t *codes, uint8_t *sf, float *scale) {
    quant_nvfp4_rows(x, rows, k, 1, codes, sf, scale);
}

/* x_hat = dec_E2M1(q) * dec_E4M3(sb) * S_t, exact in fp64. */
void fme_orc_dequant_nvfp4(const uint8_t *codes, const uint8_t *sf, const float *scale,
                           int64_t rows, int64_t k, double *out) {
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t j = 0; j < k; ++j) {
            uint8_t byte = codes[t * (k / 2) + j / 2];
            uint8_t c = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            double sb = fme_orc_e4m3_value(sf[t * (k / 16) + j / 16]);
            out[t * k + j] = fme_orc_e2m1_value(c) * sb * (double)scale[t];
        }
    }
}

/* ------------------------------------------------------------- MXFP8 ---- */

/* Scale code of one 32-block: code 0 for amax 0, else
 * clamp(floor(log2 amax) - 8 + 127, 0, 254). */
static uint8_t mx_scale_code(float amax) {
    if (amax == 0.0f)
        return 0;
    int e2;
    frexp((double)amax, &e2); /* amax = m * 2^e2, m in [0.5, 1) */
    int u = e2 - 1;          /* floor(log2 amax) */
    int code = u - 8 + 127;
    if (code < 0)
        code = 0;
    if (code > 254)
        code = 254;
    return (uint8_t)code;
}

/* The round-up scale rule (a variant, not the standard's): X = 2^ceil(log2(amax
 * / 448)), the smallest power of two with amax / X <= 448, so no element
 * saturates.  E8M0 code clamped to [0, 254]; an all-zero block gets code 0. */
static uint8_t mx_scale_code_ceil(float amax) {
    if (!(amax > 0.0f))
        return 0;
    int e2;
    const double m = frexp((double)amax / 448.0, &e2); /* amax/448 = m * 2^e2, m in [0.5, 1) */
    const int up = (m == 0.5) ? e2 - 1 : e2;            /* ceil(log2(amax / 448)) */
    const int c = up + 127;
    return (uint8_t)(c < 0 ? 0 : (c > 254 ? 254 : c));
}

/* Quantize one block of n (<= 32) values given as floats; missing values of a
 * short block count as zeros and are not written.  ceil_rule selects the
 * round-up scale instead of the standard one. */
static void mx_block(const float *v, int n, uint8_t *codes_out, int64_t code_stride,
                     uint8_t *scale_out, int ceil_rule) {
    float amax = 0.0f;
    for (int j = 0; j < n; ++j) {
        float a = fabsf(v[j]);
        if (a > amax)
            amax = a;
    }
    uint8_t sc = ceil_rule ? mx_scale_code_ceil(amax) : mx_scale_code(amax);
    *scale_out = sc;
    for (int j = 0; j < n; ++j) {
        double q = ldexp((double)v[j], 127 - (int)sc); /* x / X, exact */
        codes_out[j * code_stride] = fme_orc_e4m3_encode(q);
    }
}

/*
 * Row-wise MXFP8: blocks of 32 along each row of x [rows x cols]
 * (cols a multiple of 32).  codes [rows x cols] E4M3, sf [rows x cols/32]
 * E8M0, logical layouts.
 */
static void quant_mxfp8_rows(const uint16_t *x, int64_t rows, int64_t cols, int ceil_rule,
                             uint8_t *codes, uint8_t *sf) {
    float v[32];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < cols / 32; ++b) {
            for (int j = 0; j < 32; ++j)
                v[j] = bf16_value(x[r * cols + b * 32 + j]);
            mx_block(v, 32, codes + r * cols + b * 32, 1, sf + r * (cols / 32) + b, ceil_rule);
        }
    }
}

/*
 * Column-wise MXFP8 over groups of rows.  Group g holds rows
 * [offsets[g], offsets[g+1]) of x [rows x cols].  Its rows are laid out
 * along the padded position axis p starting at
 *   poff[g] = sum over g' < g of roundup(n_g', 128),
 * padded with zeros up to the next multiple of 128, and every column is cut
 * into blocks of 32 positions starting at poff[g].  Outputs, transposed:
 *   codes_t [cols x ld]   (position axis contiguous),
 *   sf_t    [cols x ld/32],
 *   poff    [num_groups + 1].
 * ld (a multiple of 128, at least poff[num_groups]) is the row length of the
 * outputs; positions from poff[num_groups] to ld are written as zeros.
 */
static void quant_mxfp8_cols(const uint16_t *x, int64_t rows, int64_t cols,
                             const int32_t *offsets, int32_t num_groups, int64_t ld, int ceil_rule,
                             uint8_t *codes_t, uint8_t *sf_t, int32_t *poff) {
    (void)rows;
    float v[32];
    memset(codes_t, 0, (size_t)(cols * ld));
    memset(sf_t, 0, (size_t)(cols * (ld / 32)));
    int64_t p0 = 0;
    for (int32_t g = 0; g < num_groups; ++g) {
        poff[g] = (int32_t)p0;
        int64_t n_g = offsets[g + 1] - offsets[g];
        int64_t padded = ((n_g + 127) / 128) * 128;
        for (int64_t c = 0; c < cols; ++c) {
            for (int64_t pb = 0; pb < padded; pb += 32) {
                for (int j = 0; j < 32; ++j) {
                    int64_t local = pb + j;
                    v[j] = (local < n_g) ? bf16_value(x[(offsets[g] + local) * cols + c]) : 0.0f;
                }
                mx_block(v, 32, codes_t + c * ld + p0 + pb, 1, sf_t + c * (ld / 32) + (p0 + pb) / 32,
                         ceil_rule);
            }
        }
        p0 += padded;
    }
    poff[num_groups] = (int32_t)p0;
}

void fme_orc_quant_mxfp8_rows(const uint16_t *x, int64_t rows, int64_t cols,
                              uint8_t *codes, uint8_t *sf) {
    quant_mxfp8_rows(x, rows, cols, 0, codes, sf);
}

void fme_orc_quant_mxfp8_cols(const uint16_t *x, int64_t rows, int64_t cols,
                              const int32_t *offsets, int32_t num_groups, int64_t ld,
                              uint8_t *codes_t, uint8_t *sf_t, int32_t *poff) {
    quant_mxfp8_cols(x, rows, cols, offsets, num_groups, ld, 0, codes_t, sf_t, poff);
}

/* The same two quantizers with the round-up scale rule. */
void fme_orc_quant_mxfp8_rows_ceil(const uint16_t *x, int64_t rows, int64_t cols,
                                   uint8_t *codes, uint8_t *sf) {
    quant_mxfp8_rows(x, rows, cols, 1, codes, sf);
}

void fme_orc_quant_mxfp8_cols_ceil(const uint16_t *x, int64_t rows, int64_t cols,
                                   const int32_t *offsets, int32_t num_groups, int64_t ld,
                                   uint8_t *codes_t, uint8_t *sf_t, int32_t *poff) {
    quant_mxfp8_cols(x, rows, cols, offsets, num_groups, ld, 1, codes_t, sf_t, poff);
}

/* x_hat = dec_E4M3(q) * 2^(scale - 127) for blocks of 32 along each row of a
 * [rows x cols] code matrix (cols a multiple of 32). */
void fme_orc_dequant_mxfp8(const uint8_t *codes, const uint8_t *sf, int64_t rows, int64_t cols,
                           double *out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j)
            out[r * cols + j] = fme_orc_e4m3_value(codes[r * cols + j]) *
                                fme_orc_e8m0_value(sf[r * (cols / 32) + j / 32]);
}

/* ---------------------------------------------------------------- GEMM -- */

/* y [m x n] = a [m x k] * b [n x k]^T, summed in fp64 in order of k. */
void fme_orc_gemm_abt(const double *a, const double *b, int64_t m, int64_t n, int64_t k,
                      double *y) {
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t q = 0; q < k; ++q)
                acc += a[i * k + q] * b[j * k + q];
            y[i * n + j] = acc;
        }
    }
}

/* -------------------------------------------------------------- SwiGLU -- */

/* h [rows x inter] = silu(g) * u in fp64, where row t of y_gu [rows x 2 inter]
 * (bf16) is [g_t (inter values) | u_t (inter values)] and silu(v) = v / (1 + e^-v). */
void fme_orc_swiglu(const uint16_t *y_gu, int64_t rows, int64_t inter, double *h) {
    for (int64_t t = 0; t < rows; ++t) {
        const uint16_t *row = y_gu + t * 2 * inter;
        for (int64_t j = 0; j < inter; ++j) {
            const double g = (double)bf16_value(row[j]);
            const double u = (double)bf16_value(row[inter + j]);
            h[t * inter + j] = g / (1.0 + exp(-g)) * u;
        }
    }
}

/* The same activation on fp64 rows [g | u] (the gate/up GEMM's exact outputs,
 * not rounded to bf16): h [rows x inter] = silu(g) * u in fp64. */
void fme_orc_swiglu_f64(const double *y_gu, int64_t rows, int64_t inter, double *h) {
    for (int64_t t = 0; t < rows; ++t) {
        const double *row = y_gu + t * 2 * inter;
        for (int64_t j = 0; j < inter; ++j) {
            const double g = row[j];
            const double u = row[inter + j];
            const double silu = g / (1.0 + exp(-g));
            h[t * inter + j] = silu * u;
        }
    }
}

/* d(gate/up) [rows x 2 inter] of h = silu(g) * u for the upstream gradient dh
 * [rows x inter] (bf16), in fp64: with s = 1 / (1 + e^-g) (the logistic function),
 * dh/dg = dh * u * (s + g * s * (1 - s)) and dh/du = dh * g * s; row t of the
 * result is [dg_t | du_t]. */
void fme_orc_swiglu_bwd(const uint16_t *y_gu, const uint16_t *dh, int64_t rows, int64_t inter, double *d_gu) {
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t j = 0; j < inter; ++j) {
            const double g = (double)bf16_value(y_gu[t * 2 * inter + j]);
            const double u = (double)bf16_value(y_gu[t * 2 * inter + inter + j]);
            const double d = (double)bf16_value(dh[t * inter + j]);
            const double s = 1.0 / (1.0 + exp(-g));
            d_gu[t * 2 * inter + j] = d * u * (s + g * s * (1.0 - s));
            d_gu[t * 2 * inter + inter + j] = d * g * s;
        }
    }
}

/* ------------------------------------------------------------- routing -- */

/* Stable grouping of the n assignments by expert id: offsets[e] is the number of
 * assignments to experts below e, and the assignments to expert e take grouped
 * rows offsets[e], offsets[e] + 1, ... in increasing order of a.  row_of[a] is
 * the grouped row of assignment a (-1 for an id outside [0, E)), src_row[r] the
 * assignment at grouped row r. */
void fme_orc_route(const int32_t *ids, int64_t n, int32_t num_experts, int32_t *offsets, int32_t *row_of,
                   int32_t *src_row) {
    for (int32_t e = 0; e <= num_experts; ++e)
        offsets[e] = 0;
    for (int64_t a = 0; a < n; ++a)
        if (ids[a] >= 0 && ids[a] < num_experts)
            offsets[ids[a] + 1] += 1;
    for (int32_t e = 0; e < num_experts; ++e)
        offsets[e + 1] += offsets[e];
    for (int32_t e = 0; e < num_experts; ++e) {
        int32_t next = offsets[e];
        for (int64_t a = 0; a < n; ++a) {
            if (ids[a] == e) {
                row_of[a] = next;
                src_row[next] = (int32_t)a;
                next += 1;
            }
        }
    }
    for (int64_t a = 0; a < n; ++a)
        if (ids[a] < 0 || ids[a] >= num_experts)
            row_of[a] = -1;
}

/* binary32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t bf16_round(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1;
    return (uint16_t)upper;
}

/* out[t, j] = bf16(acc), acc = 0 then acc = acc + w[t, k] * y[row_of[t, k], j]
 * for k = 0 .. top_k-1 in order, each * and + one binary32 operation; entries
 * with row_of < 0 are skipped. */
void fme_orc_combine(const uint16_t *y, const int32_t *row_of, const float *w, int64_t tokens, int32_t top_k,
                     int64_t n, uint16_t *out) {
    for (int64_t t = 0; t < tokens; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            float acc = 0.0f;
            for (int32_t k = 0; k < top_k; ++k) {
                const int32_t r = row_of[t * top_k + k];
                if (r < 0)
                    continue;
                const float prod = w[t * top_k + k] * bf16_value(y[(int64_t)r * n + j]);
                acc = acc + prod;
            }
            out[t * n + j] = bf16_round(acc);
        }
    }
}

/* ------------------------------------------------- array conveniences -- */

void fme_orc_e2m1_encode_array(const double *v, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = fme_orc_e2m1_encode(v[i]);
}

void fme_orc_e4m3_encode_array(const double *v, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = fme_orc_e4m3_encode(v[i]);
}
