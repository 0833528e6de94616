/*
 * oracle.c -- plain, slow CPU oracle for FP8 / MXFP8 quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include,
 * link or call this file; only the tests, the smoke check and the CPU
 * baseline of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Every function follows one passage of the source pages:
 *   "混合精度与 FP8 训练" (hs-black.github.io), sections 2.1-2.3 (float
 *     fields, BF16, E4M3/E5M2), 3 (binades), 4.1 (round-to-nearest-even),
 *     8.1 (why FP8 needs a scale, saturation), 8.2 (delayed vs current
 *     scaling, TE's (F8max/amax)/2^margin), 13.1 (MX blocks, E8M0).
 *   "HiFloat8：高性能训练之路" (hifloat.gccorg.com), section 1.2
 *     (eqs. 1-4: Scale = F8max/Amax, delayed Scale with 2^-N), section 2
 *     (MXFP8 1x32 blocks, rowwise and columnwise copies).
 *   "Blackwell GPU MXFP8 预训练最佳实践" (51cto.com), section 4.1 (the
 *     round-up E8M0 rule, amax = 0 gives X = -127, saturating RN cast),
 *     section 4.2 (two copies per tensor, one per reduction axis).
 *
 * Arithmetic is done in double wherever a value is compared or scaled, so
 * every comparison below is exact.  Where the definition fixes an FP32
 * intermediate (the per-tensor scale and the product x*scale), the exact
 * double result is rounded once to float; for one multiply or one divide of
 * two floats, rounding the double result to float gives the correctly
 * rounded float result (53 >= 2*24 + 2), so this is IEEE single arithmetic.
 *
 * Readings where the pages are silent:
 *   - any NaN input encodes to byte 0x7F in both formats;
 *   - +-Inf saturates to +-max like any other overflow;
 *   - the sign of zero is kept (0x80), except in an all-zero MX block;
 *   - amax is the largest |x| compared on the magnitude bits, so a NaN
 *     input makes amax NaN (largest payload wins);
 *   - an MX block whose amax is Inf or NaN gets scale byte 0xFF and all
 *     elements 0x7F;
 *   - per-tensor: amax = 0 gives scale 1, a non-finite amax gives scale 1
 *     and raises the non-finite flag, and an overflowing F8max/amax gives
 *     FLT_MAX;
 *   - dequantization: a per-tensor product value * scale_inv is rounded to
 *     FP32 first and then to the output type; an MX product value * 2^X is
 *     exact in FP32 except for overflow to Inf; BF16 output rounds to
 *     nearest, ties to even; every NaN result is the canonical quiet NaN
 *     (BF16 0x7FC0, FP32 0x7FC00000);
 *   - blockwise groups use the current-scaling scale of the group (the
 *     per-tensor special cases included); power-of-two scales round it
 *     down to the largest power of two not above it;
 *   - NVFP4: tensor scale S = fl32(448 * 6 / amax); block scale code
 *     RNE_sat_E4M3(fl32(amax_b * fl32(S / 6))); elements
 *     RNE_sat_E2M1(fl32(x * fl32(S / d))) with d the block scale's value
 *     (all zero when d = 0); a NaN element encodes as the largest code 0x7;
 *     two codes per byte, the even element in the low nibble;
 *   - quantization statistics: SQNR = 10 log10(sum x^2 / sum (x - xh)^2)
 *     with xh the FP32 value the code stands for, both sums over the
 *     elements where x and xh are finite (the rest counted apart); the
 *     zero-rate counts elements with xh = 0 and x != 0 (values that
 *     quantization flushed), next to the plain count of xh = 0;
 *   - MXFP6 elements are the OCP microscaling formats E2M3 (bias 1,
 *     largest 7.5) and E3M2 (bias 3, largest 28) -- the pages name MXFP6
 *     without defining them, so these two are parity unpinned by the
 *     pages (pinned by a binade-by-binade construction only); MXFP4 /
 *     MXFP6 blocks take destmax = the element format's largest value under
 *     the round-up rule and its exponent as e_max under the OCP rule; a
 *     non-finite block gets scale 0xFF and +0 codes (the formats have no
 *     NaN); E2M1 codes are stored two per byte (even element low), FP6
 *     codes one per byte (bits 0-5);
 *   - the block-scale layout for tensor-core MMA is NVIDIA's public
 *     128 x 4 block layout (the pages give none): parity unpinned.
 * Those readings are pinned only by their own definition ("parity unpinned"
 * by the pages); everything else is pinned by page values, closed forms and
 * library routines in tests/test_oracle_pins.py.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_E4M3 0
#define ORC_E5M2 1
#define ORC_E2M1 2
#define ORC_E2M3 3
#define ORC_E3M2 4
#define ORC_BF16 0
#define ORC_FP32 1

/* ------------------------------------------------------------------ */
/* 8-bit float formats ("混合精度与 FP8 训练" 2.1-2.2).                   */
/* E4M3: 4 exponent bits, bias 7, 3 mantissa bits, no infinities, a   */
/* single NaN pattern S.1111.111, so the top binade holds 256..448.   */
/* E5M2: IEEE style, 5 exponent bits, bias 15, 2 mantissa bits,       */
/* exponent field 31 is Inf (mantissa 0) or NaN.                      */
/* ------------------------------------------------------------------ */
static int exp_bits(int fmt) { return fmt == ORC_E4M3 ? 4 : 5; }
static int man_bits(int fmt) { return fmt == ORC_E4M3 ? 3 : 2; }
static int bias_of(int fmt) { return fmt == ORC_E4M3 ? 7 : 15; }

/* Value of an 8-bit code, straight from the field definition. */
static double code_value_def(int fmt, unsigned code)
{
    unsigned sign = (code >> 7) & 1u;
    unsigned ebits = (code >> man_bits(fmt)) & ((1u << exp_bits(fmt)) - 1u);
    unsigned mbits = code & ((1u << man_bits(fmt)) - 1u);
    unsigned emax_field = (1u << exp_bits(fmt)) - 1u;
    double mag;
    if (fmt == ORC_E4M3 && ebits == emax_field && mbits == 7u) return NAN;
    if (fmt == ORC_E5M2 && ebits == emax_field)
        return mbits ? NAN : (sign ? -INFINITY : INFINITY);
    if (ebits == 0) /* subnormal: 0.m * 2^(1-bias) */
        mag = ldexp((double)mbits, 1 - bias_of(fmt) - man_bits(fmt));
    else            /* normal: 1.m * 2^(e-bias) */
        mag = ldexp((double)((1u << man_bits(fmt)) | mbits),
                    (int)ebits - bias_of(fmt) - man_bits(fmt));
    return sign ? -mag : mag;
}

/* The definition above, tabulated once for all 256 codes of both formats
 * when the library is loaded (a cache, not a second definition). */
static double code_table[2][256];
static unsigned max_code_table[2];

__attribute__((constructor)) static void build_code_tables(void)
{
    for (int fmt = 0; fmt < 2; fmt++) {
        unsigned c;
        for (c = 0; c < 256u; c++) code_table[fmt][c] = code_value_def(fmt, c);
        c = 0x7F;
        while (!isfinite(code_table[fmt][c])) c--;
        max_code_table[fmt] = c;
    }
}

double orc_fp8_value(int fmt, unsigned code) { return code_table[fmt][code & 0xFFu]; }

/* Largest non-negative finite code: E4M3 0x7E (448), E5M2 0x7B (57344). */
unsigned orc_fp8_max_code(int fmt) { return max_code_table[fmt]; }

double orc_fp8_max(int fmt) { return orc_fp8_value(fmt, orc_fp8_max_code(fmt)); }

/*
 * Saturating round-to-nearest-even of an exact real value a
 * ("混合精度与 FP8 训练" 4.1 for RNE, 8.1 for saturation instead of
 * overflow; "Blackwell GPU MXFP8 预训练最佳实践" 4.1 for the saturating
 * RN cast).  Encoding is a search over the list of codes in value order,
 * not bit manipulation: the nearest representable value wins, and on an
 * exact tie the code whose last mantissa bit is 0 wins.
 */
unsigned orc_fp8_encode(int fmt, double a)
{
    unsigned maxc = orc_fp8_max_code(fmt);
    unsigned sign, lo, hi, c;
    double m, vlo, vhi, dlo, dhi;
    if (isnan(a)) return 0x7Fu;
    sign = signbit(a) ? 0x80u : 0u;
    m = fabs(a);
    if (m >= orc_fp8_value(fmt, maxc)) return sign | maxc; /* saturate (also Inf) */
    /* largest code lo with value(lo) <= m (values grow with the code) */
    lo = 0;
    hi = maxc; /* invariant: value(lo) <= m < value(hi) */
    while (hi - lo > 1u) {
        unsigned mid = (lo + hi) / 2u;
        if (orc_fp8_value(fmt, mid) <= m) lo = mid; else hi = mid;
    }
    vlo = orc_fp8_value(fmt, lo);
    vhi = orc_fp8_value(fmt, hi);
    dlo = m - vlo;
    dhi = vhi - m;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo & 1u) ? hi : lo; /* tie: even code */
    return sign | c;
}

/* ------------------------------------------------------------------ */
/* Input decode: BF16 is FP32 with the low 16 bits removed            */
/* ("混合精度与 FP8 训练" 2.2), so widening appends 16 zero bits.         */
/* ------------------------------------------------------------------ */
static uint32_t input_bits(const void* x, int dt, int64_t i)
{
    if (dt == ORC_BF16) return ((uint32_t)((const uint16_t*)x)[i]) << 16;
    return ((const uint32_t*)x)[i];
}

static float bits_to_float(uint32_t b)
{
    float f;
    memcpy(&f, &b, 4);
    return f;
}

static uint32_t float_to_bits(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    return b;
}

float orc_input_value(const void* x, int dt, int64_t i) { return bits_to_float(input_bits(x, dt, i)); }

/* IEEE single rounding (to nearest, ties to even) of an exact double.  C
 * leaves the conversion of an out-of-range double undefined, so overflow is
 * spelled out: at or beyond FLT_MAX + half an ulp the result is infinite. */
static float to_float(double d)
{
    const double overflow = 0x1.ffffffp127; /* FLT_MAX + 2^103 */
    if (d >= overflow) return INFINITY;
    if (d <= -overflow) return -INFINITY;
    return (float)d;
}

/* ------------------------------------------------------------------ */
/* amax = max |x_i| ("HiFloat8：高性能训练之路" 1.2 ComputeAmax;          */
/* "混合精度与 FP8 训练" 8.1).  Compared on the magnitude bits, which     */
/* orders finite values by |x| and puts NaN above Inf.                */
/* Returned as FP32 bits.                                             */
/* ------------------------------------------------------------------ */
uint32_t orc_amax_bits(const void* x, int dt, int64_t begin, int64_t end)
{
    uint32_t best = 0;
    for (int64_t i = begin; i < end; i++) {
        uint32_t mag = input_bits(x, dt, i) & 0x7FFFFFFFu;
        if (mag > best) best = mag;
    }
    return best;
}

/* ------------------------------------------------------------------ */
/* Per-tensor scale.  Current scaling: Scale = F8max / Amax (eq. 1 of */
/* "HiFloat8：高性能训练之路" 1.2); delayed scaling multiplies by 2^-N    */
/* (eqs. 3-4 there; TE's (F8max/amax)/2^margin in "混合精度与 FP8 训练"  */
/* 8.2).  FP32 arithmetic: the quotient is rounded to float, then the */
/* power-of-two factor applied and rounded again.                     */
/* ------------------------------------------------------------------ */
float orc_per_tensor_scale(uint32_t amax_bits, int fmt, int margin, int* nonfinite)
{
    float amax = bits_to_float(amax_bits);
    float s;
    if (nonfinite) *nonfinite = 0;
    if (!isfinite(amax)) {
        if (nonfinite) *nonfinite = 1;
        return 1.0f;
    }
    if (amax == 0.0f) return 1.0f;
    s = to_float(orc_fp8_max(fmt) / (double)amax);
    if (isinf(s)) s = FLT_MAX;
    s = to_float((double)s * ldexp(1.0, -margin));
    return s;
}

float orc_reciprocal(float s) { return to_float(1.0 / (double)s); }

/* ------------------------------------------------------------------ */
/* Scaled cast (eq. 2 of "HiFloat8：高性能训练之路" 1.2): q_i =           */
/* RNE_sat(fl32(x_i * scale)).  sat counts elements whose scaled       */
/* magnitude exceeds F8max (NaN excluded).                             */
/* ------------------------------------------------------------------ */
void orc_cast(const void* x, int dt, int64_t begin, int64_t end, float scale, int fmt,
              uint8_t* q, uint64_t* sat, int nthreads)
{
    double f8max = orc_fp8_max(fmt);
    uint64_t count = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) reduction(+ : count) num_threads(nthreads)
#endif
    for (int64_t i = begin; i < end; i++) {
        float y = to_float((double)orc_input_value(x, dt, i) * (double)scale);
        if (!isnan(y) && fabs((double)y) > f8max) count++;
        q[i] = (uint8_t)orc_fp8_encode(fmt, (double)y);
    }
    if (sat) *sat = count;
}

/* ------------------------------------------------------------------ */
/* MX block ("Blackwell GPU MXFP8 预训练最佳实践" 4.1; "混合精度与 FP8     */
/* 训练" 13.1).  X = ceil(log2(amax / destmax)) computed exactly: the   */
/* smallest integer X with amax <= destmax * 2^X, saturated to the     */
/* UE8M0 range [-127, 127]; the stored byte is X + 127.  amax = 0 gives */
/* X = -127 and all elements 0.  Each element is RNE_sat(v / 2^X).     */
/* ------------------------------------------------------------------ */
uint8_t orc_mx_block(const float* v, int k, int fmt, uint8_t* q)
{
    uint32_t amax = 0;
    double destmax = orc_fp8_max(fmt);
    int X, i;
    for (i = 0; i < k; i++) {
        uint32_t mag = float_to_bits(v[i]) & 0x7FFFFFFFu;
        if (mag > amax) amax = mag;
    }
    if (amax >= 0x7F800000u) { /* Inf or NaN in the block */
        for (i = 0; i < k; i++) q[i] = 0x7F;
        return 0xFF;
    }
    if (amax == 0) {
        for (i = 0; i < k; i++) q[i] = 0x00;
        return 0x00; /* X = -127 */
    }
    for (X = -127; X < 127; X++)
        if ((double)bits_to_float(amax) <= ldexp(destmax, X)) break;
    for (i = 0; i < k; i++) q[i] = (uint8_t)orc_fp8_encode(fmt, ldexp((double)v[i], -X));
    return (uint8_t)(X + 127);
}

/*
 * The same block under a choice of scale rule, with a saturation count.
 * rule 0: the round-up rule above.  rule 1: the OCP rule ("混合精度与 FP8
 * 训练" 13.1; "Blackwell GPU MXFP8 预训练最佳实践" 4.1, its formula read as
 * floor(log2 amax) - floor(log2 448)): X = floor(log2 amax) - e_max, e_max
 * the exponent of the element format's largest value (8 for E4M3, 15 for
 * E5M2), i.e. the largest integer X with 2^(X + e_max) <= amax, saturated to
 * [-127, 127].  Elements are RNE_sat(v / 2^X) either way; *sat counts those
 * whose scaled magnitude exceeds the format's maximum (the ones the
 * conversion clamps; never under rule 0).
 */
uint8_t orc_mx_block_rule(const float* v, int k, int fmt, int rule, uint8_t* q, int64_t* sat)
{
    uint32_t amax = 0;
    double destmax = orc_fp8_max(fmt);
    int emax = (int)floor(log2(destmax));
    int X, i;
    *sat = 0;
    if (rule == 0) {
        uint8_t b = orc_mx_block(v, k, fmt, q);
        if (b == 0xFF || b == 0) return b;
        for (i = 0; i < k; i++)
            if (fabs(ldexp((double)v[i], -((int)b - 127))) > destmax) (*sat)++;
        return b;
    }
    for (i = 0; i < k; i++) {
        uint32_t mag = float_to_bits(v[i]) & 0x7FFFFFFFu;
        if (mag > amax) amax = mag;
    }
    if (amax >= 0x7F800000u) {
        for (i = 0; i < k; i++) q[i] = 0x7F;
        return 0xFF;
    }
    if (amax == 0) {
        for (i = 0; i < k; i++) q[i] = 0x00;
        return 0x00;
    }
    for (X = 127; X > -127; X--)
        if (ldexp(1.0, X + emax) <= (double)bits_to_float(amax)) break;
    for (i = 0; i < k; i++) {
        double s = ldexp((double)v[i], -X);
        if (fabs(s) > destmax) (*sat)++;
        q[i] = (uint8_t)orc_fp8_encode(fmt, s);
    }
    return (uint8_t)(X + 127);
}

/* Group g covers rows [offs[g], offs[g+1]); offs == NULL means one group. */
static int64_t grp_off(const int64_t* offs, int G, int64_t rows, int g)
{
    if (!offs) return g == 0 ? 0 : rows;
    (void)G;
    return offs[g];
}

/* Number of columnwise blocks: sum over groups of ceil(n_g / 32). */
int64_t orc_mx_col_blocks(const int64_t* offs, int G, int64_t rows)
{
    int64_t t = 0;
    int g, ng = offs ? G : 1;
    for (g = 0; g < ng; g++) {
        int64_t n = grp_off(offs, ng, rows, g + 1) - grp_off(offs, ng, rows, g);
        t += (n + 31) / 32;
    }
    return t;
}

/*
 * MX quantization of a rows x cols tensor, rowwise and/or columnwise
 * ("HiFloat8：高性能训练之路" 2 and "Blackwell GPU MXFP8 预训练最佳实践"
 * 4.2: one copy per reduction axis, both from the high-precision tensor;
 * "混合精度与 FP8 训练" 13.1: MX does not commute with transposition).
 *   rowwise:    blocks x[r, 32j .. 32j+31] -> q_row[r*cols + c],
 *               s_row[r*(cols/32) + j]
 *   columnwise: per group, blocks of 32 consecutive rows starting at the
 *               group's first row (the last one may be shorter) ->
 *               q_col[c*rows + r] (the transpose), s_col[c*s_col_ld + b],
 *               b counting blocks over all groups in order.
 * dir: 1 rowwise, 2 columnwise, 3 both.
 */
void orc_mx_quantize(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* offs,
                     int G, int fmt, int dir, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                     uint8_t* s_col, int64_t s_col_ld, int nthreads)
{
    int ng = offs ? G : 1;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#endif
    if (dir & 1) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int64_t r = 0; r < rows; r++) {
            float v[32];
            for (int64_t j = 0; j < cols / 32; j++) {
                for (int i = 0; i < 32; i++) v[i] = orc_input_value(x, dt, r * cols + j * 32 + i);
                s_row[r * (cols / 32) + j] = orc_mx_block(v, 32, fmt, q_row + r * cols + j * 32);
            }
        }
    }
    if (dir & 2) {
        int64_t base = 0;
        for (int g = 0; g < ng; g++) {
            int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
            int64_t nb = (r1 - r0 + 31) / 32;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
            for (int64_t c = 0; c < cols; c++) {
                float v[32];
                uint8_t qb[32];
                for (int64_t b = 0; b < nb; b++) {
                    int64_t rs = r0 + 32 * b;
                    int k = (int)((r1 - rs) < 32 ? (r1 - rs) : 32);
                    for (int i = 0; i < k; i++) v[i] = orc_input_value(x, dt, (rs + i) * cols + c);
                    s_col[c * s_col_ld + base + b] = orc_mx_block(v, k, fmt, qb);
                    for (int i = 0; i < k; i++) q_col[c * rows + rs + i] = qb[i];
                }
            }
            base += nb;
        }
    }
}

/* orc_mx_quantize under a scale rule (see orc_mx_block_rule), also
 * returning the saturated-element counts of the rowwise (sat[0]) and
 * columnwise (sat[1]) copies. */
void orc_mx_quantize_rule(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* offs, int G,
                          int fmt, int dir, int rule, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                          uint8_t* s_col, int64_t s_col_ld, int64_t* sat, int nthreads)
{
    int ng = offs ? G : 1;
    int64_t sat_r = 0, sat_c = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#endif
    if (dir & 1) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads) reduction(+ : sat_r)
#endif
        for (int64_t r = 0; r < rows; r++) {
            float v[32];
            for (int64_t j = 0; j < cols / 32; j++) {
                int64_t n = 0;
                for (int i = 0; i < 32; i++) v[i] = orc_input_value(x, dt, r * cols + j * 32 + i);
                s_row[r * (cols / 32) + j] = orc_mx_block_rule(v, 32, fmt, rule, q_row + r * cols + j * 32, &n);
                sat_r += n;
            }
        }
    }
    if (dir & 2) {
        int64_t base = 0;
        for (int g = 0; g < ng; g++) {
            int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
            int64_t nb = (r1 - r0 + 31) / 32;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads) reduction(+ : sat_c)
#endif
            for (int64_t c = 0; c < cols; c++) {
                float v[32];
                uint8_t qb[32];
                for (int64_t b = 0; b < nb; b++) {
                    int64_t rs = r0 + 32 * b, n = 0;
                    int k = (int)((r1 - rs) < 32 ? (r1 - rs) : 32);
                    for (int i = 0; i < k; i++) v[i] = orc_input_value(x, dt, (rs + i) * cols + c);
                    s_col[c * s_col_ld + base + b] = orc_mx_block_rule(v, k, fmt, rule, qb, &n);
                    sat_c += n;
                    for (int i = 0; i < k; i++) q_col[c * rows + rs + i] = qb[i];
                }
            }
            base += nb;
        }
    }
    sat[0] = sat_r;
    sat[1] = sat_c;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Array form of orc_fp8_encode, for the tests' sweeps. */
void orc_encode_array(int fmt, const double* a, int64_t n, uint8_t* q, int nthreads)
{
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < n; i++) q[i] = (uint8_t)orc_fp8_encode(fmt, a[i]);
}

/* Encode every FP32 bit pattern in [first, first + n) with scale 1; used by
 * the exhaustive FP32 sweep (q[i] is the code of the pattern first + i). */
void orc_encode_f32_range(int fmt, uint64_t first, int64_t n, uint8_t* q, int nthreads)
{
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < n; i++)
        q[i] = (uint8_t)orc_fp8_encode(fmt, (double)bits_to_float((uint32_t)(first + (uint64_t)i)));
}

/* ------------------------------------------------------------------ */
/* Dequantization: the inverse step that de-scales an FP8 value for   */
/* use in higher precision ("HiFloat8：高性能训练之路" 1.1-1.2: the     */
/* matmul result is multiplied back by scale_inv = 1/Scale;           */
/* "Blackwell GPU MXFP8 预训练最佳实践" 4.3: without MX hardware the     */
/* blocks are dequantized and a BF16 matmul runs).                    */
/* ------------------------------------------------------------------ */

/* Nearest BF16 (ties to the even code) of a float, from the values of   */
/* the two BF16 neighbours: BF16 keeps FP32's sign and exponent and the */
/* top 7 fraction bits ("混合精度与 FP8 训练" 2.2).  Magnitudes at or    */
/* beyond the midpoint above the largest finite BF16 round to Inf (IEEE */
/* rounding with an unbounded exponent).  NaN -> 0x7FC0.                */
uint16_t orc_bf16_round(float f)
{
    uint32_t b = float_to_bits(f);
    uint32_t sign = b & 0x80000000u, mag = b & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0x7FC0;                  /* NaN */
    if (mag == 0x7F800000u) return (uint16_t)((sign | mag) >> 16);
    uint32_t lo = mag & 0xFFFF0000u;                       /* toward zero */
    if (lo == mag) return (uint16_t)((sign | mag) >> 16);  /* exact */
    uint32_t hi = lo + 0x10000u;                           /* next away from zero */
    double v = (double)bits_to_float(mag);
    double vlo = (double)bits_to_float(lo);
    double vhi = hi == 0x7F800000u ? ldexp(1.0, 128) : (double)bits_to_float(hi);
    uint32_t pick;
    if (v - vlo < vhi - v) pick = lo;
    else if (v - vlo > vhi - v) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;               /* tie: even code */
    return (uint16_t)((sign | pick) >> 16);
}

/* One dequantized value in the output type (out_dt: 0 BF16, 1 FP32):    */
/* v is the exact real result, rounded once to float, then to BF16.      */
static void put_out(void* y, int out_dt, int64_t i, double v)
{
    float f = isnan(v) ? bits_to_float(0x7FC00000u) : to_float(v);
    if (out_dt == 0) ((uint16_t*)y)[i] = orc_bf16_round(f);
    else ((uint32_t*)y)[i] = isnan(f) ? 0x7FC00000u : float_to_bits(f);
}

/* Per-tensor (per-group) dequantization of a rows x cols code array:    */
/* y = fl32(value(q) * scale_inv[g]) for the rows of group g, then the   */
/* output rounding above.  value(q) * scale_inv is exact in double.     */
void orc_dequant_per_tensor(const uint8_t* q, int64_t rows, int64_t cols, const int64_t* offs, int G,
                            int fmt, const float* scale_inv, int out_dt, void* y, int nthreads)
{
    int ng = offs ? G : 1;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#endif
    for (int g = 0; g < ng; g++) {
        int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
        double si = (double)scale_inv[g];
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int64_t i = r0 * cols; i < r1 * cols; i++)
            put_out(y, out_dt, i, orc_fp8_value(fmt, q[i]) * si);
    }
}

/* MX dequantization ("Blackwell GPU MXFP8 预训练最佳实践" 4.1: element   */
/* value times 2^X, X = byte - 127; byte 0xFF is NaN).  dir 1: rowwise   */
/* copy, q [rows][cols], s [rows][cols/32], y [rows][cols].  dir 2:      */
/* columnwise copy, q [cols][rows], s [cols][s_ld] with blocks counted   */
/* over the groups in order, y [cols][rows] (the copy's own layout).     */
void orc_mx_dequantize(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, const int64_t* offs,
                       int G, int fmt, int dir, int64_t s_ld, int out_dt, void* y, int nthreads)
{
    int ng = offs ? G : 1;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#endif
    if (dir == 1) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int64_t r = 0; r < rows; r++)
            for (int64_t c = 0; c < cols; c++) {
                unsigned byte = s[r * (cols / 32) + c / 32];
                double v = byte == 0xFFu ? NAN : ldexp(orc_fp8_value(fmt, q[r * cols + c]), (int)byte - 127);
                put_out(y, out_dt, r * cols + c, v);
            }
        return;
    }
    int64_t base = 0;
    for (int g = 0; g < ng; g++) {
        int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int64_t c = 0; c < cols; c++)
            for (int64_t r = r0; r < r1; r++) {
                unsigned byte = s[c * s_ld + base + (r - r0) / 32];
                double v = byte == 0xFFu ? NAN : ldexp(orc_fp8_value(fmt, q[c * rows + r]), (int)byte - 127);
                put_out(y, out_dt, c * rows + r, v);
            }
        base += (r1 - r0 + 31) / 32;
    }
}

/* Array form of orc_bf16_round, for the tests' sweeps. */
void orc_bf16_round_array(const float* f, int64_t n, uint16_t* out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < n; i++) out[i] = orc_bf16_round(f[i]);
}

/* ------------------------------------------------------------------ */
/* Blockwise FP8 ("混合精度与 FP8 训练" 10.2-10.5): one FP32 scale per    */
/* group of gr rows x gc columns -- 1x128 for activations (128 channels */
/* of one token), 128x128 for weights, 128x1 for the transposed copy of */
/* an activation.  The scale is the current-scaling scale of the group  */
/* (Scale = F8max / amax, eq. 1 of "HiFloat8：高性能训练之路" 1.2, taken  */
/* online per group, 10.3), optionally rounded down to a power of two   */
/* (10.4: scales that are integer powers of 2).                         */
/* q = RNE_sat(fl32(x * scale)); the stored scale is scale_inv =        */
/* fl32(1 / scale), one per group, row-major over the group grid        */
/* [ceil(rows / gr)][ceil(cols / gc)].  Codes keep x's layout.          */
/* ------------------------------------------------------------------ */
float orc_pow2_floor(float s)
{
    int e;
    double m = frexp((double)s, &e); /* s = m * 2^e, m in [0.5, 1) */
    (void)m;
    return to_float(ldexp(1.0, e - 1));
}

void orc_blockwise(const void* x, int dt, int64_t rows, int64_t cols, int fmt, int gr, int gc, int pow2,
                   uint8_t* q, float* scale_inv, int nthreads)
{
    int64_t nbr = (rows + gr - 1) / gr, nbc = (cols + gc - 1) / gc;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t b = 0; b < nbr * nbc; b++) {
        int64_t br = b / nbc, bc = b % nbc;
        int64_t r0 = br * gr, r1 = r0 + gr < rows ? r0 + gr : rows;
        int64_t c0 = bc * gc, c1 = c0 + gc < cols ? c0 + gc : cols;
        uint32_t amax = 0;
        for (int64_t r = r0; r < r1; r++)
            for (int64_t c = c0; c < c1; c++) {
                uint32_t mag = input_bits(x, dt, r * cols + c) & 0x7FFFFFFFu;
                if (mag > amax) amax = mag;
            }
        int nf;
        float s = orc_per_tensor_scale(amax, fmt, 0, &nf);
        if (pow2) s = orc_pow2_floor(s);
        for (int64_t r = r0; r < r1; r++)
            for (int64_t c = c0; c < c1; c++) {
                double v = (double)orc_input_value(x, dt, r * cols + c);
                q[r * cols + c] = (uint8_t)orc_fp8_encode(fmt, (double)to_float(v * (double)s));
            }
        scale_inv[b] = orc_reciprocal(s);
    }
}

/* ------------------------------------------------------------------ */
/* NVFP4 ("混合精度与 FP8 训练" 13.2): E2M1 elements (1 sign, 2 exponent  */
/* bits with bias 1, 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6), one    */
/* E4M3 scale per 16 elements, and one FP32 scale for the tensor (the    */
/* second level, because E4M3 alone lacks the range).                    */
/* ------------------------------------------------------------------ */
double orc_e2m1_value(unsigned code)
{
    unsigned sign = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - 1);
    return sign ? -mag : mag;
}

/* Nearest E2M1 code (ties to the even code), saturating at 6; a NaN
 * encodes as the largest code 0x7. */
unsigned orc_e2m1_encode(double a)
{
    if (isnan(a)) return 0x7u;
    unsigned sign = signbit(a) ? 0x8u : 0u;
    double m = fabs(a);
    if (m >= 6.0) return sign | 0x7u;
    unsigned lo = 0;
    while (lo < 7u && orc_e2m1_value(lo + 1) <= m) lo++;
    if (orc_e2m1_value(lo) == m || lo == 7u) return sign | lo;
    double dl = m - orc_e2m1_value(lo), dh = orc_e2m1_value(lo + 1) - m;
    unsigned c = dl < dh ? lo : dh < dl ? lo + 1 : ((lo & 1u) ? lo + 1 : lo);
    return sign | c;
}

/* The tensor-level scale S = fl32(448 * 6 / amax) (the E4M3 maximum times
 * the E2M1 maximum over the tensor's amax), with the per-tensor special
 * cases: amax 0 or non-finite -> 1, a quotient above FLT_MAX -> FLT_MAX. */
float orc_nvfp4_tensor_scale(uint32_t amax_bits)
{
    if (amax_bits == 0 || amax_bits >= 0x7F800000u) return 1.0f;
    double q = 448.0 * 6.0 / (double)bits_to_float(amax_bits);
    float s = to_float(q);
    return isinf(s) ? FLT_MAX : s;
}

/* One block of k <= 16 values under tensor scale S: block scale code
 * RNE_sat_E4M3(fl32(amax_b * fl32(S / 6))), its value d; elements
 * RNE_sat_E2M1(fl32(x * fl32(S / d))), or all +0 when d = 0.  Returns the
 * scale code. */
uint8_t orc_nvfp4_block(const float* v, int k, float S, uint8_t* q)
{
    uint32_t amax = 0;
    for (int i = 0; i < k; i++) {
        uint32_t mag = float_to_bits(v[i]) & 0x7FFFFFFFu;
        if (mag > amax) amax = mag;
    }
    float t = to_float((double)S / 6.0);
    float sval = to_float((double)bits_to_float(amax) * (double)t);
    uint8_t code = (uint8_t)orc_fp8_encode(ORC_E4M3, (double)sval);
    double d = orc_fp8_value(ORC_E4M3, code);
    if (d == 0.0 || isnan(d)) {
        for (int i = 0; i < k; i++) q[i] = 0;
        return code;
    }
    float r = to_float((double)S / d);
    for (int i = 0; i < k; i++) q[i] = (uint8_t)orc_e2m1_encode((double)to_float((double)v[i] * (double)r));
    return code;
}

/* NVFP4 of a rows x cols tensor (cols % 16 == 0), rowwise 1x16 blocks:
 * q [rows][cols / 2] with element 2i in the low nibble, s [rows][cols / 16]
 * E4M3 codes, *S_out the tensor scale. */
void orc_nvfp4(const void* x, int dt, int64_t rows, int64_t cols, uint8_t* q, uint8_t* s, float* S_out, int nthreads)
{
    float S = orc_nvfp4_tensor_scale(orc_amax_bits(x, dt, 0, rows * cols));
    *S_out = S;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t r = 0; r < rows; r++) {
        float v[16];
        uint8_t qb[16];
        for (int64_t j = 0; j < cols / 16; j++) {
            for (int i = 0; i < 16; i++) v[i] = orc_input_value(x, dt, r * cols + 16 * j + i);
            s[r * (cols / 16) + j] = orc_nvfp4_block(v, 16, S, qb);
            for (int i = 0; i < 8; i++) q[r * (cols / 2) + 8 * j + i] = (uint8_t)(qb[2 * i] | (qb[2 * i + 1] << 4));
        }
    }
}

/* ------------------------------------------------------------------ */
/* Quantization-error statistics ("昇腾 Ascend 950 低精度格式", appendix */
/* 3.4: the SQNR and the zero-rate of quantized weights, activations   */
/* and KV cache, compared between formats).  For input x and the FP32  */
/* value xh its code stands for, over the elements where both are      */
/* finite: signal = sum x^2 and noise = sum (x - xh)^2 (SQNR = 10      */
/* log10(signal / noise) dB); the other elements are counted as        */
/* non-finite.  n_zero counts xh == 0; n_flushed counts xh == 0 with   */
/* x != 0 (a NaN x is not zero): the values quantization set to zero.  */
/* Plain double sums in element order.                                 */
/* sums[0] signal, sums[1] noise; counts[0] n, [1] n_zero,             */
/* [2] n_flushed, [3] n_nonfinite.                                     */
/* ------------------------------------------------------------------ */
static void stats_add(double* sums, int64_t* counts, float x, float xh)
{
    counts[0]++;
    if (xh == 0.0f) {
        counts[1]++;
        if (!(x == 0.0f)) counts[2]++;
    }
    if (!isfinite(x) || !isfinite(xh)) {
        counts[3]++;
        return;
    }
    double e = (double)x - (double)xh;
    sums[0] += (double)x * (double)x;
    sums[1] += e * e;
}

/* The FP32 value an MX code stands for: value(q) * 2^X, exact in double,
 * rounded once to float (so only a product of 2^128 or more changes: it
 * becomes Inf); scale byte 0xFF is NaN. */
static float mx_value_f32(int fmt, unsigned code, unsigned byte)
{
    if (byte == 0xFFu) return NAN;
    double v = orc_fp8_value(fmt, code);
    return isnan(v) ? NAN : to_float(ldexp(v, (int)byte - 127));
}

/* Statistics of the per-tensor (per-group) copy q of x: xh =
 * fl32(value(q) * scale_inv[g]) for the rows of group g. */
void orc_qstats_per_tensor(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* offs, int G,
                           int fmt, const uint8_t* q, const float* scale_inv, double* sums, int64_t* counts)
{
    int ng = offs ? G : 1;
    sums[0] = sums[1] = 0.0;
    counts[0] = counts[1] = counts[2] = counts[3] = 0;
    for (int g = 0; g < ng; g++) {
        int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
        double si = (double)scale_inv[g];
        for (int64_t i = r0 * cols; i < r1 * cols; i++) {
            double v = orc_fp8_value(fmt, q[i]);
            float xh = isnan(v) || isnan(si) ? NAN : to_float(v * si);
            stats_add(sums, counts, orc_input_value(x, dt, i), xh);
        }
    }
}

/* Statistics of one MX copy of x (layouts as orc_mx_dequantize): dir 1
 * the rowwise copy, dir 2 the columnwise copy, whose element (c, r)
 * pairs with x[r][c].  Elements are visited in x's row-major order. */
void orc_qstats_mx(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* offs, int G, int fmt,
                   int dir, const uint8_t* q, const uint8_t* s, int64_t s_ld, double* sums, int64_t* counts)
{
    int ng = offs ? G : 1;
    sums[0] = sums[1] = 0.0;
    counts[0] = counts[1] = counts[2] = counts[3] = 0;
    int64_t base = 0;
    for (int g = 0; g < ng; g++) {
        int64_t r0 = grp_off(offs, ng, rows, g), r1 = grp_off(offs, ng, rows, g + 1);
        for (int64_t r = r0; r < r1; r++)
            for (int64_t c = 0; c < cols; c++) {
                float xh;
                if (dir == 1)
                    xh = mx_value_f32(fmt, q[r * cols + c], s[r * (cols / 32) + c / 32]);
                else
                    xh = mx_value_f32(fmt, q[c * rows + r], s[c * s_ld + base + (r - r0) / 32]);
                stats_add(sums, counts, orc_input_value(x, dt, r * cols + c), xh);
            }
        base += (r1 - r0 + 31) / 32;
    }
}

/* ------------------------------------------------------------------ */
/* MXFP4 and MXFP6 ("混合精度与 FP8 训练" 13.1: an MX block is k = 32    */
/* elements and an E8M0 scale, e_max of E2M1 is 2; 13.2: E2M1 holds 0,  */
/* 0.5, 1, 1.5, 2, 3, 4, 6 and negatives; "Blackwell GPU MXFP8 预训练最  */
/* 佳实践" 3.2: Blackwell's block-scaled types MXFP8, MXFP6, MXFP4).     */
/* The pages name MXFP6 but not its elements; they are read here as the */
/* OCP microscaling pair E2M3 (bias 1, largest 7.5) and E3M2 (bias 3,   */
/* largest 28).  All three formats have subnormals and no Inf or NaN; a */
/* code is a sign bit above the magnitude bits (bit 3 for E2M1, bit 5   */
/* for the FP6 formats).                                                */
/* ------------------------------------------------------------------ */
static int lp_ebits(int fmt) { return fmt == ORC_E3M2 ? 3 : 2; }
static int lp_mbits(int fmt) { return fmt == ORC_E2M1 ? 1 : fmt == ORC_E2M3 ? 3 : 2; }
static unsigned lp_top(int fmt) { return (1u << (lp_ebits(fmt) + lp_mbits(fmt))) - 1u; }

/* Value of a code from its fields: exponent field 0 is subnormal. */
double orc_lp_value(int fmt, unsigned code)
{
    int eb = lp_ebits(fmt), mb = lp_mbits(fmt), bias = (1 << (eb - 1)) - 1;
    unsigned sign = (code >> (eb + mb)) & 1u;
    unsigned e = (code >> mb) & ((1u << eb) - 1u), m = code & ((1u << mb) - 1u);
    double f = ldexp((double)m, -mb);
    double mag = e == 0 ? ldexp(f, 1 - bias) : ldexp(1.0 + f, (int)e - bias);
    return sign ? -mag : mag;
}

/* Nearest code of a real value, ties to the even code, saturating at the
 * largest magnitude; the sign of zero is kept.  (NaN is never encoded: an
 * MX block holding one is marked by its scale.) */
unsigned orc_lp_encode(int fmt, double a)
{
    unsigned top = lp_top(fmt), sign = signbit(a) ? top + 1u : 0u;
    double m = fabs(a);
    if (isnan(a)) return 0u;
    if (m >= orc_lp_value(fmt, top)) return sign | top;
    unsigned lo = 0;
    while (orc_lp_value(fmt, lo + 1) <= m) lo++;
    if (orc_lp_value(fmt, lo) == m) return sign | lo;
    double dl = m - orc_lp_value(fmt, lo), dh = orc_lp_value(fmt, lo + 1) - m;
    unsigned c = dl < dh ? lo : dh < dl ? lo + 1 : ((lo & 1u) ? lo + 1 : lo);
    return sign | c;
}

/*
 * One MX block of k <= 32 values with E2M1, E2M3 or E3M2 elements, under
 * scale rule 0 (round-up: the smallest X with amax <= destmax * 2^X) or 1
 * (OCP: X = floor(log2 amax) - e_max), X saturated to [-127, 127]; destmax
 * is the format's largest value (6, 7.5, 28) and e_max its exponent (2, 2,
 * 4).  Elements are the nearest codes of v / 2^X (exact), saturating;
 * *sat counts |v / 2^X| > destmax.  amax 0: byte 0 and all codes +0;
 * amax Inf or NaN: byte 0xFF and all codes +0 (the scale marks the block).
 */
uint8_t orc_mxlp_block(const float* v, int k, int fmt, int rule, uint8_t* q, int64_t* sat)
{
    uint32_t amax = 0;
    double destmax = orc_lp_value(fmt, lp_top(fmt));
    int emax = (int)floor(log2(destmax));
    int X, i;
    *sat = 0;
    for (i = 0; i < k; i++) {
        uint32_t mag = float_to_bits(v[i]) & 0x7FFFFFFFu;
        if (mag > amax) amax = mag;
    }
    if (amax >= 0x7F800000u || amax == 0) {
        for (i = 0; i < k; i++) q[i] = 0;
        return amax ? 0xFF : 0x00;
    }
    double a = (double)bits_to_float(amax);
    if (rule == 0) {
        for (X = -127; X < 127; X++)
            if (a <= ldexp(destmax, X)) break;
    } else {
        for (X = 127; X > -127; X--)
            if (ldexp(1.0, X + emax) <= a) break;
    }
    for (i = 0; i < k; i++) {
        double sv = ldexp((double)v[i], -X);
        if (fabs(sv) > destmax) (*sat)++;
        q[i] = (uint8_t)orc_lp_encode(fmt, sv);
    }
    return (uint8_t)(X + 127);
}

/* Code i of a copy's row, stored two per byte (E2M1: element 2j in the low
 * nibble of byte j) or one per byte (FP6: bits 0-5). */
static void lp_put(uint8_t* row, int fmt, int64_t i, uint8_t code)
{
    if (fmt != ORC_E2M1) {
        row[i] = code;
        return;
    }
    uint8_t* b = row + i / 2;
    *b = (i & 1) ? (uint8_t)((*b & 0x0F) | (code << 4)) : (uint8_t)((*b & 0xF0) | code);
}

/*
 * MXFP4 / MXFP6 quantization of a rows x cols tensor (cols % 32 == 0):
 * dir 1 rowwise blocks x[r][32j .. 32j+31]; dir 2 columnwise blocks of 32
 * rows (the last one shorter), stored transposed; 3 both.
 *   E2M1: q_row [rows][cols / 2], q_col [cols][rows / 2] (rows even)
 *   FP6:  q_row [rows][cols],     q_col [cols][rows]
 *   s_row [rows][cols / 32], s_col [cols][ceil(rows / 32)]
 * sat[0], sat[1]: the rowwise and columnwise saturation counts.
 */
void orc_mxlp_quantize(const void* x, int dt, int64_t rows, int64_t cols, int fmt, int dir, int rule,
                       uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int64_t* sat)
{
    float v[32];
    uint8_t qb[32];
    int64_t s1, nb = (rows + 31) / 32;
    int64_t rlen = fmt == ORC_E2M1 ? cols / 2 : cols, clen = fmt == ORC_E2M1 ? rows / 2 : rows;
    sat[0] = sat[1] = 0;
    if (dir & 1)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t j = 0; j < cols / 32; j++) {
                for (int i = 0; i < 32; i++) v[i] = orc_input_value(x, dt, r * cols + 32 * j + i);
                s_row[r * (cols / 32) + j] = orc_mxlp_block(v, 32, fmt, rule, qb, &s1);
                sat[0] += s1;
                for (int i = 0; i < 32; i++) lp_put(q_row + r * rlen, fmt, 32 * j + i, qb[i]);
            }
    if (dir & 2)
        for (int64_t c = 0; c < cols; c++)
            for (int64_t b = 0; b < nb; b++) {
                int k = rows - 32 * b < 32 ? (int)(rows - 32 * b) : 32;
                for (int i = 0; i < k; i++) v[i] = orc_input_value(x, dt, (32 * b + i) * cols + c);
                s_col[c * nb + b] = orc_mxlp_block(v, k, fmt, rule, qb, &s1);
                sat[1] += s1;
                for (int i = 0; i < k; i++) lp_put(q_col + c * clen, fmt, 32 * b + i, qb[i]);
            }
}

/* ------------------------------------------------------------------ */
/* Block-scale layout for block-scaled tensor-core MMA.  The pages give */
/* none ("Blackwell GPU MXFP8 预训练最佳实践" 3.2 only says Blackwell's  */
/* tensor cores take the MX types natively); this follows NVIDIA's      */
/* public description of the scale-factor layout for block-scaled GEMM  */
/* operands: the scale array (rows x scale_cols, e.g. the rowwise MX    */
/* scales [rows][cols / 32]) is padded to multiples of 128 rows and 4   */
/* columns and cut into 128 x 4 blocks of 512 bytes, stored block row   */
/* by block row; inside a block, element (r, c) sits at byte            */
/* (r % 32) * 16 + (r / 32) * 4 + c.  Padding bytes are 0.  Parity      */
/* unpinned by the pages.                                                */
/* ------------------------------------------------------------------ */
void orc_mma_scale_layout(const uint8_t* s, int64_t rows, int64_t scale_cols, int64_t s_ld, uint8_t* out)
{
    int64_t R = (rows + 127) / 128 * 128, C = (scale_cols + 3) / 4 * 4;
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) {
            int64_t block = (r / 128) * (C / 4) + c / 4;
            int64_t rr = r % 128, cc = c % 4;
            int64_t off = block * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc;
            out[off] = (r < rows && c < scale_cols) ? s[r * s_ld + c] : 0;
        }
}
