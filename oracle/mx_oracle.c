/*
 * mx_oracle.c -- the CPU oracle for MX block-scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the MX hot path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  The product library
 * never links, calls or includes anything from here, and nothing here includes
 * anything from the product.
 *
 * Sources (web pages; cited by title and section):
 *   [Dialect]  "A Dialect Is a Set of Co-Designed Decisions: Designing for MX
 *              Quantization in MLIR" -- sections "What block scaling is",
 *              "The type: !mx.tensor", "The four ops", "The block axis",
 *              "The accumulator operand".
 *   [Layout]   "Bit Layout" (MXFP4 community format pages) -- sections
 *              "The E2M1 element", "The E8M0 shared scale",
 *              "Block structure and packing", "Reference encode and decode".
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 floor(log2 amax) is the exact integer exponent of amax (frexp), not a
 *      rounded float log2.
 *   R2 ties go to the lower magnitude (first index of the argmin), for both
 *      element formats.
 *   R3 E4M3FN is the OCP "finite + NaN" 8-bit float: bias 7, largest finite
 *      448, codes S.1111.111 are NaN, no infinities; emax = 8.
 *   R4 a block holding a NaN or an infinity gets scale 0xFF and codes 0.
 *   R5 scale bytes for the GEMM are exact powers of two; products are formed
 *      from the exact dequantized values in binary64.
 *   R6 quantizing along the first axis writes its outputs in the layout of
 *      the transposed tensor ([N, K] codes and scales), the operand layout of
 *      block_matmul.
 *   R7 dequantize to bfloat16 is the exact value rounded to nearest, ties to
 *      even (the IEEE conversion; the pages name only the output type).
 *   R8 the f32 right-hand operand of the pages' first block_matmul is
 *      row-major [K, N].
 *   R9 fold_scale accepts only a positive finite power of two 2^j; the scale
 *      byte saturates at 0 and 254 and 0xFF stays 0xFF.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 *
 * Arithmetic is binary64 unless stated.  Build: plain C99, -O2, no fast-math;
 * OpenMP (if present) only splits independent rows across threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MXO_E2M1 1
#define MXO_E4M3 2
#define MXO_BLOCK 32

/* ---------------------------------------------------------------------------
 * Element formats.
 * ------------------------------------------------------------------------- */

/* The eight nonnegative E2M1 magnitudes, ascending; the index is the 3-bit
 * code without its sign ([Layout] "Reference encode and decode", magnitude
 * table; the same values follow from the bit formula in "The E2M1 element"). */
static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Magnitude of an E4M3FN code (sign stripped), reading R3.
 * Exponent field E (4 bits), mantissa M (3 bits), bias 7:
 *   E == 0 : M/8 * 2^(1-7)          (subnormal)
 *   E >  0 : (1 + M/8) * 2^(E-7)    (normal)
 * The 7-bit code 0x7F (E=15, M=7) is NaN. */
static double e4m3_magnitude(int c7)
{
    int E = (c7 >> 3) & 0xF;
    int M = c7 & 0x7;
    if (c7 == 0x7F) return NAN;
    if (E == 0) return ldexp((double)M, -9);
    return ldexp((double)(8 + M), E - 10);
}

/* Number of finite nonnegative grid points and the largest power-of-two
 * exponent of the element format ("emax"):
 *   E2M1: 8 points (codes 0..7), emax 2: 6.0 lies in the 2^2 binade
 *         ([Layout] "Reference encode and decode", closing remarks).
 *   E4M3: 127 points (codes 0..126), emax 8: 448 lies in the 2^8 binade (R3). */
static int grid_size(int fmt) { return fmt == MXO_E2M1 ? 8 : 127; }
static int emax_of(int fmt) { return fmt == MXO_E2M1 ? 2 : 8; }
static double grid_value(int fmt, int i)
{
    return fmt == MXO_E2M1 ? E2M1_GRID[i] : e4m3_magnitude(i);
}
static int sign_bit_of(int fmt) { return fmt == MXO_E2M1 ? 0x8 : 0x80; }

/* Decode one element code to its value (before the block scale).
 * E2M1: sign is bit 3, magnitude index bits 0..2 ([Layout] "The E2M1 element").
 * E4M3: sign is bit 7 (R3). */
double mxo_decode_element(int fmt, int code)
{
    if (fmt == MXO_E2M1) {
        double m = E2M1_GRID[code & 0x7];
        return (code & 0x8) ? -m : m;
    }
    if (fmt == MXO_E4M3) {
        double m = e4m3_magnitude(code & 0x7F);
        return (code & 0x80) ? -m : m;
    }
    return NAN;
}

/* E8M0 scale byte -> value: 2^(byte-127); 0xFF is NaN
 * ([Layout] "The E8M0 shared scale"). */
double mxo_decode_scale(int byte)
{
    if (byte == 0xFF) return NAN;
    return ldexp(1.0, byte - 127);
}

/* floor(log2 v) for finite v > 0, exactly (reading R1).  frexp gives
 * v = f * 2^ex with f in [0.5, 1), so floor(log2 v) = ex - 1; this holds for
 * subnormal v as well. */
int mxo_floor_log2(double v)
{
    int ex = 0;
    (void)frexp(v, &ex);
    return ex - 1;
}

/* ---------------------------------------------------------------------------
 * quantize_block ([Dialect] "The four ops": quantize_block; [Layout]
 * "Reference encode and decode").  One block of 32 values -> 32 unpacked codes
 * and one E8M0 byte.
 *
 * Steps, in the pages' order:
 *   1. amax = max |x_i|; an all-zero block gives codes 0 and scale 127.
 *   2. e = floor(log2 amax) - emax, clipped to [-127, 127].
 *   3. y_i = |x_i| / 2^e.
 *   4. idx_i = argmin_j |y_i - grid_j|, first index on ties (R2).
 *   5. code_i = idx_i with the sign bit set when x_i < 0.
 *   6. scale byte = e + 127.
 *
 * Exactness of step 4 in binary64: y_i = |x_i| * 2^-e is exact (x_i is a
 * binary32 value and the scaling is a power of two).  If the nearest grid
 * point g* is nonzero then y_i is at least half of g*, hence at least half the
 * smallest nonzero grid value, so y_i
 * has its lowest bit at 2^-33 or above, every grid value has its lowest bit
 * at 2^-9 or above and its highest below 2^9: every |y_i - g| needs at most
 * 42 significant bits and is exact.  If g* is zero then d* = y_i is exact and
 * it is the first index, so no earlier index can tie it.  The argmin over the
 * binary64 distances is therefore the argmin over the real distances.
 * ------------------------------------------------------------------------- */
static void quantize_block(const float* x, int fmt, uint8_t* codes, uint8_t* scale)
{
    int i, j;
    double amax = 0.0;

    /* Reading R4: a non-finite input poisons the block. */
    for (i = 0; i < MXO_BLOCK; ++i) {
        if (!isfinite(x[i])) {
            for (j = 0; j < MXO_BLOCK; ++j) codes[j] = 0;
            *scale = 0xFF;
            return;
        }
    }

    for (i = 0; i < MXO_BLOCK; ++i) {
        double a = fabs((double)x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) {
        for (i = 0; i < MXO_BLOCK; ++i) codes[i] = 0;
        *scale = 127;
        return;
    }

    int e = mxo_floor_log2(amax) - emax_of(fmt);
    if (e < -127) e = -127;
    if (e > 127) e = 127;

    const int n = grid_size(fmt);
    for (i = 0; i < MXO_BLOCK; ++i) {
        double y = ldexp(fabs((double)x[i]), -e);
        int best = 0;
        double best_d = fabs(y - grid_value(fmt, 0));
        for (j = 1; j < n; ++j) {
            double d = fabs(y - grid_value(fmt, j));
            if (d < best_d) { /* strict: equal distance keeps the lower index */
                best_d = d;
                best = j;
            }
        }
        int code = best;
        if (x[i] < 0.0f) code |= sign_bit_of(fmt);
        codes[i] = (uint8_t)code;
    }
    *scale = (uint8_t)(e + 127);
}

/* Packing ([Layout] "Block structure and packing"): two E2M1 codes per
 * byte, element 2k in the low nibble and element 2k+1 in the high nibble.
 * E4M3 codes are one byte each. */
static void store_codes(int fmt, const uint8_t* unpacked, int64_t first_elem, uint8_t* row_codes)
{
    int i;
    if (fmt == MXO_E4M3) {
        for (i = 0; i < MXO_BLOCK; ++i) row_codes[first_elem + i] = unpacked[i];
        return;
    }
    for (i = 0; i < MXO_BLOCK; i += 2) {
        uint8_t lo = unpacked[i] & 0x0F;
        uint8_t hi = unpacked[i + 1] & 0x0F;
        row_codes[(first_elem + i) / 2] = (uint8_t)((hi << 4) | lo);
    }
}

static int load_code(int fmt, const uint8_t* row_codes, int64_t k)
{
    if (fmt == MXO_E4M3) return row_codes[k];
    uint8_t b = row_codes[k / 2];
    return (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

static int64_t row_code_bytes(int fmt, int64_t cols)
{
    return fmt == MXO_E2M1 ? cols / 2 : cols;
}

static int check_shape(int fmt, int64_t rows, int64_t cols)
{
    /* The type's verifier: the block size must divide the last dimension
     * ([Dialect] "The type: !mx.tensor"). */
    if (fmt != MXO_E2M1 && fmt != MXO_E4M3) return 2;
    if (rows < 0 || cols < 0 || cols % MXO_BLOCK != 0) return 1;
    return 0;
}

/* Quantize a row-major [rows, cols] binary32 tensor along its last axis.
 * codes: row-major, cols/2 bytes per row (E2M1) or cols bytes per row (E4M3).
 * scales: row-major [rows, cols/32] bytes.
 * Returns 0, 1 (bad shape) or 2 (bad format). */
int mxo_quantize(const float* x, int64_t rows, int64_t cols, int fmt,
                 uint8_t* codes, uint8_t* scales)
{
    int rc = check_shape(fmt, rows, cols);
    if (rc) return rc;
    const int64_t nb = cols / MXO_BLOCK;
    const int64_t cb = row_code_bytes(fmt, cols);
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t b;
        for (b = 0; b < nb; ++b) {
            uint8_t blk[MXO_BLOCK];
            uint8_t s;
            quantize_block(x + r * cols + b * MXO_BLOCK, fmt, blk, &s);
            store_codes(fmt, blk, b * MXO_BLOCK, codes + r * cb);
            scales[r * nb + b] = s;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * dequantize_block ([Dialect] "The four ops": dequantize_block; [Layout]
 * "The E8M0 shared scale" and "Reference encode and decode").
 * value = element * 2^(byte-127); byte 0xFF makes every element of the block
 * NaN.  The product is formed in binary64 (exact: at most 4 significant bits
 * times a power of two) and rounded once to binary32 (exact unless it
 * overflows binary32).
 * ------------------------------------------------------------------------- */
int mxo_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                   int fmt, float* y)
{
    int rc = check_shape(fmt, rows, cols);
    if (rc) return rc;
    const int64_t nb = cols / MXO_BLOCK;
    const int64_t cb = row_code_bytes(fmt, cols);
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t k;
        for (k = 0; k < cols; ++k) {
            int s = scales[r * nb + k / MXO_BLOCK];
            double v = mxo_decode_element(fmt, load_code(fmt, codes + r * cb, k)) * mxo_decode_scale(s);
            y[r * cols + k] = (float)v;
        }
    }
    return 0;
}

/* Exact dequantized value of element k of a row, in binary64 (reading R5). */
static double deq_exact(int fmt, const uint8_t* row_codes, const uint8_t* row_scales, int64_t k)
{
    return mxo_decode_element(fmt, load_code(fmt, row_codes, k)) *
           mxo_decode_scale(row_scales[k / MXO_BLOCK]);
}

/* ---------------------------------------------------------------------------
 * block_matmul ([Dialect] "The four ops" and "The accumulator operand"):
 *   C[m,n] <- C[m,n] + sum_k A[m,k] * B[k,n]
 * with both operands block-scaled along the reduction axis K ([Dialect]
 * "The block axis").  B is given as its transpose Bt [N, K] so that its blocks
 * run along its own last axis, K.
 *
 * Outputs, per (m, n):
 *   ref[m,n]  = C0[m,n] + sum_k deqA[m,k] * deqB[n,k]   (binary64 sum of exact
 *               binary64 products)
 *   sabs[m,n] = sum_k |deqA[m,k] * deqB[n,k]|           (the scale the parity
 *               tolerance is stated against)
 * ------------------------------------------------------------------------- */
static void matmul_entry(int a_fmt, const uint8_t* a_codes, const uint8_t* a_scales,
                         int b_fmt, const uint8_t* b_codes, const uint8_t* b_scales,
                         int64_t K, int64_t m, int64_t n, double c0,
                         double* ref, double* sabs)
{
    const int64_t nb = K / MXO_BLOCK;
    const uint8_t* ra = a_codes + m * row_code_bytes(a_fmt, K);
    const uint8_t* rb = b_codes + n * row_code_bytes(b_fmt, K);
    const uint8_t* sa = a_scales + m * nb;
    const uint8_t* sb = b_scales + n * nb;
    double acc = c0, s = 0.0;
    int64_t k;
    for (k = 0; k < K; ++k) {
        double p = deq_exact(a_fmt, ra, sa, k) * deq_exact(b_fmt, rb, sb, k);
        acc += p;
        s += fabs(p);
    }
    *ref = acc;
    *sabs = s;
}

int mxo_block_matmul(const uint8_t* a_codes, const uint8_t* a_scales, int a_fmt,
                     const uint8_t* b_codes, const uint8_t* b_scales, int b_fmt,
                     int64_t M, int64_t N, int64_t K, const float* C0,
                     double* ref, double* sabs)
{
    if (check_shape(a_fmt, M, K) || check_shape(b_fmt, N, K) || N < 0) return 1;
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int64_t n;
        for (n = 0; n < N; ++n)
            matmul_entry(a_fmt, a_codes, a_scales, b_fmt, b_codes, b_scales, K, m, n,
                         (double)C0[m * N + n], &ref[m * N + n], &sabs[m * N + n]);
    }
    return 0;
}

/* The same definition evaluated at chosen entries only: entry i is
 * (ms[i], ns[i]) with starting accumulator c0[i]; a_codes/a_scales hold the
 * rows of A named by ms (row ms[i] is at position a_row[i]) and likewise for
 * B.  Used where the full product is too large for a CPU. */
int mxo_block_matmul_entries(const uint8_t* a_codes, const uint8_t* a_scales, int a_fmt,
                             const uint8_t* b_codes, const uint8_t* b_scales, int b_fmt,
                             int64_t K, const int64_t* a_row, const int64_t* b_row,
                             const float* c0, int64_t count, double* ref, double* sabs)
{
    if (check_shape(a_fmt, 1, K) || check_shape(b_fmt, 1, K) || count < 0) return 1;
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < count; ++i)
        matmul_entry(a_fmt, a_codes, a_scales, b_fmt, b_codes, b_scales, K, a_row[i], b_row[i],
                     (double)c0[i], &ref[i], &sabs[i]);
    return 0;
}

/* ---------------------------------------------------------------------------
 * The block axis ([Dialect] "The block axis"): blocking is along the reduction
 * axis, which for the right-hand operand of a product is its FIRST axis.
 * Quantize a row-major [rows, cols] tensor in blocks of 32 consecutive rows of
 * one column.  The outputs are laid out as the transposed tensor's would be:
 * codes [cols, rows] (row c holds column c's codes, packed as usual) and scales
 * [cols, rows/32], so that the result is directly a [N, K] operand.
 * Returns 0, 1 (bad shape: rows % 32 != 0) or 2 (bad format).
 * ------------------------------------------------------------------------- */
int mxo_quantize_axis0(const float* x, int64_t rows, int64_t cols, int fmt,
                       uint8_t* codes, uint8_t* scales)
{
    int rc = check_shape(fmt, cols, rows);
    if (rc) return rc;
    const int64_t nb = rows / MXO_BLOCK;
    const int64_t cb = row_code_bytes(fmt, rows);
    int64_t c;
#pragma omp parallel for schedule(static)
    for (c = 0; c < cols; ++c) {
        int64_t b;
        for (b = 0; b < nb; ++b) {
            float blockv[MXO_BLOCK];
            uint8_t blk[MXO_BLOCK];
            uint8_t s;
            int i;
            for (i = 0; i < MXO_BLOCK; ++i) blockv[i] = x[(b * MXO_BLOCK + i) * cols + c];
            quantize_block(blockv, fmt, blk, &s);
            store_codes(fmt, blk, b * MXO_BLOCK, codes + c * cb);
            scales[c * nb + b] = s;
        }
    }
    return 0;
}

/* Round a binary32 value to the nearest bfloat16 (8 significant bits, the
 * binary32 exponent range), ties to even -- the IEEE conversion; NaN stays NaN
 * (quiet).  Returns the bfloat16 bit pattern. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t keep = u >> 16;          /* truncated result */
    const uint32_t rest = u & 0xFFFFu;       /* dropped 16 bits */
    uint32_t r = keep;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1u; /* carry may reach Inf: correct */
    return (uint16_t)r;
}

/* dequantize_block with a bfloat16 result: the exact value (as in
 * mxo_dequantize: element * 2^(byte-127), 0xFF -> NaN) rounded once to the
 * nearest bfloat16, ties to even.  The value fits binary32 exactly (at most 4
 * significant bits, exponent within binary32's range or beyond its largest
 * finite value, where binary32 and bfloat16 both give infinity), so rounding
 * the binary32 value is rounding the exact one. */
int mxo_dequantize_bf16(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                        int fmt, uint16_t* y)
{
    int rc = check_shape(fmt, rows, cols);
    if (rc) return rc;
    const int64_t nb = cols / MXO_BLOCK;
    const int64_t cb = row_code_bytes(fmt, cols);
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t k;
        for (k = 0; k < cols; ++k) {
            int s = scales[r * nb + k / MXO_BLOCK];
            double v = mxo_decode_element(fmt, load_code(fmt, codes + r * cb, k)) * mxo_decode_scale(s);
            y[r * cols + k] = f32_to_bf16_rne((float)v);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * block_matmul as the pages' first version states it ([Dialect] "The four
 * ops": the left operand an MX tensor, the right one plain f32): 
 *   C[m,n] <- C0[m,n] + sum_k deqA[m,k] * B[k,n]
 * with B row-major [K, N].  Each product is exact in binary64 (at most 4
 * significant bits times a binary32 value); the sum is formed in binary64 in
 * k order.  sabs is sum_k |deqA * B|, the scale of the parity tolerance.
 * ------------------------------------------------------------------------- */
int mxo_block_matmul_f32b(const uint8_t* a_codes, const uint8_t* a_scales, int a_fmt,
                          const float* B, int64_t M, int64_t N, int64_t K, const float* C0,
                          double* ref, double* sabs)
{
    if (check_shape(a_fmt, M, K) || N < 0) return 1;
    const int64_t nb = K / MXO_BLOCK;
    const int64_t cb = row_code_bytes(a_fmt, K);
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int64_t n;
        for (n = 0; n < N; ++n) {
            double acc = (double)C0[m * N + n], s = 0.0;
            int64_t k;
            for (k = 0; k < K; ++k) {
                double p = deq_exact(a_fmt, a_codes + m * cb, a_scales + m * nb, k) * (double)B[k * N + n];
                acc += p;
                s += fabs(p);
            }
            ref[m * N + n] = acc;
            sabs[m * N + n] = s;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * fold_scale ([Dialect] "The four ops": multiply an MX tensor by a scalar):
 * for a scalar 2^j the product is the same codes with every scale byte
 * increased by j, since an E8M0 byte is the exponent of a power of two
 * ([Layout] "The E8M0 shared scale").  The byte saturates at 0 (2^-127) and
 * 254 (2^127) -- the nearest representable scales -- and 0xFF (NaN) stays
 * 0xFF.  A scalar that is not a positive power of two is not foldable.
 * ------------------------------------------------------------------------- */
void mxo_fold_scale(uint8_t* scales, int64_t count, int j)
{
    int64_t i;
    for (i = 0; i < count; ++i) {
        int b = scales[i];
        if (b == 0xFF) continue;
        b += j;
        if (b < 0) b = 0;
        if (b > 254) b = 254;
        scales[i] = (uint8_t)b;
    }
}

/* The exponent j of a foldable scalar (a positive finite power of two,
 * subnormal ones included), or -1000 when the scalar is not foldable. */
int mxo_fold_exponent(double scalar)
{
    if (!(scalar > 0.0) || !isfinite(scalar)) return -1000;
    int ex;
    double f = frexp(scalar, &ex);
    if (f != 0.5) return -1000;
    return ex - 1;
}

int mxo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void mxo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
