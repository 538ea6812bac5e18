/*
 * Plain CPU oracle for the tiled contraction D = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a separate shared
 * library that only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load.  It shares no code, header, table or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * Everything here is written from definitions, for a reader to check by eye:
 *   - the number formats (bfloat16, OCP FP8 E4M3FN, OCP E8M0 scale) are
 *     decoded from their bit-field definitions with ldexp, no bit casting;
 *   - the product follows "tcgen05.mma", section "Examples" (page 5 of the
 *     TIRx tile-operation guides): B is stored as (N, K) and the result is
 *     a @ b.T, i.e. ref[i][j] = sum over k of a[i][k] * b[j][k];
 *   - the k sum runs in ascending k, one float64 accumulator per output;
 *   - mag[i][j] = sum over k of |a[i][k] * b[j][k]| is computed in the same
 *     pass; it scales the tolerance of the comparison;
 *   - the optional elementwise epilogue adds a constant to the float64 sum
 *     ("Tile Operands and Execution", section "A Load, Compute, and Store
 *     Example": an add-one applied to every register element);
 *   - block scaling (".block_scale", "tcgen05.mma" section "Weight-stationary
 *     and block scaling") is taken in its plain MX reading: every element of
 *     A (resp. B) is multiplied by 2^(e - 127) where e is the E8M0 byte of
 *     its row and of its 32-element K block; for FP4 (E2M1) operands the
 *     scale is E8M0 per 32 elements (MXFP4) or UE4M3 per 16 (NVFP4).
 *
 * Parallelism: OpenMP over output rows only; each output keeps its own
 * ascending-k sum, so the thread count never changes a result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TGO_OK 0
#define TGO_ERR_ARG 1
#define TGO_ERR_NOMEM 2

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * exponent 0: subnormal, value = f/128 * 2^-126; exponent 255: inf / NaN. */
double tgo_bf16_to_f64(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xFF;
    int frac = bits & 0x7F;
    double v;
    if (expo == 0xFF) {
        v = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        v = ldexp((double)frac / 128.0, -126);
    } else {
        v = ldexp(1.0 + (double)frac / 128.0, expo - 127);
    }
    return sign ? -v : v;
}

/* FP8 E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits.
 * exponent 0: subnormal, value = f/8 * 2^-6.  No infinities; the only NaN
 * encodings are S.1111.111.  Largest finite magnitude 1.75 * 2^8 = 448. */
double tgo_e4m3fn_to_f64(uint8_t bits)
{
    int sign = (bits >> 7) & 1;
    int expo = (bits >> 3) & 0xF;
    int frac = bits & 0x7;
    double v;
    if (expo == 0xF && frac == 0x7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexp((double)frac / 8.0, -6);
    } else {
        v = ldexp(1.0 + (double)frac / 8.0, expo - 7);
    }
    return sign ? -v : v;
}

/* E8M0 scale: 8 exponent bits, no sign, no fraction; value 2^(e-127),
 * e = 255 is NaN. */
double tgo_e8m0_to_f64(uint8_t bits)
{
    if (bits == 0xFF) return NAN;
    return ldexp(1.0, (int)bits - 127);
}

/* FP4 E2M1 (OCP MX element format): 1 sign bit, 2 exponent bits (bias 1),
 * 1 fraction bit, in the low 4 bits of `nibble`.  exponent 0: subnormal,
 * value = f/2 * 2^0; otherwise (1 + f/2) * 2^(e-1).  No infinities or NaNs;
 * the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double tgo_e2m1_to_f64(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int expo = (nibble >> 1) & 0x3;
    int frac = nibble & 0x1;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac / 2.0, 0);
    } else {
        v = ldexp(1.0 + (double)frac / 2.0, expo - 1);
    }
    return sign ? -v : v;
}

/* UE4M3 scale (the unsigned use of E4M3 for NVFP4 block scales): the
 * E4M3FN definition with the sign bit required to be 0; a set sign bit or
 * the NaN code 0x7F decodes to NaN. */
double tgo_ue4m3_to_f64(uint8_t bits)
{
    if (bits & 0x80) return NAN;
    return tgo_e4m3fn_to_f64(bits);
}

/* ------------------------------------------------------------------------ */
/* The contraction over decoded operands                                     */
/* ------------------------------------------------------------------------ */

/* ref/mag are [nrows, ncols] row-major.  a_rows[r] is decoded row rows[r] of
 * A (length K); b_rows[c] is decoded row cols[c] of B (length K). */
static void dot_grid(const double *a_rows, const double *b_rows, int64_t nrows,
                     int64_t ncols, int64_t K, double add, double *ref,
                     double *mag)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < nrows; ++r) {
        const double *a = a_rows + r * K;
        for (int64_t c = 0; c < ncols; ++c) {
            const double *b = b_rows + c * K;
            double s = 0.0, m = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = a[k] * b[k];
                s += p;
                m += fabs(p);
            }
            ref[r * ncols + c] = s + add;
            mag[r * ncols + c] = m;
        }
    }
}

static int check_index_list(const int64_t *idx, int64_t n, int64_t bound)
{
    if (n < 0) return 0;
    if (idx == NULL) return 1;
    for (int64_t i = 0; i < n; ++i)
        if (idx[i] < 0 || idx[i] >= bound) return 0;
    return 1;
}

/* Row r of the selection: idx[r] if a list is given, else r. */
static int64_t pick(const int64_t *idx, int64_t r) { return idx ? idx[r] : r; }

/*
 * bf16 GEMM oracle.  A is [M, K] with row stride lda (elements), B is [N, K]
 * with row stride ldb; both hold raw bfloat16 bit patterns.  rows/cols
 * select which outputs to compute (NULL = all M rows / all N columns, with
 * nrows = M / ncols = N).  ref and mag receive [nrows, ncols] float64.
 * `add` is the epilogue constant (0 for a plain product).
 */
int tgo_gemm_bf16(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                  int64_t M, int64_t N, int64_t K, double add,
                  const int64_t *rows, int64_t nrows, const int64_t *cols,
                  int64_t ncols, double *ref, double *mag)
{
    if (!A || !B || !ref || !mag || M < 0 || N < 0 || K < 0 || lda < K || ldb < K)
        return TGO_ERR_ARG;
    if (!check_index_list(rows, nrows, M) || !check_index_list(cols, ncols, N))
        return TGO_ERR_ARG;
    if (!rows && nrows != M) return TGO_ERR_ARG;
    if (!cols && ncols != N) return TGO_ERR_ARG;
    if (nrows == 0 || ncols == 0) return TGO_OK;
    if (K == 0) {
        for (int64_t i = 0; i < nrows * ncols; ++i) { ref[i] = add; mag[i] = 0.0; }
        return TGO_OK;
    }
    double *ad = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    double *bd = (double *)malloc(sizeof(double) * (size_t)(ncols * K));
    if (!ad || !bd) { free(ad); free(bd); return TGO_ERR_NOMEM; }
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t k = 0; k < K; ++k)
            ad[r * K + k] = tgo_bf16_to_f64(A[pick(rows, r) * lda + k]);
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t k = 0; k < K; ++k)
            bd[c * K + k] = tgo_bf16_to_f64(B[pick(cols, c) * ldb + k]);
    dot_grid(ad, bd, nrows, ncols, K, add, ref, mag);
    free(ad);
    free(bd);
    return TGO_OK;
}

/*
 * Block-scaled MXFP8 GEMM oracle.  A is [M, K] E4M3FN bytes (row stride lda),
 * B is [N, K] E4M3FN bytes (row stride ldb).  SFA is [M, K/32] E8M0 bytes
 * (row stride ld_sfa), SFB is [N, K/32] (row stride ld_sfb).  The decoded
 * operand is a[i][k] = e4m3(A[i][k]) * 2^(SFA[i][k/32] - 127), likewise b.
 * K must be a multiple of 32.  Output selection as in tgo_gemm_bf16.
 */
int tgo_gemm_mxfp8(const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                   const uint8_t *SFA, int64_t ld_sfa, const uint8_t *SFB,
                   int64_t ld_sfb, int64_t M, int64_t N, int64_t K, double add,
                   const int64_t *rows, int64_t nrows, const int64_t *cols,
                   int64_t ncols, double *ref, double *mag)
{
    if (!A || !B || !SFA || !SFB || !ref || !mag || M < 0 || N < 0 || K < 0)
        return TGO_ERR_ARG;
    if (K % 32 != 0 || lda < K || ldb < K || ld_sfa < K / 32 || ld_sfb < K / 32)
        return TGO_ERR_ARG;
    if (!check_index_list(rows, nrows, M) || !check_index_list(cols, ncols, N))
        return TGO_ERR_ARG;
    if (!rows && nrows != M) return TGO_ERR_ARG;
    if (!cols && ncols != N) return TGO_ERR_ARG;
    if (nrows == 0 || ncols == 0) return TGO_OK;
    if (K == 0) {
        for (int64_t i = 0; i < nrows * ncols; ++i) { ref[i] = add; mag[i] = 0.0; }
        return TGO_OK;
    }
    double *ad = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    double *bd = (double *)malloc(sizeof(double) * (size_t)(ncols * K));
    if (!ad || !bd) { free(ad); free(bd); return TGO_ERR_NOMEM; }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = pick(rows, r);
        for (int64_t k = 0; k < K; ++k)
            ad[r * K + k] = tgo_e4m3fn_to_f64(A[i * lda + k]) *
                            tgo_e8m0_to_f64(SFA[i * ld_sfa + k / 32]);
    }
    for (int64_t c = 0; c < ncols; ++c) {
        int64_t j = pick(cols, c);
        for (int64_t k = 0; k < K; ++k)
            bd[c * K + k] = tgo_e4m3fn_to_f64(B[j * ldb + k]) *
                            tgo_e8m0_to_f64(SFB[j * ld_sfb + k / 32]);
    }
    dot_grid(ad, bd, nrows, ncols, K, add, ref, mag);
    free(ad);
    free(bd);
    return TGO_OK;
}

/*
 * Block-scaled FP4 GEMM oracle ("tcgen05.mma", Block-scaled opcodes with
 * .scale_vec::2X / ::4X).  A is [M, K/2] bytes (row stride lda bytes) of
 * packed E2M1 values: element k of a row is the low nibble of byte k/2 when
 * k is even and the high nibble when k is odd.  B is [N, K/2] likewise.
 * scale_kind 0 (MXFP4): SFA is [M, K/32] E8M0 bytes, one per 32 consecutive
 * K elements; scale_kind 1 (NVFP4): SFA is [M, K/16] UE4M3 bytes, one per 16.
 * The decoded operand is a[i][k] = e2m1(A[i][k]) * scale(SFA[i][k / block]),
 * likewise b; the product and the output selection are as in tgo_gemm_bf16.
 */
int tgo_gemm_fp4(const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                 const uint8_t *SFA, int64_t ld_sfa, const uint8_t *SFB,
                 int64_t ld_sfb, int64_t M, int64_t N, int64_t K, int scale_kind,
                 double add, const int64_t *rows, int64_t nrows,
                 const int64_t *cols, int64_t ncols, double *ref, double *mag)
{
    int64_t block;
    if (scale_kind == 0) block = 32;
    else if (scale_kind == 1) block = 16;
    else return TGO_ERR_ARG;
    if (!A || !B || !SFA || !SFB || !ref || !mag || M < 0 || N < 0 || K < 0)
        return TGO_ERR_ARG;
    if (K % block != 0 || 2 * lda < K || 2 * ldb < K || ld_sfa < K / block ||
        ld_sfb < K / block)
        return TGO_ERR_ARG;
    if (!check_index_list(rows, nrows, M) || !check_index_list(cols, ncols, N))
        return TGO_ERR_ARG;
    if (!rows && nrows != M) return TGO_ERR_ARG;
    if (!cols && ncols != N) return TGO_ERR_ARG;
    if (nrows == 0 || ncols == 0) return TGO_OK;
    if (K == 0) {
        for (int64_t i = 0; i < nrows * ncols; ++i) { ref[i] = add; mag[i] = 0.0; }
        return TGO_OK;
    }
    double *ad = (double *)malloc(sizeof(double) * (size_t)(nrows * K));
    double *bd = (double *)malloc(sizeof(double) * (size_t)(ncols * K));
    if (!ad || !bd) { free(ad); free(bd); return TGO_ERR_NOMEM; }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = pick(rows, r);
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = A[i * lda + k / 2];
            uint8_t nib = (k % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
            uint8_t sb = SFA[i * ld_sfa + k / block];
            double sc = scale_kind == 0 ? tgo_e8m0_to_f64(sb) : tgo_ue4m3_to_f64(sb);
            ad[r * K + k] = tgo_e2m1_to_f64(nib) * sc;
        }
    }
    for (int64_t c = 0; c < ncols; ++c) {
        int64_t j = pick(cols, c);
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = B[j * ldb + k / 2];
            uint8_t nib = (k % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
            uint8_t sb = SFB[j * ld_sfb + k / block];
            double sc = scale_kind == 0 ? tgo_e8m0_to_f64(sb) : tgo_ue4m3_to_f64(sb);
            bd[c * K + k] = tgo_e2m1_to_f64(nib) * sc;
        }
    }
    dot_grid(ad, bd, nrows, ncols, K, add, ref, mag);
    free(ad);
    free(bd);
    return TGO_OK;
}

/* out[j][i] = in[i][j] on raw 16-bit patterns; in is [rows, cols] with row
 * stride ld_in, out is [cols, rows] with row stride ld_out. */
int tgo_transpose_b16(const uint16_t *in, int64_t ld_in, uint16_t *out,
                      int64_t ld_out, int64_t rows, int64_t cols)
{
    if (!in || !out || rows < 0 || cols < 0 || ld_in < cols || ld_out < rows)
        return TGO_ERR_ARG;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j)
            out[j * ld_out + i] = in[i * ld_in + j];
    return TGO_OK;
}

/* Number of OpenMP threads a parallel region will use (1 without OpenMP). */
int tgo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void tgo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Elementwise decoders over arrays (same definitions as above). */
void tgo_decode_bf16(const uint16_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tgo_bf16_to_f64(in[i]);
}

void tgo_decode_e4m3fn(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tgo_e4m3fn_to_f64(in[i]);
}

void tgo_decode_e8m0(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tgo_e8m0_to_f64(in[i]);
}

void tgo_decode_e2m1(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tgo_e2m1_to_f64(in[i]);
}

void tgo_decode_ue4m3(const uint8_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tgo_ue4m3_to_f64(in[i]);
}
