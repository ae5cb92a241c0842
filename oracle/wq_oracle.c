/*
 * wq_oracle.c -- the ORACLE for the W4A16 dequantise-GEMM  C = A . deq(B)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * bench's cpu_baseline / reference arm may load this library.  The product
 * (the CUDA library under weight_only_bit_w4a16_gb300/) never links, loads or
 * calls it, and the two share no code, header, table or constant.
 *
 * Plain, slow and written to be checked by eye:
 *   - every code and every scale byte is decoded bit by bit, or through the
 *     explicit e2m1 table, into an fp64 value;
 *   - the weight is the exact fp64 product of the decoded pieces (exact for
 *     all three formats: at most 5 + 8 significant bits, far inside fp64
 *     range);
 *   - C[m,n] = sum over k ascending of double(a[m,k]) * w[n,k] in fp64, and
 *     the tolerance scale S[m,n] = sum over k of |a[m,k] * w[n,k]|;
 *   - the bf16 image of a weight is rounded to nearest-even directly from the
 *     exact fp64 value (no detour through fp32).
 *
 * Sources (page title, then section / symbol on it):
 *   [P1] example_dequant_gemm_bf16_fp4_hopper.py (TileLang example),
 *        _tir_u8_to_f4_to_bf16 and simple_dequant_bf16_fp4: the e2m1 bit
 *        fields (sign = bit 3, exponent = bits 2..1, mantissa = bit 0, bias 1)
 *        and the nibble order (element j of a row lives in byte j/2, nibble
 *        j%2, so the even index is the LOW nibble).
 *   [P3] Matmul2dFp4 (Mojo / MAX API docs), run and run_smem_decode: packed
 *        (N, K/2) uint8, scales (N, K/16) float8_e4m3fn, weight =
 *        decode_e2m1 * |scale|.
 *   [P4] megakernel_int4_weight_decode.py (KBench task spec), "The weight
 *        format" and the Precision section: two codes per uint8, the even
 *        input index in the low nibble; per group of 128 consecutive inputs a
 *        bf16 scale and a uint8 zero point; value = (code - zero) * scale,
 *        the zero point subtracted first.
 *   MXFP4 uses the OCP Microscaling (MX) definition of the scale: an e8m0
 *   byte E meaning 2^(E-127), 0xFF = NaN, one scale per 32 elements.
 *
 * Readings where the pages are silent or disagree (each also listed in the
 * design notes):
 *   - e2m1 exponent 0 is subnormal (code 1 = 0.5, code 0 = 0); [P1]'s helper
 *     has no subnormal case and would give 0.75 / 0.5 -- treated as a defect.
 *   - NVFP4 applies |e4m3(scale)| ([P3] wording); the sign bit is ignored.
 *   - e4m3fn: bias 7, exponent 0 subnormal, S.1111.111 is NaN, no infinity.
 *   - e8m0 0x00 is 2^-127 (not zero); 0xFF is NaN.
 *   - int4 zero is read as a full uint8 (the KBench spec's weight format gives 0..15).
 *   - No second-level per-tensor NVFP4 scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Format codes of the oracle's own interface (Python passes these ints). */
enum { WQO_NVFP4 = 0, WQO_MXFP4 = 1, WQO_INT4 = 2 };

/* e2m1 value table indexed by the 4-bit code s.ee.m: [P1] bit fields, with
 * exponent field 0 read as subnormal (m * 0.5).  Codes 8..15 are the negated
 * codes 0..7 (code 8 is -0). */
static const double E2M1[16] = {
    +0.0, +0.5, +1.0, +1.5, +2.0, +3.0, +4.0, +6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double wqo_e2m1(int code) { return E2M1[code & 0xF]; }

/* float8_e4m3fn ([P3] scale type): 1 sign, 4 exponent (bias 7), 3 mantissa. */
double wqo_e4m3(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 0xF, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;               /* the only NaN pattern */
    if (e == 0) v = ldexp((double)m / 8.0, -6);       /* subnormal */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* e8m0 (OCP MX scale): 2^(E-127); 0xFF is NaN. */
double wqo_e8m0(int byte)
{
    byte &= 0xFF;
    if (byte == 0xFF) return NAN;
    return ldexp(1.0, byte - 127);
}

/* bfloat16 bits: 1 sign, 8 exponent (bias 127), 7 mantissa ([P4] scale). */
double wqo_bf16(int bits)
{
    int s = (bits >> 15) & 1, e = (bits >> 7) & 0xFF, m = bits & 0x7F;
    double v;
    if (e == 0xFF) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m / 128.0, -126);   /* subnormal */
    else v = ldexp(1.0 + (double)m / 128.0, e - 127);
    return s ? -v : v;
}

/* Round an fp64 value to the nearest bfloat16, ties to even mantissa,
 * overflow to +-inf, NaN to the quiet NaN 0x7FC0 (sign kept).  Works on the
 * exact value: the quantum of the binade (2^(E-7), or 2^-133 below 2^-126) is
 * applied with nearbyint() in the default ties-to-even mode. */
int wqo_round_bf16(double x)
{
    int sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x), r;
    int e2, E, q, bits;
    if (isnan(x)) return sign | 0x7FC0;
    if (isinf(x)) return sign | 0x7F80;
    if (ax == 0.0) return sign;
    frexp(ax, &e2);                 /* ax in [2^(e2-1), 2^e2) */
    E = e2 - 1;                     /* ax in [2^E, 2^(E+1)) */
    q = (E < -126) ? -133 : E - 7;  /* spacing of bf16 values near ax */
    r = nearbyint(ldexp(ax, -q));   /* integer multiple of the spacing */
    if (E < -126) {
        bits = (int)r;              /* subnormal; r == 128 carries to 2^-126 */
    } else {
        /* r in [128, 256]; 256 carries into the exponent field */
        double bexp = (double)(E + 127) * 128.0 + (r - 128.0);
        if (bexp >= 255.0 * 128.0) return sign | 0x7F80;    /* overflow */
        bits = (int)bexp;
    }
    return sign | bits;
}

/* 4-bit code of element (n, k): byte k/2 of row n, LOW nibble for even k
 * ([P1] simple_dequant_bf16_fp4 indexing; [P4] "The weight format"). */
static int code_at(const uint8_t* packed, int K, int n, int k)
{
    uint8_t byte = packed[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
    return (k & 1) ? (byte >> 4) & 0xF : byte & 0xF;
}

/* Exact fp64 weight w[n,k] of one element. */
double wqo_weight(const uint8_t* packed, const void* scales, const uint8_t* zeros,
                  int N, int K, int fmt, int group, int n, int k)
{
    int c = code_at(packed, K, n, k);
    size_t gi = (size_t)n * (size_t)(K / group) + (size_t)(k / group);
    (void)N;
    if (fmt == WQO_NVFP4)
        return E2M1[c] * fabs(wqo_e4m3(((const uint8_t*)scales)[gi]));
    if (fmt == WQO_MXFP4)
        return E2M1[c] * wqo_e8m0(((const uint8_t*)scales)[gi]);
    /* WQO_INT4: subtract the zero point, then multiply by the scale ([P4]) */
    return ((double)c - (double)zeros[gi]) * wqo_bf16(((const uint16_t*)scales)[gi]);
}

/* Decode the whole (N, K) weight: W64 gets the exact values (may be NULL),
 * Wbf16 the round-to-nearest-even bf16 bits (may be NULL). */
void wqo_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros,
                 int N, int K, int fmt, int group, double* W64, uint16_t* Wbf16)
{
    long long nk = (long long)N * K, i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nk; ++i) {
        int n = (int)(i / K), k = (int)(i % K);
        double w = wqo_weight(packed, scales, zeros, N, K, fmt, group, n, k);
        if (W64) W64[i] = w;
        if (Wbf16) Wbf16[i] = (uint16_t)wqo_round_bf16(w);
    }
}

/* C[i, j] = sum_k double(A[rows[i], k]) * w[cols[j], k] and
 * S[i, j] = sum_k |A[rows[i], k] * w[cols[j], k]|, k ascending, fp64.
 * A is (M, K) bf16 bits, row-major.  rows == NULL means all M rows,
 * cols == NULL all N columns.  C and S are (nrows, ncols), row-major.
 * Columns are handled in blocks so that only a block of decoded weights is
 * held at a time. */
void wqo_gemm(const uint16_t* A, const uint8_t* packed, const void* scales,
              const uint8_t* zeros, int M, int N, int K, int fmt, int group,
              const int* rows, int nrows, const int* cols, int ncols,
              double* C, double* S)
{
    const int NB = 64;   /* columns decoded per block */
    double* a64;
    double* wblk;
    int i, jb;
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    a64 = (double*)malloc(sizeof(double) * (size_t)nrows * (size_t)K);
    wblk = (double*)malloc(sizeof(double) * (size_t)NB * (size_t)K);
    if (!a64 || !wblk) { free(a64); free(wblk); return; }
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int m = rows ? rows[i] : i, k;
        for (k = 0; k < K; ++k)
            a64[(size_t)i * K + k] = wqo_bf16(A[(size_t)m * K + k]);
    }
    for (jb = 0; jb < ncols; jb += NB) {
        int nb = (ncols - jb < NB) ? ncols - jb : NB, t;
        long long p, np;
#pragma omp parallel for schedule(static)
        for (t = 0; t < nb; ++t) {
            int n = cols ? cols[jb + t] : jb + t, k;
            for (k = 0; k < K; ++k)
                wblk[(size_t)t * K + k] =
                    wqo_weight(packed, scales, zeros, N, K, fmt, group, n, k);
        }
        np = (long long)nrows * nb;
#pragma omp parallel for schedule(dynamic, 16)
        for (p = 0; p < np; ++p) {
            int ii = (int)(p / nb), t = (int)(p % nb), k;
            const double* ar = a64 + (size_t)ii * K;
            const double* wr = wblk + (size_t)t * K;
            double c = 0.0, s = 0.0;
            for (k = 0; k < K; ++k) {
                double term = ar[k] * wr[k];
                c += term;
                s += fabs(term);
            }
            C[(size_t)ii * ncols + jb + t] = c;
            S[(size_t)ii * ncols + jb + t] = s;
        }
    }
    free(a64);
    free(wblk);
}

/* Thread control for the CPU baseline (reports how many threads ran). */
int wqo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void wqo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
