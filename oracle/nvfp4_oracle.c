/*
 * CPU oracle for the masked, block-scaled NVFP4 grouped GEMM-NT.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or table with the CUDA
 * library; it has its own copy of every format table.
 *
 * What it computes (the operation FlashInfer calls grouped_gemm_nt_masked, as
 * described on "The CuteDSL Gamble: Chasing Kernel Efficiency on Blackwell
 * GPUs", sections "The Message" and "Output Knowledge Created": a masked,
 * batched GEMM whose two operands each come as (data, scale factors), with a
 * per-expert mask masked_m, a scale-factor vector size, and an optional alpha
 * applied at the output):
 *
 *   for g < G, m < masked_m[g], n < N:
 *     C[g][m][n] = bf16_rne( alpha[g] * sum_{k<K} a(g,m,k) * b(g,n,k) )
 *     a(g,m,k)   = e2m1(A code of element k of row m) * e4m3(A_sf[g][m][k/16])
 *     b(g,n,k)   = e2m1(B code of element k of row n) * e4m3(B_sf[g][n][k/16])
 *   rows m >= masked_m[g] of C are not written.
 *
 * The pages name NVFP4 (a 4-bit floating-point format with a scale per block
 * of elements; same page, "Input Knowledge Required") but never define its
 * encodings.  The
 * readings taken here are the public OCP Microscaling definitions:
 *   - e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 *     exponent 0 is subnormal with value mantissa * 0.5.
 *   - e4m3 ("fn" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 *     mantissa; exponent 0 is subnormal (mantissa * 2^-9); 0x7F/0xFF are NaN;
 *     there is no infinity.
 *   - packing: element k of a row lives in byte k/2, even k in the low nibble.
 *   - scale layout: one e4m3 byte per 16 consecutive K elements, row-major
 *     [G][rows][K/16] (sf_vec_size = 16).
 *   - bf16 output: one rounding, fp64 -> bf16, round to nearest, ties to even.
 *
 * Accumulation is in fp64.  Every product of two e2m1 values and two e4m3
 * scales is exact in fp64 (at most 4 + 8 significant bits), so with
 * power-of-two scales the sum is exact in any order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* e2m1 code -> value, written from the bit-field definition (OCP FP4 E2M1). */
double nvfp4o_e2m1_value(int code) {
    int sign = (code >> 3) & 1;
    int exp = (code >> 1) & 3;
    int man = code & 1;
    double mag = (exp == 0) ? 0.5 * man : ldexp(1.0 + 0.5 * man, exp - 1);
    return sign ? -mag : mag;
}

/* e4m3 ("fn") byte -> value, from the bit-field definition (OCP FP8 E4M3). */
double nvfp4o_e4m3_value(int byte) {
    int sign = (byte >> 7) & 1;
    int exp = (byte >> 3) & 15;
    int man = byte & 7;
    double mag;
    if (exp == 15 && man == 7) return NAN;
    if (exp == 0) mag = ldexp((double)man, -9);
    else mag = ldexp(1.0 + man / 8.0, exp - 7);
    return sign ? -mag : mag;
}

/* fp64 -> bf16 bits, one rounding to nearest with ties to even.  bf16 has an
 * 8-bit exponent (bias 127) and 7 stored mantissa bits: in the binade
 * [2^e, 2^(e+1)) the spacing is 2^(e-7), and below 2^-126 it is 2^-133. */
uint16_t nvfp4o_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    if (isinf(x)) return signbit(x) ? 0xFF80 : 0x7F80;
    int E;
    frexp(x, &E);                 /* |x| in [2^(E-1), 2^E) */
    int e = E - 1;
    if (e < -126) e = -126;
    double q = ldexp(1.0, e - 7);
    double r = nearbyint(x / q) * q;   /* x/q is exact: q is a power of two */
    const double bf16_max = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max) return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* The 16 e2m1 values as a lookup table, indexed by the 4-bit code: codes
 * 0..7 are +0, 0.5, 1, 1.5, 2, 3, 4, 6 (OCP FP4 E2M1), codes 8..15 the same
 * magnitudes negated (8 is -0).  Elements are decoded through this table;
 * the bit-field function above is the independent statement it is pinned
 * against. */
static const double kE2M1[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double nvfp4o_e2m1_table(int code) { return kE2M1[code & 15]; }

/* Value of element k of the packed row `row` (K/2 bytes). */
static double elem(const uint8_t* row, const uint8_t* sf_row, int k) {
    int byte = row[k >> 1];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    return kE2M1[code] * nvfp4o_e4m3_value(sf_row[k >> 4]);
}

int nvfp4o_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full oracle.  Plain layouts:
 *   A    u8 [G][M_max][K/2]    A_sf u8 [G][M_max][K/16]
 *   B    u8 [G][N][K/2]        B_sf u8 [G][N][K/16]
 *   alpha f32 [G], masked_m i32 [G]
 *   C    u16 (bf16 bits) [G][M_max][N], in/out: only valid rows are written.
 *   ref64 (optional, may be NULL) f64 [G][M_max][N]: the unrounded
 *        alpha*sum for valid rows; other entries are left as they were.
 * Each operand is first decoded into a dense fp64 matrix (code value times
 * its block scale); C is then alpha times the plain product A_g * B_g^T.
 * Returns 0, or -1 for bad arguments.
 */
int nvfp4o_gemm(const uint8_t* A, const uint8_t* A_sf, const uint8_t* B,
                const uint8_t* B_sf, const float* alpha, const int32_t* masked_m,
                uint16_t* C, double* ref64, int G, int M_max, int N, int K,
                int nthreads) {
    if (G <= 0 || M_max <= 0 || N <= 0 || K <= 0 || (K % 16) != 0) return -1;
    for (int g = 0; g < G; g++)
        if (masked_m[g] < 0 || masked_m[g] > M_max) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const size_t kb = (size_t)K / 2, ks = (size_t)K / 16;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)N * K);
    double* Ad = (double*)malloc(sizeof(double) * (size_t)M_max * K);
    if (!Bd || !Ad) { free(Bd); free(Ad); return -2; }
    for (int g = 0; g < G; g++) {
        int mm = masked_m[g];
        if (mm == 0) continue;
        /* decode B_g and the valid rows of A_g */
        #pragma omp parallel for schedule(static)
        for (int n = 0; n < N; n++) {
            const uint8_t* row = B + ((size_t)g * N + n) * kb;
            const uint8_t* srow = B_sf + ((size_t)g * N + n) * ks;
            for (int k = 0; k < K; k++) Bd[(size_t)n * K + k] = elem(row, srow, k);
        }
        #pragma omp parallel for schedule(static)
        for (int m = 0; m < mm; m++) {
            const uint8_t* row = A + ((size_t)g * M_max + m) * kb;
            const uint8_t* srow = A_sf + ((size_t)g * M_max + m) * ks;
            for (int k = 0; k < K; k++) Ad[(size_t)m * K + k] = elem(row, srow, k);
        }
        double al = (double)alpha[g];
        #pragma omp parallel for collapse(2) schedule(dynamic, 16)
        for (int m = 0; m < mm; m++) {
            for (int n = 0; n < N; n++) {
                const double* a = Ad + (size_t)m * K;
                const double* b = Bd + (size_t)n * K;
                double acc = 0.0;
                for (int k = 0; k < K; k++) acc += a[k] * b[k];
                double v = al * acc;
                size_t o = ((size_t)g * M_max + m) * N + n;
                if (ref64) ref64[o] = v;
                C[o] = nvfp4o_bf16_rne(v);
            }
        }
    }
    free(Bd);
    free(Ad);
    return 0;
}

/*
 * Sampled oracle: for each of `count` triples idx[3i..3i+2] = (g, m, n) it
 * writes out[i] = alpha[g] * sum_k a(g,m,k) b(g,n,k) in fp64 (unrounded),
 * decoding elements on the fly.  The caller picks only valid (g, m, n).
 */
int nvfp4o_gemm_sampled(const uint8_t* A, const uint8_t* A_sf, const uint8_t* B,
                        const uint8_t* B_sf, const float* alpha,
                        const int64_t* idx, int64_t count, double* out,
                        int G, int M_max, int N, int K, int nthreads) {
    if (G <= 0 || M_max <= 0 || N <= 0 || K <= 0 || (K % 16) != 0) return -1;
    for (int64_t i = 0; i < count; i++) {
        int64_t g = idx[3 * i], m = idx[3 * i + 1], n = idx[3 * i + 2];
        if (g < 0 || g >= G || m < 0 || m >= M_max || n < 0 || n >= N) return -1;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const size_t kb = (size_t)K / 2, ks = (size_t)K / 16;
    #pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; i++) {
        int64_t g = idx[3 * i], m = idx[3 * i + 1], n = idx[3 * i + 2];
        const uint8_t* arow = A + ((size_t)g * M_max + m) * kb;
        const uint8_t* asf = A_sf + ((size_t)g * M_max + m) * ks;
        const uint8_t* brow = B + ((size_t)g * N + n) * kb;
        const uint8_t* bsf = B_sf + ((size_t)g * N + n) * ks;
        double acc = 0.0;
        for (int k = 0; k < K; k++) acc += elem(arow, asf, k) * elem(brow, bsf, k);
        out[i] = (double)alpha[g] * acc;
    }
    return 0;
}
