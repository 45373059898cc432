/*
 * Reference oracle for the bf16 -> fp32 tiled GEMM: TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load this file's shared object.  The product path (the CUDA
 * library) never calls it, and it shares no source with that library.
 *
 * What it computes.  The contraction every page of the method is about,
 * written out from its plain definition:
 *
 *     C_b[i][j] = sum_{k=0}^{K-1} A_b[i][k] * B_b[k][j]
 *
 *   - LuisaCompute "Pipelines and stage boundaries", section "Stage boundaries
 *     are lexical": the k-tile example accumulates acc = mma(a, b, acc) over
 *     the k tiles of A and B.
 *   - LuisaCompute "Execution Nests and coordinates", section "Dimensions and
 *     spaces": A carries dims (m, reduction), B (reduction, n), C (m, n).
 *   - OCANNL "Module Ir.Schedule", Tensorize: the micro-kernel body is
 *     d[i, j] += a[i, k] * b[k, j].
 *
 * The tiling, padding, pipelining and split-K of the method all reach this
 * same mathematical value; they only change the rounding order (OCANNL
 * "Module Ir.Schedule", Interchange and the two-pass split reduction license
 * that reassociation).  So the oracle has no tiles, no pad and no split: one
 * i-k-j triple loop whose accumulator is an fp64 row buffer, and a dot-product
 * form for sampled entries (k ascending).
 *
 * Precision.  Inputs are bf16 bit patterns (uint16).  Widening bf16 -> fp32 ->
 * fp64 is exact (a bf16 value is the top half of an fp32 pattern).  A product
 * of two bf16 values has at most 16 significant bits and is exact in fp64, so
 * the only rounding is in the fp64 running sum.
 *
 * Layout.  Row-major, element strides: A_b[i][k] = A[b*sA + i*lda + k],
 * B_b[k][j] = B[b*sB + k*ldb + j], C_b[i][j] = C[b*sC + i*ldc + j].
 *
 * Build: plain C99 + OpenMP, compiled with -ffp-contract=off so that x86 and
 * aarch64 builds produce identical bits (no fused multiply-add contraction).
 * OpenMP splits the (b, i) rows; each row's sum order is fixed, so the result
 * does not depend on the thread count.
 */
#include <stdint.h>
#include <string.h>

static double widen_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Full product.  Returns 0 on success, -1 on a negative extent or stride
 * smaller than its row length.  C is overwritten (no accumulation into it). */
int oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *C,
                    int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc,
                    int64_t batch, int64_t sA, int64_t sB, int64_t sC)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0) return -1;
    if (lda < K || ldb < N || ldc < N) return -1;
    const int64_t rows = batch * M;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t b = r / M;
        const int64_t i = r % M;
        const uint16_t *a_row = A + b * sA + i * lda;
        double *c_row = C + b * sC + i * ldc;
        for (int64_t j = 0; j < N; ++j) c_row[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = widen_bf16(a_row[k]);
            const uint16_t *b_row = B + b * sB + k * ldb;
            for (int64_t j = 0; j < N; ++j) c_row[j] += a * widen_bf16(b_row[j]);
        }
    }
    return 0;
}

/* Sampled entries: out[t] = C_{bi[t]}[ii[t]][jj[t]], each one dot product
 * over k = 0 .. K-1 in ascending order.  Returns -1 on an index outside the
 * problem. */
int oracle_gemm_entries_f64(const uint16_t *A, const uint16_t *B,
                            int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb,
                            int64_t batch, int64_t sA, int64_t sB,
                            const int64_t *bi, const int64_t *ii, const int64_t *jj,
                            int64_t count, double *out)
{
    for (int64_t t = 0; t < count; ++t)
        if (bi[t] < 0 || bi[t] >= batch || ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N)
            return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t *a_row = A + bi[t] * sA + ii[t] * lda;
        const uint16_t *b_col = B + bi[t] * sB + jj[t];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += widen_bf16(a_row[k]) * widen_bf16(b_col[k * ldb]);
        out[t] = acc;
    }
    return 0;
}

/* Thread count OpenMP will use for the loops above (for reporting). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
