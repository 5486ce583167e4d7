/*
 * fp64 GEMM oracle: C = A . B and Cabs = |A| . |B| from exactly dequantised operands.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Plain loops, fp64 accumulation in
 * increasing k, no blocking and no reordering; OpenMP only splits the output rows.
 * Compiled with -ffp-contract=off so the multiply and the add round separately on every
 * host.
 *
 * Operand layouts (row-major, leading dimensions in elements):
 *   A: M x K, lda >= K
 *   B: K x N with ldb >= N when b_kn != 0, else N x K with ldb >= K
 * Outputs: for each requested row r (index rows[r] of A) the full row of C and Cabs,
 * stored densely as nrows x N.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

void oracle_gemm_rows_f64(const double* A, int64_t lda, const double* B, int64_t ldb,
                          int b_kn, int64_t N, int64_t K, const int64_t* rows,
                          int64_t nrows, double* C, double* Cabs) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const double* a = A + rows[r] * lda;
        double* c = C + r * N;
        double* cab = Cabs + r * N;
        for (int64_t j = 0; j < N; ++j) {
            c[j] = 0.0;
            cab[j] = 0.0;
        }
        if (b_kn) {
            for (int64_t k = 0; k < K; ++k) {
                const double av = a[k];
                const double aa = fabs(av);
                const double* b = B + k * ldb;
                for (int64_t j = 0; j < N; ++j) {
                    c[j] += av * b[j];
                    cab[j] += aa * fabs(b[j]);
                }
            }
        } else {
            for (int64_t j = 0; j < N; ++j) {
                const double* b = B + j * ldb;
                double s = 0.0, sa = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    s += a[k] * b[k];
                    sa += fabs(a[k]) * fabs(b[k]);
                }
                c[j] = s;
                cab[j] = sa;
            }
        }
    }
}

/* Single entries C[i][j] for a list of (i, j) pairs. */
void oracle_gemm_entries_f64(const double* A, int64_t lda, const double* B, int64_t ldb,
                             int b_kn, int64_t K, const int64_t* ii, const int64_t* jj,
                             int64_t n, double* C, double* Cabs) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < n; ++p) {
        const double* a = A + ii[p] * lda;
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double bv = b_kn ? B[k * ldb + jj[p]] : B[jj[p] * ldb + k];
            s += a[k] * bv;
            sa += fabs(a[k]) * fabs(bv);
        }
        C[p] = s;
        Cabs[p] = sa;
    }
}
