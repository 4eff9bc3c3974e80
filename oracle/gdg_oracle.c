/*
 * fp64 CPU oracle of the ragged BF16 grouped GEMM -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code with the CUDA library: it is a
 * plain, slow, obviously correct restatement of the computation table of the
 * "Cake ragged BF16 grouped GEMM (experimental)" docs page:
 *
 *   fwd    Y[s_e:t_e]  = X[s_e:t_e] @ W[e].T          -> [rows, N]
 *   dgrad  dX[s_e:t_e] = G[s_e:t_e] @ W[e]  (W as stored) -> [rows, K]
 *   wgrad  dW[e]       = G[s_e:t_e].T @ X[s_e:t_e]    -> [E, N, K]
 *
 * with group e covering rows [s_e, t_e): s_e = offs[e-1] (0 for e = 0) and
 * t_e = offs[e] for cumulative ends, or s_e = m_indptr[e], t_e =
 * m_indptr[e+1] for the leading-zero form (same page, intro paragraph).
 * An empty group gives an exactly zero weight gradient (same paragraph).
 *
 * Inputs are raw bf16 bit patterns; each value is widened exactly to double
 * and every sum runs in ascending index order in double precision.  Rows
 * that belong to no group are never written by fwd / dgrad.  Offsets must
 * be non-decreasing and inside [0, rows]; anything else is rejected (-1).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OFFS_ENDS 0
#define OFFS_INDPTR 1

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Group row ranges from the offsets; -1 when they are not a valid
 * non-decreasing partition of a sub-range of [0, rows]. */
int gdg_oracle_bounds(const int32_t* offs, int offs_kind, int E, int64_t rows,
                      int64_t* start, int64_t* end) {
    if (E < 1 || rows < 0 || (offs_kind != OFFS_ENDS && offs_kind != OFFS_INDPTR)) return -1;
    int64_t prev = (offs_kind == OFFS_ENDS) ? 0 : (int64_t)offs[0];
    if (prev < 0 || prev > rows) return -1;
    for (int e = 0; e < E; ++e) {
        int64_t t = (offs_kind == OFFS_ENDS) ? (int64_t)offs[e] : (int64_t)offs[e + 1];
        if (t < prev || t > rows) return -1;
        start[e] = prev;
        end[e] = t;
        prev = t;
    }
    return 0;
}

/* Group of row i, or -1 if the row lies outside every group. */
static int group_of_row(const int64_t* start, const int64_t* end, int E, int64_t i) {
    for (int e = 0; e < E; ++e)
        if (i >= start[e] && i < end[e]) return e;
    return -1;
}

/* Y[i, n] = sum_k x(i, k) w(e, n, k) for one row i of group e. */
static void fwd_row(const uint16_t* X, const uint16_t* W, int e, int64_t i, int N, int K,
                    double* yrow) {
    const uint16_t* xr = X + i * (int64_t)K;
    for (int n = 0; n < N; ++n) {
        const uint16_t* wr = W + ((int64_t)e * N + n) * (int64_t)K;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += bf16_to_double(xr[k]) * bf16_to_double(wr[k]);
        yrow[n] = acc;
    }
}

/* dX[i, k] = sum_n g(i, n) w(e, n, k): W is used as stored, [N, K]. */
static void dgrad_row(const uint16_t* G, const uint16_t* W, int e, int64_t i, int N, int K,
                      double* dxrow) {
    const uint16_t* gr = G + i * (int64_t)N;
    for (int k = 0; k < K; ++k) dxrow[k] = 0.0;
    for (int n = 0; n < N; ++n) {
        double g = bf16_to_double(gr[n]);
        const uint16_t* wr = W + ((int64_t)e * N + n) * (int64_t)K;
        for (int k = 0; k < K; ++k) dxrow[k] += g * bf16_to_double(wr[k]);
    }
}

int gdg_oracle_fwd(const uint16_t* X, const uint16_t* W, const int32_t* offs, int offs_kind,
                   int64_t rows, int E, int N, int K, double* Y) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    for (int e = 0; e < E; ++e) {
        int64_t s = st[e], t = en[e];
        #pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = s; i < t; ++i) fwd_row(X, W, e, i, N, K, Y + i * (int64_t)N);
    }
    free(st);
    return 0;
}

int gdg_oracle_dgrad(const uint16_t* G, const uint16_t* W, const int32_t* offs, int offs_kind,
                     int64_t rows, int E, int N, int K, double* dX) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    for (int e = 0; e < E; ++e) {
        int64_t s = st[e], t = en[e];
        #pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = s; i < t; ++i) dgrad_row(G, W, e, i, N, K, dX + i * (int64_t)K);
    }
    free(st);
    return 0;
}

/* dW[e, n, k] = sum over rows i of group e, ascending, of g(i, n) x(i, k);
 * exactly 0 for an empty group. */
int gdg_oracle_wgrad(const uint16_t* G, const uint16_t* X, const int32_t* offs, int offs_kind,
                     int64_t rows, int E, int N, int K, double* dW) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    for (int e = 0; e < E; ++e) {
        int64_t s = st[e], t = en[e];
        #pragma omp parallel for schedule(dynamic, 1)
        for (int n = 0; n < N; ++n) {
            double* out = dW + ((int64_t)e * N + n) * (int64_t)K;
            for (int k = 0; k < K; ++k) out[k] = 0.0;
            for (int64_t i = s; i < t; ++i) {
                double g = bf16_to_double(G[i * (int64_t)N + n]);
                const uint16_t* xr = X + i * (int64_t)K;
                for (int k = 0; k < K; ++k) out[k] += g * bf16_to_double(xr[k]);
            }
        }
    }
    free(st);
    return 0;
}

/* Sampled forms for large shapes: the same sums, evaluated only where asked.
 * row_group[j] receives the group of row_ids[j] (-1: no group, row skipped). */
int gdg_oracle_fwd_rows(const uint16_t* X, const uint16_t* W, const int32_t* offs, int offs_kind,
                        int64_t rows, int E, int N, int K, const int64_t* row_ids,
                        int64_t n_ids, double* Yrows, int32_t* row_group) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_ids; ++j) {
        int e = (row_ids[j] >= 0 && row_ids[j] < rows) ? group_of_row(st, en, E, row_ids[j]) : -1;
        row_group[j] = e;
        if (e >= 0) fwd_row(X, W, e, row_ids[j], N, K, Yrows + j * (int64_t)N);
    }
    free(st);
    return 0;
}

int gdg_oracle_dgrad_rows(const uint16_t* G, const uint16_t* W, const int32_t* offs,
                          int offs_kind, int64_t rows, int E, int N, int K,
                          const int64_t* row_ids, int64_t n_ids, double* dXrows,
                          int32_t* row_group) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_ids; ++j) {
        int e = (row_ids[j] >= 0 && row_ids[j] < rows) ? group_of_row(st, en, E, row_ids[j]) : -1;
        row_group[j] = e;
        if (e >= 0) dgrad_row(G, W, e, row_ids[j], N, K, dXrows + j * (int64_t)K);
    }
    free(st);
    return 0;
}

/* ids are flat indices e*N*K + n*K + k into dW. */
int gdg_oracle_wgrad_entries(const uint16_t* G, const uint16_t* X, const int32_t* offs,
                             int offs_kind, int64_t rows, int E, int N, int K,
                             const int64_t* ids, int64_t n_ids, double* vals) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    const int64_t NK = (int64_t)N * K;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t j = 0; j < n_ids; ++j) {
        int64_t id = ids[j];
        int e = (int)(id / NK);
        int n = (int)((id % NK) / K);
        int k = (int)(id % K);
        double acc = 0.0;
        for (int64_t i = st[e]; i < en[e]; ++i)
            acc += bf16_to_double(G[i * (int64_t)N + n]) * bf16_to_double(X[i * (int64_t)K + k]);
        vals[j] = acc;
    }
    free(st);
    return 0;
}

/* Whole dW rows dW[e, n, :] for the listed (e, n) pairs (pair j = ids[2j], ids[2j+1]);
 * the same ascending-row sums as gdg_oracle_wgrad. */
int gdg_oracle_wgrad_rows(const uint16_t* G, const uint16_t* X, const int32_t* offs,
                          int offs_kind, int64_t rows, int E, int N, int K,
                          const int64_t* ids, int64_t n_ids, double* vals) {
    int64_t* st = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)E);
    if (!st) return -2;
    int64_t* en = st + E;
    if (gdg_oracle_bounds(offs, offs_kind, E, rows, st, en)) { free(st); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_ids; ++j) {
        int e = (int)ids[2 * j], n = (int)ids[2 * j + 1];
        double* out = vals + j * (int64_t)K;
        for (int k = 0; k < K; ++k) out[k] = 0.0;
        for (int64_t i = st[e]; i < en[e]; ++i) {
            double g = bf16_to_double(G[i * (int64_t)N + n]);
            const uint16_t* xr = X + i * (int64_t)K;
            for (int k = 0; k < K; ++k) out[k] += g * bf16_to_double(xr[k]);
        }
    }
    free(st);
    return 0;
}

int gdg_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
