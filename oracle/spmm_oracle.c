/*
 * spmm_oracle.c -- plain CPU reference for C = A_sparse * B_dense.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (the definition the fast kernels must reproduce): for every
 * element (i, k, a) that the sparse format stores, C[i][n] += a * B[k][n] for
 * every output column n.  Products and sums are in fp64 (int64 for int8
 * operands) and each output row is summed in stored order, which for all four
 * formats is ascending k.  This equals densify(A) @ B exactly up to rounding
 * order, since explicitly stored zeros add exact zeros.
 *   - SpMM over block-sparse (BCSR) and row-window (WCSR) operands:
 *     "AsyncSparse: Accelerating Sparse Matrix-Matrix Multiplication on
 *     Asynchronous GPU Architectures", abstract and Fig. 2 (BCSR vs WCSR).
 *   - 2:4 semi-structured and tile-vector-wise (TVW) operands:
 *     "Accelerating Sparse DNNs Based on Tiled GEMM", abstract (tile-wise
 *     pruning at global-memory level, 2:4 inside the sparse tensor core).
 *
 * Readings where the pages are silent (format layouts, padding rules) are the
 * ones listed in the repository's design notes; each builder below states the
 * reading it implements.  Every function is a direct transcription of the
 * definition: no blocking, no fusion, no reordering beyond "ascending k".
 *
 * Element encodings: dtype 0 = bf16 bits (uint16), 1 = fp16 bits (uint16),
 * 2 = int8, 3 = fp8 E4M3 bits (uint8), 4 = fp8 E5M2 bits (uint8).  A stored
 * element is "zero" iff it compares equal to 0 in IEEE arithmetic (so -0.0 is
 * zero, NaN is nonzero); for int8 iff it is 0.
 *
 * The 8-bit floating-point types are the ones the pages pair with 2:4 on
 * recent GPUs ("Spense", abstract on the "sparse FP4 GEMM" search page: 2:4
 * sparse tensor cores on B200 in FP8; "SlideSparse", same page: FP8 among its
 * precisions).  The pages do not define the encodings; the reading taken is
 * the two 8-bit formats of the OCP 8-bit floating-point specification, which
 * is what the tensor core's e4m3 / e5m2 operand types implement:
 *   E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0 is
 *         subnormal (m * 2^-9); S.1111.111 is NaN; no infinities (max 448).
 *   E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits; exponent field 0 is
 *         subnormal (m * 2^-16); exponent field 31 is infinity (m = 0) or NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_I8 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4 };
enum { ORC_OK = 0, ORC_ERR_SHAPE = 2, ORC_ERR_FORMAT = 4 };

/* ------------------------------------------------------------------ values */

double orc_decode_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_decode_f16(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* OCP E4M3: (-1)^s * 2^(e-7) * (1 + m/8) for e = 1..15 (except e = 15, m = 7:
 * NaN), (-1)^s * m * 2^-9 for e = 0. */
double orc_decode_e4m3(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(m + 8), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP E5M2: (-1)^s * 2^(e-15) * (1 + m/4) for e = 1..30, m * 2^-16 for e = 0,
 * infinity (m = 0) or NaN for e = 31. */
double orc_decode_e5m2(uint8_t b) {
    int sign = b >> 7, e = (b >> 2) & 31, m = b & 3;
    double v;
    if (e == 0)
        v = ldexp((double)m, -16);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 4), e - 17);        /* (1 + m/4) * 2^(e-15) */
    return sign ? -v : v;
}

static int is_byte_type(int dtype) { return dtype == ORC_I8 || dtype == ORC_E4M3 || dtype == ORC_E5M2; }

static int esize(int dtype) { return is_byte_type(dtype) ? 1 : 2; }

static double get_f(const void *p, int64_t idx, int dtype) {
    if (dtype == ORC_BF16) return orc_decode_bf16(((const uint16_t *)p)[idx]);
    if (dtype == ORC_F16) return orc_decode_f16(((const uint16_t *)p)[idx]);
    if (dtype == ORC_E4M3) return orc_decode_e4m3(((const uint8_t *)p)[idx]);
    if (dtype == ORC_E5M2) return orc_decode_e5m2(((const uint8_t *)p)[idx]);
    return (double)((const int8_t *)p)[idx];
}

static int64_t get_i(const void *p, int64_t idx) { return (int64_t)((const int8_t *)p)[idx]; }

static int is_zero(const void *p, int64_t idx, int dtype) {
    if (dtype == ORC_I8) return ((const int8_t *)p)[idx] == 0;
    if (dtype == ORC_E4M3 || dtype == ORC_E5M2) return (((const uint8_t *)p)[idx] & 0x7F) == 0;
    return (((const uint16_t *)p)[idx] & 0x7FFF) == 0;   /* +0.0 or -0.0 */
}

static void copy_elem(void *dst, int64_t di, const void *src, int64_t si, int dtype) {
    if (is_byte_type(dtype)) ((uint8_t *)dst)[di] = ((const uint8_t *)src)[si];
    else ((uint16_t *)dst)[di] = ((const uint16_t *)src)[si];
}

static void zero_elem(void *dst, int64_t di, int dtype) {
    if (is_byte_type(dtype)) ((uint8_t *)dst)[di] = 0;
    else ((uint16_t *)dst)[di] = 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Output selection shared by every SpMM below: rows [r0, r1) of C and either
 * all N columns (cols == NULL, ncols == N) or the listed columns.  The result
 * block is (r1 - r0) x ncols, row-major with leading dimension ncols. */
#define OUTCOL(j) (cols ? cols[j] : (j))

/* ================================================================== BCSR
 * Reading: A (M x K) is cut into bh x bw blocks; a block is stored iff one of
 * its entries is nonzero.  Block rows ascending, block columns ascending in a
 * row.  row_ptr[M/bh + 1], col_idx[nnzb] (block-column index), vals[nnzb][bh][bw]
 * row-major inside a block.  M % bh == 0 and K % bw == 0 are required.
 */
static int block_nonzero(const void *A, int64_t ld, int64_t br, int64_t bc, int bh, int bw, int dtype) {
    for (int r = 0; r < bh; r++)
        for (int c = 0; c < bw; c++)
            if (!is_zero(A, (br * bh + r) * ld + bc * bw + c, dtype)) return 1;
    return 0;
}

int64_t orc_bcsr_count(const void *A, int64_t M, int64_t K, int64_t ld, int bh, int bw, int dtype,
                       int32_t *row_ptr) {
    if (bh <= 0 || bw <= 0 || M % bh || K % bw) return -ORC_ERR_SHAPE;
    int64_t gm = M / bh, gk = K / bw, n = 0;
    row_ptr[0] = 0;
    for (int64_t br = 0; br < gm; br++) {
        for (int64_t bc = 0; bc < gk; bc++) n += block_nonzero(A, ld, br, bc, bh, bw, dtype);
        row_ptr[br + 1] = (int32_t)n;
    }
    return n;
}

int orc_bcsr_fill(const void *A, int64_t M, int64_t K, int64_t ld, int bh, int bw, int dtype,
                  const int32_t *row_ptr, int32_t *col_idx, void *vals) {
    if (bh <= 0 || bw <= 0 || M % bh || K % bw) return ORC_ERR_SHAPE;
    int64_t gm = M / bh, gk = K / bw;
    for (int64_t br = 0; br < gm; br++) {
        int64_t j = row_ptr[br];
        for (int64_t bc = 0; bc < gk; bc++) {
            if (!block_nonzero(A, ld, br, bc, bh, bw, dtype)) continue;
            col_idx[j] = (int32_t)bc;
            for (int r = 0; r < bh; r++)
                for (int c = 0; c < bw; c++)
                    copy_elem(vals, (j * bh + r) * bw + c, A, (br * bh + r) * ld + bc * bw + c, dtype);
            j++;
        }
    }
    return ORC_OK;
}

void orc_bcsr_densify(int64_t M, int64_t K, int bh, int bw, int dtype, const int32_t *row_ptr,
                      const int32_t *col_idx, const void *vals, void *D) {
    memset(D, 0, (size_t)(M * K * esize(dtype)));
    for (int64_t br = 0; br < M / bh; br++)
        for (int64_t j = row_ptr[br]; j < row_ptr[br + 1]; j++)
            for (int r = 0; r < bh; r++)
                for (int c = 0; c < bw; c++)
                    copy_elem(D, (br * bh + r) * K + (int64_t)col_idx[j] * bw + c, vals,
                              (j * bh + r) * bw + c, dtype);
}

/* C[i][n] = sum over stored blocks j of block row i/bh, over c in [0, bw):
 *           vals[j][i % bh][c] * B[col_idx[j]*bw + c][n]   (fp64). */
void orc_bcsr_spmm(int64_t M, int64_t K, int bh, int bw, int dtype, const int32_t *row_ptr,
                   const int32_t *col_idx, const void *vals, const void *B, int64_t ldb,
                   int64_t r0, int64_t r1, const int64_t *cols, int64_t ncols, double *C) {
    (void)M; (void)K;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = r0; i < r1; i++) {
        double *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0.0;
        int64_t br = i / bh, r = i % bh;
        for (int64_t j = row_ptr[br]; j < row_ptr[br + 1]; j++)
            for (int c = 0; c < bw; c++) {
                double a = get_f(vals, (j * bh + r) * bw + c, dtype);
                int64_t k = (int64_t)col_idx[j] * bw + c;
                for (int64_t q = 0; q < ncols; q++) out[q] += a * get_f(B, k * ldb + OUTCOL(q), dtype);
            }
    }
}

/* ================================================================== CSR
 * Row-wise CSR SpMM, the textbook special case (used as the h = 1 check of
 * the row-window format and as a plain reference for CSR inputs). */
int orc_csr_check(int64_t M, int64_t K, const int32_t *row_ptr, const int32_t *col) {
    if (row_ptr[0] != 0) return ORC_ERR_FORMAT;
    for (int64_t i = 0; i < M; i++) {
        if (row_ptr[i + 1] < row_ptr[i]) return ORC_ERR_FORMAT;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; e++) {
            if (col[e] < 0 || col[e] >= K) return ORC_ERR_FORMAT;
            if (e > row_ptr[i] && col[e] <= col[e - 1]) return ORC_ERR_FORMAT;
        }
    }
    return ORC_OK;
}

void orc_csr_spmm(int64_t M, int dtype, const int32_t *row_ptr, const int32_t *col, const void *val,
                  const void *B, int64_t ldb, int64_t r0, int64_t r1, const int64_t *cols,
                  int64_t ncols, double *C) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = r0; i < r1; i++) {
        double *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0.0;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; e++) {
            double a = get_f(val, e, dtype);
            for (int64_t q = 0; q < ncols; q++) out[q] += a * get_f(B, (int64_t)col[e] * ldb + OUTCOL(q), dtype);
        }
    }
}

/* ================================================================== WCSR
 * Reading (row windows): rows are grouped into windows of h consecutive rows
 * (the last window may be shorter).  Per window w:
 *   wcols[wcol_ptr[w] .. wcol_ptr[w+1])   the window's distinct columns, ascending
 *   T_w = number of distinct columns; they form ceil(T_w / 16) column tiles;
 *   the window is split into U_w = max(1, ceil(T_w / (16*S))) work units, unit
 *   u covering column slots [16*S*u, 16*S*(u+1)).
 * Per stored nonzero (window-major; inside a window unit-major, then row, then
 * column):  lrow = row - h*w,  slot = index of its column in the window's wcols,
 * val = its value.  wnz_ptr[w] = first nonzero of window w (equals the CSR
 * row_ptr at row h*w); unit_ptr[w] = first unit of window w; for unit u:
 * unit_win[u] = its window, unit_nz_ptr[u] = its first nonzero.
 */
static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static int64_t window_unique(const int32_t *row_ptr, const int32_t *col, int64_t rb, int64_t re,
                             int32_t *tmp) {
    int64_t n = 0;
    for (int64_t e = row_ptr[rb]; e < row_ptr[re]; e++) tmp[n++] = col[e];
    qsort(tmp, (size_t)n, sizeof(int32_t), cmp_i32);
    int64_t u = 0;
    for (int64_t i = 0; i < n; i++)
        if (u == 0 || tmp[i] != tmp[u - 1]) tmp[u++] = tmp[i];
    return u;
}

static int64_t find_slot(const int32_t *w, int64_t n, int32_t c) {
    int64_t lo = 0, hi = n;                     /* first index with w[idx] >= c */
    while (lo < hi) { int64_t mid = (lo + hi) / 2; if (w[mid] < c) lo = mid + 1; else hi = mid; }
    return lo;
}

int orc_wcsr_sizes(int64_t M, int64_t K, const int32_t *row_ptr, const int32_t *col, int h, int S,
                   int64_t *n_wcols, int64_t *n_units) {
    if (h <= 0 || h > 256 || S <= 0) return ORC_ERR_SHAPE;
    if (orc_csr_check(M, K, row_ptr, col) != ORC_OK) return ORC_ERR_FORMAT;
    int64_t nw = (M + h - 1) / h, tw = 0, tu = 0, span = 16 * (int64_t)S;
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(row_ptr[M] + 1));
    for (int64_t w = 0; w < nw; w++) {
        int64_t rb = w * h, re = rb + h < M ? rb + h : M;
        int64_t T = window_unique(row_ptr, col, rb, re, tmp);
        tw += T;
        tu += T ? (T + span - 1) / span : 1;
    }
    free(tmp);
    *n_wcols = tw;
    *n_units = tu;
    return ORC_OK;
}

int orc_wcsr_fill(int64_t M, int64_t K, int dtype, const int32_t *row_ptr, const int32_t *col,
                  const void *val, int h, int S, int32_t *wcol_ptr, int32_t *wcols, int32_t *wnz_ptr,
                  int32_t *unit_ptr, int32_t *unit_win, int32_t *unit_nz_ptr, uint8_t *lrow,
                  int32_t *slot, void *wval) {
    if (h <= 0 || h > 256 || S <= 0) return ORC_ERR_SHAPE;
    if (orc_csr_check(M, K, row_ptr, col) != ORC_OK) return ORC_ERR_FORMAT;
    int64_t nw = (M + h - 1) / h, span = 16 * (int64_t)S;
    int64_t cw = 0, cu = 0, cz = 0;
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(row_ptr[M] + 1));
    for (int64_t w = 0; w < nw; w++) {
        int64_t rb = w * h, re = rb + h < M ? rb + h : M;
        int32_t *wc = wcols + cw;
        /* collect and de-duplicate in scratch, then copy the T distinct columns */
        int64_t T = window_unique(row_ptr, col, rb, re, tmp);
        for (int64_t t = 0; t < T; t++) wc[t] = tmp[t];
        int64_t U = T ? (T + span - 1) / span : 1;
        wcol_ptr[w] = (int32_t)cw;
        wnz_ptr[w] = (int32_t)cz;
        unit_ptr[w] = (int32_t)cu;
        for (int64_t u = 0; u < U; u++) {
            unit_win[cu + u] = (int32_t)w;
            unit_nz_ptr[cu + u] = (int32_t)cz;
            for (int64_t r = rb; r < re; r++)
                for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; e++) {
                    int64_t s = find_slot(wc, T, col[e]);
                    if (s / span != u) continue;
                    lrow[cz] = (uint8_t)(r - rb);
                    slot[cz] = (int32_t)s;
                    copy_elem(wval, cz, val, e, dtype);
                    cz++;
                }
        }
        cw += T;
        cu += U;
    }
    free(tmp);
    wcol_ptr[nw] = (int32_t)cw;
    wnz_ptr[nw] = (int32_t)cz;
    unit_ptr[nw] = (int32_t)cu;
    unit_nz_ptr[cu] = (int32_t)cz;
    return ORC_OK;
}

/* Back to CSR (round-trip check): every window's nonzeros regrouped by row,
 * columns ascending. */
void orc_wcsr_to_csr(int64_t M, int h, int dtype, const int32_t *wcol_ptr, const int32_t *wcols,
                     const int32_t *wnz_ptr, const uint8_t *lrow, const int32_t *slot,
                     const void *wval, int32_t *row_ptr, int32_t *col, void *val) {
    int64_t nw = (M + h - 1) / h;
    int64_t *cnt = (int64_t *)calloc((size_t)M + 1, sizeof(int64_t));
    for (int64_t w = 0; w < nw; w++)
        for (int64_t e = wnz_ptr[w]; e < wnz_ptr[w + 1]; e++) cnt[w * h + lrow[e] + 1]++;
    row_ptr[0] = 0;
    for (int64_t i = 0; i < M; i++) row_ptr[i + 1] = (int32_t)(row_ptr[i] + cnt[i + 1]);
    /* columns ascending inside a row: visit each window's slots in ascending
     * order and append to the row's cursor */
    int64_t *cur = (int64_t *)malloc(sizeof(int64_t) * (size_t)(M + 1));
    for (int64_t i = 0; i < M; i++) cur[i] = row_ptr[i];
    for (int64_t w = 0; w < nw; w++) {
        int64_t T = wcol_ptr[w + 1] - wcol_ptr[w];
        for (int64_t s = 0; s < T; s++)
            for (int64_t e = wnz_ptr[w]; e < wnz_ptr[w + 1]; e++) {
                if (slot[e] != s) continue;
                int64_t i = w * h + lrow[e];
                col[cur[i]] = wcols[wcol_ptr[w] + s];
                copy_elem(val, cur[i], wval, e, dtype);
                cur[i]++;
            }
    }
    free(cur);
    free(cnt);
}

/* C[i][n] = sum over the stored nonzeros of row i (window i/h, lrow i%h), in
 * stored order: val * B[wcols[wcol_ptr[w] + slot]][n]. */
void orc_wcsr_spmm(int64_t M, int h, int dtype, const int32_t *wcol_ptr, const int32_t *wcols,
                   const int32_t *wnz_ptr, const uint8_t *lrow, const int32_t *slot, const void *wval,
                   const void *B, int64_t ldb, int64_t r0, int64_t r1, const int64_t *cols,
                   int64_t ncols, double *C) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = r0; i < r1; i++) {
        double *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0.0;
        int64_t w = i / h;
        for (int64_t e = wnz_ptr[w]; e < wnz_ptr[w + 1]; e++) {
            if (w * h + lrow[e] != i) continue;
            double a = get_f(wval, e, dtype);
            int64_t k = wcols[wcol_ptr[w] + slot[e]];
            for (int64_t q = 0; q < ncols; q++) out[q] += a * get_f(B, k * ldb + OUTCOL(q), dtype);
        }
    }
}

/* ================================================================== 2:4
 * Reading: in every group of 4 consecutive K entries at most 2 are nonzero.
 * Stored per row: vals[K/2] (the two kept entries of group g at 2g, 2g+1) and
 * meta[K/8] bytes; group g's nibble is idx0 | idx1 << 2 with idx0 < idx1 the
 * kept positions inside the group; groups 2j and 2j+1 share byte j (low, high
 * nibble).  A group with fewer than 2 nonzeros keeps its nonzero positions
 * plus the lowest-index zero positions.  K % 4 != 0 -> shape error; more than
 * 2 nonzeros in a group -> format error.
 */
static int compress_group(const void *src, int64_t base, int64_t stride, int dtype, int *i0, int *i1) {
    int nz[4], n = 0;
    for (int p = 0; p < 4; p++)
        if (!is_zero(src, base + p * stride, dtype)) nz[n++] = p;
    if (n > 2) return ORC_ERR_FORMAT;
    int keep[4] = {0, 0, 0, 0};
    for (int t = 0; t < n; t++) keep[nz[t]] = 1;
    for (int p = 0; p < 4 && n < 2; p++)
        if (!keep[p]) { keep[p] = 1; n++; }
    int t = 0, idx[2];
    for (int p = 0; p < 4; p++)
        if (keep[p]) idx[t++] = p;
    *i0 = idx[0];
    *i1 = idx[1];
    return ORC_OK;
}

int orc_compress24(const void *A, int64_t M, int64_t K, int64_t ld, int dtype, void *vals, uint8_t *meta) {
    if (K % 4) return ORC_ERR_SHAPE;
    int64_t G = K / 4, lm = (K + 7) / 8;
    for (int64_t i = 0; i < M; i++) {
        for (int64_t j = 0; j < lm; j++) meta[i * lm + j] = 0;
        for (int64_t g = 0; g < G; g++) {
            int i0, i1;
            if (compress_group(A, i * ld + 4 * g, 1, dtype, &i0, &i1) != ORC_OK) return ORC_ERR_FORMAT;
            copy_elem(vals, i * (K / 2) + 2 * g, A, i * ld + 4 * g + i0, dtype);
            copy_elem(vals, i * (K / 2) + 2 * g + 1, A, i * ld + 4 * g + i1, dtype);
            meta[i * lm + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
        }
    }
    return ORC_OK;
}

/* Magnitude of element idx as an unsigned key that orders by |a|: |v| for int8
 * (0..128); for bf16/fp16/fp8 the bit pattern without its sign bit, which orders
 * finite values and infinities by magnitude and puts NaN above every number. */
static unsigned mag_key(const void *p, int64_t idx, int dtype) {
    if (dtype == ORC_I8) {
        int v = ((const int8_t *)p)[idx];
        return (unsigned)(v < 0 ? -v : v);
    }
    if (dtype == ORC_E4M3 || dtype == ORC_E5M2) return ((const uint8_t *)p)[idx] & 0x7Fu;
    return ((const uint16_t *)p)[idx] & 0x7FFFu;
}

/* Magnitude pruning into 2:4 ("Accelerating Sparse DNNs Based on Tiled GEMM",
 * abstract: pruning into the sparse tensor core's 2:4 pattern).  Reading: in
 * every group of 4 consecutive K entries keep the two of largest magnitude,
 * ties going to the lower index; store them in ascending index order with the
 * nibble idx0 | idx1 << 2, exactly as the 2:4 format stores a group. */
int orc_prune24(const void *A, int64_t M, int64_t K, int64_t ld, int dtype, void *vals, uint8_t *meta) {
    if (K % 4) return ORC_ERR_SHAPE;
    int64_t G = K / 4, lm = (K + 7) / 8;
    for (int64_t i = 0; i < M; i++) {
        for (int64_t j = 0; j < lm; j++) meta[i * lm + j] = 0;
        for (int64_t g = 0; g < G; g++) {
            int64_t base = i * ld + 4 * g;
            int first = 0; /* largest key, lowest index among equals */
            for (int q = 1; q < 4; q++)
                if (mag_key(A, base + q, dtype) > mag_key(A, base + first, dtype)) first = q;
            int second = -1; /* largest of the other three, lowest index among equals */
            for (int q = 0; q < 4; q++) {
                if (q == first) continue;
                if (second < 0 || mag_key(A, base + q, dtype) > mag_key(A, base + second, dtype)) second = q;
            }
            int i0 = first < second ? first : second, i1 = first < second ? second : first;
            copy_elem(vals, i * (K / 2) + 2 * g, A, base + i0, dtype);
            copy_elem(vals, i * (K / 2) + 2 * g + 1, A, base + i1, dtype);
            meta[i * lm + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
        }
    }
    return ORC_OK;
}

/* Magnitude pruning into the tile-vector-wise format ("Accelerating Sparse DNNs
 * Based on Tiled GEMM", abstract: tile-wise column selection, 2:4 inside).
 * The kept columns of each row tile are an input (ascending, inside [0, K));
 * entries outside them are dropped, and each group of 4 consecutive kept
 * columns keeps its two largest magnitudes (ties to the lower index), as in
 * orc_prune24.  Groups past a tile's kept count are padding: value 0, nibble
 * (0, 1). */
int orc_prune_tvw(const void *A, int64_t M, int64_t K, int64_t ld, int dtype, int tile_rows,
                  const int32_t *tile_ptr, const int32_t *cols, int64_t Kp, void *vals, uint8_t *meta) {
    if (tile_rows <= 0 || Kp % 8) return ORC_ERR_SHAPE;
    int64_t nt = (M + tile_rows - 1) / tile_rows, lm = Kp / 8;
    for (int64_t t = 0; t < nt; t++) {
        int64_t kb = tile_ptr[t], Kt = tile_ptr[t + 1] - kb;
        if (Kt < 0 || Kt % 4 || Kt > Kp) return ORC_ERR_SHAPE;
        for (int64_t q = 0; q < Kt; q++) {
            if (cols[kb + q] < 0 || cols[kb + q] >= K) return ORC_ERR_FORMAT;
            if (q && cols[kb + q] <= cols[kb + q - 1]) return ORC_ERR_FORMAT;
        }
        int64_t rb = t * tile_rows, re = rb + tile_rows < M ? rb + tile_rows : M;
        for (int64_t i = rb; i < re; i++) {
            for (int64_t j = 0; j < lm; j++) meta[i * lm + j] = 0;
            for (int64_t g = 0; g < Kp / 4; g++) {
                int i0 = 0, i1 = 1;
                if (4 * g < Kt) {
                    int64_t at[4];
                    for (int p = 0; p < 4; p++) at[p] = i * ld + cols[kb + 4 * g + p];
                    int first = 0;
                    for (int q = 1; q < 4; q++)
                        if (mag_key(A, at[q], dtype) > mag_key(A, at[first], dtype)) first = q;
                    int second = -1;
                    for (int q = 0; q < 4; q++) {
                        if (q == first) continue;
                        if (second < 0 || mag_key(A, at[q], dtype) > mag_key(A, at[second], dtype)) second = q;
                    }
                    i0 = first < second ? first : second;
                    i1 = first < second ? second : first;
                    copy_elem(vals, i * (Kp / 2) + 2 * g, A, at[i0], dtype);
                    copy_elem(vals, i * (Kp / 2) + 2 * g + 1, A, at[i1], dtype);
                } else {
                    zero_elem(vals, i * (Kp / 2) + 2 * g, dtype);
                    zero_elem(vals, i * (Kp / 2) + 2 * g + 1, dtype);
                }
                meta[i * lm + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
            }
        }
    }
    return ORC_OK;
}

/* ================================================================== (2n-2):2n
 * "SlideSparse" (abstract): a (2n-2):2n block is rewritten as n-1 overlapping
 * 2:4 windows and the activations are rearranged to match.  Group g of a row
 * is columns 2n g .. 2n g + 2n - 1 (at most 2n - 2 nonzero); window j of the
 * group (0 <= j < n - 1) covers the group's positions 2j .. 2j + 3, i.e. the
 * pairs j and j + 1, so pair 0 and pair n - 1 lie in one window each and every
 * other pair in two.
 *
 * Lifted order (a reading; the pages fix none): with G = K / 2n groups, the
 * lifted operand has K' = 4 (n - 1) G columns, window j of group g occupying
 * lifted columns 4 (j G + g) .. 4 (j G + g) + 3 ("window planes": all groups'
 * window 0, then all groups' window 1, ...).  Lifted column 4 (j G + g) + p
 * therefore reads original column 2n g + 2j + p; the same map lifts B's rows.
 *
 * Assignment of the nonzeros to windows (a reading; the pages state only that
 * the decomposition is exact): windows are filled in order j = 0, 1, ...;
 * window j first takes every nonzero of pair j that window j - 1 left (no later
 * window covers them), then the nonzeros of pair j + 1 in ascending position
 * while it holds fewer than two.  This earliest-deadline order places every
 * nonzero whenever the group has at most 2n - 2 of them (pairs a..b reach
 * windows a-1..b, which hold at least as many entries as the pairs unless the
 * range is the whole group).  Each window then holds at most two nonzeros, so
 * the lifted matrix is 2:4 and compresses with the ordinary 2:4 rule. */

/* Original column of lifted column q (window planes). */
static int64_t slide_src(int64_t q, int64_t G, int n) {
    int64_t w = q / 4, p = q % 4, j = w / G, g = w % G;
    return 2 * n * g + 2 * j + p;
}

int64_t orc_slide_src(int64_t q, int64_t K, int n) { return slide_src(q, K / (2 * n), n); }

/* dense A (M x K, leading dim ld) -> dense lifted L (M x K', leading dim K'),
 * every nonzero of A placed in exactly one window, zeros elsewhere. */
int orc_slide_decompose(const void *A, int64_t M, int64_t K, int64_t ld, int dtype, int n, void *L) {
    if (n < 2 || n > 32 || K % (2 * n)) return ORC_ERR_SHAPE;
    int64_t G = K / (2 * n), Kl = 4 * (n - 1) * G;
    for (int64_t i = 0; i < M; i++) {
        for (int64_t q = 0; q < Kl; q++) zero_elem(L, i * Kl + q, dtype);
        for (int64_t g = 0; g < G; g++) {
            int64_t base = i * ld + 2 * n * g;
            int nzc = 0, placed[64] = {0};
            for (int t = 0; t < 2 * n; t++) nzc += !is_zero(A, base + t, dtype);
            if (nzc > 2 * n - 2) return ORC_ERR_FORMAT;
            for (int j = 0; j < n - 1; j++) {
                int held = 0;
                for (int t = 2 * j; t < 2 * j + 4; t++) {
                    if (placed[t] || is_zero(A, base + t, dtype)) continue;
                    if (held == 2) break; /* only pair j + 1 can be left for window j + 1 */
                    placed[t] = 1;
                    held++;
                    copy_elem(L, i * Kl + 4 * (j * G + g) + (t - 2 * j), A, base + t, dtype);
                }
            }
            for (int t = 0; t < 2 * n; t++)
                if (!placed[t] && !is_zero(A, base + t, dtype)) return ORC_ERR_FORMAT;
        }
    }
    return ORC_OK;
}

void orc_densify24(int64_t M, int64_t K, int dtype, const void *vals, const uint8_t *meta, void *D) {
    int64_t G = K / 4, lm = (K + 7) / 8;
    memset(D, 0, (size_t)(M * K * esize(dtype)));
    for (int64_t i = 0; i < M; i++)
        for (int64_t g = 0; g < G; g++) {
            int nib = (meta[i * lm + g / 2] >> (4 * (g % 2))) & 15;
            copy_elem(D, i * K + 4 * g + (nib & 3), vals, i * (K / 2) + 2 * g, dtype);
            copy_elem(D, i * K + 4 * g + (nib >> 2), vals, i * (K / 2) + 2 * g + 1, dtype);
        }
}

/* Float 2:4 SpMM (fp64 accumulate): bf16/fp16, and fp8 E4M3/E5M2 with B of
 * the same type.  For E4M3 the result is exact: every value is a multiple of
 * 2^-9 below 2^9, so every product is a multiple of 2^-18 below 2^18 and, for
 * K below 2^17, every partial sum is a multiple of 2^-18 below 2^35, which
 * fp64 holds exactly. */
void orc_spmm24_f64(int64_t M, int64_t K, int dtype, const void *vals, const uint8_t *meta,
                    const void *B, int64_t ldb, int64_t r0, int64_t r1, const int64_t *cols,
                    int64_t ncols, double *C) {
    (void)M;
    int64_t G = K / 4, lm = (K + 7) / 8;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = r0; i < r1; i++) {
        double *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0.0;
        for (int64_t g = 0; g < G; g++) {
            int nib = (meta[i * lm + g / 2] >> (4 * (g % 2))) & 15;
            for (int t = 0; t < 2; t++) {
                double a = get_f(vals, i * (K / 2) + 2 * g + t, dtype);
                int64_t k = 4 * g + (t ? (nib >> 2) : (nib & 3));
                for (int64_t q = 0; q < ncols; q++) out[q] += a * get_f(B, k * ldb + OUTCOL(q), dtype);
            }
        }
    }
}

/* int8 2:4 SpMM, exact in int64. */
void orc_spmm24_i64(int64_t M, int64_t K, const int8_t *vals, const uint8_t *meta, const int8_t *B,
                    int64_t ldb, int64_t r0, int64_t r1, const int64_t *cols, int64_t ncols, int64_t *C) {
    (void)M;
    int64_t G = K / 4, lm = (K + 7) / 8;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = r0; i < r1; i++) {
        int64_t *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0;
        for (int64_t g = 0; g < G; g++) {
            int nib = (meta[i * lm + g / 2] >> (4 * (g % 2))) & 15;
            for (int t = 0; t < 2; t++) {
                int64_t a = get_i(vals, i * (K / 2) + 2 * g + t);
                int64_t k = 4 * g + (t ? (nib >> 2) : (nib & 3));
                for (int64_t q = 0; q < ncols; q++) out[q] += a * get_i(B, k * ldb + OUTCOL(q));
            }
        }
    }
}

/* ================================================================== TVW
 * Reading (tile-vector-wise): rows are cut into tiles of tile_rows rows; tile t
 * keeps the ascending column list cols[tile_ptr[t] .. tile_ptr[t+1]) (Kt
 * entries, Kt % 4 == 0; the kept set is an input).  Inside a tile every row is
 * 2:4 over its kept columns taken in ascending order (group g = kept columns
 * 4g..4g+3).  Stored: vals[M][Kp/2], meta[M][Kp/8] with a common pitch
 * Kp >= max Kt (Kp % 8 == 0); entries past a tile's Kt are value 0 with the
 * nibble for positions (0, 1).  A nonzero outside the kept set, unsorted or
 * out-of-range kept columns, or more than 2 nonzeros in a group -> format error.
 */
int orc_tvw_build(const void *A, int64_t M, int64_t K, int64_t ld, int dtype, int tile_rows,
                  const int32_t *tile_ptr, const int32_t *cols, int64_t Kp, void *vals, uint8_t *meta) {
    if (tile_rows <= 0 || Kp % 8) return ORC_ERR_SHAPE;
    int64_t nt = (M + tile_rows - 1) / tile_rows, lm = Kp / 8;
    for (int64_t t = 0; t < nt; t++) {
        int64_t kb = tile_ptr[t], Kt = tile_ptr[t + 1] - kb;
        if (Kt < 0 || Kt % 4 || Kt > Kp) return ORC_ERR_SHAPE;
        for (int64_t q = 0; q < Kt; q++) {
            if (cols[kb + q] < 0 || cols[kb + q] >= K) return ORC_ERR_FORMAT;
            if (q && cols[kb + q] <= cols[kb + q - 1]) return ORC_ERR_FORMAT;
        }
        int64_t rb = t * tile_rows, re = rb + tile_rows < M ? rb + tile_rows : M;
        for (int64_t i = rb; i < re; i++) {
            /* every nonzero of the row must sit in a kept column */
            int64_t nz_all = 0, nz_kept = 0;
            for (int64_t k = 0; k < K; k++) nz_all += !is_zero(A, i * ld + k, dtype);
            for (int64_t q = 0; q < Kt; q++) nz_kept += !is_zero(A, i * ld + cols[kb + q], dtype);
            if (nz_all != nz_kept) return ORC_ERR_FORMAT;
            for (int64_t j = 0; j < lm; j++) meta[i * lm + j] = 0;
            for (int64_t g = 0; g < Kp / 4; g++) {
                int i0 = 0, i1 = 1;
                if (4 * g < Kt) {
                    int nz[4], n = 0, keep[4] = {0, 0, 0, 0}, idx[2], c = 0;
                    for (int p = 0; p < 4; p++)
                        if (!is_zero(A, i * ld + cols[kb + 4 * g + p], dtype)) nz[n++] = p;
                    if (n > 2) return ORC_ERR_FORMAT;
                    for (int s = 0; s < n; s++) keep[nz[s]] = 1;
                    for (int p = 0; p < 4 && n < 2; p++)
                        if (!keep[p]) { keep[p] = 1; n++; }
                    for (int p = 0; p < 4; p++)
                        if (keep[p]) idx[c++] = p;
                    i0 = idx[0];
                    i1 = idx[1];
                    copy_elem(vals, i * (Kp / 2) + 2 * g, A, i * ld + cols[kb + 4 * g + i0], dtype);
                    copy_elem(vals, i * (Kp / 2) + 2 * g + 1, A, i * ld + cols[kb + 4 * g + i1], dtype);
                } else {
                    zero_elem(vals, i * (Kp / 2) + 2 * g, dtype);
                    zero_elem(vals, i * (Kp / 2) + 2 * g + 1, dtype);
                }
                meta[i * lm + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
            }
        }
    }
    return ORC_OK;
}

void orc_tvw_densify(int64_t M, int64_t K, int dtype, int tile_rows, const int32_t *tile_ptr,
                     const int32_t *cols, int64_t Kp, const void *vals, const uint8_t *meta, void *D) {
    int64_t lm = Kp / 8;
    memset(D, 0, (size_t)(M * K * esize(dtype)));
    for (int64_t i = 0; i < M; i++) {
        int64_t t = i / tile_rows, kb = tile_ptr[t], Kt = tile_ptr[t + 1] - kb;
        for (int64_t g = 0; g < Kt / 4; g++) {
            int nib = (meta[i * lm + g / 2] >> (4 * (g % 2))) & 15;
            copy_elem(D, i * K + cols[kb + 4 * g + (nib & 3)], vals, i * (Kp / 2) + 2 * g, dtype);
            copy_elem(D, i * K + cols[kb + 4 * g + (nib >> 2)], vals, i * (Kp / 2) + 2 * g + 1, dtype);
        }
    }
}

/* C[i][n] = sum over the kept groups of row i's tile, in ascending kept-column
 * order: vals * B[cols[tile_ptr[t] + 4g + idx]][n]   (fp64). */
void orc_tvw_spmm(int64_t M, int dtype, int tile_rows, const int32_t *tile_ptr, const int32_t *cols,
                  int64_t Kp, const void *vals, const uint8_t *meta, const void *B, int64_t ldb,
                  int64_t r0, int64_t r1, const int64_t *ocols, int64_t ncols, double *C) {
    (void)M;
    int64_t lm = Kp / 8;
    const int64_t *colsel = ocols;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = r0; i < r1; i++) {
        double *out = C + (i - r0) * ncols;
        for (int64_t j = 0; j < ncols; j++) out[j] = 0.0;
        int64_t t = i / tile_rows, kb = tile_ptr[t], Kt = tile_ptr[t + 1] - kb;
        for (int64_t g = 0; g < Kt / 4; g++) {
            int nib = (meta[i * lm + g / 2] >> (4 * (g % 2))) & 15;
            for (int s = 0; s < 2; s++) {
                double a = get_f(vals, i * (Kp / 2) + 2 * g + s, dtype);
                int64_t k = cols[kb + 4 * g + (s ? (nib >> 2) : (nib & 3))];
                for (int64_t q = 0; q < ncols; q++)
                    out[q] += a * get_f(B, k * ldb + (colsel ? colsel[q] : q), dtype);
            }
        }
    }
}

/* ================================================================== permutation
 * "SMaT" (abstract): the sparse matrix is permuted to minimise the number of
 * nonzero blocks before the block-sparse multiply; the method's reference list
 * cites Cuthill and McKee, "Reducing the bandwidth of sparse symmetric
 * matrices".  Reading (the pages name no algorithm): symmetric Reverse
 * Cuthill-McKee on the pattern of A + A^T of a square A (i ~ j iff i != j and
 * A[i][j] or A[j][i] is stored), applied to rows and columns alike:
 * A' = P A P^T with A'[i][j] = A[perm[i]][perm[j]].
 *   degree(i) = number of distinct neighbours of i;
 *   while nodes remain: start at the unvisited node of least degree (lowest
 *   index on ties) and run a breadth-first search in which every dequeued node
 *   appends its unvisited neighbours in ascending (degree, index) order;
 *   perm = the visiting order reversed. */
static const int32_t *rcm_deg;
static int rcm_cmp(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    if (rcm_deg[x] != rcm_deg[y]) return rcm_deg[x] < rcm_deg[y] ? -1 : 1;
    return (x > y) - (x < y);
}

int orc_rcm(int64_t n, const int32_t *row_ptr, const int32_t *col, int32_t *perm) {
    if (n <= 0) return ORC_OK;
    /* dense boolean adjacency of the symmetrised pattern (test sizes only) */
    uint8_t *adj = calloc((size_t)(n * n), 1);
    int32_t *deg = calloc((size_t)n, sizeof(int32_t));
    int32_t *order = malloc(sizeof(int32_t) * (size_t)n);
    int32_t *nb = malloc(sizeof(int32_t) * (size_t)n);
    uint8_t *seen = calloc((size_t)n, 1);
    int rc = ORC_OK;
    if (!adj || !deg || !order || !nb || !seen) {
        rc = ORC_ERR_SHAPE;
        goto done;
    }
    for (int64_t i = 0; i < n; i++)
        for (int32_t e = row_ptr[i]; e < row_ptr[i + 1]; e++) {
            int64_t j = col[e];
            if (j < 0 || j >= n) {
                rc = ORC_ERR_FORMAT;
                goto done;
            }
            if (j != i) adj[i * n + j] = adj[j * n + i] = 1;
        }
    for (int64_t i = 0; i < n; i++)
        for (int64_t j = 0; j < n; j++) deg[i] += adj[i * n + j];
    rcm_deg = deg;
    int64_t head = 0, tail = 0;
    while (tail < n) {
        int64_t s = -1;
        for (int64_t i = 0; i < n; i++)
            if (!seen[i] && (s < 0 || deg[i] < deg[s])) s = i;
        seen[s] = 1;
        order[tail++] = (int32_t)s;
        while (head < tail) {
            int64_t v = order[head++], m = 0;
            for (int64_t j = 0; j < n; j++)
                if (adj[v * n + j] && !seen[j]) nb[m++] = (int32_t)j;
            qsort(nb, (size_t)m, sizeof(int32_t), rcm_cmp);
            for (int64_t t = 0; t < m; t++) {
                seen[nb[t]] = 1;
                order[tail++] = nb[t];
            }
        }
    }
    for (int64_t i = 0; i < n; i++) perm[i] = order[n - 1 - i];
done:
    free(adj);
    free(deg);
    free(order);
    free(nb);
    free(seen);
    return rc;
}

/* A'[i][j] = A[perm[i]][perm[j]] (n x n, leading dims ld / n). */
void orc_permute_sym(int64_t n, int64_t ld, int dtype, const void *A, const int32_t *perm, void *out) {
    for (int64_t i = 0; i < n; i++)
        for (int64_t j = 0; j < n; j++) copy_elem(out, i * n + j, A, perm[i] * ld + perm[j], dtype);
}

/* ================================================================== SDDMM
 * "Magicube" (abstract: SpMM and SDDMM, the two sparse operations the library
 * supports).  Reading (the page gives no definition): the sampled dense-dense
 * product, out[e] = sum_k A[i][k] * Bt[j][k] for every stored entry e = (i, j)
 * of a CSR pattern, i.e. (A B) at the pattern's positions with B = Bt^T given
 * as Bt (N x K, row-major; attention's Q K^T has this form).  The pattern's
 * values are not used.  Products and sums in fp64, ascending k. */
void orc_sddmm(int64_t M, int64_t K, int dtype, const int32_t *row_ptr, const int32_t *col, const void *A,
               const void *Bt, double *out) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < M; i++)
        for (int32_t e = row_ptr[i]; e < row_ptr[i + 1]; e++) {
            int64_t j = col[e];
            double s = 0.0;
            for (int64_t k = 0; k < K; k++) s += get_f(A, i * K + k, dtype) * get_f(Bt, j * K + k, dtype);
            out[e] = s;
        }
}

/* The quantized SDDMM ("Magicube", abstract: SpMM and SDDMM on low-precision
 * integers): int8 A and Bt, every product and sum in int64, so out[e] is the
 * exact integer sum_k A[i][k] * Bt[j][k] at every stored (i, j). */
void orc_sddmm_i64(int64_t M, int64_t K, const int32_t *row_ptr, const int32_t *col, const int8_t *A,
                   const int8_t *Bt, int64_t *out) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < M; i++)
        for (int32_t e = row_ptr[i]; e < row_ptr[i + 1]; e++) {
            int64_t j = col[e];
            int64_t s = 0;
            for (int64_t k = 0; k < K; k++) s += (int64_t)A[i * K + k] * (int64_t)Bt[j * K + k];
            out[e] = s;
        }
}
