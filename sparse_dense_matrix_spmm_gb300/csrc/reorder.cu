// reorder.cu -- permuting a square sparse matrix before the block-sparse
// multiply ("SMaT", abstract: the sparse matrix is permuted to minimise the
// number of nonzero blocks), with Reverse Cuthill-McKee as the permutation
// (Cuthill and McKee, "Reducing the bandwidth of sparse symmetric matrices",
// in that page's reference list).
//
//   spmm_rcm_order       the order, on the host: a breadth-first search whose
//                        visiting order depends on every earlier step, run once
//                        per matrix in O(nnz log nnz)
//   spmm_permute_sym     A' = P A P^T on the device (dense, any 8/16-bit type)
//   spmm_permute_rows    row gather / scatter on the device (1, 2 or 4-byte elements)
//   spmm_bcsr_permuted   C = P^T (A' (P B)): gather B's rows, the BCSR kernel on
//                        A', scatter C's rows (inside the BCSR epilogue for
//                        64-row blocks, else as a second pass)
#include <algorithm>
#include <vector>

#include "internal.h"

namespace spmm {
namespace {

// dst row i <- src row perm[i] (gather) or dst row perm[i] <- src row i (scatter).
// `vec`: rows, pitches and base addresses allow 16-byte copies.
__global__ void permute_rows_kernel(const uint8_t* __restrict__ src, int64_t lds, uint8_t* __restrict__ dst,
                                    int64_t ldd, int64_t rows, int64_t row_bytes, const int32_t* __restrict__ perm,
                                    int scatter, int vec, int* err) {
    const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * (vec ? 16 : 1);
    if (c >= row_bytes) return;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const int32_t p = __ldg(perm + r);
        if (p < 0 || p >= rows) {
            if (c == 0) atomicOr(err, SPMM_DEVERR_INDEX);
            continue;
        }
        const int64_t rs = scatter ? r : p, rd = scatter ? p : r;
        if (vec)
            *reinterpret_cast<uint4*>(dst + rd * ldd + c) = __ldcs(reinterpret_cast<const uint4*>(src + rs * lds + c));
        else
            dst[rd * ldd + c] = src[rs * lds + c];
    }
}

// out[i][j] = A[perm[i]][perm[j]]; one thread per output element of a row.
template <typename T>
__global__ void permute_sym_kernel(const T* __restrict__ A, int64_t n, int64_t ld, const int32_t* __restrict__ perm,
                                   T* __restrict__ out, int64_t ldo, int* err) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int32_t pj = __ldg(perm + j);
    for (int64_t i = blockIdx.y; i < n; i += gridDim.y) {
        const int32_t pi = __ldg(perm + i);
        const bool ok = pi >= 0 && pi < n && pj >= 0 && pj < n;
        if (!ok) atomicOr(err, SPMM_DEVERR_INDEX);
        out[i * ldo + j] = ok ? A[pi * ld + pj] : T(0);
    }
}

}  // namespace

spmm_status rcm_order_host(int64_t n, const int32_t* row_ptr, const int32_t* col, int32_t* perm) {
    if (row_ptr[0] != 0) return SPMM_ERR_FORMAT;
    // symmetrised adjacency without self loops: count, place, then sort and
    // deduplicate every row
    std::vector<int64_t> start(static_cast<size_t>(n) + 1, 0);
    for (int64_t i = 0; i < n; ++i) {
        if (row_ptr[i + 1] < row_ptr[i]) return SPMM_ERR_FORMAT;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            const int64_t j = col[e];
            if (j < 0 || j >= n) return SPMM_ERR_FORMAT;
            if (j == i) continue;
            ++start[i + 1];
            ++start[j + 1];
        }
    }
    for (int64_t i = 0; i < n; ++i) start[i + 1] += start[i];
    std::vector<int32_t> adj(static_cast<size_t>(start[n]));
    std::vector<int64_t> fill(start.begin(), start.end() - 1);
    for (int64_t i = 0; i < n; ++i)
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            const int64_t j = col[e];
            if (j == i) continue;
            adj[fill[i]++] = static_cast<int32_t>(j);
            adj[fill[j]++] = static_cast<int32_t>(i);
        }
    std::vector<int32_t> deg(static_cast<size_t>(n));
    std::vector<int64_t> end(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) {
        auto b = adj.begin() + start[i], e = adj.begin() + start[i + 1];
        std::sort(b, e);
        end[i] = std::unique(b, e) - adj.begin();
        deg[i] = static_cast<int32_t>(end[i] - start[i]);
    }
    auto before = [&](int32_t x, int32_t y) { return deg[x] != deg[y] ? deg[x] < deg[y] : x < y; };
    // start nodes in (degree, index) order; the next start is the first unvisited one
    std::vector<int32_t> starts(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) starts[i] = static_cast<int32_t>(i);
    std::sort(starts.begin(), starts.end(), before);
    std::vector<uint8_t> seen(static_cast<size_t>(n), 0);
    std::vector<int32_t> order;
    order.reserve(static_cast<size_t>(n));
    std::vector<int32_t> nb;
    size_t head = 0, next_start = 0;
    while (order.size() < static_cast<size_t>(n)) {
        while (seen[starts[next_start]]) ++next_start;
        const int32_t s = starts[next_start];
        seen[s] = 1;
        order.push_back(s);
        while (head < order.size()) {
            const int32_t v = order[head++];
            nb.clear();
            for (int64_t e = start[v]; e < end[v]; ++e)
                if (!seen[adj[e]]) nb.push_back(adj[e]);
            std::sort(nb.begin(), nb.end(), before);
            for (int32_t u : nb) {
                seen[u] = 1;
                order.push_back(u);
            }
        }
    }
    for (int64_t i = 0; i < n; ++i) perm[i] = order[static_cast<size_t>(n - 1 - i)];
    return SPMM_OK;
}

spmm_status run_permute_rows(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int32_t elem_bytes, const int32_t* perm, bool scatter, int* err, cudaStream_t s) {
    if (rows == 0 || cols == 0) return SPMM_OK;
    const int64_t rb = cols * elem_bytes, sb = lds * elem_bytes, db = ldd * elem_bytes;
    const int vec = (rb % 16 == 0 && sb % 16 == 0 && db % 16 == 0 && aligned16(src) && aligned16(dst)) ? 1 : 0;
    const int64_t per_row = vec ? rb / 16 : rb;
    const dim3 grid(static_cast<unsigned>((per_row + 255) / 256), static_cast<unsigned>(rows < 65535 ? rows : 65535));
    trace_begin(SPMM_KERNEL_PERMUTE, s);
    permute_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), sb, static_cast<uint8_t*>(dst), db,
                                             rows, rb, perm, scatter ? 1 : 0, vec, err);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_PERMUTE, s);
    return cuda_status(e);
}

spmm_status run_permute_sym(const void* dense, int64_t n, int64_t ld, int32_t dtype, const int32_t* perm, void* out,
                            int64_t ldo, int* err, cudaStream_t s) {
    if (n == 0) return SPMM_OK;
    const dim3 grid(static_cast<unsigned>((n + 255) / 256), static_cast<unsigned>(n < 65535 ? n : 65535));
    if (dtype == SPMM_I8)
        permute_sym_kernel<int8_t><<<grid, 256, 0, s>>>(static_cast<const int8_t*>(dense), n, ld, perm,
                                                        static_cast<int8_t*>(out), ldo, err);
    else
        permute_sym_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(dense), n, ld, perm,
                                                          static_cast<uint16_t*>(out), ldo, err);
    return cuda_status(cudaGetLastError());
}

// Workspace of the permuted product: B' (K rows, pitch N rounded up to 8
// elements) then C' (M rows, pitch N rounded up to 4), each 256-byte aligned.
size_t bcsr_permuted_ws_bytes(const spmm_bcsr_t* A, int64_t N) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int64_t nb = (N + 7) / 8 * 8, nc = (N + 3) / 4 * 4;
    return al(static_cast<size_t>(A->K) * nb * 2) + al(static_cast<size_t>(A->M) * nc * 4);
}

spmm_status launch_bcsr_permuted(const spmm_bcsr_t* A, const int32_t* perm, const void* B, int64_t ldb, float* C,
                                 int64_t ldc, int64_t N, void* ws, cudaStream_t s) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    const int64_t nb = (N + 7) / 8 * 8, nc = (N + 3) / 4 * 4;
    uint8_t* w = static_cast<uint8_t*>(ws);
    void* Bp = w;
    float* Cp = reinterpret_cast<float*>(w + ((static_cast<size_t>(A->K) * nb * 2 + 255) & ~size_t(255)));
    spmm_status st = run_permute_rows(B, ldb, Bp, nb, A->K, N, 2, perm, false, dev->err, s);
    if (st != SPMM_OK) return st;
    // 64-row blocks and 16-byte aligned C rows: the BCSR epilogue writes each row
    // straight to C row perm[r]; otherwise C' is scattered by a second pass
    if (A->bh == 64 && ldc % 4 == 0 && aligned16(C) && A->nnzb > 0) return launch_bcsr(A, Bp, nb, C, ldc, N, s, perm);
    st = launch_bcsr(A, Bp, nb, Cp, nc, N, s);
    if (st != SPMM_OK) return st;
    return run_permute_rows(Cp, nc, C, ldc, A->M, N, 4, perm, true, dev->err, s);
}

}  // namespace spmm
