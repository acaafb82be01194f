// api.cu -- the extern "C" boundary: argument validation, per-device state,
// tensor-map encoding and dispatch to the kernels of each format.
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "sm103.cuh"

namespace spmm {

// Sticky per-device error word (SPMM_DEVERR_* bits), written by kernels.
__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxKernelSlots = 32;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
bool g_attr_done[kMaxDevices][kMaxKernelSlots];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

__global__ void timeout_selftest_kernel(int* err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // Nothing ever arrives on this barrier: the wait must give up by itself.
    if (threadIdx.x == 0) ptx::mbar_wait(b, 0, timeout_ns, err, SPMM_DEVERR_TIMEOUT);
    __syncthreads();
}

// ---------------------------------------------------------------- tracing
struct TraceRec {
    int kernel;
    cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;        // records of the current session
std::vector<cudaEvent_t> g_ev_pool;   // events reused across sessions
size_t g_ev_used = 0;
int g_open_kernel = 0;
cudaEvent_t g_open_ev = nullptr;

cudaEvent_t take_event() {
    if (g_ev_used == g_ev_pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_ev_pool.push_back(e);
    }
    return g_ev_pool[g_ev_used++];
}

}  // namespace

void trace_begin(int kernel, cudaStream_t s) {
    if (!g_trace_on) return;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    cudaEvent_t e = take_event();
    if (!e) return;
    cudaEventRecord(e, s);
    g_open_kernel = kernel;
    g_open_ev = e;
}

void trace_end(int kernel, cudaStream_t s) {
    if (!g_trace_on) return;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (!g_open_ev || g_open_kernel != kernel) return;
    cudaEvent_t e = take_event();
    if (!e) return;
    cudaEventRecord(e, s);
    g_trace.push_back({kernel, g_open_ev, e});
    g_open_ev = nullptr;
}

const DeviceInfo* device_info() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_info_ok[d]) {
        DeviceInfo info;
        if (cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) !=
            cudaSuccess)
            return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        info.err = static_cast<int*>(p);
        g_info[d] = info;
        g_info_ok[d] = true;
    }
    return &g_info[d];
}

bool set_smem_attr_once(const void* kernel, int bytes, int slot) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices || slot < 0 || slot >= kMaxKernelSlots)
        return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_attr_done[d][slot]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        g_attr_done[d][slot] = true;
    }
    return true;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    std::memset(map, 0, sizeof(*map));
    return f(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[3],
                    const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
    cuuint32_t bx[3] = {box[0], box[1], box[2]};
    cuuint32_t estr[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    return f(map, type, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_4d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    return f(map, type, 4, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
spmm_status check_24(const spmm_24_t* A, int64_t N) {
    if (!A) return SPMM_ERR_NULL;
    if (!dtype_24(A->dtype)) return SPMM_ERR_DTYPE;
    if (A->vals16 && A->dtype != SPMM_I8) return SPMM_ERR_DTYPE;  // pre-widened values: int8 only
    if (A->M < 0 || A->K <= 0 || N < 0) return SPMM_ERR_SHAPE;
    if (A->K % (is_fp8(A->dtype) ? 256 : 128)) return SPMM_ERR_SHAPE;  // whole K steps of the kernel
    if (A->M >= (int64_t(1) << 31) || A->K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    return SPMM_OK;
}

}  // namespace

// Every check spmm_24 makes before it launches, except the workspace's.
spmm_status check_24_call(const spmm_24_t* A, const void* B, int64_t ldb, const void* C, int64_t ldc, int64_t N) {
    spmm_status st = check_24(A, N);
    if (st != SPMM_OK) return st;
    if (A->M > 0 && N > 0 && (!B || !C)) return SPMM_ERR_NULL;
    if (A->M > 0 && (!A->vals || !A->meta)) return SPMM_ERR_NULL;
    if (ldb < N || ldc < N || !aligned16(A->vals) || !aligned16(A->meta)) return SPMM_ERR_SHAPE;
    if (A->vals16 && !aligned16(A->vals16)) return SPMM_ERR_SHAPE;
    // B is read by TMA (not for int8, which is widened first): 16-byte aligned rows
    if (A->dtype != SPMM_I8 && ((ldb * dtype_bytes(A->dtype)) % 16 || !aligned16(B))) return SPMM_ERR_SHAPE;
    return SPMM_OK;
}

}  // namespace spmm

using namespace spmm;

extern "C" {

const char* spmm_status_string(spmm_status s) {
    switch (s) {
        case SPMM_OK: return "ok";
        case SPMM_ERR_NULL: return "null pointer";
        case SPMM_ERR_SHAPE: return "invalid shape, leading dimension or alignment";
        case SPMM_ERR_DTYPE: return "unsupported dtype";
        case SPMM_ERR_FORMAT: return "invalid sparse format data";
        case SPMM_ERR_WORKSPACE: return "workspace missing or too small";
        case SPMM_ERR_TIMEOUT: return "device pipeline wait timed out";
        case SPMM_ERR_CUDA: return "CUDA error";
        case SPMM_ERR_UNSUPPORTED: return "unsupported configuration";
    }
    return "unknown status";
}

int spmm_version(void) { return 100; }

spmm_status spmm_last_device_error(int32_t* bits) {
    if (!bits) return SPMM_ERR_NULL;
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SPMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, dev->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SPMM_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SPMM_ERR_CUDA;
    *bits = v;
    return SPMM_OK;
}

spmm_status spmm_selftest_timeout(uint64_t timeout_ns, spmm_stream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (timeout_ns > 4000000000ull) return SPMM_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    timeout_selftest_kernel<<<1, 32, 0, s>>>(dev->err, timeout_ns);
    if (cudaGetLastError() != cudaSuccess) return SPMM_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

spmm_status spmm_trace_enable(int32_t on) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    g_trace.clear();
    g_ev_used = 0;
    g_open_ev = nullptr;
    g_trace_on = on != 0;
    return SPMM_OK;
}

spmm_status spmm_trace_read(int32_t kernel, int64_t* launches, double* total_ms) {
    if (!launches || !total_ms) return SPMM_ERR_NULL;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    int64_t n = 0;
    double ms = 0.0;
    for (const TraceRec& r : g_trace) {
        if (r.kernel != kernel) continue;
        if (cudaEventSynchronize(r.b) != cudaSuccess) return SPMM_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return SPMM_ERR_CUDA;
        ms += t;
        ++n;
    }
    *launches = n;
    *total_ms = ms;
    return SPMM_OK;
}

static spmm_status check_bcsr(const spmm_bcsr_t* A, int64_t N) {
    if (!A) return SPMM_ERR_NULL;
    if (A->dtype != SPMM_BF16 && A->dtype != SPMM_F16) return SPMM_ERR_DTYPE;
    if (A->M < 0 || A->K <= 0 || N < 0 || A->bh <= 0 || A->bw <= 0 || A->nnzb < 0) return SPMM_ERR_SHAPE;
    if (A->M % A->bh || A->K % A->bw) return SPMM_ERR_SHAPE;
    if (A->nnzb > 0 && !aligned16(A->vals)) return SPMM_ERR_SHAPE;
    if (A->nnzb > 0 && (!A->row_ptr || !A->col_idx || !A->vals)) return SPMM_ERR_NULL;
    if (A->bh % 16 || A->bh > 256 || (A->bw != 16 && A->bw != 32 && A->bw != 64)) return SPMM_ERR_UNSUPPORTED;
    if (A->nnzb * A->bh >= (int64_t(1) << 31) || A->K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    return SPMM_OK;
}

spmm_status spmm_bcsr(const spmm_bcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                      spmm_stream_t stream) {
    if (!A) return SPMM_ERR_NULL;
    if (A->M > 0 && N > 0 && (!B || !C)) return SPMM_ERR_NULL;  // an empty C needs no buffers
    const spmm_status st = check_bcsr(A, N);
    if (st != SPMM_OK) return st;
    if (ldb < N || ldc < N || (ldb * 2) % 16 || !aligned16(B)) return SPMM_ERR_SHAPE;
    return launch_bcsr(A, B, ldb, C, ldc, N, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- SDDMM

spmm_status spmm_sddmm(const spmm_csr_t* S, int64_t K, const void* A, int64_t lda, const void* Bt, int64_t ldbt,
                       void* out, spmm_stream_t stream) {
    if (!S) return SPMM_ERR_NULL;
    if (S->dtype != SPMM_BF16 && S->dtype != SPMM_F16 && S->dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    // one 16-byte load covers 8 16-bit or 16 int8 elements
    const int64_t e = S->dtype == SPMM_I8 ? 16 : 8;
    if (S->M < 0 || S->K < 0 || S->nnz < 0 || K <= 0 || K % e || lda < K || ldbt < K || lda % e || ldbt % e)
        return SPMM_ERR_SHAPE;
    // int8: every sum is exact in int32 while K * 128 * 128 < 2^31
    if (S->dtype == SPMM_I8 && K * 16384 >= (int64_t(1) << 31)) return SPMM_ERR_SHAPE;
    if (S->nnz == 0) return SPMM_OK;
    if (!S->row_ptr || !S->col || !A || !Bt || !out) return SPMM_ERR_NULL;
    if (S->M == 0 || !aligned16(A) || !aligned16(Bt)) return SPMM_ERR_SHAPE;
    if (S->M >= (int64_t(1) << 31) || S->K >= (int64_t(1) << 31) || S->nnz >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    return launch_sddmm(S, K, A, lda, Bt, ldbt, out, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- permutation

spmm_status spmm_rcm_order(int64_t n, const int32_t* row_ptr, const int32_t* col, int32_t* perm) {
    if (n < 0) return SPMM_ERR_SHAPE;
    if (n == 0) return SPMM_OK;
    if (!row_ptr || !perm || (row_ptr[n] > 0 && !col)) return SPMM_ERR_NULL;
    if (n >= (int64_t(1) << 31)) return SPMM_ERR_UNSUPPORTED;
    return rcm_order_host(n, row_ptr, col, perm);
}

spmm_status spmm_permute_sym(const void* dense, int64_t n, int64_t ld, int32_t dtype, const int32_t* perm, void* out,
                             int64_t ldo, spmm_stream_t stream) {
    if (n > 0 && (!dense || !perm || !out)) return SPMM_ERR_NULL;
    if (dtype != SPMM_BF16 && dtype != SPMM_F16 && dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (n < 0 || ld < n || ldo < n) return SPMM_ERR_SHAPE;
    if (n >= (int64_t(1) << 31)) return SPMM_ERR_UNSUPPORTED;
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    return run_permute_sym(dense, n, ld, dtype, perm, out, ldo, dev->err, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_permute_rows(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                              int32_t elem_bytes, const int32_t* perm, int32_t scatter, spmm_stream_t stream) {
    if (rows > 0 && cols > 0 && (!src || !dst || !perm)) return SPMM_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return SPMM_ERR_DTYPE;
    if (rows < 0 || cols < 0 || lds < cols || ldd < cols) return SPMM_ERR_SHAPE;
    if (rows >= (int64_t(1) << 31)) return SPMM_ERR_UNSUPPORTED;
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    return run_permute_rows(src, lds, dst, ldd, rows, cols, elem_bytes, perm, scatter != 0, dev->err,
                            reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_bcsr_permuted_workspace_size(const spmm_bcsr_t* A, int64_t N, size_t* bytes) {
    if (!bytes) return SPMM_ERR_NULL;
    const spmm_status st = check_bcsr(A, N);
    if (st != SPMM_OK) return st;
    *bytes = bcsr_permuted_ws_bytes(A, N);
    return SPMM_OK;
}

spmm_status spmm_bcsr_permuted(const spmm_bcsr_t* A, const int32_t* perm, const void* B, int64_t ldb, float* C,
                               int64_t ldc, int64_t N, void* workspace, size_t workspace_bytes,
                               spmm_stream_t stream) {
    if (!A) return SPMM_ERR_NULL;
    if (A->M > 0 && N > 0 && (!B || !C || !perm)) return SPMM_ERR_NULL;
    const spmm_status st = check_bcsr(A, N);
    if (st != SPMM_OK) return st;
    if (A->M != A->K || ldb < N || ldc < N) return SPMM_ERR_SHAPE;
    const size_t need = bcsr_permuted_ws_bytes(A, N);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return SPMM_ERR_WORKSPACE;
    return launch_bcsr_permuted(A, perm, B, ldb, C, ldc, N, workspace, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- builders

spmm_status spmm_build_bcsr_count(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t bh, int32_t bw,
                                  int32_t dtype, int32_t* row_ptr, int64_t* nnzb, spmm_stream_t stream) {
    if (!row_ptr || !nnzb || (M > 0 && K > 0 && !dense)) return SPMM_ERR_NULL;
    if (dtype != SPMM_BF16 && dtype != SPMM_F16 && dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || bh <= 0 || bw <= 0 || M % bh || K % bw || ld < K) return SPMM_ERR_SHAPE;
    if (K / bw > 40000 || M / bh >= (int64_t(1) << 31)) return SPMM_ERR_UNSUPPORTED;
    return run_bcsr_count(dense, M, K, ld, bh, bw, dtype, row_ptr, nnzb, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_build_bcsr_fill(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t bh, int32_t bw,
                                 int32_t dtype, const int32_t* row_ptr, int32_t* col_idx, void* vals,
                                 spmm_stream_t stream) {
    if (!row_ptr || (M > 0 && K > 0 && !dense)) return SPMM_ERR_NULL;
    if (dtype != SPMM_BF16 && dtype != SPMM_F16 && dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || bh <= 0 || bw <= 0 || M % bh || K % bw || ld < K) return SPMM_ERR_SHAPE;
    if (K / bw > 8000) return SPMM_ERR_UNSUPPORTED;
    return run_bcsr_fill(dense, M, K, ld, bh, bw, dtype, row_ptr, col_idx, vals,
                         reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_compress_24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                             uint8_t* meta, spmm_stream_t stream) {
    if (M > 0 && K > 0 && (!dense || !vals || !meta)) return SPMM_ERR_NULL;
    if (!dtype_24(dtype)) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || K % 8 || ld < K) return SPMM_ERR_SHAPE;
    return run_compress24(dense, M, K, ld, dtype, vals, meta, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_prune_24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                          uint8_t* meta, spmm_stream_t stream) {
    if (M > 0 && K > 0 && (!dense || !vals || !meta)) return SPMM_ERR_NULL;
    if (!dtype_24(dtype)) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || K % 8 || ld < K) return SPMM_ERR_SHAPE;
    return run_prune24(dense, M, K, ld, dtype, vals, meta, reinterpret_cast<cudaStream_t>(stream));
}

static spmm_status tvw_build_checked(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype,
                                     int32_t tile_rows, const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles,
                                     int64_t Kp, void* vals, uint8_t* meta, bool prune, spmm_stream_t stream) {
    if (M > 0 && (!dense || !tile_ptr || !vals || !meta)) return SPMM_ERR_NULL;
    if (dtype != SPMM_BF16 && dtype != SPMM_F16 && dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || ld < K || tile_rows <= 0 || Kp < 0 || Kp % 8) return SPMM_ERR_SHAPE;
    if (n_tiles != (M + tile_rows - 1) / tile_rows) return SPMM_ERR_SHAPE;
    if (M == 0) return SPMM_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // tile_ptr is small: check it on the host (starts at 0, monotone, Kt % 4 == 0, Kt <= Kp)
    std::vector<int32_t> tp(static_cast<size_t>(n_tiles + 1));
    if (cudaMemcpyAsync(tp.data(), tile_ptr, tp.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    if (tp[0] != 0) return SPMM_ERR_FORMAT;
    for (int64_t t = 0; t < n_tiles; ++t) {
        const int64_t kt = int64_t(tp[t + 1]) - tp[t];
        if (kt < 0 || kt % 4 || kt > Kp) return SPMM_ERR_FORMAT;
    }
    if (tp[n_tiles] > 0 && !cols) return SPMM_ERR_NULL;
    return run_build_tvw(dense, M, K, ld, dtype, tile_rows, tile_ptr, cols, n_tiles, Kp, vals, meta, prune, s);
}

spmm_status spmm_build_tvw(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t tile_rows,
                           const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles, int64_t Kp, void* vals,
                           uint8_t* meta, spmm_stream_t stream) {
    return tvw_build_checked(dense, M, K, ld, dtype, tile_rows, tile_ptr, cols, n_tiles, Kp, vals, meta, false,
                             stream);
}

spmm_status spmm_prune_tvw(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t tile_rows,
                           const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles, int64_t Kp, void* vals,
                           uint8_t* meta, spmm_stream_t stream) {
    return tvw_build_checked(dense, M, K, ld, dtype, tile_rows, tile_ptr, cols, n_tiles, Kp, vals, meta, true,
                             stream);
}

spmm_status spmm_build_slide(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t n,
                             void* vals, uint8_t* meta, spmm_stream_t stream) {
    if (M > 0 && K > 0 && (!dense || !vals || !meta)) return SPMM_ERR_NULL;
    if (dtype != SPMM_BF16 && dtype != SPMM_F16 && dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (M < 0 || K < 0 || ld < K || n < 2 || n > 8 || K % (4 * n)) return SPMM_ERR_SHAPE;
    return run_build_slide(dense, M, K, ld, dtype, n, vals, meta, reinterpret_cast<cudaStream_t>(stream));
}

static spmm_status check_csr(const spmm_csr_t* A, int32_t h, int32_t S) {
    if (!A) return SPMM_ERR_NULL;
    if (A->dtype != SPMM_BF16 && A->dtype != SPMM_F16) return SPMM_ERR_DTYPE;
    if (A->M < 0 || A->K <= 0 || A->nnz < 0 || h <= 0 || h > 256 || S <= 0) return SPMM_ERR_SHAPE;
    if (A->M >= (int64_t(1) << 31) || A->K >= (int64_t(1) << 31) || A->nnz >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    if (!A->row_ptr || (A->nnz > 0 && (!A->col || !A->val))) return SPMM_ERR_NULL;
    return SPMM_OK;
}

spmm_status spmm_build_wcsr_workspace_size(const spmm_csr_t* A, int32_t h, size_t* bytes) {
    if (!bytes) return SPMM_ERR_NULL;
    spmm_status st = check_csr(A, h, 1);
    if (st != SPMM_OK) return st;
    *bytes = wcsr_build_ws_bytes(A->M, A->nnz, h);
    return SPMM_OK;
}

spmm_status spmm_build_wcsr_count(const spmm_csr_t* A, int32_t h, int32_t S, void* workspace, size_t workspace_bytes,
                                  int64_t* n_wcols, int64_t* n_units, spmm_stream_t stream) {
    if (!n_wcols || !n_units) return SPMM_ERR_NULL;
    spmm_status st = check_csr(A, h, S);
    if (st != SPMM_OK) return st;
    if (!workspace || workspace_bytes < wcsr_build_ws_bytes(A->M, A->nnz, h) || !aligned16(workspace))
        return SPMM_ERR_WORKSPACE;
    return run_wcsr_count(A, h, S, workspace, n_wcols, n_units, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_build_wcsr_fill(const spmm_csr_t* A, int32_t h, int32_t S, void* workspace, size_t workspace_bytes,
                                 spmm_wcsr_t* out, spmm_stream_t stream) {
    if (!out) return SPMM_ERR_NULL;
    spmm_status st = check_csr(A, h, S);
    if (st != SPMM_OK) return st;
    if (!workspace || workspace_bytes < wcsr_build_ws_bytes(A->M, A->nnz, h) || !aligned16(workspace))
        return SPMM_ERR_WORKSPACE;
    const int64_t nw = (A->M + h - 1) / h;
    if (!out->wcol_ptr || !out->wnz_ptr || !out->unit_ptr || !out->unit_nz_ptr) return SPMM_ERR_NULL;
    if (A->nnz > 0 && (!out->wcols || !out->lrow || !out->slot || !out->val || !out->unit_win))
        return SPMM_ERR_NULL;
    out->M = A->M;
    out->K = A->K;
    out->nnz = A->nnz;
    out->h = h;
    out->S = S;
    out->dtype = A->dtype;
    out->n_windows = nw;
    return run_wcsr_fill(A, h, S, workspace, out, reinterpret_cast<cudaStream_t>(stream));
}

static spmm_status check_wcsr(const spmm_wcsr_t* A) {
    if (!A) return SPMM_ERR_NULL;
    if (A->dtype != SPMM_BF16 && A->dtype != SPMM_F16) return SPMM_ERR_DTYPE;
    if (A->M < 0 || A->K <= 0 || A->nnz < 0 || A->h <= 0 || A->S <= 0) return SPMM_ERR_SHAPE;
    if (A->n_windows != (A->M + A->h - 1) / A->h || A->n_units < A->n_windows) return SPMM_ERR_SHAPE;
    if (A->h > wcsr_max_h()) return SPMM_ERR_UNSUPPORTED;
    return SPMM_OK;
}

spmm_status spmm_wcsr_workspace_size(const spmm_wcsr_t* A, int64_t N, size_t* bytes) {
    if (!bytes) return SPMM_ERR_NULL;
    spmm_status st = check_wcsr(A);
    if (st != SPMM_OK) return st;
    if (N < 0) return SPMM_ERR_SHAPE;
    *bytes = wcsr_spmm_ws_bytes(A, N);
    return SPMM_OK;
}

spmm_status spmm_wcsr(const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                      void* workspace, size_t workspace_bytes, spmm_stream_t stream) {
    spmm_status st = check_wcsr(A);
    if (st != SPMM_OK) return st;
    if (A->M > 0 && N > 0 && (!B || !C)) return SPMM_ERR_NULL;
    if (N < 0 || ldb < N || ldc < N || (ldb * 2) % 16 || !aligned16(B)) return SPMM_ERR_SHAPE;
    if (A->M > 0 && (!A->wcol_ptr || !A->unit_ptr || !A->unit_win || !A->unit_nz_ptr)) return SPMM_ERR_NULL;
    if (A->nnz > 0 && (!A->wcols || !A->lrow || !A->slot || !A->val)) return SPMM_ERR_NULL;
    if (!workspace || workspace_bytes < wcsr_spmm_ws_bytes(A, N) || !aligned16(workspace))
        return SPMM_ERR_WORKSPACE;
    return launch_wcsr(A, B, ldb, C, ldc, N, workspace, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_24_workspace_size(const spmm_24_t* A, int64_t N, size_t* bytes) {
    if (!bytes) return SPMM_ERR_NULL;
    spmm_status st = check_24(A, N);
    if (st != SPMM_OK) return st;
    *bytes = spmm24_workspace_bytes(A, N);
    return SPMM_OK;
}

spmm_status spmm_widen_24(const spmm_24_t* A, void* vals16, spmm_stream_t stream) {
    spmm_status st = check_24(A, 0);
    if (st != SPMM_OK) return st;
    if (A->dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (A->M == 0) return SPMM_OK;
    if (!A->vals || !vals16) return SPMM_ERR_NULL;
    if (!aligned16(A->vals) || !aligned16(vals16)) return SPMM_ERR_SHAPE;
    return widen_values_24(A->vals, A->M, A->K / 2, vals16, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_24(const spmm_24_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                    void* workspace, size_t workspace_bytes, spmm_stream_t stream) {
    spmm_status st = check_24_call(A, B, ldb, C, ldc, N);
    if (st != SPMM_OK) return st;
    const size_t need = spmm24_workspace_bytes(A, N);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return SPMM_ERR_WORKSPACE;
    return launch_spmm24(A, B, ldb, C, ldc, N, workspace, reinterpret_cast<cudaStream_t>(stream));
}

static spmm_status check_slide(const spmm_slide_t* A, int64_t N) {
    if (!A) return SPMM_ERR_NULL;
    if (A->dtype != SPMM_BF16 && A->dtype != SPMM_F16 && A->dtype != SPMM_I8) return SPMM_ERR_DTYPE;
    if (A->M < 0 || A->K <= 0 || N < 0 || A->n < 2 || A->n > 8) return SPMM_ERR_SHAPE;
    if (A->K % (64 * A->n)) return SPMM_ERR_SHAPE;
    if (A->M >= (int64_t(1) << 31) || A->K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    return SPMM_OK;
}

spmm_status spmm_slide_workspace_size(const spmm_slide_t* A, int64_t N, size_t* bytes) {
    if (!bytes) return SPMM_ERR_NULL;
    spmm_status st = check_slide(A, N);
    if (st != SPMM_OK) return st;
    *bytes = slide_workspace_bytes(A, N);
    return SPMM_OK;
}

spmm_status spmm_slide(const spmm_slide_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                       void* workspace, size_t workspace_bytes, spmm_stream_t stream) {
    spmm_status st = check_slide(A, N);
    if (st != SPMM_OK) return st;
    if (A->M > 0 && N > 0 && (!B || !C)) return SPMM_ERR_NULL;
    if (A->M > 0 && (!A->vals || !A->meta)) return SPMM_ERR_NULL;
    if (ldb < N || ldc < N || !aligned16(A->vals) || !aligned16(A->meta)) return SPMM_ERR_SHAPE;
    if (A->dtype != SPMM_I8 && ((ldb * 2) % 16 || !aligned16(B))) return SPMM_ERR_SHAPE;
    const size_t need = slide_workspace_bytes(A, N);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return SPMM_ERR_WORKSPACE;
    return launch_slide(A, B, ldb, C, ldc, N, workspace, reinterpret_cast<cudaStream_t>(stream));
}

spmm_status spmm_tvw(const spmm_tvw_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                     spmm_stream_t stream) {
    if (!A) return SPMM_ERR_NULL;
    if (A->M > 0 && N > 0 && (!B || !C)) return SPMM_ERR_NULL;
    if (A->dtype != SPMM_BF16 && A->dtype != SPMM_F16) return SPMM_ERR_DTYPE;
    if (A->M < 0 || A->K <= 0 || N < 0 || A->Kp < 0 || A->tile_rows <= 0) return SPMM_ERR_SHAPE;
    if (A->n_tiles != (A->M + A->tile_rows - 1) / A->tile_rows) return SPMM_ERR_SHAPE;
    if (A->M > 0 && (!A->tile_ptr || !A->cols || !A->vals || !A->meta)) return SPMM_ERR_NULL;
    if (ldb < N || ldc < N || (ldb * 2) % 16 || !aligned16(B) || !aligned16(A->vals) || !aligned16(A->meta))
        return SPMM_ERR_SHAPE;
    if (A->tile_rows != 128 || A->Kp % 128 || A->Kp == 0) return SPMM_ERR_UNSUPPORTED;
    if (A->M >= (int64_t(1) << 31) || A->K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    return launch_tvw(A, B, ldb, C, ldc, N, reinterpret_cast<cudaStream_t>(stream));
}
}  // extern "C"
