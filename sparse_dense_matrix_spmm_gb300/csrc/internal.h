// internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "spmm_gb300.h"

namespace spmm {

// Per-device facts and the device address of the sticky error word.
struct DeviceInfo {
    int sms = 0;
    int max_smem_optin = 0;
    int* err = nullptr;  // device address of the error word (SPMM_DEVERR_* bits)
};

// Facts for the current device; nullptr if the CUDA runtime is unusable.
const DeviceInfo* device_info();

// Default bound on any single pipeline wait inside a kernel.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// 2-D tiled tensor map: `inner` elements per row (contiguous), `outer` rows,
// `row_bytes` between rows; box of box_inner x box_outer elements.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle);

// 3-D tiled tensor map: dims[0] contiguous, byte strides of dims 1 and 2, box
// of box[0] x box[1] x box[2] elements.  Returns false if the driver rejects it.
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[3],
                    const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle);

// 4-D tiled tensor map: dims[0] contiguous, byte strides of dims 1-3.
bool encode_tmap_4d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle);

inline spmm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline CUtensorMapDataType half_type(int32_t dtype) {
    return dtype == SPMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Element types of the 2:4 operand: bf16, fp16, int8, fp8 E4M3 / E5M2.
inline bool dtype_24(int32_t dtype) {
    return dtype == SPMM_BF16 || dtype == SPMM_F16 || dtype == SPMM_I8 || dtype == SPMM_E4M3 || dtype == SPMM_E5M2;
}
inline int dtype_bytes(int32_t dtype) { return (dtype == SPMM_BF16 || dtype == SPMM_F16) ? 2 : 1; }
inline bool is_fp8(int32_t dtype) { return dtype == SPMM_E4M3 || dtype == SPMM_E5M2; }

// Argument checks shared by spmm_24 and spmm_24_noalloc (everything except the
// workspace): status of the first failing check, SPMM_OK otherwise.
spmm_status check_24_call(const spmm_24_t* A, const void* B, int64_t ldb, const void* C, int64_t ldc, int64_t N);

// Tracing hooks: no-ops unless spmm_trace_enable(1) is in effect.
void trace_begin(int kernel, cudaStream_t s);
void trace_end(int kernel, cudaStream_t s);

// Raise a kernel's dynamic shared memory limit once per device.
bool set_smem_attr_once(const void* kernel, int bytes, int slot);

// Kernel launchers implemented in the per-format translation units.  Arguments
// are already validated by the C-ABI layer.
// row_perm (device, M entries): C row row_perm[r] receives row r; only for
// 64-row blocks with 16-byte aligned C rows (else SPMM_ERR_UNSUPPORTED).
spmm_status launch_bcsr(const spmm_bcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        cudaStream_t stream, const int32_t* row_perm = nullptr);

size_t spmm24_workspace_bytes(const spmm_24_t* A, int64_t N);
// int8 stored values (rows x kv, pitch kv) widened to fp16 into dst (pitch kv).
spmm_status widen_values_24(const void* vals, int64_t rows, int64_t kv, void* dst, cudaStream_t stream);
spmm_status launch_spmm24(const spmm_24_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                          void* ws, cudaStream_t stream);
size_t slide_workspace_bytes(const spmm_slide_t* A, int64_t N);
spmm_status launch_slide(const spmm_slide_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                         void* ws, cudaStream_t stream);
spmm_status launch_tvw(const spmm_tvw_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                       cudaStream_t stream);

size_t wcsr_build_ws_bytes(int64_t M, int64_t nnz, int32_t h);
spmm_status run_wcsr_count(const spmm_csr_t* A, int32_t h, int32_t S, void* ws, int64_t* n_wcols, int64_t* n_units,
                           cudaStream_t s);
spmm_status run_wcsr_fill(const spmm_csr_t* A, int32_t h, int32_t S, void* ws, spmm_wcsr_t* out, cudaStream_t s);
size_t wcsr_spmm_ws_bytes(const spmm_wcsr_t* A, int64_t N);
spmm_status launch_wcsr(const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        void* ws, cudaStream_t s);
int wcsr_max_h();
// Whether spmm_wcsr runs this operand's window products on the tensor core
// (enough nonzeros per distinct window column) or on CUDA cores.
bool wcsr_uses_tensor_core(const spmm_wcsr_t* A);

spmm_status run_bcsr_count(const void* dense, int64_t M, int64_t K, int64_t ld, int bh, int bw, int32_t dtype,
                           int32_t* row_ptr, int64_t* nnzb, cudaStream_t s);
spmm_status run_bcsr_fill(const void* dense, int64_t M, int64_t K, int64_t ld, int bh, int bw, int32_t dtype,
                          const int32_t* row_ptr, int32_t* col_idx, void* vals, cudaStream_t s);
spmm_status run_compress24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                           uint8_t* meta, cudaStream_t s);
spmm_status run_prune24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                        uint8_t* meta, cudaStream_t stream);
spmm_status run_build_tvw(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t tile_rows,
                          const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles, int64_t Kp, void* vals,
                          uint8_t* meta, bool prune, cudaStream_t s);
spmm_status run_build_slide(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t n,
                            void* vals, uint8_t* meta, cudaStream_t s);

spmm_status launch_sddmm(const spmm_csr_t* S, int64_t K, const void* A, int64_t lda, const void* Bt, int64_t ldbt,
                         void* out, cudaStream_t s);
spmm_status rcm_order_host(int64_t n, const int32_t* row_ptr, const int32_t* col, int32_t* perm);
spmm_status run_permute_rows(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int32_t elem_bytes, const int32_t* perm, bool scatter, int* err, cudaStream_t s);
spmm_status run_permute_sym(const void* dense, int64_t n, int64_t ld, int32_t dtype, const int32_t* perm, void* out,
                            int64_t ldo, int* err, cudaStream_t s);
size_t bcsr_permuted_ws_bytes(const spmm_bcsr_t* A, int64_t N);
spmm_status launch_bcsr_permuted(const spmm_bcsr_t* A, const int32_t* perm, const void* B, int64_t ldb, float* C,
                                 int64_t ldc, int64_t N, void* ws, cudaStream_t s);

}  // namespace spmm
