// noalloc.cu -- a 2:4 SpMM entry point that never allocates device memory.
//
// spmm_24 takes a caller-provided workspace because int8 operands are widened
// to fp16 before they reach the tensor core.  Some callers cannot obtain one:
// code that runs inside another runtime and is handed only its input and
// output buffers, services that reserve all device memory at start-up and
// forbid allocation afterwards, or latency-critical paths that cannot afford
// the implicit synchronisation of cudaMalloc.  spmm_24_noalloc serves them by
// placing that scratch in a fixed array that lives in the library's own device
// image.  Every GPU that loads this library holds the array until the process
// exits.
#include <mutex>

#include "internal.h"

// The scratch: file-scope, 256-byte aligned, fixed size.  Host code must not use
// this name as a device address (on the host it is only a stand-in symbol); it
// asks the runtime for the device address instead (scratch_address below).
static constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace spmm {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];
bool g_ready[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per
// device with that device current and kept for the process's lifetime (a
// cudaDeviceReset would leave the kept address pointing into the old context;
// the library is not meant to be used across one).
spmm_status scratch_address(void** out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return SPMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SPMM_ERR_CUDA;
        g_addr[d] = p;
        g_ready[d] = true;
    }
    *out = g_addr[d];
    return SPMM_OK;
}

}  // namespace
}  // namespace spmm

using namespace spmm;

extern "C" spmm_status spmm_24_noalloc(const spmm_24_t* A, const void* B, int64_t ldb, void* C, int64_t ldc,
                                       int64_t N, spmm_stream_t stream) {
    // the same checks spmm_24 makes, from the one shared function
    const spmm_status chk = check_24_call(A, B, ldb, C, ldc, N);
    if (chk != SPMM_OK) return chk;
    // Same scratch as spmm_24 would ask for; refuse anything larger than the array.
    const size_t need = spmm24_workspace_bytes(A, N);
    if (need > kNoAllocScratchBytes) return SPMM_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        const spmm_status st = scratch_address(&scratch);
        if (st != SPMM_OK) return st;
    }
    return launch_spmm24(A, B, ldb, C, ldc, N, scratch, reinterpret_cast<cudaStream_t>(stream));
}
