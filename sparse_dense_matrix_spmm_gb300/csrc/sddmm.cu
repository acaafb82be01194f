// sddmm.cu -- sampled dense-dense product, the second sparse operation of
// "Magicube" (abstract: SpMM and SDDMM on low-precision integers): out[e] =
// sum_k A[i][k] * Bt[j][k] for every stored entry e = (i, j) of a CSR pattern;
// fp16/bf16 in with fp32 out, or int8 in with exact int32 out (four-way byte
// dot products, dp4a, summed in int32).
//
// A dot product of two contiguous K-vectors per output: HBM- and
// gather-bound work for CUDA cores, not a contraction for the tensor core.
// Each warp takes a fixed slice of the nonzero array (so one long row does not
// serialise on one warp), finds the slice's first row by a 32-way search in
// row_ptr (about log32(M) rounds of dependent loads, so slices are long), and
// preloads the slice's (row, column) pairs with coalesced loads into shared
// memory, where the lane groups read them.  Four lanes form one output's group:
// each lane loads E elements (16 bytes: E = 8 for 16-bit types, 16 for int8)
// of A's row and of Bt's row per step, K / (4 E) steps, and the group sums by
// two shuffle rounds.  Each lane keeps kIlp outputs in flight to hide the
// latency of the Bt row gathers.  The kernel is bound by instruction issue, and
// few lanes per output spend few shuffles on it (measured at K = 128 on the
// 65536^2 log-normal pattern: 4 lanes 53.9 us fp16 / 33.4 us int8, 16 and 8
// lanes 70.3 / 37.5 us, 2 lanes 58.0 / 39.6 us, 1 lane 92.8 / 56.0 us).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace spmm {
namespace {

constexpr int kIlp = 4;
constexpr int kLanes = 4;     // lanes per output
// entries per warp: passes of (32 / kLanes) * kIlp entries amortise the slice's
// binary search (128 entries measured best at 16 lanes per output too)
constexpr int kSliceEntries = 128;
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float dot8(uint4 a, uint4 b);
template <>
__device__ __forceinline__ float dot8<__half>(uint4 a, uint4 b) {
    const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&x[i]));
        const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&y[i]));
        s = fmaf(p.x, q.x, s);
        s = fmaf(p.y, q.y, s);
    }
    return s;
}
template <>
__device__ __forceinline__ float dot8<__nv_bfloat16>(uint4 a, uint4 b) {
    const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // a bf16 is the high half of an fp32
        s = fmaf(__uint_as_float(x[i] << 16), __uint_as_float(y[i] << 16), s);
        s = fmaf(__uint_as_float(x[i] & 0xFFFF0000u), __uint_as_float(y[i] & 0xFFFF0000u), s);
    }
    return s;
}

// int8: sixteen signed byte products per 16-byte pair, four per dp4a, summed
// in int32 (exact: |sum| <= K * 16384 < 2^31, checked on the host).
__device__ __forceinline__ int dot16_i8(uint4 a, uint4 b) {
    int s = 0;
    s = __dp4a(static_cast<int>(a.x), static_cast<int>(b.x), s);
    s = __dp4a(static_cast<int>(a.y), static_cast<int>(b.y), s);
    s = __dp4a(static_cast<int>(a.z), static_cast<int>(b.z), s);
    s = __dp4a(static_cast<int>(a.w), static_cast<int>(b.w), s);
    return s;
}

// Per element type: elements per 16-byte load, accumulator / output type.
template <typename T>
struct Sd {
    static constexpr int E = 8;
    using Acc = float;
    __device__ static Acc dot(uint4 a, uint4 b) { return dot8<T>(a, b); }
};
template <>
struct Sd<int8_t> {
    static constexpr int E = 16;
    using Acc = int;
    __device__ static Acc dot(uint4 a, uint4 b) { return dot16_i8(a, b); }
};

struct SddmmArgs {
    const int32_t* row_ptr;
    const int32_t* col;
    int64_t M, N, K, nnz;
    const uint8_t* A;   // element pitch lda, elements of the kernel's type
    int64_t lda;
    const uint8_t* Bt;
    int64_t ldb;
    void* out;          // fp32, or int32 for int8
    int* err;
};

// Four CTAs (32 warps) per SM: the register cap of 64 fits the kernel without
// spills and keeps a third more gathers in flight than the 80 registers it
// takes unbounded (measured at K = 128 with 16 lanes per output: 68 us against
// 79 us for fp16, 38 us against 48 us for int8; five or more CTAs spilled and ran
// slower).
template <typename T, int L>
__global__ void __launch_bounds__(kThreads, 4) sddmm_kernel(const SddmmArgs a) {
    using Acc = typename Sd<T>::Acc;
    constexpr int E = Sd<T>::E;
    constexpr int G = 32 / L;                   // outputs per warp per pass
    constexpr int kPer = G * kIlp;              // entries per pass
    constexpr int kPasses = kSliceEntries / kPer;
    constexpr int kSlice = kPer * kPasses;      // entries per warp
    static_assert(kPasses > 0 && kSlice == kSliceEntries, "whole passes per slice");
    constexpr int kRegs = kSlice / 32;          // (row, column) pairs each lane preloads
    static_assert(kSlice % 32 == 0, "whole warp loads of the slice's indices");
    const int lane = threadIdx.x & 31, sub = lane / L, sl = lane % L;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t e0 = warp_id * kSlice;
    if (e0 >= a.nnz) return;
    const int64_t e1 = e0 + kSlice < a.nnz ? e0 + kSlice : a.nnz;
    // row of e0: the last i with row_ptr[i] <= e0, by a 32-way search (each round
    // the lanes probe 32 points of [lo, hi) and keep the interval that holds it)
    int64_t lo = 0, hi = a.M;  // row_ptr[lo] <= e0 < row_ptr[hi] (row_ptr[M] = nnz > e0)
    while (hi - lo > 1) {
        const int64_t step = (hi - lo + 31) / 32;
        const int64_t probe = lo + step * lane;
        const bool le = probe < hi && __ldg(a.row_ptr + probe) <= e0;
        const int k = 31 - __clz(__ballot_sync(0xffffffffu, le));  // last probe at or below e0 (lane 0 always is)
        lo = lo + step * k;
        hi = lo + step < hi ? lo + step : hi;
    }
    // Preload the slice's (row, column) pairs into this warp's shared arrays, lane l
    // writing entries e0 + l + 32 t (coalesced loads), so the passes below wait on
    // no index load.  Rows: the lanes
    // load the ends of 32 consecutive rows rb .. rb + 31 (one coalesced load); an
    // entry before the last of those ends lies in row rb + (number of ends at or
    // before it), found by a 5-step search over the 32 sorted ends.  Entries past
    // the window retry with the next 32 rows.  Each group of 32 entries starts
    // at the row of its first entry, so one window usually serves it.
    constexpr int64_t kPastEnd = int64_t(1) << 62;  // row ends beyond row M - 1
    __shared__ int32_t s_row[kThreads / 32][kSlice], s_col[kThreads / 32][kSlice];
    int32_t* pr_s = s_row[threadIdx.x >> 5];
    int32_t* pc_s = s_col[threadIdx.x >> 5];
    int64_t rb = lo;  // a row at or before the group's first entry
#pragma unroll
    for (int t = 0; t < kRegs; ++t) {
        const int64_t e = e0 + lane + 32 * t;
        const bool live = e < e1;
        int64_t row = -1;
        for (int64_t w = rb;; w += 32) {  // ends: the row ends advance to row_ptr[M] = nnz > e
            const int64_t end_l = w + lane + 1 <= a.M ? __ldg(a.row_ptr + w + lane + 1) : kPastEnd;
            const int64_t last = __shfl_sync(0xffffffffu, end_l, 31);
            int c = 0;  // every lane searches (uniform shuffles); the result counts where it applies
#pragma unroll
            for (int bit = 16; bit > 0; bit >>= 1) {
                const int64_t v = __shfl_sync(0xffffffffu, end_l, c + bit - 1);
                if (v <= e) c += bit;
            }
            if (live && row < 0 && e < last) row = w + c;
            if (__all_sync(0xffffffffu, !live || row >= 0) || w + 32 >= a.M) break;
        }
        pr_s[lane + 32 * t] = row >= 0 ? static_cast<int32_t>(row) : 0;
        pc_s[lane + 32 * t] = live && row >= 0 ? __ldg(a.col + e) : -1;
        // the next group starts at or after this group's last row
        const int64_t last_row = __shfl_sync(0xffffffffu, row, 31);
        rb = last_row >= 0 ? last_row : rb;
    }
    Acc* __restrict__ out = static_cast<Acc*>(a.out);
    __syncwarp();  // the slice's pairs are in shared memory for every lane
    auto fetch = [&](int p, int32_t (&jj)[kIlp], int32_t (&ri)[kIlp], bool (&ok)[kIlp]) {
#pragma unroll
        for (int u = 0; u < kIlp; ++u) {
            const int base = p * kPer + u * G;
            jj[u] = pc_s[base + sub];
            ri[u] = pr_s[base + sub];
            const bool live = e0 + base + sub < e1;
            ok[u] = live && jj[u] >= 0 && jj[u] < a.N;
            if (live && !ok[u] && sl == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);
        }
    };
    auto finish = [&](int p, Acc (&acc)[kIlp], const bool (&ok)[kIlp]) {
#pragma unroll
        for (int u = 0; u < kIlp; ++u) {
#pragma unroll
            for (int o = L / 2; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
            const int64_t e = e0 + p * kPer + u * G + sub;
            if (sl == 0 && e < e1) out[e] = ok[u] ? acc[u] : Acc(0);
        }
    };
#pragma unroll 1
    for (int p = 0; p < kPasses; ++p) {
        int32_t jj[kIlp], ri[kIlp];
        bool ok[kIlp];
        Acc acc[kIlp];
        fetch(p, jj, ri, ok);
#pragma unroll
        for (int u = 0; u < kIlp; ++u) acc[u] = Acc(0);
        for (int64_t k0 = 0; k0 < a.K; k0 += E * L) {
            const int64_t k = k0 + E * sl;
            if (k >= a.K) continue;
            uint4 x[kIlp], y[kIlp];
#pragma unroll
            for (int u = 0; u < kIlp; ++u)
                if (ok[u]) {
                    x[u] = __ldg(reinterpret_cast<const uint4*>(a.A + (static_cast<int64_t>(ri[u]) * a.lda + k) * sizeof(T)));
                    y[u] = __ldg(reinterpret_cast<const uint4*>(a.Bt + (static_cast<int64_t>(jj[u]) * a.ldb + k) * sizeof(T)));
                }
#pragma unroll
            for (int u = 0; u < kIlp; ++u)
                if (ok[u]) acc[u] += Sd<T>::dot(x[u], y[u]);
        }
        finish(p, acc, ok);
    }
}


}  // namespace

spmm_status launch_sddmm(const spmm_csr_t* S, int64_t K, const void* A, int64_t lda, const void* Bt, int64_t ldbt,
                         void* out, cudaStream_t s) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (S->nnz == 0) return SPMM_OK;
    SddmmArgs a{};
    a.row_ptr = S->row_ptr;
    a.col = S->col;
    a.M = S->M;
    a.N = S->K;
    a.K = K;
    a.nnz = S->nnz;
    a.A = static_cast<const uint8_t*>(A);
    a.lda = lda;
    a.Bt = static_cast<const uint8_t*>(Bt);
    a.ldb = ldbt;
    a.out = out;
    a.err = dev->err;
    const int64_t warps = (S->nnz + kSliceEntries - 1) / kSliceEntries;
    const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks >= (int64_t(1) << 31)) return SPMM_ERR_UNSUPPORTED;
    trace_begin(SPMM_KERNEL_SDDMM, s);
    const unsigned grid = static_cast<unsigned>(blocks);
    if (S->dtype == SPMM_I8)
        sddmm_kernel<int8_t, kLanes><<<grid, kThreads, 0, s>>>(a);
    else if (S->dtype == SPMM_BF16)
        sddmm_kernel<__nv_bfloat16, kLanes><<<grid, kThreads, 0, s>>>(a);
    else
        sddmm_kernel<__half, kLanes><<<grid, kThreads, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_SDDMM, s);
    return cuda_status(e);
}

}  // namespace spmm
