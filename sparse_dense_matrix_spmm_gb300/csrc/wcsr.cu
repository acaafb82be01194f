// wcsr.cu -- row-window CSR: the GPU builder (CSR -> windows, units) and SpMM.
//
// "AsyncSparse" (abstract; Fig. 2): for irregular sparsity the WCSR kernel
// loads the sparse operand per row window and splits large windows across
// thread blocks for load balance.
//
// Builder.  Every output position comes from binary searches over the sorted
// rows of a window and from prefix sums, so the result is bit-exact with the
// format definition (see include/spmm_gb300.h) and independent of scheduling:
//   count:  first[e]    = 1 iff no earlier row of e's window holds col[e]
//           fpre[e]     = exclusive prefix of first[] inside e's row, rowfirst[r] its total
//           T_w = sum of rowfirst over the window, U_w = max(1, ceil(T_w / 16S)); scans
//   fill:   slot(e)     = sum over the window's rows r' of the number of first
//                         occurrences in r' with a column below col[e]
//           wcols[wcol_ptr[w] + slot(e)] = col[e] for first occurrences
//           position of e = window start + nonzeros of earlier units + nonzeros of
//                           earlier rows in e's unit + rank inside its row segment
//
// SpMM: three kernels, chosen from the format's counts (wcsr_uses_tensor_core).
//  - Windows whose columns hold about one nonzero each (the synthetic power-law
//    workload: windows ~6% dense) run on CUDA cores (cc::wcsr_spmm_kernel): a
//    dense tile per window would gather as many B rows as the plain product.
//    Each nonzero gathers one B row (N * 2 bytes) from L2; with one CTA per work
//    unit the kernel is bound by instruction issue and by the chain of dependent
//    loads per unit (unit header, window header and nonzeros, column list, B
//    rows), so occupancy (8 CTAs of 4 warps per SM) and instructions per nonzero
//    decide its rate.  The CTA stages the unit's sparse operand in shared memory
//    as {column, local row | value} (all of a thread's slots requested before
//    any column is resolved), then cuts it into eight contiguous streams, one
//    per half-warp.  The 16 lanes of a half read one B row per load (8 columns,
//    16 bytes, each), accumulate with one mixed-precision FMA per element
//    (16-bit operands, fp32 accumulator; the same result as converting both and
//    using fmaf), write rows that lie inside the stream into a shared-memory
//    tile, and hand the two rows at the stream's ends to a fix-up that adds them
//    in stream order, so every sum has a fixed order.  Rows never decrease along
//    a stream, so a batch whose last entry is on the current row needs no
//    per-entry row test.  The first wave of CTAs prefetches the format arrays
//    and B into L2 with bulk prefetches.
//  - Windows that reuse their columns run their window products on the tensor
//    core: per 16 column slots, the 16 gathered B rows (128 output columns on
//    the MMA's M) times the window's value tile (window rows on N), fp32 in
//    TMEM.  Windows of at most 16 rows take the streaming kernel
//    (ts::wcsr_ts_kernel: preparation, gathers, MMA issue and epilogue in
//    separate warps over a persistent item sequence), taller ones the per-item
//    kernel (tc::wcsr_tc_kernel: four warpgroups, each on its own items).
// In every kernel, unsplit windows write C directly; a split window's units
// write partial tiles to the workspace, and the last unit to finish (an
// arrival counter tagged with the call's generation, so the workspace needs no
// clearing) sums them in unit order.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "sm103.cuh"

namespace spmm {

__device__ int g_wcsr_build_error;  // data-dependent builder errors (SPMM_DEVERR_FORMAT)

namespace {

constexpr int kMaxH = 64;   // largest window height the SpMM kernel accepts (MMA N <= 64)

std::mutex g_mu;

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int32_t v) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < v) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ bool contains(const int32_t* a, int n, int32_t v) {
    const int p = lower_bound_i32(a, n, v);
    return p < n && a[p] == v;
}

// ---------------------------------------------------------------- validation
__global__ void csr_check_kernel(const int32_t* rp, const int32_t* col, int64_t M, int64_t K, int64_t nnz,
                                 int* err) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r == 0 && (rp[0] != 0 || rp[M] != nnz)) atomicOr(err, SPMM_DEVERR_FORMAT);
    if (r >= M) return;
    const int32_t b = rp[r], e = rp[r + 1];
    if (e < b || b < 0 || e > nnz) {
        atomicOr(err, SPMM_DEVERR_FORMAT);
        return;
    }
    for (int32_t i = b; i < e; ++i) {
        const int32_t c = col[i];
        if (c < 0 || c >= K || (i > b && col[i - 1] >= c)) {
            atomicOr(err, SPMM_DEVERR_FORMAT);
            return;
        }
    }
}

// ---------------------------------------------------------------- count phase
// One warp per row: first-occurrence flags, their exclusive prefix, row totals.
__global__ void wcsr_first_kernel(const int32_t* rp, const int32_t* col, int64_t M, int h, int32_t* fpre,
                                  int32_t* rowfirst) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x & 31;
    if (r >= M) return;
    const int64_t r0 = (r / h) * h;
    const int32_t b = rp[r], L = rp[r + 1] - b;
    int32_t carry = 0;
    for (int32_t base = 0; base < L; base += 32) {
        const int32_t i = base + lane;
        bool first = i < L;
        const int32_t c = first ? col[b + i] : 0;
        for (int64_t q = r0; q < r && first; ++q)
            if (contains(col + rp[q], rp[q + 1] - rp[q], c)) first = false;
        const unsigned m = __ballot_sync(0xffffffffu, first);
        if (i < L) fpre[b + i] = carry + __popc(m & ((1u << lane) - 1u));
        carry += __popc(m);
    }
    if (lane == 0) rowfirst[r] = carry;
}

// One thread per window: distinct columns and work units.
__global__ void wcsr_window_kernel(const int32_t* rowfirst, int64_t M, int h, int64_t span, int64_t nw,
                                   int32_t* wT, int32_t* wU) {
    const int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (w >= nw) return;
    const int64_t r0 = w * h, r1 = (M < r0 + h) ? M : r0 + h;
    int64_t T = 0;
    for (int64_t r = r0; r < r1; ++r) T += rowfirst[r];
    wT[w] = static_cast<int32_t>(T);
    wU[w] = static_cast<int32_t>(T ? (T + span - 1) / span : 1);
}

// ---------------------------------------------------------------- fill phase
__device__ __forceinline__ int32_t firsts_below(const int32_t* rp, const int32_t* col, const int32_t* fpre,
                                                const int32_t* rowfirst, int64_t q, int32_t c) {
    const int32_t b = rp[q], L = rp[q + 1] - b;
    const int p = lower_bound_i32(col + b, L, c);
    return p < L ? fpre[b + p] : rowfirst[q];
}

// One warp per row: slot of every nonzero, and the window's distinct columns.
__global__ void wcsr_slot_kernel(const int32_t* rp, const int32_t* col, const int32_t* fpre,
                                 const int32_t* rowfirst, const int32_t* wcol_ptr, int64_t M, int h,
                                 int32_t* slot_ws, int32_t* wcols) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x & 31;
    if (r >= M) return;
    const int64_t w = r / h, r0 = w * h, r1 = (M < r0 + h) ? M : r0 + h;
    const int32_t b = rp[r], L = rp[r + 1] - b;
    for (int32_t i = lane; i < L; i += 32) {
        const int32_t c = col[b + i];
        int32_t s = 0;
        for (int64_t q = r0; q < r1; ++q) s += firsts_below(rp, col, fpre, rowfirst, q, c);
        slot_ws[b + i] = s;
        const int32_t next = (i + 1 < L) ? fpre[b + i + 1] : rowfirst[r];
        if (next - fpre[b + i] == 1) wcols[wcol_ptr[w] + s] = c;
    }
}

// Number of nonzeros of row q whose slot is below `lim`.
__device__ __forceinline__ int32_t slots_below(const int32_t* rp, const int32_t* slot_ws, int64_t q, int64_t lim) {
    const int32_t b = rp[q], L = rp[q + 1] - b;
    const int32_t v = lim > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(lim);
    return lower_bound_i32(slot_ws + b, L, v);
}

// One warp per row: final position of every nonzero (unit, row, column order).
template <typename T>
__global__ void wcsr_place_kernel(const int32_t* rp, const T* val, const int32_t* slot_ws, int64_t M, int h,
                                  int64_t span, uint8_t* lrow, int32_t* slot, T* wval) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x & 31;
    if (r >= M) return;
    const int64_t w = r / h, r0 = w * h, r1 = (M < r0 + h) ? M : r0 + h;
    const int32_t b = rp[r], L = rp[r + 1] - b;
    const int32_t wstart = rp[r0];
    for (int32_t i = lane; i < L; i += 32) {
        const int32_t s = slot_ws[b + i];
        const int64_t u = s / span;
        int64_t pos = wstart;
        for (int64_t q = r0; q < r1; ++q) {
            const int32_t lo = slots_below(rp, slot_ws, q, u * span);
            pos += lo;                                                  // earlier units
            if (q < r) pos += slots_below(rp, slot_ws, q, (u + 1) * span) - lo;  // earlier rows, same unit
            else if (q == r) pos += i - lo;                             // rank inside the row segment
        }
        lrow[pos] = static_cast<uint8_t>(r - r0);
        slot[pos] = s;
        wval[pos] = val[b + i];
    }
}

// One thread per window: window offsets and the unit list.
__global__ void wcsr_units_kernel(const int32_t* rp, const int32_t* slot_ws, const int32_t* unit_ptr, int64_t M,
                                  int h, int64_t span, int64_t nw, int32_t* wnz_ptr, int32_t* unit_win,
                                  int32_t* unit_nz_ptr) {
    const int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (w > nw) return;
    if (w == nw) {
        wnz_ptr[nw] = rp[M];
        unit_nz_ptr[unit_ptr[nw]] = rp[M];
        return;
    }
    const int64_t r0 = w * h, r1 = (M < r0 + h) ? M : r0 + h;
    wnz_ptr[w] = rp[r0];
    for (int32_t u = unit_ptr[w]; u < unit_ptr[w + 1]; ++u) {
        const int64_t k = u - unit_ptr[w];
        int64_t pos = rp[r0];
        for (int64_t q = r0; q < r1; ++q) pos += slots_below(rp, slot_ws, q, k * span);
        unit_win[u] = static_cast<int32_t>(w);
        unit_nz_ptr[u] = static_cast<int32_t>(pos);
    }
}

// ---------------------------------------------------------------- scan (single CTA)
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* a, int64_t n) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += 1024) {
        const int64_t i = base + tid;
        const int32_t v = i < n ? a[i] : 0;
        int32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t s = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const int32_t before = carry + (wid ? warp_sums[wid - 1] : 0) + x - v;
        if (i < n) a[i] = before;
        __syncthreads();
        if (tid == 1023) carry = before + v;
        __syncthreads();
    }
}

// Open this call's generation on a tagged counter (gen << 32 | count): the first
// caller that sees an older tag resets the count to 0; everyone returns once
// the word carries this call's tag.  Exactly one reset happens per call, and it
// happens before any increment of that call, because increments come only
// from threads that saw the new tag.
__device__ __forceinline__ bool open_tag(unsigned long long* w, uint32_t gen, int* err) {
    unsigned long long cur = atomicAdd(w, 0ull);
#pragma unroll 1
    for (int it = 0; it < (1 << 20); ++it) {
        if (static_cast<uint32_t>(cur >> 32) == gen) return true;
        const unsigned long long prev = atomicCAS(w, cur, static_cast<unsigned long long>(gen) << 32);
        if (prev == cur) return true;
        cur = prev;
    }
    atomicOr(err, SPMM_DEVERR_TIMEOUT);
    return false;
}

// ---------------------------------------------------------------- SpMM on CUDA cores
// For windows whose column slots hold about one nonzero each (no column reuse
// inside the window), a dense tile per window is ~6% full and the tensor
// core gathers as many B rows as the plain product does; this kernel keeps
// the gathers and does the multiply-adds on CUDA cores.  One CTA per work
// unit, 8 CTAs of 4 warps per SM, so many units' chains of dependent loads
// (unit header -> window header and nonzeros -> column list -> B rows) are in
// flight at once.
namespace cc {

constexpr int kWarps = 4;     // several CTAs per SM: one CTA's staging overlaps the others' gathers
constexpr int kMinBlocks = 8; // resident CTAs per SM the register budget is sized for (64 registers)
constexpr int kThreads = kWarps * 32;
constexpr int kSlab = 128;    // output columns per pass (8 per lane of a half-warp)
static_assert(kThreads >= kSlab, "the boundary fix-up gives one thread to each slab column");
constexpr int kPfArrays = 10;

struct WcsrArgs {
    const int32_t* wcol_ptr;
    const int32_t* wcols;
    const int32_t* unit_ptr;
    const int32_t* unit_win;
    const int32_t* unit_nz_ptr;
    const uint8_t* lrow;
    const int32_t* slot;
    const void* val;
    const void* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
    int64_t M, K, N;
    int32_t h;
    int32_t b_vec;    // B rows can be read as 16-byte pieces (16-byte aligned base, ldb % 8 == 0, K * ldb < 2^31)
    int32_t c_vec;    // C and the partials can be written as float4 (aligned base, ldc % 4 == 0, N % 4 == 0)
    float* partial;   // [n_units][h][N]
    unsigned long long* ticket;  // [n_windows * nslabs] arrival counters (generation-tagged; slab 0's word)
    int32_t nslabs;
    uint32_t gen;     // this call's generation tag (never 0)
    int* err;
    // L2 warm-up: the first pf_ctas CTAs each prefetch their share of these
    // arrays (format arrays and B), so later index and B-row loads hit L2
    // instead of paying an HBM round trip each.
    const void* pf_ptr[kPfArrays];
    int64_t pf_bytes[kPfArrays];
    int32_t pf_n, pf_ctas;
};

constexpr int kStage = 1024;                   // nonzeros whose operand is staged in shared memory at once
constexpr int kPerThread = kStage / kThreads;  // staged entries per thread
constexpr int kBatch = 4;                      // entries per half-warp batch: 4 B-row loads in flight per half
constexpr int kStreams = 2 * kWarps;           // one stream of staged entries per half-warp
constexpr int kBnd = 2 * kStreams;             // fix-up slots: first and last row of every stream
static_assert(kStage % kThreads == 0, "staging gives every thread the same number of entries");

// acc[i] += v * x_i for the eight 16-bit values x_0..x_7 packed in r, with v the
// low 16 bits of pk: one mixed-precision FMA per element (the 16-bit product is
// exact in fp32, so this equals converting both operands and using fmaf).
template <typename T>
__device__ __forceinline__ void fma8(float (&acc)[8], uint32_t pk, const uint4& r);
#define SPMM_WCSR_FMA8(TY)                                                                                  \
    asm("{\n\t.reg .b16 v, t, x0, x1, x2, x3, x4, x5, x6, x7;\n\t"                                          \
        "mov.b32 {v, t}, %8;\n\t"                                                                          \
        "mov.b32 {x0, x1}, %9;\n\tmov.b32 {x2, x3}, %10;\n\tmov.b32 {x4, x5}, %11;\n\tmov.b32 {x6, x7}, %12;\n\t" \
        "fma.rn.f32." TY " %0, v, x0, %0;\n\tfma.rn.f32." TY " %1, v, x1, %1;\n\t"                          \
        "fma.rn.f32." TY " %2, v, x2, %2;\n\tfma.rn.f32." TY " %3, v, x3, %3;\n\t"                          \
        "fma.rn.f32." TY " %4, v, x4, %4;\n\tfma.rn.f32." TY " %5, v, x5, %5;\n\t"                          \
        "fma.rn.f32." TY " %6, v, x6, %6;\n\tfma.rn.f32." TY " %7, v, x7, %7;\n\t}"                         \
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]), \
          "+f"(acc[7])                                                                                      \
        : "r"(pk), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w))
template <>
__device__ __forceinline__ void fma8<__half>(float (&acc)[8], uint32_t pk, const uint4& r) {
    SPMM_WCSR_FMA8("f16");
}
template <>
__device__ __forceinline__ void fma8<__nv_bfloat16>(float (&acc)[8], uint32_t pk, const uint4& r) {
    SPMM_WCSR_FMA8("bf16");
}
#undef SPMM_WCSR_FMA8

__device__ __forceinline__ void store8(float* dst, const float (&acc)[8]) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// This lane's 8 columns of B row `col` (16 bytes).  FULL: one vector load, with
// Bv = B as 16-byte pieces already offset to this lane's columns and ldv = ldb / 8
// (the host guarantees K * ldb < 2^31, so the offset fits 32 bits).  Otherwise
// element loads of the `valid` columns at B + col * ldb + ncol.
template <typename T, bool FULL>
__device__ __forceinline__ uint4 load_b8(const uint4* Bv, uint32_t ldv, const T* B, int64_t ldb, int64_t ncol,
                                         int valid, int col) {
    if (FULL) return __ldg(Bv + static_cast<uint32_t>(col) * ldv);
    const uint16_t* q = reinterpret_cast<const uint16_t*>(B + static_cast<int64_t>(col) * ldb + ncol);
    uint32_t e[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) e[t] = t < valid ? static_cast<uint32_t>(q[t]) : 0u;
    return make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
}

// One half-warp's stream of staged entries [j_lo, j_end): the 16 lanes of the
// half read 128 columns of one B row per load (8 columns, 16 bytes, per lane),
// BATCH loads in flight (fewer on the element-wise path for ragged or unaligned
// B), and accumulate fp32 per row in registers.  A row finished inside the
// stream goes straight into the tile; the stream's first and last rows, which
// may continue in the neighbouring streams, go to the stream's two fix-up
// slots.  Entries are {column, local row << 16 | value bits}; rows change
// rarely, so the change test is a warp vote around a rarely taken branch.
template <typename T, bool FULL, int BATCH = FULL ? kBatch : 4>
__device__ __forceinline__ void wcsr_stream(const T* B, int64_t ldb, int64_t ncol, int valid, const int2* s_ent,
                                            int j_lo, int j_end, float* tile, float* bnd, int* bnd_row, int stream,
                                            int hl) {
    const uint4* Bv = reinterpret_cast<const uint4*>(B) + (FULL ? ncol / 8 : 0);
    const uint32_t ldv = static_cast<uint32_t>(ldb / 8);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    int cur = -1;
    bool first_seg = true;
    for (int j0 = j_lo;; j0 += BATCH) {
        if (!__any_sync(0xffffffffu, j0 < j_end)) break;
        uint4 raw[BATCH];
        uint32_t pk[BATCH];
        if (__all_sync(0xffffffffu, j0 + BATCH <= j_end)) {
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int2 e = s_ent[j0 + b];
                pk[b] = static_cast<uint32_t>(e.y);
                raw[b] = load_b8<T, FULL>(Bv, ldv, B, ldb, ncol, valid, e.x);
            }
        } else {
            // past the stream's end: value 0 on the stream's last row (adds nothing,
            // and rows stay non-decreasing through the batch)
            const uint32_t tail = j0 < j_end ? (static_cast<uint32_t>(s_ent[j_end - 1].y) & 0xFFFF0000u)
                                             : static_cast<uint32_t>(cur) << 16;
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const bool live = j0 + b < j_end;
                const int2 e = live ? s_ent[j0 + b] : make_int2(0, static_cast<int>(tail));
                pk[b] = static_cast<uint32_t>(e.y);
                raw[b] = live ? load_b8<T, FULL>(Bv, ldv, B, ldb, ncol, valid, e.x) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // Rows never decrease along a stream: if the batch's last entry is still on
        // the current row, so is every entry of the batch.
        if (__all_sync(0xffffffffu, (static_cast<int>(pk[BATCH - 1]) >> 16) == cur)) {
#pragma unroll
            for (int b = 0; b < BATCH; ++b) fma8<T>(acc, pk[b], raw[b]);
            continue;
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int rr = static_cast<int>(pk[b]) >> 16;
            if (__any_sync(0xffffffffu, rr != cur)) {
                if (rr != cur) {
                    if (cur >= 0) {
                        // a finished segment: the stream's first row goes to its fix-up
                        // slot, any later one lies wholly inside this stream
                        float* dst = first_seg ? bnd + (2 * stream) * kSlab : tile + cur * kSlab;
                        store8(dst + 8 * hl, acc);
                        if (first_seg && hl == 0) bnd_row[2 * stream] = cur;
                        first_seg = false;
                    }
                    cur = rr;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                }
            }
            fma8<T>(acc, pk[b], raw[b]);
        }
    }
    if (cur >= 0) {
        // the stream's last segment may continue in the next stream
        const int k = first_seg ? 0 : 1;
        store8(bnd + (2 * stream + k) * kSlab + 8 * hl, acc);
        if (hl == 0) bnd_row[2 * stream + k] = cur;
    }
}

// Stage entries [st0, st0 + n_st) of the nonzero arrays (at most COUNT per
// thread) as {column, local row << 16 | value bits}; invalid entries become value
// 0 on row 0, column 0 and are reported.  All of a thread's slots are requested
// before any column is resolved through the window's column list.
template <int COUNT>
__device__ __forceinline__ void stage_entries(const WcsrArgs& a, int32_t st0, int n_st, int32_t wbase, int32_t T_w,
                                              int nrows, int2* s_ent, int tid) {
    const uint16_t* val = static_cast<const uint16_t*>(a.val);
    uint32_t lr[COUNT], v[COUNT];
    int32_t sl[COUNT], c[COUNT];
#pragma unroll
    for (int k = 0; k < COUNT; ++k) {
        const int i = tid + k * kThreads;
        lr[k] = 0u;
        sl[k] = -1;
        v[k] = 0u;
        if (i < n_st) {
            lr[k] = a.lrow[st0 + i];
            sl[k] = a.slot[st0 + i];
            v[k] = val[st0 + i];
        }
    }
#pragma unroll
    for (int k = 0; k < COUNT; ++k) c[k] = (sl[k] >= 0 && sl[k] < T_w) ? a.wcols[wbase + sl[k]] : -1;
#pragma unroll
    for (int k = 0; k < COUNT; ++k) {
        const int i = tid + k * kThreads;
        if (i < n_st) {
            const bool ok = static_cast<int>(lr[k]) < nrows && c[k] >= 0 && c[k] < a.K;
            if (!ok) atomicOr(a.err, SPMM_DEVERR_INDEX);
            s_ent[i] = ok ? make_int2(c[k], static_cast<int>((lr[k] << 16) | v[k])) : make_int2(0, 0);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, kMinBlocks) wcsr_spmm_kernel(const WcsrArgs a) {
    extern __shared__ float sm[];
    // tile[h][kSlab] | bnd[kBnd][kSlab] | s_ent[kStage] | bnd_row[kBnd]
    float* tile = sm;
    float* bnd = tile + a.h * kSlab;
    int2* s_ent = reinterpret_cast<int2*>(bnd + kBnd * kSlab);
    int* bnd_row = reinterpret_cast<int*>(s_ent + kStage);
    __shared__ int s_last;

    const int u = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int stream = 2 * warp + half;
    if (u < a.pf_ctas && tid < a.pf_n) {
        // this CTA's share of array `tid`, shrunk to 16-byte boundaries inside it
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(a.pf_ptr[tid]);
        const int64_t n = a.pf_bytes[tid];
        const uintptr_t lo = (b0 + n * u / a.pf_ctas + 15) & ~uintptr_t(15);
        uintptr_t hi = (b0 + n * (u + 1) / a.pf_ctas) & ~uintptr_t(15);
        const uintptr_t end = (b0 + n) & ~uintptr_t(15);
        if (hi > end) hi = end;
        for (uintptr_t x = lo; x < hi; x += 65536u)
            ptx::bulk_prefetch_l2(reinterpret_cast<const void*>(x), static_cast<uint32_t>(hi - x < 65536u ? hi - x : 65536u));
    }
    const int w = a.unit_win[u];
    const int32_t nz0 = a.unit_nz_ptr[u], nz1 = a.unit_nz_ptr[u + 1];
    const T* B = static_cast<const T*>(a.B);
    if (w < 0 || static_cast<int64_t>(w) * a.h >= a.M) {  // malformed unit list: skip the unit
        if (tid == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);
        return;
    }
    const int64_t r0 = static_cast<int64_t>(w) * a.h;
    const int64_t rem = a.M - r0;
    const int nrows = rem < a.h ? static_cast<int>(rem) : a.h;
    const int units_in_window = a.unit_ptr[w + 1] - a.unit_ptr[w];
    const bool split = units_in_window > 1;
    const int32_t wbase = a.wcol_ptr[w], T_w = a.wcol_ptr[w + 1] - wbase;
    const bool one_stage = nz1 - nz0 <= kStage;
    const bool full_vec = a.b_vec != 0;

    for (int64_t n0 = 0; n0 < a.N; n0 += kSlab) {
        const int64_t ncol = n0 + 8 * hl;
        const int64_t left = a.N - ncol;
        const int valid = left >= 8 ? 8 : (left > 0 ? static_cast<int>(left) : 0);
        const bool full = full_vec && n0 + kSlab <= a.N;
        for (int i = tid; i < a.h * (kSlab / 4); i += kThreads)
            reinterpret_cast<float4*>(tile)[i] = make_float4(0.f, 0.f, 0.f, 0.f);

        for (int32_t st0 = nz0; st0 < nz1; st0 += kStage) {
            const int n_st = (nz1 - st0 < kStage) ? nz1 - st0 : kStage;
            if (!(one_stage && n0 > 0)) {
                // stage the sparse operand: resolved column, packed (local row, value)
                if (n_st <= 2 * kThreads)
                    stage_entries<2>(a, st0, n_st, wbase, T_w, nrows, s_ent, tid);
                else
                    stage_entries<kPerThread>(a, st0, n_st, wbase, T_w, nrows, s_ent, tid);
            }
            if (tid < kBnd) bnd_row[tid] = -1;
            __syncthreads();

            // whole batches per stream, so at most one stream ends in a partial batch
            const int per = ((n_st + kStreams - 1) / kStreams + kBatch - 1) / kBatch * kBatch;
            const int j_lo = stream * per;
            const int j_end = min(n_st, j_lo + per);
            if (full)
                wcsr_stream<T, true>(B, a.ldb, ncol, valid, s_ent, j_lo, j_end, tile, bnd, bnd_row, stream, hl);
            else
                wcsr_stream<T, false>(B, a.ldb, ncol, valid, s_ent, j_lo, j_end, tile, bnd, bnd_row, stream, hl);
            __syncthreads();
            // stream-boundary rows, added in stream order: thread t owns column t of the slab
            for (int k = 0; k < kBnd; ++k) {
                const int r = bnd_row[k];
                if (r >= 0) tile[r * kSlab + tid] += bnd[k * kSlab + tid];
            }
            __syncthreads();
        }

        if (!split) {
            for (int i = tid; i < nrows * (kSlab / 4); i += kThreads) {
                const int r = i / (kSlab / 4), q = i % (kSlab / 4);
                const int64_t col = n0 + 4 * q;
                const float4 v = *reinterpret_cast<const float4*>(tile + r * kSlab + 4 * q);
                float* cp = a.C + (r0 + r) * a.ldc + col;
                if (col + 4 <= a.N && a.c_vec) {
                    __stcs(reinterpret_cast<float4*>(cp), v);
                } else {
                    const float e[4] = {v.x, v.y, v.z, v.w};
                    for (int t = 0; t < 4 && col + t < a.N; ++t) cp[t] = e[t];
                }
            }
        } else {
            float* part = a.partial + static_cast<int64_t>(u) * a.h * a.N;
            for (int i = tid; i < nrows * (kSlab / 4); i += kThreads) {
                const int r = i / (kSlab / 4), q = i % (kSlab / 4);
                const int64_t col = n0 + 4 * q;
                const float4 v = *reinterpret_cast<const float4*>(tile + r * kSlab + 4 * q);
                float* pp = part + static_cast<int64_t>(r) * a.N + col;
                if (col + 4 <= a.N && a.c_vec) {
                    __stcg(reinterpret_cast<float4*>(pp), v);
                } else {
                    const float e[4] = {v.x, v.y, v.z, v.w};
                    for (int t = 0; t < 4 && col + t < a.N; ++t) __stcg(pp + t, e[t]);
                }
            }
        }
        __syncthreads();
    }

    if (!split) return;
    // last unit of the window to finish sums the partials in unit order
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        unsigned long long* t = a.ticket + static_cast<int64_t>(w) * a.nslabs;
        int last = 0;
        if (open_tag(t, a.gen, a.err)) {
            const unsigned long long old = atomicAdd(t, 1ull);
            last = static_cast<int>(old & 0xffffffffull) == units_in_window - 1;
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int u0 = a.unit_ptr[w];
    const int U = units_in_window;
    if (a.c_vec) {
        // four float4 positions per thread per pass, units two at a time: eight
        // independent loads in flight, summed in unit order
        const int64_t nv = static_cast<int64_t>(nrows) * a.N / 4;
        const int64_t stride_u = static_cast<int64_t>(a.h) * a.N / 4;  // float4s per unit partial
        const float4* pv = reinterpret_cast<const float4*>(a.partial) + static_cast<int64_t>(u0) * stride_u;
        for (int64_t i0 = tid; i0 < nv; i0 += 4 * kThreads) {
            float4 s[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) s[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < U; k0 += 2) {
                float4 x[4][2];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int64_t i = i0 + q * kThreads;
                        x[q][kk] = (k0 + kk < U && i < nv) ? __ldcg(pv + (k0 + kk) * stride_u + i)
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        if (k0 + kk < U) {
                            s[q].x += x[q][kk].x;
                            s[q].y += x[q][kk].y;
                            s[q].z += x[q][kk].z;
                            s[q].w += x[q][kk].w;
                        }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t i = i0 + q * kThreads;
                if (i < nv) {
                    const int64_t r = (4 * i) / a.N, c = (4 * i) % a.N;
                    *reinterpret_cast<float4*>(a.C + (r0 + r) * a.ldc + c) = s[q];
                }
            }
        }
    } else {
        for (int64_t i = tid; i < static_cast<int64_t>(nrows) * a.N; i += kThreads) {
            const int64_t r = i / a.N, c = i % a.N;
            float s = 0.f;
            for (int k = 0; k < U; ++k) s += __ldcg(a.partial + (static_cast<int64_t>(u0 + k) * a.h + r) * a.N + c);
            a.C[(r0 + r) * a.ldc + c] = s;
        }
    }
}

}  // namespace cc


// ---------------------------------------------------------------- SpMM on the tensor core
// Tensor-core row-window product.  For one work item (a unit, i.e. a window or
// one split of it, and one 128-column slab of B) the unit's column slots are
// taken 16 at a time (a "K step"):
//     D (128 x h) += G^T (128 x 16) * W^T (16 x h)
// where G holds the 16 gathered B rows of the step's slots (the slab's 128
// columns are the MMA's M dimension) and W is the dense h x 16 tile of the
// window's values at those slots (zero where a row has no nonzero).  D lives in
// TMEM as 128 lanes (output columns) x h columns (window rows), so each lane
// of the epilogue holds one output column of all h rows and stores it
// coalesced.
//
// One CTA per SM, four warpgroups, each working through its own items:
//   - the warpgroup's 128 threads copy the unit's column list and place its
//     nonzeros into the W tiles of up to 32 K steps (a "chunk") in shared memory;
//   - per stage of four K steps, warp q of the warpgroup gathers step q's 16 B
//     rows (16-byte loads) into a 128-byte-swizzled stage buffer (two buffers);
//   - after a named barrier, one thread issues the stage's MMAs and commits them
//     to the buffer's mbarrier;
//   - at the end of the item the four warps read their TMEM lane quarter and
//     write C (or, for a split window, a partial tile; the last unit of the
//     window sums the partials in unit order).
// All synchronisation inside a warpgroup is a named barrier or an mbarrier the
// MMAs arrive on; warpgroups share nothing but the TMEM allocation.
namespace tc {

constexpr int kWG = 4;                   // warpgroups per CTA
constexpr int kThreads = 128 * kWG;
constexpr int kSteps = 4;                // K steps per stage, one per warp of the warpgroup
constexpr int kSlab = 128;               // output columns per item (the MMA's M)
constexpr uint32_t kStepBytes = 16 * kSlab * 2;        // 16 gathered rows of 256 bytes
constexpr uint32_t kStageBytes = kSteps * kStepBytes;  // 16 KB
constexpr uint32_t kWBytes = 16384;      // W tiles of one chunk
constexpr int kMaxNp = 64;               // window rows rounded up to 16 (MMA N), at most 64
constexpr int kChunkSlots = 512;         // column slots of one chunk, at most (Np = 16: 32 steps)
constexpr uint32_t kColBytes = kChunkSlots * 4;
constexpr uint32_t kWGBytes = 2 * kStageBytes + kWBytes + kColBytes;  // 50 KB, 1024-aligned
static_assert(kWGBytes % 1024 == 0, "swizzle alignment of every warpgroup's stage buffers");

struct Args {
    const int32_t* wcol_ptr;
    const int32_t* wcols;
    const int32_t* unit_ptr;
    const int32_t* unit_win;
    const int32_t* unit_nz_ptr;
    const uint8_t* lrow;
    const int32_t* slot;
    const uint16_t* val;
    const uint16_t* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
    int64_t M, K, N;
    int32_t h, S, Np, nslabs;
    int64_t n_windows, n_units, n_items;
    int32_t b_vec;                  // B rows readable as 16-byte pieces
    uint32_t idesc;
    uint32_t gen;                   // this call's generation tag (never 0)
    unsigned long long* ticket;     // [n_windows * nslabs] arrival counters of split windows
    float* partial;                 // [n_units][h][N]
    int* err;
    uint64_t timeout_ns;
    // L2 warm-up: every CTA prefetches its share of these arrays at the start
    const void* pf_ptr[10];
    int64_t pf_bytes[10];
    int32_t pf_n;
};

__host__ __device__ constexpr int smem_bytes() { return 1024 + kWG * static_cast<int>(kWGBytes) + 8 * 3 * kWG + 16 + 16 * kWG; }

// Named barrier over `count` threads that also ANDs a per-thread flag: every
// thread gets the same answer, so a warpgroup leaves its loop together when
// any of its bounded waits gave up.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
using ptx::st_shared_v4;

// Columns n .. n+7 of B row `row` (this lane's 16-byte piece of the slab), zero
// past N or for row < 0; one vector load when the piece is whole and aligned.
__device__ __forceinline__ uint4 load_piece(const Args& a, int row, int64_t n) {
    if (row < 0) return make_uint4(0u, 0u, 0u, 0u);
    const uint16_t* p = a.B + static_cast<int64_t>(row) * a.ldb + n;
    if (a.b_vec && n + 8 <= a.N) return __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t e[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) e[t] = (n + t < a.N) ? static_cast<uint32_t>(__ldg(p + t)) : 0u;
    return make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
}

// One item's header.
struct Item {
    int32_t u, w, n0, r0, nrows, wbase, slot0, Tu, nk, nz0, nz1, U, u0;
    bool ok;
};

__device__ __forceinline__ Item load_item(const Args& a, int64_t id) {
    Item it{};
    const int64_t u = id / a.nslabs;
    it.u = static_cast<int32_t>(u);
    it.n0 = static_cast<int32_t>((id - u * a.nslabs) * kSlab);
    const int w = __ldg(a.unit_win + u);
    it.ok = w >= 0 && w < a.n_windows;
    if (!it.ok) return it;
    const int32_t up0 = __ldg(a.unit_ptr + w), up1 = __ldg(a.unit_ptr + w + 1);
    const int32_t wb = __ldg(a.wcol_ptr + w), we = __ldg(a.wcol_ptr + w + 1);
    const int32_t z0 = __ldg(a.unit_nz_ptr + u), z1 = __ldg(a.unit_nz_ptr + u + 1);
    const int64_t span = 16 * static_cast<int64_t>(a.S);
    const int64_t sl0 = span * (u - up0);
    int64_t tu = static_cast<int64_t>(we - wb) - sl0;
    tu = tu < 0 ? 0 : (tu > span ? span : tu);
    const int64_t r0 = static_cast<int64_t>(w) * a.h;
    it.w = w;
    it.r0 = static_cast<int32_t>(r0);
    it.nrows = static_cast<int32_t>(a.M - r0 < a.h ? a.M - r0 : a.h);
    it.wbase = wb;
    it.slot0 = static_cast<int32_t>(sl0);
    it.Tu = static_cast<int32_t>(tu);
    it.nk = static_cast<int32_t>((tu + 15) / 16);
    it.nz0 = z0;
    it.nz1 = z1 < z0 ? z0 : z1;
    it.U = up1 - up0;
    it.u0 = up0;
    return it;
}

__global__ void __launch_bounds__(kThreads, 1) wcsr_tc_kernel(const Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int wg = warp / 4, q = warp % 4;  // q: the warp's TMEM lane quarter and its step in every stage
    const int tw = threadIdx.x % 128;       // thread within the warpgroup
    uint8_t* wgs = smem + wg * kWGBytes;    // [stage 0 | stage 1 | W tiles | column list]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWG * kWGBytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * kWG);
    int* s_last = reinterpret_cast<int*>(tslot + 4) + wg;
    const uint32_t sw = ptx::smem_u32(wgs);
    const uint32_t w_tiles = sw + 2 * kStageBytes;
    int32_t* collist = reinterpret_cast<int32_t*>(wgs + 2 * kStageBytes + kWBytes);
    const uint32_t sdone0 = ptx::smem_u32(bars + 3 * wg), sdone1 = sdone0 + 8, adone = sdone0 + 16;
    const uint32_t bar_id = 1 + wg;
    const uint32_t tstep = static_cast<uint32_t>(a.Np) * 32u;  // one K step's W tile
    const int chunk_steps = static_cast<int>(kWBytes / tstep) < kChunkSlots / 16 ? static_cast<int>(kWBytes / tstep)
                                                                                  : kChunkSlots / 16;
    const uint32_t tmem_cols = kWG * a.Np <= 64 ? 64u : (kWG * a.Np <= 128 ? 128u : 256u);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 3 * kWG; ++i) ptx::mbar_init(ptx::smem_u32(bars + i), 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), tmem_cols);
        ptx::tmem_relinquish();
    }
    if (threadIdx.x < a.pf_n) {
        // L2 warm-up: this CTA's share of one of the format arrays or B
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(a.pf_ptr[threadIdx.x]);
        const int64_t n = a.pf_bytes[threadIdx.x];
        const uintptr_t lo = (b0 + n * blockIdx.x / gridDim.x + 15) & ~uintptr_t(15);
        uintptr_t hi = (b0 + n * (blockIdx.x + 1) / gridDim.x) & ~uintptr_t(15);
        const uintptr_t end = (b0 + n) & ~uintptr_t(15);
        if (hi > end) hi = end;
        for (uintptr_t x = lo; x < hi; x += 65536u)
            ptx::bulk_prefetch_l2(reinterpret_cast<const void*>(x), static_cast<uint32_t>(hi - x < 65536u ? hi - x : 65536u));
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t dacc = tmem + static_cast<uint32_t>(wg * a.Np);

    // A operand: the gathered rows, M = 128 columns x K = 16 slots, MN-major,
    // 128-byte swizzle, two 64-column chunks 2 KB apart.  B operand: the W tile,
    // N = Np rows x K = 16 slots, K-major without swizzle: (row, slot) at
    // (row / 8) 256 + (slot / 8) 128 + (row % 8) 16 + (slot % 8) 2.
    const uint64_t adesc0 = ptx::smem_desc(sw, 2048u, 1024u, ptx::SWZ_128B);
    const uint64_t bdesc0 = ptx::smem_desc(w_tiles, 128u, 256u, ptx::SWZ_NONE);
    const int hl = lane & 15, hi = lane >> 4;
    const uint32_t piece_off = static_cast<uint32_t>(hl / 8) * 2048u;
    const int gq = hl % 8;
    const int64_t nwg = static_cast<int64_t>(gridDim.x) * kWG;
    int sc = 0, ic = 0;  // stages and items of this warpgroup so far
    bool ok = true;
    Item nxt = load_item(a, static_cast<int64_t>(blockIdx.x) * kWG + wg < a.n_items
                                ? static_cast<int64_t>(blockIdx.x) * kWG + wg : 0);
    for (int64_t id = static_cast<int64_t>(blockIdx.x) * kWG + wg; id < a.n_items && ok; id += nwg) {
        const Item it = nxt;
        if (id + nwg < a.n_items) nxt = load_item(a, id + nwg);  // next item's header, in flight meanwhile
        if (!it.ok) {
            if (tw == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);  // malformed unit list: skip the unit
            continue;
        }
        const int64_t n = static_cast<int64_t>(it.n0) + 8 * hl;
        for (int c0 = 0; c0 < it.nk && ok; c0 += chunk_steps) {
            const int cs = it.nk - c0 < chunk_steps ? it.nk - c0 : chunk_steps;
            // the W tiles and column list are rewritten: the last stage's MMAs must be done
            const bool free_ok = sc == 0 || ptx::mbar_wait((sc - 1) % 2 ? sdone1 : sdone0,
                                                           static_cast<uint32_t>((sc - 1) / 2) & 1u, a.timeout_ns,
                                                           a.err, SPMM_DEVERR_TIMEOUT);
            if (!bar_and(bar_id, 128, free_ok)) {
                ok = false;
                break;
            }
            for (uint32_t o = 16u * tw; o < static_cast<uint32_t>(cs) * tstep; o += 16u * 128u)
                st_shared_v4(w_tiles + o, make_uint4(0u, 0u, 0u, 0u));
            {
                // at most 4 slots per thread (a chunk has at most 512): all loads in flight together
                int cv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = tw + 128 * k, sl = 16 * c0 + e;
                    cv[k] = (e < 16 * cs && sl < it.Tu) ? __ldg(a.wcols + it.wbase + it.slot0 + sl) : -1;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = tw + 128 * k, sl = 16 * c0 + e;
                    if (e < 16 * cs) {
                        const bool good = cv[k] >= 0 && cv[k] < a.K;
                        if (sl < it.Tu && !good) atomicOr(a.err, SPMM_DEVERR_INDEX);
                        collist[e] = good ? cv[k] : -1;
                    }
                }
            }
            ptx::named_barrier(bar_id, 128);
            // the chunk's nonzeros into their W tiles, eight per thread loaded together
            const int lo = 16 * c0, hiw = 16 * (c0 + cs);
            for (int e0 = it.nz0 + tw; e0 < it.nz1; e0 += 128 * 8) {
                int lr[8], sl[8];
                uint16_t v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int e = e0 + 128 * k;
                    lr[k] = 255;
                    sl[k] = -1;
                    v[k] = 0;
                    if (e < it.nz1) {
                        lr[k] = a.lrow[e];
                        sl[k] = __ldg(a.slot + e) - it.slot0;
                        v[k] = __ldg(a.val + e);
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (e0 + 128 * k >= it.nz1) continue;
                    if (sl[k] < 0 || sl[k] >= it.Tu || lr[k] >= it.nrows) {
                        if (c0 == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);  // skipped, reported once
                        continue;
                    }
                    if (sl[k] < lo || sl[k] >= hiw) continue;
                    const int kk = sl[k] - lo, kx = kk & 15;
                    st_shared_u16(w_tiles + (kk >> 4) * tstep + (lr[k] >> 3) * 256u + (kx >> 3) * 128u +
                                      (lr[k] & 7) * 16u + (kx & 7) * 2u,
                                  v[k]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_barrier(bar_id, 128);
            // stages of the chunk: warp q gathers step 4 j + q (its 16 rows are
            // loaded while the buffer's previous MMAs are waited for)
            const int nst = (cs + kSteps - 1) / kSteps;
            for (int j = 0; j < nst; ++j) {
                const int b = sc % 2;
                const uint32_t sdone = b ? sdone1 : sdone0;
                uint4 r[8];
                {
                    const int ks = kSteps * j + q;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int col = ks < cs ? collist[16 * ks + 2 * t + hi] : -1;
                        r[t] = load_piece(a, col, n);
                    }
                }
                // buffer b was last read by the MMAs of stage sc - 2
                const bool buf_ok = sc < 2 || ptx::mbar_wait(sdone, static_cast<uint32_t>((sc - 2) / 2) & 1u,
                                                             a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
                if (buf_ok && kSteps * j + q < cs) {
                    const uint32_t dst = sw + b * kStageBytes + q * kStepBytes + piece_off;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int s = 2 * t + hi;  // slot within the step
                        st_shared_v4(dst + s * 128u + (static_cast<uint32_t>(gq ^ (s & 7)) << 4), r[t]);
                    }
                    ptx::fence_proxy_async_smem();
                }
                ptx::tc_fence_before();
                if (!bar_and(bar_id, 128, buf_ok)) {
                    ok = false;
                    break;
                }
                if (tw == 0) {
                    ptx::tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>((b * kStageBytes) >> 4);
                    const int nq = cs - kSteps * j < kSteps ? cs - kSteps * j : kSteps;
                    for (int qq = 0; qq < nq; ++qq)
                        ptx::mma_f16(dacc, adesc0 + so + static_cast<uint64_t>(qq) * (kStepBytes >> 4),
                                     bdesc0 + static_cast<uint64_t>(kSteps * j + qq) * (tstep >> 4), a.idesc,
                                     (c0 + kSteps * j + qq > 0) ? 1u : 0u);
                    ptx::mma_commit(sdone);
                }
                ++sc;
            }
        }
        if (!ok) break;
        // ---- epilogue: this warp's lane quarter = output columns 32 q .. 32 q + 31 of the slab
        if (tw == 0) ptx::mma_commit(adone);  // arrives once every MMA issued so far is done
        const bool acc_ok = ptx::mbar_wait(adone, static_cast<uint32_t>(ic) & 1u, a.timeout_ns, a.err,
                                           SPMM_DEVERR_TIMEOUT);
        if (!bar_and(bar_id, 128, acc_ok)) {
            ok = false;
            break;
        }
        ++ic;
        ptx::tc_fence_after();
        const int64_t ncol = static_cast<int64_t>(it.n0) + 32 * q + lane;
        const bool split = it.U > 1;
        float* base = split ? a.partial + static_cast<int64_t>(it.u) * a.h * a.N
                            : a.C + static_cast<int64_t>(it.r0) * a.ldc;
        const int64_t ld = split ? a.N : a.ldc;
        const uint32_t tl = dacc + (static_cast<uint32_t>(32 * q) << 16);
        for (int c = 0; c < a.Np / 16; ++c) {
            uint32_t v[16];
            if (it.nk > 0) {
                ptx::tmem_ld16(tl + 16 * c, v);
                ptx::tmem_ld_wait();
            } else {
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] = 0u;  // a window without nonzeros
            }
            if (ncol < a.N) {
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int rr = 16 * c + t;
                    if (rr < it.nrows) {
                        float* p = base + rr * ld + ncol;
                        if (split) __stcg(p, __uint_as_float(v[t]));
                        else __stcs(p, __uint_as_float(v[t]));
                    }
                }
            }
        }
        ptx::tc_fence_before();
        if (!split) continue;
        // Split window: the last of its units (arrival counter) sums the partials
        // of all units in unit order, so the result does not depend on timing.
        __threadfence();
        ptx::named_barrier(bar_id, 128);
        if (tw == 0) {
            unsigned long long* t = a.ticket + static_cast<int64_t>(it.w) * a.nslabs + it.n0 / kSlab;
            int last = 0;
            if (open_tag(t, a.gen, a.err)) {
                const unsigned long long old = atomicAdd(t, 1ull);
                last = static_cast<int>(old & 0xffffffffull) == it.U - 1;
            }
            *s_last = last;
        }
        ptx::named_barrier(bar_id, 128);
        if (!*s_last) continue;
        __threadfence();
        if (ncol < a.N) {
            // 8 rows at a time: those rows of one unit are loaded together, the
            // units are added in unit order
            for (int rb = 0; rb < it.nrows; rb += 8) {
                float acc[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) acc[t] = 0.f;
                for (int k = 0; k < it.U; ++k) {
                    const float* pp = a.partial + (static_cast<int64_t>(it.u0 + k) * a.h + rb) * a.N + ncol;
                    float x[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) x[t] = rb + t < it.nrows ? __ldcg(pp + t * a.N) : 0.f;
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[t] += x[t];
                }
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    if (rb + t < it.nrows) a.C[(static_cast<int64_t>(it.r0) + rb + t) * a.ldc + ncol] = acc[t];
            }
        }
    }
    // leave no MMA in flight (after a timeout too): wait, bounded, for the last commit
    if (sc > 0 && tw == 0) {
        ptx::mma_commit(adone);
        ptx::mbar_wait(adone, static_cast<uint32_t>(ic) & 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace tc

// ---------------------------------------------------------------- streaming tensor-core product
// The same window products as tc::wcsr_tc_kernel (D (128 x Np) += G (128 x 16)
// W^T (16 x Np) per 16 column slots), with the work split by role instead of by
// item, so that the gathers of later items proceed while earlier items are
// prepared, multiplied and written out.  One CTA per SM, persistent over items
// (unit, 128-column slab); windows of at most 16 rows (Np = 16).
//   warps 0-7   preparation, one item per warp at a time (item i to warp i % 8,
//               its own item slot): the unit header, its column list, its
//               values into the slot's W tiles (all steps of the item: at most
//               32, 16 KB), then the item record.  Each item's chain of dependent
//               loads is several L2 round trips, so eight are prepared at once.
//   warps 8-15  gathers: items alternate between two rings of 8 stages (4 KB
//               each), one per MMA issuer; step t of a ring's sequence of (item,
//               K step) goes to warp 8 + t % 8, which copies the step's 16 B rows
//               into stage t % 8 of that ring with 16-byte cp.async copies (no
//               registers held: both rings can be in flight).
//   warps 16-17 MMA issuers, items alternating between them: one thread each
//               issues its items' steps (M = 128 output columns, N = 16 window
//               rows, K = 16 slots) into the item's accumulator (two per issuer
//               in TMEM) and commits each stage back to the gathers.  With one
//               issuer its per-step waits and issue latency bounded the kernel
//               (clustered windows: 76 us against 62 us with two).
//   warps 18-21 epilogue: per item, read the accumulator (TMEM lane quarter =
//               32 output columns) and write C, or a partial tile and the
//               split-window fix-up as in tc::wcsr_tc_kernel.
// Every stage has exactly one filling warp and one consuming issuer, so no
// party can run two phases ahead of a parity wait (a shared ring let one issuer
// take a stage two fills early).  An item slot is reused once its gathers, both
// issuers and its epilogue have all let go of it; every wait is bounded.
namespace ts {

constexpr int kPrepWarps = 8, kGatherWarps = 8, kEpiWarps = 4;
constexpr int kIssuers = 2;  // MMA-issuing warps (alternate items, own stage ring, two accumulators each)
constexpr int kGroup = 1;    // steps whose stages are waited for together before their MMAs (more: slower)
constexpr int kGatherWarp0 = kPrepWarps, kMmaWarp = kGatherWarp0 + kGatherWarps, kEpiWarp0 = kMmaWarp + kIssuers;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kSlab = 128;
constexpr int kNp = 16;                                  // MMA N: windows of at most 16 rows
constexpr int kSlots = kPrepWarps;                       // item slots: one per preparing warp
constexpr int kAcc = 2 * kIssuers;                       // TMEM accumulators (two per issuer)
constexpr int kStages = 16;                              // gather stages, split into one ring per issuer
constexpr int kRing = kStages / kIssuers;                // so every stage has one filler and one consumer
static_assert(kStages % kIssuers == 0 && kGroup <= kRing, "ring split");
// gathering warp g fills the steps t with t % kGatherWarps == g; a stage filled by two warps
// could see one of them two fills ahead of the other, which a parity wait cannot tell apart
static_assert(kRing % kGatherWarps == 0, "one filling warp per stage");
constexpr uint32_t kStepBytes = 16 * kSlab * 2;          // 16 gathered rows of 256 bytes
constexpr uint32_t kTile = kNp * 32;                     // one step's W tile (16 rows x 16 slots, fp16)
constexpr int kMaxSteps = 32;                            // 512 column slots per unit at most (S <= 32)
constexpr uint32_t kWBytes = kMaxSteps * kTile;          // 16 KB per item slot
constexpr uint32_t kColBytes = kMaxSteps * 16 * 4;       // 2 KB per item slot
constexpr uint32_t kRingOff = 0;
constexpr uint32_t kWOff = kRingOff + kStages * kStepBytes;
constexpr uint32_t kColOff = kWOff + kSlots * kWBytes;
constexpr uint32_t kRecOff = kColOff + kSlots * kColBytes;
constexpr uint32_t kBarOff = kRecOff + kSlots * 64;
// barriers: item_full, item_empty [kSlots]; stage_full, stage_empty [kStages]; acc_full, acc_empty [kAcc];
// done [kIssuers]
constexpr int kBars = 2 * kSlots + 2 * kStages + 2 * kAcc + kIssuers;
constexpr uint32_t kSmem = 1024 + kBarOff + 8 * kBars + 16 + 16;
static_assert(kStepBytes % 1024 == 0 && kWOff % 1024 == 0, "swizzle alignment of the stages");
static_assert(kSmem <= 232448, "shared memory per block");
// item_empty: every gathering warp, every MMA issuer (each reads the step count) and every epilogue warp
constexpr int kItemUsers = kGatherWarps + kIssuers + kEpiWarps;
static_assert(kAcc % kIssuers == 0, "issuer j owns accumulators j, j + kIssuers, ...");

struct Rec {
    int32_t u, w, n0, r0, nrows, Tu, nk, U, u0, ok;
};

__global__ void __launch_bounds__(kThreads, 1) wcsr_ts_kernel(const tc::Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t s0 = ptx::smem_u32(smem);
    const uint32_t bar0 = s0 + kBarOff;
    auto item_full = [&](int i) { return bar0 + 8u * i; };
    auto item_empty = [&](int i) { return bar0 + 8u * (kSlots + i); };
    auto stage_full = [&](int s) { return bar0 + 8u * (2 * kSlots + s); };
    auto stage_empty = [&](int s) { return bar0 + 8u * (2 * kSlots + kStages + s); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * kSlots + 2 * kStages + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kSlots + 2 * kStages + kAcc + b); };
    auto done_bar = [&](int j) { return bar0 + 8u * (2 * kSlots + 2 * kStages + 2 * kAcc + j); };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kBars);
    int* s_last = reinterpret_cast<int*>(smem + kBarOff + 8 * kBars + 16);
    Rec* recs = reinterpret_cast<Rec*>(smem + kRecOff);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            ptx::mbar_init(item_full(i), 1);
            ptx::mbar_init(item_empty(i), kItemUsers);
        }
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(stage_full(s), 32);  // one cp.async arrival per lane of the gathering warp
            ptx::mbar_init(stage_empty(s), 1);
        }
        for (int b = 0; b < kAcc; ++b) {
            ptx::mbar_init(acc_full(b), 1);
            ptx::mbar_init(acc_empty(b), kEpiWarps);
        }
        for (int j = 0; j < kIssuers; ++j) ptx::mbar_init(done_bar(j), 1);
        ptx::fence_mbar_init();
    }
    constexpr uint32_t kTmemCols = kAcc * kNp <= 32 ? 32u : (kAcc * kNp <= 64 ? 64u : 128u);
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), kTmemCols);
        ptx::tmem_relinquish();
    }
    if (threadIdx.x < a.pf_n) {
        // L2 warm-up: this CTA's share of one of the format arrays or B
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(a.pf_ptr[threadIdx.x]);
        const int64_t n = a.pf_bytes[threadIdx.x];
        const uintptr_t lo = (b0 + n * blockIdx.x / gridDim.x + 15) & ~uintptr_t(15);
        uintptr_t hi = (b0 + n * (blockIdx.x + 1) / gridDim.x) & ~uintptr_t(15);
        const uintptr_t end = (b0 + n) & ~uintptr_t(15);
        if (hi > end) hi = end;
        for (uintptr_t x = lo; x < hi; x += 65536u)
            ptx::bulk_prefetch_l2(reinterpret_cast<const void*>(x), static_cast<uint32_t>(hi - x < 65536u ? hi - x : 65536u));
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    const int64_t first = blockIdx.x, stride = gridDim.x;

    if (warp < kPrepWarps) {
        // -------------------------------------------------------- preparation
        const int pw = warp;  // this warp prepares items pw, pw + kPrepWarps, ... in slot pw
        bool ok = true;
        for (int ic = pw; ok && first + static_cast<int64_t>(ic) * stride < a.n_items; ic += kPrepWarps) {
            const int64_t id = first + static_cast<int64_t>(ic) * stride;
            const int slot = ic % kSlots;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(item_empty(slot), (static_cast<uint32_t>(ic / kSlots) & 1u) ^ 1u,
                                                        a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT))) {
                ok = false;
                break;
            }
            const tc::Item it = tc::load_item(a, id);
            const int nk = it.ok ? it.nk : 0;
            int32_t* cols = reinterpret_cast<int32_t*>(smem + kColOff + slot * kColBytes);
            const uint32_t wt = s0 + kWOff + slot * kWBytes;
            // the column list (at most 16 slots per lane, all loads in flight together)
            int cv[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int e = lane + 32 * k;
                cv[k] = (e < 16 * nk && e < it.Tu) ? __ldg(a.wcols + it.wbase + it.slot0 + e) : -1;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int e = lane + 32 * k;
                if (e < 16 * nk) {
                    const bool good = cv[k] >= 0 && cv[k] < a.K;
                    if (e < it.Tu && !good) atomicOr(a.err, SPMM_DEVERR_INDEX);
                    cols[e] = good ? cv[k] : -1;
                }
            }
            for (uint32_t o = 16u * lane; o < static_cast<uint32_t>(nk) * kTile; o += 16u * 32u)
                ptx::st_shared_v4(wt + o, make_uint4(0u, 0u, 0u, 0u));
            __syncwarp();
            // the unit's nonzeros into their W tiles, eight per lane loaded together
            if (it.ok) {
                for (int e0 = it.nz0 + lane; e0 < it.nz1; e0 += 32 * 8) {
                    int lr[8], sl[8];
                    uint16_t v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int e = e0 + 32 * k;
                        lr[k] = 255;
                        sl[k] = -1;
                        v[k] = 0;
                        if (e < it.nz1) {
                            lr[k] = a.lrow[e];
                            sl[k] = __ldg(a.slot + e) - it.slot0;
                            v[k] = __ldg(a.val + e);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (e0 + 32 * k >= it.nz1) continue;
                        if (sl[k] < 0 || sl[k] >= it.Tu || lr[k] >= it.nrows) {
                            atomicOr(a.err, SPMM_DEVERR_INDEX);  // skipped
                            continue;
                        }
                        const int kx = sl[k] & 15;
                        tc::st_shared_u16(wt + (sl[k] >> 4) * kTile + (lr[k] >> 3) * 256u + (kx >> 3) * 128u +
                                              (lr[k] & 7) * 16u + (kx & 7) * 2u,
                                          v[k]);
                    }
                }
            } else if (lane == 0) {
                atomicOr(a.err, SPMM_DEVERR_INDEX);  // malformed unit list: the item is skipped
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                recs[slot] = Rec{it.u, it.w, it.n0, it.r0, it.nrows, it.Tu, nk, it.U, it.u0, it.ok ? 1 : 0};
                ptx::mbar_arrive(item_full(slot));
            }
        }
    } else if (warp < kMmaWarp) {
        // -------------------------------------------------------- gathers
        const int g = warp - kGatherWarp0;
        const int hl = lane & 15, hi = lane >> 4, gq = hl % 8;
        const uint32_t piece_off = static_cast<uint32_t>(hl / 8) * 2048u;
        int ic = 0;
        int64_t tr[kIssuers];  // steps of earlier items, per ring
#pragma unroll
        for (int r = 0; r < kIssuers; ++r) tr[r] = 0;
        bool ok = true;
        for (int64_t id = first; id < a.n_items && ok; id += stride, ++ic) {
            const int slot = ic % kSlots, ring = ic % kIssuers;
            int64_t t0 = tr[0];
#pragma unroll
            for (int r = 1; r < kIssuers; ++r)
                if (ring == r) t0 = tr[r];
            // every wait's outcome is made warp-uniform, so the warp leaves together
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(item_full(slot), static_cast<uint32_t>(ic / kSlots) & 1u,
                                                        a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT))) {
                ok = false;
                break;
            }
            const int nk = recs[slot].nk;
            const int64_t n = static_cast<int64_t>(recs[slot].n0) + 8 * hl;
            const int32_t* cols = reinterpret_cast<const int32_t*>(smem + kColOff + slot * kColBytes);
            for (int k = static_cast<int>((g - t0 % kGatherWarps + kGatherWarps) % kGatherWarps); k < nk;
                 k += kGatherWarps) {
                const int64_t t = t0 + k;
                const int s = ring * kRing + static_cast<int>(t % kRing);
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(stage_empty(s), (static_cast<uint32_t>(t / kRing) & 1u) ^ 1u,
                                                            a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT))) {
                    ok = false;
                    break;
                }
                // this lane's 8 pieces (16 bytes each) of rows 2 j + hi; zero-filled for
                // slots past the unit's columns and columns past N
                const uint32_t dst = s0 + kRingOff + s * kStepBytes + piece_off;
                const int64_t left = a.N - n;
                const uint32_t nb = left >= 8 ? 16u : (left > 0 ? static_cast<uint32_t>(left) * 2u : 0u);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int sr = 2 * j + hi;  // slot within the step
                    const int col = cols[16 * k + sr];
                    const uint16_t* src = col >= 0 && nb ? a.B + static_cast<int64_t>(col) * a.ldb + n : a.B;
                    ptx::cp_async16(dst + sr * 128u + (static_cast<uint32_t>(gq ^ (sr & 7)) << 4), src,
                                    col >= 0 ? nb : 0u);
                }
                ptx::cp_async_arrive_noinc(stage_full(s));
            }
#pragma unroll
            for (int r = 0; r < kIssuers; ++r)
                if (ring == r) tr[r] = t0 + nk;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(item_empty(slot));
        }
        ptx::cp_async_wait<0>();  // no copy into shared memory outstanding at exit
    } else if (warp < kEpiWarp0) {
        // -------------------------------------------------------- MMA issuers
        // issuer j takes items j, j + kIssuers, ... and their steps from ring j; it
        // waits for each group of kGroup stages before one proxy fence and their MMAs
        const int j = warp - kMmaWarp;
        if (lane == 0) {
            const uint64_t adesc0 = ptx::smem_desc(s0 + kRingOff, 2048u, 1024u, ptx::SWZ_128B);
            int ic = 0;
            int64_t t = 0;
            bool ok = true;
            for (int64_t id = first; id < a.n_items && ok; id += stride, ++ic) {
                const int slot = ic % kSlots;
                if (!ptx::mbar_wait(item_full(slot), static_cast<uint32_t>(ic / kSlots) & 1u, a.timeout_ns, a.err,
                                    SPMM_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                const int nk = recs[slot].nk;
                if (ic % kIssuers != j) {  // another issuer's item
                    ptx::mbar_arrive(item_empty(slot));
                    continue;
                }
                const int b = ic % kAcc;
                if (!ptx::mbar_wait(acc_empty(b), (static_cast<uint32_t>(ic / kAcc) & 1u) ^ 1u, a.timeout_ns, a.err,
                                    SPMM_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t bdesc0 = ptx::smem_desc(s0 + kWOff + slot * kWBytes, 128u, 256u, ptx::SWZ_NONE);
                const uint32_t d = tmem + static_cast<uint32_t>(b * kNp);
                for (int k0 = 0; k0 < nk && ok; k0 += kGroup) {
                    const int kn = nk - k0 < kGroup ? nk - k0 : kGroup;
                    for (int k = k0; k < k0 + kn; ++k) {
                        const int64_t tt = t + k;
                        if (!ptx::mbar_wait(stage_full(j * kRing + static_cast<int>(tt % kRing)),
                                            static_cast<uint32_t>(tt / kRing) & 1u, a.timeout_ns, a.err,
                                            SPMM_DEVERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    ptx::tc_fence_after();
                    ptx::fence_proxy_async_smem();  // the stages arrived through cp.async (generic proxy)
                    for (int k = k0; k < k0 + kn; ++k) {
                        const int s = j * kRing + static_cast<int>((t + k) % kRing);
                        ptx::mma_f16(d, adesc0 + static_cast<uint64_t>(s) * (kStepBytes >> 4),
                                     bdesc0 + static_cast<uint64_t>(k) * (kTile >> 4), a.idesc, k > 0 ? 1u : 0u);
                        ptx::mma_commit(stage_empty(s));
                    }
                }
                if (!ok) break;
                t += nk;
                ptx::mma_commit(acc_full(b));
                ptx::mbar_arrive(item_empty(slot));
            }
            // leave no MMA in flight (after a timeout too)
            ptx::mma_commit(done_bar(j));
            ptx::mbar_wait(done_bar(j), 0, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter: output columns 32 q .. 32 q + 31 of the slab
        const int et = threadIdx.x - 32 * kEpiWarp0;  // 0 .. 127
        int ic = 0;
        bool ok = true;
        for (int64_t id = first; id < a.n_items && ok; id += stride, ++ic) {
            const int slot = ic % kSlots, b = ic % kAcc;
            const bool waited = ptx::mbar_wait(item_full(slot), static_cast<uint32_t>(ic / kSlots) & 1u, a.timeout_ns,
                                               a.err, SPMM_DEVERR_TIMEOUT) &&
                                ptx::mbar_wait(acc_full(b), static_cast<uint32_t>(ic / kAcc) & 1u, a.timeout_ns, a.err,
                                               SPMM_DEVERR_TIMEOUT);
            if (!tc::bar_and(2, 32 * kEpiWarps, waited)) {  // the four warps leave together
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const Rec it = recs[slot];
            const int64_t ncol = static_cast<int64_t>(it.n0) + 32 * q + lane;
            const bool split = it.U > 1;
            float* base = split ? a.partial + static_cast<int64_t>(it.u) * a.h * a.N
                                : a.C + static_cast<int64_t>(it.r0) * a.ldc;
            const int64_t ld = split ? a.N : a.ldc;
            uint32_t v[16];
            if (it.nk > 0) {
                ptx::tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * kNp), v);
                ptx::tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0u;  // a window without nonzeros
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(acc_empty(b));
                ptx::mbar_arrive(item_empty(slot));
            }
            if (!it.ok) continue;
            if (ncol < a.N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < it.nrows) {
                        float* p = base + j * ld + ncol;
                        if (split)
                            __stcg(p, __uint_as_float(v[j]));
                        else
                            __stcs(p, __uint_as_float(v[j]));
                    }
            }
            if (!split) continue;
            // split window: the last of its units (arrival counter) sums the partials
            // of all units in unit order
            __threadfence();
            ptx::named_barrier(2, 32 * kEpiWarps);
            if (et == 0) {
                unsigned long long* tk = a.ticket + static_cast<int64_t>(it.w) * a.nslabs + it.n0 / kSlab;
                int last = 0;
                if (open_tag(tk, a.gen, a.err)) {
                    const unsigned long long old = atomicAdd(tk, 1ull);
                    last = static_cast<int>(old & 0xffffffffull) == it.U - 1;
                }
                *s_last = last;
            }
            ptx::named_barrier(2, 32 * kEpiWarps);
            const int last = *s_last;
            ptx::named_barrier(2, 32 * kEpiWarps);  // s_last is rewritten by the next split item
            if (!last) continue;
            __threadfence();
            if (ncol < a.N) {
                for (int rb = 0; rb < it.nrows; rb += 8) {
                    float acc[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
                    for (int k = 0; k < it.U; ++k) {
                        const float* pp = a.partial + (static_cast<int64_t>(it.u0 + k) * a.h + rb) * a.N + ncol;
                        float x[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) x[j] = rb + j < it.nrows ? __ldcg(pp + j * a.N) : 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] += x[j];
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (rb + j < it.nrows) a.C[(static_cast<int64_t>(it.r0) + rb + j) * a.ldc + ncol] = acc[j];
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace ts

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct BuildWs {
    int32_t *fpre, *rowfirst, *wT, *wU, *slot_ws;
};

BuildWs carve(void* ws, int64_t M, int64_t nnz, int64_t nw) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    BuildWs b;
    b.fpre = reinterpret_cast<int32_t*>(p);
    p += align256(sizeof(int32_t) * (nnz + 1));
    b.rowfirst = reinterpret_cast<int32_t*>(p);
    p += align256(sizeof(int32_t) * (M + 1));
    b.wT = reinterpret_cast<int32_t*>(p);
    p += align256(sizeof(int32_t) * (nw + 1));
    b.wU = reinterpret_cast<int32_t*>(p);
    p += align256(sizeof(int32_t) * (nw + 1));
    b.slot_ws = reinterpret_cast<int32_t*>(p);
    return b;
}

}  // namespace

size_t wcsr_build_ws_bytes(int64_t M, int64_t nnz, int32_t h) {
    const int64_t nw = (M + h - 1) / h;
    return align256(4 * (nnz + 1)) + align256(4 * (M + 1)) + 2 * align256(4 * (nw + 1)) + align256(4 * (nnz + 1));
}

spmm_status run_wcsr_count(const spmm_csr_t* A, int32_t h, int32_t S, void* ws, int64_t* n_wcols, int64_t* n_units,
                           cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_mu);
    void* ep = nullptr;
    if (cudaGetSymbolAddress(&ep, g_wcsr_build_error) != cudaSuccess) return SPMM_ERR_CUDA;
    int* err = static_cast<int*>(ep);
    const int64_t M = A->M, nnz = A->nnz, nw = (M + h - 1) / h, span = 16 * static_cast<int64_t>(S);
    BuildWs b = carve(ws, M, nnz, nw);
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SPMM_ERR_CUDA;
    csr_check_kernel<<<static_cast<unsigned>((M + 256) / 256), 256, 0, s>>>(A->row_ptr, A->col, M, A->K, nnz, err);
    int e = 0;
    if (cudaMemcpyAsync(&e, err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    if (e) return SPMM_ERR_FORMAT;
    if (M > 0) {
        wcsr_first_kernel<<<static_cast<unsigned>((M * 32 + 255) / 256), 256, 0, s>>>(A->row_ptr, A->col, M, h,
                                                                                      b.fpre, b.rowfirst);
        wcsr_window_kernel<<<static_cast<unsigned>((nw + 255) / 256), 256, 0, s>>>(b.rowfirst, M, h, span, nw, b.wT,
                                                                                   b.wU);
    }
    if (cudaMemsetAsync(b.wT + nw, 0, sizeof(int32_t), s) != cudaSuccess ||
        cudaMemsetAsync(b.wU + nw, 0, sizeof(int32_t), s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    scan_kernel<<<1, 1024, 0, s>>>(b.wT, nw + 1);
    scan_kernel<<<1, 1024, 0, s>>>(b.wU, nw + 1);
    if (cudaGetLastError() != cudaSuccess) return SPMM_ERR_CUDA;
    int32_t tot[2] = {0, 0};
    if (cudaMemcpyAsync(&tot[0], b.wT + nw, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&tot[1], b.wU + nw, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    *n_wcols = tot[0];
    *n_units = tot[1];
    return SPMM_OK;
}

spmm_status run_wcsr_fill(const spmm_csr_t* A, int32_t h, int32_t S, void* ws, spmm_wcsr_t* out, cudaStream_t s) {
    const int64_t M = A->M, nnz = A->nnz, nw = (M + h - 1) / h, span = 16 * static_cast<int64_t>(S);
    BuildWs b = carve(ws, M, nnz, nw);
    if (cudaMemcpyAsync(out->wcol_ptr, b.wT, 4 * (nw + 1), cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(out->unit_ptr, b.wU, 4 * (nw + 1), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    if (M > 0) {
        const unsigned gw = static_cast<unsigned>((M * 32 + 255) / 256);
        wcsr_slot_kernel<<<gw, 256, 0, s>>>(A->row_ptr, A->col, b.fpre, b.rowfirst, b.wT, M, h, b.slot_ws,
                                            out->wcols);
        // values are copied bit for bit (both 16-bit types)
        wcsr_place_kernel<uint16_t><<<gw, 256, 0, s>>>(A->row_ptr, static_cast<const uint16_t*>(A->val),
                                                       b.slot_ws, M, h, span, out->lrow, out->slot,
                                                       static_cast<uint16_t*>(out->val));
    }
    wcsr_units_kernel<<<static_cast<unsigned>((nw + 1 + 255) / 256), 256, 0, s>>>(
        A->row_ptr, b.slot_ws, b.wU, M, h, span, nw, out->wnz_ptr, out->unit_win, out->unit_nz_ptr);
    return cuda_status(cudaGetLastError());
}

namespace {

// Workspace of the SpMM: one arrival counter per (window, 128-column slab)
// and the partial tiles of split windows.  The counters carry the generation
// tag of the call that last used them, so the workspace needs no clearing
// between calls, and a call that stopped early (a timed-out wait) leaves
// nothing that a later call would misread.
struct SpmmWs {
    unsigned long long* ticket;
    float* partial;
};

size_t wcsr_nslabs(int64_t N) { return static_cast<size_t>((N + tc::kSlab - 1) / tc::kSlab); }

size_t wcsr_ticket_bytes(const spmm_wcsr_t* A, int64_t N) {
    return align256(sizeof(unsigned long long) * static_cast<size_t>(A->n_windows) * wcsr_nslabs(N));
}

SpmmWs carve_spmm(void* ws, const spmm_wcsr_t* A, int64_t N) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    SpmmWs w;
    p += 256;
    w.ticket = reinterpret_cast<unsigned long long*>(p);
    p += wcsr_ticket_bytes(A, N);
    w.partial = reinterpret_cast<float*>(p);
    return w;
}

std::atomic<uint32_t> g_call_gen{0};

}  // namespace

size_t wcsr_spmm_ws_bytes(const spmm_wcsr_t* A, int64_t N) {
    return 256 + wcsr_ticket_bytes(A, N) + align256(sizeof(float) * static_cast<size_t>(A->n_units) * A->h * N);
}

namespace {

// L2 warm-up set shared by both kernels: the format arrays, and B when its rows
// are not much wider than N.
template <typename Args>
void warmup_set(Args& a, const spmm_wcsr_t* A, const void* B, int64_t ldb, int64_t N) {
    int n = 0;
    auto add = [&](const void* p, int64_t bytes) {
        if (p && bytes >= 16 && n < 10) {
            a.pf_ptr[n] = p;
            a.pf_bytes[n] = bytes;
            ++n;
        }
    };
    add(A->unit_win, 4 * A->n_units);
    add(A->unit_nz_ptr, 4 * (A->n_units + 1));
    add(A->unit_ptr, 4 * (A->n_windows + 1));
    add(A->wcol_ptr, 4 * (A->n_windows + 1));
    add(A->lrow, A->nnz);
    add(A->slot, 4 * A->nnz);
    add(A->val, 2 * A->nnz);
    add(A->wcols, 4 * A->n_wcols);
    if (ldb <= 2 * N && A->K * ldb * 2 <= (int64_t(64) << 20)) add(B, A->K * ldb * 2);
    a.pf_n = n;
}

uint32_t next_gen() {
    uint32_t gen = ++g_call_gen;
    if (gen == 0) gen = ++g_call_gen;
    return gen;
}

spmm_status launch_wcsr_tc(const DeviceInfo* dev, const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C,
                           int64_t ldc, int64_t N, void* ws, cudaStream_t s) {
    tc::Args a{};
    a.wcol_ptr = A->wcol_ptr;
    a.wcols = A->wcols;
    a.unit_ptr = A->unit_ptr;
    a.unit_win = A->unit_win;
    a.unit_nz_ptr = A->unit_nz_ptr;
    a.lrow = A->lrow;
    a.slot = A->slot;
    a.val = static_cast<const uint16_t*>(A->val);
    a.B = static_cast<const uint16_t*>(B);
    a.ldb = ldb;
    a.C = C;
    a.ldc = ldc;
    a.M = A->M;
    a.K = A->K;
    a.N = N;
    a.h = A->h;
    a.S = A->S;
    a.Np = (A->h + 15) / 16 * 16;
    a.nslabs = static_cast<int32_t>(wcsr_nslabs(N));
    a.n_windows = A->n_windows;
    a.n_units = A->n_units;
    a.n_items = A->n_units * a.nslabs;
    a.b_vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 8 == 0);
    a.idesc = ptx::idesc_f16(128, a.Np, A->dtype == SPMM_BF16, true, false, false);
    a.gen = next_gen();
    const SpmmWs w = carve_spmm(ws, A, N);
    a.ticket = w.ticket;
    a.partial = w.partial;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;
    warmup_set(a, A, B, ldb, N);
    // one CTA (four warpgroups) per SM, no more than there are items for
    const int64_t need = (a.n_items + tc::kWG - 1) / tc::kWG;
    const unsigned grid = static_cast<unsigned>(need < dev->sms ? need : dev->sms);
    const int smem = tc::smem_bytes();
    if (dev->max_smem_optin < smem) return SPMM_ERR_UNSUPPORTED;
    if (!set_smem_attr_once(reinterpret_cast<const void*>(tc::wcsr_tc_kernel), smem, 16)) return SPMM_ERR_CUDA;
    trace_begin(SPMM_KERNEL_WCSR, s);
    tc::wcsr_tc_kernel<<<grid, tc::kThreads, smem, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WCSR, s);
    return cuda_status(e);
}

spmm_status launch_wcsr_ts(const DeviceInfo* dev, const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C,
                           int64_t ldc, int64_t N, void* ws, cudaStream_t s) {
    tc::Args a{};
    a.wcol_ptr = A->wcol_ptr;
    a.wcols = A->wcols;
    a.unit_ptr = A->unit_ptr;
    a.unit_win = A->unit_win;
    a.unit_nz_ptr = A->unit_nz_ptr;
    a.lrow = A->lrow;
    a.slot = A->slot;
    a.val = static_cast<const uint16_t*>(A->val);
    a.B = static_cast<const uint16_t*>(B);
    a.ldb = ldb;
    a.C = C;
    a.ldc = ldc;
    a.M = A->M;
    a.K = A->K;
    a.N = N;
    a.h = A->h;
    a.S = A->S;
    a.Np = ts::kNp;
    a.nslabs = static_cast<int32_t>(wcsr_nslabs(N));
    a.n_windows = A->n_windows;
    a.n_units = A->n_units;
    a.n_items = A->n_units * a.nslabs;
    a.b_vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 8 == 0);
    a.idesc = ptx::idesc_f16(128, ts::kNp, A->dtype == SPMM_BF16, true, false, false);
    a.gen = next_gen();
    const SpmmWs w = carve_spmm(ws, A, N);
    a.ticket = w.ticket;
    a.partial = w.partial;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;
    warmup_set(a, A, B, ldb, N);
    const unsigned grid = static_cast<unsigned>(a.n_items < dev->sms ? a.n_items : dev->sms);
    const int smem = static_cast<int>(ts::kSmem);
    if (dev->max_smem_optin < smem) return SPMM_ERR_UNSUPPORTED;
    if (!set_smem_attr_once(reinterpret_cast<const void*>(ts::wcsr_ts_kernel), smem, 21)) return SPMM_ERR_CUDA;
    trace_begin(SPMM_KERNEL_WCSR, s);
    ts::wcsr_ts_kernel<<<grid, ts::kThreads, smem, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WCSR, s);
    return cuda_status(e);
}

spmm_status launch_wcsr_cc(const DeviceInfo* dev, const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C,
                           int64_t ldc, int64_t N, void* ws, cudaStream_t s) {
    cc::WcsrArgs a{};
    a.wcol_ptr = A->wcol_ptr;
    a.wcols = A->wcols;
    a.unit_ptr = A->unit_ptr;
    a.unit_win = A->unit_win;
    a.unit_nz_ptr = A->unit_nz_ptr;
    a.lrow = A->lrow;
    a.slot = A->slot;
    a.val = A->val;
    a.B = B;
    a.ldb = ldb;
    a.C = C;
    a.ldc = ldc;
    a.M = A->M;
    a.K = A->K;
    a.N = N;
    a.h = A->h;
    const SpmmWs w = carve_spmm(ws, A, N);
    a.ticket = w.ticket;
    a.partial = w.partial;
    a.nslabs = static_cast<int32_t>(wcsr_nslabs(N));
    a.gen = next_gen();
    a.err = dev->err;
    warmup_set(a, A, B, ldb, N);
    const int64_t wave = static_cast<int64_t>(dev->sms) * cc::kMinBlocks;
    a.pf_ctas = static_cast<int32_t>(A->n_units < wave ? A->n_units : wave);
    a.b_vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 8 == 0) && (A->K * ldb < (int64_t(1) << 31));
    a.c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0) && (N % 4 == 0);
    auto smem_for = [](int h) {
        return static_cast<int>(sizeof(float) * (h * cc::kSlab + cc::kBnd * cc::kSlab) + sizeof(int2) * cc::kStage +
                                sizeof(int) * cc::kBnd);
    };
    const int smem = smem_for(A->h), smem_max = smem_for(kMaxH);
    const void* kern = A->dtype == SPMM_BF16 ? reinterpret_cast<const void*>(cc::wcsr_spmm_kernel<__nv_bfloat16>)
                                             : reinterpret_cast<const void*>(cc::wcsr_spmm_kernel<__half>);
    if (!set_smem_attr_once(kern, smem_max, A->dtype == SPMM_BF16 ? 4 : 5)) return SPMM_ERR_CUDA;
    trace_begin(SPMM_KERNEL_WCSR, s);
    if (A->dtype == SPMM_BF16)
        cc::wcsr_spmm_kernel<__nv_bfloat16><<<static_cast<unsigned>(A->n_units), cc::kThreads, smem, s>>>(a);
    else
        cc::wcsr_spmm_kernel<__half><<<static_cast<unsigned>(A->n_units), cc::kThreads, smem, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WCSR, s);
    return cuda_status(e);
}

}  // namespace

// When the window products run on the tensor core.  That kernel gathers each
// B row once per window column, so it needs column reuse (several nonzeros per
// distinct window column) to gather fewer rows than the CUDA-core kernel, which
// gathers one per nonzero; and its time per work unit is dominated by a fixed
// chain of dependent loads, so units must carry enough nonzeros to amortise
// it.  Measured on GB300 (65536 x 65536, 128 columns of B): with 4 to 16
// nonzeros per window column but 256 per unit the CUDA-core kernel is 5-13%
// faster; with 8 to 16 per column and 512 to 1024 per unit the tensor core is
// 1.26-1.66x faster; with ~1 per column it is 2.4x slower.
constexpr double kTensorCoreReuse = 4.0;      // nonzeros per distinct window column
constexpr double kTensorCoreUnitNnz = 384.0;  // nonzeros per work unit

spmm_status launch_wcsr(const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        void* ws, cudaStream_t s) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    if (!wcsr_uses_tensor_core(A)) return launch_wcsr_cc(dev, A, B, ldb, C, ldc, N, ws, s);
    // windows of at most 16 rows and at most 32 steps per unit: the streaming kernel
    // (clustered windows, 65536 x 65536, N = 128: 62 us against 66); B rows start on
    // 16-byte boundaries (checked by the entry point), as its 16-byte copies need
    if (A->h <= ts::kNp && A->S <= ts::kMaxSteps) return launch_wcsr_ts(dev, A, B, ldb, C, ldc, N, ws, s);
    return launch_wcsr_tc(dev, A, B, ldb, C, ldc, N, ws, s);
}

bool wcsr_uses_tensor_core(const spmm_wcsr_t* A) {
    const double nnz = static_cast<double>(A->nnz);
    return A->n_wcols > 0 && A->n_units > 0 && nnz >= kTensorCoreReuse * static_cast<double>(A->n_wcols) &&
           nnz >= kTensorCoreUnitNnz * static_cast<double>(A->n_units);
}

int wcsr_max_h() { return kMaxH; }

}  // namespace spmm
