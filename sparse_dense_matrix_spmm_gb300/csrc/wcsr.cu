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
// SpMM.  On the synthetic power-law workload the windows are about 6% dense
// (uniform columns), so the contraction per window is not a dense tile: the
// kernel runs on CUDA cores and is bound by gathering B rows (N * 2 bytes per
// nonzero) from L2, which is latency-bound: throughput is the bytes in flight
// per SM over the L2 round trip, so occupancy decides it.  One CTA (4 warps,
// 8 CTAs per SM) per work unit.  The CTA first stages the
// unit's sparse operand in shared memory (local row, column resolved through
// the window's column list, value), then cuts it into equal chunks, one per
// warp.  Each warp keeps 16 B-row loads in flight, accumulates fp32 per row in
// registers (lane = 4 columns of a 128-column slab), writes rows that lie inside its
// chunk straight into a shared-memory tile, and hands the two rows at its
// chunk's ends to a fix-up that adds them in warp order, so every sum has a
// fixed order.  Unsplit windows write C from the tile; a split window's units
// write partial tiles to the workspace, and the last unit to finish (ticket
// counter) sums them in unit order and resets the counter.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"

namespace spmm {

__device__ int g_wcsr_build_error;  // data-dependent builder errors (SPMM_DEVERR_FORMAT)

namespace {

constexpr int kWarps = 4;   // 8 CTAs per SM: one CTA's staging overlaps the others' gathers
constexpr int kThreads = kWarps * 32;
constexpr int kSlab = 128;  // output columns per pass (4 per lane)
static_assert(kThreads >= kSlab, "the boundary fix-up gives one thread to each slab column");
constexpr int kMaxH = 64;   // largest window height the SpMM kernel accepts

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

// ---------------------------------------------------------------- SpMM
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
    float* partial;   // [n_units][h][N]
    int32_t* ticket;  // [n_windows]
    int* err;
};

template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// value bits (low half of a packed word) -> fp32
template <typename T>
__device__ __forceinline__ float low_to_f(uint32_t pk);
template <>
__device__ __forceinline__ float low_to_f<__half>(uint32_t pk) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(pk & 0xFFFFu)));
}
template <>
__device__ __forceinline__ float low_to_f<__nv_bfloat16>(uint32_t pk) {
    return __uint_as_float(pk << 16);
}

constexpr int kStage = 1024;  // nonzeros whose operand is staged in shared memory at once
constexpr int kBatch = 16;    // B-row loads in flight per warp
constexpr int kPad = kWarps * kBatch;

// One warp's chunk of staged entries [j_lo, j_hi) (a multiple of kBatch long):
// gather B rows, accumulate per row, store finished rows in the tile and the
// chunk's end rows in the fix-up slots.
template <typename T, bool FULL>
__device__ __forceinline__ void wcsr_chunk(const T* B, int64_t ldb, int64_t ncol, int valid, const int* s_col,
                                           const uint32_t* s_pk, int j_lo, int j_hi, float* tile, float* bnd,
                                           int* bnd_row, int warp, int lane) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int cur = -1;
    bool first_seg = true;
    for (int j0 = j_lo; j0 < j_hi; j0 += kBatch) {
        uint2 raw[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const T* p = B + static_cast<int64_t>(s_col[j0 + b]) * ldb + ncol;
            if (FULL) {
                raw[b] = __ldg(reinterpret_cast<const uint2*>(p));
            } else {
                const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
                const uint32_t e0 = valid > 0 ? q[0] : 0u, e1 = valid > 1 ? q[1] : 0u;
                const uint32_t e2 = valid > 2 ? q[2] : 0u, e3 = valid > 3 ? q[3] : 0u;
                raw[b] = make_uint2(e0 | (e1 << 16), e2 | (e3 << 16));
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const uint32_t pk = s_pk[j0 + b];
            const int rr = static_cast<int>(pk >> 16);
            if (rr != cur) {
                if (cur >= 0) {
                    // a finished segment: the chunk's first row goes to the fix-up,
                    // any later one lies wholly inside this chunk
                    float* dst = first_seg ? bnd + (warp * 2) * kSlab : tile + cur * kSlab;
                    *reinterpret_cast<float4*>(dst + 4 * lane) = acc;
                    if (first_seg && lane == 0) bnd_row[warp * 2] = cur;
                    first_seg = false;
                }
                cur = rr;
                acc = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const float v = low_to_f<T>(pk);
            const float2 lo = unpack2<T>(raw[b].x), hi = unpack2<T>(raw[b].y);
            acc.x += v * lo.x;
            acc.y += v * lo.y;
            acc.z += v * hi.x;
            acc.w += v * hi.y;
        }
    }
    if (cur >= 0) {
        // the chunk's last segment may continue in the next chunk
        const int k = first_seg ? 0 : 1;
        *reinterpret_cast<float4*>(bnd + (warp * 2 + k) * kSlab + 4 * lane) = acc;
        if (lane == 0) bnd_row[warp * 2 + k] = cur;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 8) wcsr_spmm_kernel(const WcsrArgs a) {
    extern __shared__ float sm[];
    // tile[h][kSlab] | bnd[2*kWarps][kSlab] | bnd_row[2*kWarps] | s_col[kStage+kPad] | s_pk[kStage+kPad]
    float* tile = sm;
    float* bnd = tile + a.h * kSlab;
    int* bnd_row = reinterpret_cast<int*>(bnd + 2 * kWarps * kSlab);
    int* s_col = bnd_row + 2 * kWarps;
    uint32_t* s_pk = reinterpret_cast<uint32_t*>(s_col + kStage + kPad);
    __shared__ int s_last;

    const int u = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = a.unit_win[u];
    if (w < 0 || static_cast<int64_t>(w) * a.h >= a.M) {  // malformed unit list: skip the unit
        if (threadIdx.x == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);
        return;
    }
    const int64_t r0 = static_cast<int64_t>(w) * a.h;
    const int64_t rem = a.M - r0;
    const int nrows = rem < a.h ? static_cast<int>(rem) : a.h;
    const int units_in_window = a.unit_ptr[w + 1] - a.unit_ptr[w];
    const bool split = units_in_window > 1;
    const int32_t wbase = a.wcol_ptr[w], T_w = a.wcol_ptr[w + 1] - wbase;
    const int32_t nz0 = a.unit_nz_ptr[u], nz1 = a.unit_nz_ptr[u + 1];
    const uint16_t* val = static_cast<const uint16_t*>(a.val);
    const T* B = static_cast<const T*>(a.B);

    for (int64_t n0 = 0; n0 < a.N; n0 += kSlab) {
        const int64_t ncol = n0 + 4 * lane;
        const int64_t left = a.N - ncol;
        const int valid = left >= 4 ? 4 : (left > 0 ? static_cast<int>(left) : 0);
        const bool full = n0 + kSlab <= a.N;
        for (int i = threadIdx.x; i < a.h * kSlab; i += kThreads) tile[i] = 0.f;

        for (int32_t st0 = nz0; st0 < nz1; st0 += kStage) {
            const int n_st = (nz1 - st0 < kStage) ? nz1 - st0 : kStage;
            const int per = ((n_st + kWarps - 1) / kWarps + kBatch - 1) / kBatch * kBatch;
            // stage the sparse operand: resolved column, packed (local row, value);
            // invalid entries become value 0 on row 0, column 0
            for (int i = threadIdx.x; i < n_st; i += kThreads) {
                const int32_t e = st0 + i;
                const int lr = a.lrow[e];
                const int32_t sl = a.slot[e];
                const int32_t c = (sl >= 0 && sl < T_w) ? a.wcols[wbase + sl] : -1;
                const bool ok = lr < nrows && c >= 0 && c < a.K;
                if (!ok) atomicOr(a.err, SPMM_DEVERR_INDEX);
                s_col[i] = ok ? c : 0;
                s_pk[i] = ok ? ((static_cast<uint32_t>(lr) << 16) | val[e]) : 0u;
            }
            __syncthreads();
            // pad every chunk to whole batches: value-0 copies of the last entry
            for (int i = n_st + threadIdx.x; i < kWarps * per; i += kThreads) {
                s_col[i] = s_col[n_st - 1];
                s_pk[i] = s_pk[n_st - 1] & 0xFFFF0000u;
            }
            if (threadIdx.x < 2 * kWarps) bnd_row[threadIdx.x] = -1;
            __syncthreads();

            const int j_lo = warp * per, j_hi = j_lo + per;
            if (full)
                wcsr_chunk<T, true>(B, a.ldb, ncol, valid, s_col, s_pk, j_lo, j_hi, tile, bnd, bnd_row, warp, lane);
            else
                wcsr_chunk<T, false>(B, a.ldb, ncol, valid, s_col, s_pk, j_lo, j_hi, tile, bnd, bnd_row, warp, lane);
            __syncthreads();
            // chunk-boundary rows, added in warp order: thread t owns column t of the slab
            if (threadIdx.x < kSlab) {
                for (int k = 0; k < 2 * kWarps; ++k) {
                    const int r = bnd_row[k];
                    if (r >= 0) tile[r * kSlab + threadIdx.x] += bnd[k * kSlab + threadIdx.x];
                }
            }
            __syncthreads();
        }

        if (!split) {
            for (int i = threadIdx.x; i < nrows * (kSlab / 4); i += kThreads) {
                const int r = i / (kSlab / 4), q = i % (kSlab / 4);
                const int64_t col = n0 + 4 * q;
                const float4 v = *reinterpret_cast<const float4*>(tile + r * kSlab + 4 * q);
                float* cp = a.C + (r0 + r) * a.ldc + col;
                if (col + 4 <= a.N && (reinterpret_cast<uintptr_t>(cp) & 15) == 0) {
                    __stcs(reinterpret_cast<float4*>(cp), v);
                } else {
                    const float e[4] = {v.x, v.y, v.z, v.w};
                    for (int t = 0; t < 4 && col + t < a.N; ++t) cp[t] = e[t];
                }
            }
        } else {
            float* part = a.partial + static_cast<int64_t>(u) * a.h * a.N;
            for (int i = threadIdx.x; i < nrows * kSlab; i += kThreads) {
                const int r = i / kSlab, q = i % kSlab;
                if (n0 + q < a.N) __stcg(part + static_cast<int64_t>(r) * a.N + n0 + q, tile[i]);
            }
        }
        __syncthreads();
    }

    if (!split) return;
    // last unit of the window to finish sums the partials in unit order
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int t = atomicAdd(a.ticket + w, 1);
        s_last = (t == units_in_window - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int u0 = a.unit_ptr[w];
    for (int64_t i = threadIdx.x; i < static_cast<int64_t>(nrows) * a.N; i += kThreads) {
        const int64_t r = i / a.N, c = i % a.N;
        float s = 0.f;
        for (int k = 0; k < units_in_window; ++k)
            s += __ldcg(a.partial + (static_cast<int64_t>(u0 + k) * a.h + r) * a.N + c);
        a.C[(r0 + r) * a.ldc + c] = s;
    }
    if (threadIdx.x == 0) a.ticket[w] = 0;  // ready for the next call
}

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

size_t wcsr_spmm_ws_bytes(const spmm_wcsr_t* A, int64_t N) {
    return align256(sizeof(int32_t) * static_cast<size_t>(A->n_windows)) +
           align256(sizeof(float) * static_cast<size_t>(A->n_units) * A->h * N);
}

spmm_status launch_wcsr(const spmm_wcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        void* ws, cudaStream_t s) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    WcsrArgs a{};
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
    a.ticket = static_cast<int32_t*>(ws);
    a.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                         align256(sizeof(int32_t) * static_cast<size_t>(A->n_windows)));
    a.err = dev->err;
    const int smem = static_cast<int>(sizeof(float) * (A->h * kSlab + kWarps * 2 * kSlab) + sizeof(int) * kWarps * 2 +
                                      (kStage + kPad) * (sizeof(int) + sizeof(uint32_t)));
    const int smem_max = static_cast<int>(sizeof(float) * (kMaxH * kSlab + kWarps * 2 * kSlab) +
                                          sizeof(int) * kWarps * 2 + (kStage + kPad) * (sizeof(int) + sizeof(uint32_t)));
    const void* kern = A->dtype == SPMM_BF16 ? reinterpret_cast<const void*>(wcsr_spmm_kernel<__nv_bfloat16>)
                                             : reinterpret_cast<const void*>(wcsr_spmm_kernel<__half>);
    if (!set_smem_attr_once(kern, smem_max, A->dtype == SPMM_BF16 ? 4 : 5)) return SPMM_ERR_CUDA;
    trace_begin(SPMM_KERNEL_WCSR, s);
    if (A->dtype == SPMM_BF16)
        wcsr_spmm_kernel<__nv_bfloat16><<<static_cast<unsigned>(A->n_units), kThreads, smem, s>>>(a);
    else
        wcsr_spmm_kernel<__half><<<static_cast<unsigned>(A->n_units), kThreads, smem, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WCSR, s);
    return cuda_status(e);
}

int wcsr_max_h() { return kMaxH; }

}  // namespace spmm
