// builders.cu -- GPU format builders: dense -> BCSR, dense -> 2:4, dense -> TVW,
// (2n-2):2n -> lifted 2:4 windows.
//
// Every builder is bit-exact with respect to its format definition: stored
// values are copied bit for bit, and the order of stored items comes from
// prefix sums (never from atomics), so the output does not depend on thread
// scheduling.  A stored element is "zero" iff it compares equal to zero
// (16-bit types: (bits & 0x7FFF) == 0, so -0.0 is zero and NaN is not).
#include <mutex>

#include "internal.h"

namespace spmm {

__device__ int g_build_error;  // data-dependent builder errors (SPMM_DEVERR_FORMAT)

namespace {

std::mutex g_build_mu;  // builders share g_build_error: one at a time per process

template <typename T>
__device__ __forceinline__ bool nz(T v);
template <>
__device__ __forceinline__ bool nz<uint16_t>(uint16_t v) { return (v & 0x7FFFu) != 0; }
template <>
__device__ __forceinline__ bool nz<int8_t>(int8_t v) { return v != 0; }
// fp8 (E4M3 / E5M2) bit patterns: zero iff every bit but the sign is 0
template <>
__device__ __forceinline__ bool nz<uint8_t>(uint8_t v) { return (v & 0x7Fu) != 0; }

// ---------------------------------------------------------------- scan
// In-place exclusive prefix sum of a[0..n) with one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(int32_t* a, int64_t n) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += 1024) {
        const int64_t i = base + tid;
        int32_t v = i < n ? a[i] : 0;
        int32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t s = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, s, o);
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

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* total, int32_t* sh /* >= 33 ints */) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = (blockDim.x + 31) >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t s = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh[lane] = s;
    }
    __syncthreads();
    const int32_t r = (wid ? sh[wid - 1] : 0) + x - v;
    if (total) *total = sh[nw - 1];
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------- BCSR
// One CTA per block row; flags[bc] = 1 iff block (br, bc) holds a nonzero.
template <typename T>
__device__ void bcsr_flags(const T* dense, int64_t ld, int br, int bh, int gk, int bw, uint8_t* flags) {
    for (int bc = threadIdx.x; bc < gk; bc += blockDim.x) flags[bc] = 0;
    __syncthreads();
    const int64_t K = static_cast<int64_t>(gk) * bw;
    const int64_t total = static_cast<int64_t>(bh) * K;
    const T* base = dense + static_cast<int64_t>(br) * bh * ld;
    for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
        const int64_t r = e / K, c = e % K;
        if (nz<T>(base[r * ld + c])) flags[c / bw] = 1;  // benign same-value race
    }
    __syncthreads();
}

// Any element of a 16-byte piece nonzero (the rule of nz, per element).
template <typename T>
__device__ __forceinline__ bool nz16(const uint4& v);
template <>
__device__ __forceinline__ bool nz16<uint16_t>(const uint4& v) { return ((v.x | v.y | v.z | v.w) & 0x7FFF7FFFu) != 0u; }
template <>
__device__ __forceinline__ bool nz16<int8_t>(const uint4& v) { return (v.x | v.y | v.z | v.w) != 0u; }

// The same flags from 16-byte pieces (VEC: rows and block columns 16-byte
// aligned, bh * K / 8 < 2^31): consecutive threads read consecutive pieces of
// a row, four loads in flight per thread, and a piece's block column comes
// from 32-bit arithmetic.
template <typename T>
__device__ void bcsr_flags_vec(const T* dense, int64_t ld, int br, int bh, int gk, int bw, uint8_t* flags) {
    for (int bc = threadIdx.x; bc < gk; bc += blockDim.x) flags[bc] = 0;
    __syncthreads();
    constexpr int E = 16 / static_cast<int>(sizeof(T));
    const int ppr = gk * (bw / E), ppb = bw / E;  // pieces per row, per block column
    const int total = bh * ppr;
    const T* base = dense + static_cast<int64_t>(br) * bh * ld;
#pragma unroll 4
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / ppr, pc = i - r * ppr;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<int64_t>(r) * ld) + pc);
        if (nz16<T>(v)) flags[pc / ppb] = 1;  // benign same-value race
    }
    __syncthreads();
}

template <typename T, bool VEC>
__global__ void bcsr_count_kernel(const T* dense, int64_t ld, int bh, int bw, int gk, int32_t* row_ptr) {
    extern __shared__ uint8_t flags[];
    __shared__ int32_t sh[33];
    const int br = blockIdx.x;
    if constexpr (VEC)
        bcsr_flags_vec<T>(dense, ld, br, bh, gk, bw, flags);
    else
        bcsr_flags<T>(dense, ld, br, bh, gk, bw, flags);
    int32_t cnt = 0;
    for (int bc = threadIdx.x; bc < gk; bc += blockDim.x) cnt += flags[bc];
    int32_t total = 0;
    block_exclusive_scan(cnt, &total, sh);
    if (threadIdx.x == 0) row_ptr[br] = total;
}

template <typename T, bool VEC>
__global__ void bcsr_fill_kernel(const T* dense, int64_t ld, int bh, int bw, int gk, const int32_t* row_ptr,
                                 int32_t* col_idx, T* vals) {
    extern __shared__ uint8_t smem[];
    uint8_t* flags = smem;
    int32_t* pos = reinterpret_cast<int32_t*>(smem + ((gk + 15) & ~15));
    __shared__ int32_t sh[33];
    const int br = blockIdx.x;
    if constexpr (VEC)
        bcsr_flags_vec<T>(dense, ld, br, bh, gk, bw, flags);
    else
        bcsr_flags<T>(dense, ld, br, bh, gk, bw, flags);
    // positions of the stored blocks inside this block row, in ascending bc
    const int per = (gk + blockDim.x - 1) / blockDim.x;
    const int b0 = min(gk, static_cast<int>(threadIdx.x) * per), b1 = min(gk, b0 + per);
    int32_t cnt = 0;
    for (int bc = b0; bc < b1; ++bc) cnt += flags[bc];
    int32_t run = block_exclusive_scan(cnt, nullptr, sh);
    for (int bc = b0; bc < b1; ++bc) {
        pos[bc] = run;
        run += flags[bc];
    }
    __syncthreads();
    const int64_t first = row_ptr[br];
    for (int bc = threadIdx.x; bc < gk; bc += blockDim.x)
        if (flags[bc]) col_idx[first + pos[bc]] = bc;
    const int64_t blk = static_cast<int64_t>(bh) * bw;
    const int64_t K = static_cast<int64_t>(gk) * bw;
    const T* base = dense + static_cast<int64_t>(br) * bh * ld;
    if constexpr (VEC) {
        // the stored blocks' 16-byte pieces, in the same order as the flag pass
        constexpr int E = 16 / static_cast<int>(sizeof(T));
        const int ppr = gk * (bw / E), ppb = bw / E;
        const int total = bh * ppr;
#pragma unroll 4
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int r = i / ppr, pc = i - r * ppr, bc = pc / ppb;
            if (!flags[bc]) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<int64_t>(r) * ld) + pc);
            *reinterpret_cast<uint4*>(vals + (first + pos[bc]) * blk + static_cast<int64_t>(r) * bw + (pc - bc * ppb) * E) = v;
        }
    } else {
        for (int64_t e = threadIdx.x; e < static_cast<int64_t>(bh) * K; e += blockDim.x) {
            const int64_t r = e / K, c = e % K;
            const int bc = static_cast<int>(c / bw);
            if (!flags[bc]) continue;
            vals[(first + pos[bc]) * blk + r * bw + (c % bw)] = base[r * ld + c];
        }
    }
}

// One CTA per block row; 1024 threads keep enough 16-byte loads in flight when
// a matrix has only a few hundred block rows.
constexpr int kBcsrBuildThreads = 1024;

// 16-byte pieces for the BCSR builders: aligned base and row pitch, block
// columns a whole number of pieces, piece indices of a block row in 32 bits.
bool bcsr_vec(const void* dense, int64_t ld, int64_t K, int bh, int bw, int es, const void* vals) {
    return reinterpret_cast<uintptr_t>(dense) % 16 == 0 && (ld * es) % 16 == 0 && (bw * es) % 16 == 0 &&
           (vals == nullptr || reinterpret_cast<uintptr_t>(vals) % 16 == 0) &&
           static_cast<int64_t>(bh) * K * es / 16 < (int64_t(1) << 31);
}

// ---------------------------------------------------------------- 2:4
// Eight consecutive elements (two 4-groups) as one 16-byte (16-bit types) or
// 8-byte (int8) access when `vec` (base and pitch aligned), else element-wise;
// four stored values likewise as one 8- or 4-byte store.
template <typename T>
__device__ __forceinline__ void load8(const T* src, bool vec, T (&v)[8]) {
    if (vec) {
        if constexpr (sizeof(T) == 2) {
            const uint4 w = *reinterpret_cast<const uint4*>(src);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = static_cast<T>(u[i] & 0xFFFFu);
                v[2 * i + 1] = static_cast<T>(u[i] >> 16);
            }
        } else {
            const uint2 w = *reinterpret_cast<const uint2*>(src);
            const uint32_t u[2] = {w.x, w.y};
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = static_cast<T>((u[i / 4] >> (8 * (i % 4))) & 0xFFu);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = src[i];
    }
}
template <typename T>
__device__ __forceinline__ void store4(T* dst, bool vec, const T (&v)[4]) {
    if (vec) {
        if constexpr (sizeof(T) == 2) {
            const uint32_t lo = static_cast<uint16_t>(v[0]) | (static_cast<uint32_t>(static_cast<uint16_t>(v[1])) << 16);
            const uint32_t hi = static_cast<uint16_t>(v[2]) | (static_cast<uint32_t>(static_cast<uint16_t>(v[3])) << 16);
            *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
        } else {
            uint32_t w = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) w |= static_cast<uint32_t>(static_cast<uint8_t>(v[i])) << (8 * i);
            *reinterpret_cast<uint32_t*>(dst) = w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = v[i];
    }
}

// Keep the nonzero positions of a 4-group, padded with the lowest-index zero
// positions; nibble = idx0 | idx1 << 2.  Returns false on > 2 nonzeros.
__device__ __forceinline__ bool pick2(unsigned mask, int& i0, int& i1) {
    if (__popc(mask) > 2) return false;
    unsigned keep = mask;
    for (int p = 0; p < 4 && __popc(keep) < 2; ++p) keep |= 1u << p;  // lowest zero positions
    i0 = __ffs(keep) - 1;
    i1 = __ffs(keep & ~(1u << i0)) - 1;
    return true;
}

// One thread per (row, meta byte) = 2 groups = 8 dense columns.
template <typename T>
__global__ void compress24_kernel(const T* __restrict__ dense, int64_t M, int64_t K, int64_t ld,
                                  T* __restrict__ vals, uint8_t* __restrict__ meta, int vec, int* err) {
    // grid: x over the row's meta bytes, y over rows (strided when M exceeds the grid)
    const int64_t nb = K / 8;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= nb) return;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        T x[8], out[4];
        load8<T>(dense + i * ld + 8 * j, vec != 0, x);
        uint8_t byte = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            unsigned mask = 0;
#pragma unroll
            for (int p = 0; p < 4; ++p)
                if (nz<T>(x[4 * h + p])) mask |= 1u << p;
            int i0 = 0, i1 = 1;
            if (!pick2(mask, i0, i1)) {
                atomicOr(err, SPMM_DEVERR_FORMAT);
                i0 = 0;
                i1 = 1;
            }
            out[2 * h] = x[4 * h + i0];
            out[2 * h + 1] = x[4 * h + i1];
            byte |= static_cast<uint8_t>((i0 | (i1 << 2)) << (4 * h));
        }
        store4<T>(vals + i * (K / 2) + 4 * j, vec != 0, out);
        meta[i * nb + j] = byte;
    }
}

// Magnitude pruning into 2:4 ("Accelerating Sparse DNNs Based on Tiled GEMM",
// abstract: pruning into the sparse tensor core's 2:4 pattern): per 4-group the
// two entries of largest magnitude, ties to the lower index, stored in
// ascending index order.  The magnitude key is |v| for int8 and the bits
// without the sign for bf16/fp16 (orders |a|; NaN above every number).
template <typename T>
__device__ __forceinline__ unsigned mag_key(T v);
template <>
__device__ __forceinline__ unsigned mag_key<int8_t>(int8_t v) {
    return static_cast<unsigned>(v < 0 ? -static_cast<int>(v) : static_cast<int>(v));
}
template <>
__device__ __forceinline__ unsigned mag_key<uint16_t>(uint16_t v) {
    return v & 0x7FFFu;
}
template <>
__device__ __forceinline__ unsigned mag_key<uint8_t>(uint8_t v) {  // fp8: bits without the sign
    return v & 0x7Fu;
}

// The two positions of largest key (lowest index among equals), ascending.
__device__ __forceinline__ void top2(const unsigned (&key)[4], int& i0, int& i1) {
    int first = 0;
#pragma unroll
    for (int p = 1; p < 4; ++p)
        if (key[p] > key[first]) first = p;
    int second = first == 0 ? 1 : 0;
#pragma unroll
    for (int p = 0; p < 4; ++p)
        if (p != first && p > second && key[p] > key[second]) second = p;
    i0 = min(first, second);
    i1 = max(first, second);
}

// One thread per (row, meta byte) = 2 groups = 8 dense columns.
template <typename T>
__global__ void prune24_kernel(const T* __restrict__ dense, int64_t M, int64_t K, int64_t ld, T* __restrict__ vals,
                               uint8_t* __restrict__ meta, int vec) {
    // grid: x over the row's meta bytes, y over rows (strided when M exceeds the grid)
    const int64_t nb = K / 8;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= nb) return;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        T x[8], out[4];
        load8<T>(dense + i * ld + 8 * j, vec != 0, x);
        uint8_t byte = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            unsigned key[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) key[p] = mag_key<T>(x[4 * h + p]);
            int i0, i1;
            top2(key, i0, i1);
            out[2 * h] = x[4 * h + i0];
            out[2 * h + 1] = x[4 * h + i1];
            byte |= static_cast<uint8_t>((i0 | (i1 << 2)) << (4 * h));
        }
        store4<T>(vals + i * (K / 2) + 4 * j, vec != 0, out);
        meta[i * nb + j] = byte;
    }
}

// ---------------------------------------------------------------- (2n-2):2n
// Four consecutive elements as one 8-byte (16-bit types) or 4-byte (int8) load
// when `vec`, else element-wise.
template <typename T>
__device__ __forceinline__ void load4(const T* src, bool vec, T* v) {
    if (vec) {
        if constexpr (sizeof(T) == 2) {
            const uint2 w = *reinterpret_cast<const uint2*>(src);
            v[0] = static_cast<T>(w.x & 0xFFFFu);
            v[1] = static_cast<T>(w.x >> 16);
            v[2] = static_cast<T>(w.y & 0xFFFFu);
            v[3] = static_cast<T>(w.y >> 16);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = static_cast<T>((w >> (8 * i)) & 0xFFu);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = src[i];
    }
}

// y[i] for a runtime i < 4 by selects, keeping y in registers.
template <typename T>
__device__ __forceinline__ T sel4(const T* y, int i) {
    T r = y[0];
    r = i == 1 ? y[1] : r;
    r = i == 2 ? y[2] : r;
    r = i == 3 ? y[3] : r;
    return r;
}

// (2n-2):2n -> n-1 overlapping 2:4 windows per group ("SlideSparse", abstract:
// sliding window decomposition).  Window j of group g covers the group's
// positions 2j .. 2j+3 and is stored as 2:4 group j G + g of the lifted row
// (window planes: every group's window 0, then every group's window 1, ...).
// Windows are filled in order j = 0, 1, ...: first the nonzeros of pair j that
// window j-1 left, then those of pair j+1 while the window holds fewer than
// two; this places every nonzero of a group with at most 2n-2 of them.  A
// window's stored pair is its nonzero positions padded with its lowest other
// positions (value +0).  One thread per (row, two groups): groups 2q and 2q+1
// share metadata byte (j G) / 2 + q of every plane j, so each thread writes
// whole bytes.  `vec`: bit 0 = vector loads, bit 1 = vector stores.
template <typename T, int NN>
__global__ void slide_build_kernel(const T* __restrict__ dense, int64_t M, int64_t G, int64_t ld,
                                   T* __restrict__ vals, uint8_t* __restrict__ meta, int vec, int* err) {
    constexpr int W = NN - 1;  // windows per group
    const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (q >= G / 2) return;
    const int64_t lv = 2 * W * G;  // stored values per row: K' / 2
    const int64_t lm = W * G / 2;  // metadata bytes per row: K' / 8
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        T x[4 * NN];
#pragma unroll
        for (int c = 0; c < NN; ++c) load4<T>(dense + i * ld + 4 * NN * q + 4 * c, (vec & 1) != 0, x + 4 * c);
        uint8_t byte[W];
        T out[W][4];
#pragma unroll
        for (int j = 0; j < W; ++j) byte[j] = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const T* y = x + 2 * NN * h;
            unsigned mask = 0;
#pragma unroll
            for (int p = 0; p < 2 * NN; ++p)
                if (nz<T>(y[p])) mask |= 1u << p;
            unsigned placed = 0;
#pragma unroll
            for (int j = 0; j < W; ++j) {
                unsigned keep = 0;
                int held = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int pos = 2 * j + t;
                    if ((((mask & ~placed) >> pos) & 1u) && held < 2) {
                        placed |= 1u << pos;
                        keep |= 1u << t;
                        ++held;
                    }
                }
                int i0 = 0, i1 = 1;
                pick2(keep, i0, i1);  // keep holds at most two positions
                out[j][2 * h] = ((keep >> i0) & 1u) ? sel4<T>(y + 2 * j, i0) : T(0);
                out[j][2 * h + 1] = ((keep >> i1) & 1u) ? sel4<T>(y + 2 * j, i1) : T(0);
                byte[j] |= static_cast<uint8_t>((i0 | (i1 << 2)) << (4 * h));
            }
            if (__popc(mask) > 2 * NN - 2 || (mask & ~placed) != 0) atomicOr(err, SPMM_DEVERR_FORMAT);
        }
#pragma unroll
        for (int j = 0; j < W; ++j) {
            store4<T>(vals + i * lv + 2 * (j * G + 2 * q), (vec & 2) != 0, out[j]);
            meta[i * lm + (j * G) / 2 + q] = byte[j];
        }
    }
}

// ---------------------------------------------------------------- TVW
// Kept columns of every tile must be ascending and inside [0, K).
__global__ void tvw_check_cols_kernel(const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles, int64_t K,
                                      int* err) {
    const int64_t t = blockIdx.x;
    if (t >= n_tiles) return;
    const int32_t b = tile_ptr[t], e = tile_ptr[t + 1];
    for (int32_t q = b + threadIdx.x; q < e; q += blockDim.x) {
        const int32_t c = cols[q];
        if (c < 0 || c >= K || (q > b && cols[q - 1] >= c)) atomicOr(err, SPMM_DEVERR_FORMAT);
    }
}

// One CTA per row.  Every nonzero of the row must sit in a kept column; then
// each group of 4 kept columns is compressed to 2:4.
// PRUNE (magnitude pruning into TVW): entries outside the kept columns are
// dropped instead of rejected, and each group of 4 kept columns keeps its two
// largest magnitudes instead of requiring at most two nonzeros.
template <typename T, bool PRUNE>
__global__ void tvw_build_kernel(const T* dense, int64_t M, int64_t K, int64_t ld, int tile_rows,
                                 const int32_t* tile_ptr, const int32_t* cols, int64_t Kp, T* vals, uint8_t* meta,
                                 int* err) {
    __shared__ int32_t sh[33];
    const int64_t i = blockIdx.x;
    const int64_t t = i / tile_rows;
    const int32_t kb = tile_ptr[t], Kt = tile_ptr[t + 1] - kb;
    const T* row = dense + i * ld;
    if (!PRUNE) {
        int32_t all = 0, kept = 0;
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) all += nz<T>(row[k]);
        for (int32_t q = threadIdx.x; q < Kt; q += blockDim.x) {
            const int32_t c = cols[kb + q];
            if (c >= 0 && c < K) kept += nz<T>(row[c]);
        }
        int32_t tall = 0, tkept = 0;
        block_exclusive_scan(all, &tall, sh);
        block_exclusive_scan(kept, &tkept, sh);
        if (threadIdx.x == 0 && tall != tkept) atomicOr(err, SPMM_DEVERR_FORMAT);
    }
    const int64_t nb = Kp / 8;
    for (int64_t j = threadIdx.x; j < nb; j += blockDim.x) {
        uint8_t byte = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t g = 2 * j + h;
            int i0 = 0, i1 = 1;
            if (4 * g < Kt) {
                T v[4];
                unsigned mask = 0, key[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int32_t c = cols[kb + 4 * g + p];
                    v[p] = (c >= 0 && c < K) ? row[c] : T(0);
                    if (nz<T>(v[p])) mask |= 1u << p;
                    key[p] = mag_key<T>(v[p]);
                }
                if (PRUNE) {
                    top2(key, i0, i1);
                } else if (!pick2(mask, i0, i1)) {
                    atomicOr(err, SPMM_DEVERR_FORMAT);
                    i0 = 0;
                    i1 = 1;
                }
                vals[i * (Kp / 2) + 2 * g] = v[i0];
                vals[i * (Kp / 2) + 2 * g + 1] = v[i1];
            } else {
                vals[i * (Kp / 2) + 2 * g] = T(0);
                vals[i * (Kp / 2) + 2 * g + 1] = T(0);
            }
            byte |= static_cast<uint8_t>((i0 | (i1 << 2)) << (4 * h));
        }
        meta[i * nb + j] = byte;
    }
}

int* build_err_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_build_error) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

// Clear the builder error word before a launch, read it back after.
spmm_status build_begin(int* e, cudaStream_t s) { return cuda_status(cudaMemsetAsync(e, 0, sizeof(int), s)); }
spmm_status build_end(int* e, cudaStream_t s) {
    int v = 0;
    if (cudaGetLastError() != cudaSuccess) return SPMM_ERR_CUDA;
    if (cudaMemcpyAsync(&v, e, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPMM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPMM_ERR_CUDA;
    return v ? SPMM_ERR_FORMAT : SPMM_OK;
}

}  // namespace

spmm_status run_bcsr_count(const void* dense, int64_t M, int64_t K, int64_t ld, int bh, int bw, int32_t dtype,
                           int32_t* row_ptr, int64_t* nnzb, cudaStream_t s) {
    const int nbr = static_cast<int>(M / bh), gk = static_cast<int>(K / bw);
    const int smem = gk;
    if (nbr > 0 && gk > 0) {
        const bool vec = bcsr_vec(dense, ld, K, bh, bw, dtype == SPMM_I8 ? 1 : 2, nullptr);
        if (dtype == SPMM_I8 && vec)
            bcsr_count_kernel<int8_t, true>
                <<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const int8_t*>(dense), ld, bh, bw, gk, row_ptr);
        else if (dtype == SPMM_I8)
            bcsr_count_kernel<int8_t, false>
                <<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const int8_t*>(dense), ld, bh, bw, gk, row_ptr);
        else if (vec)
            bcsr_count_kernel<uint16_t, true>
                <<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const uint16_t*>(dense), ld, bh, bw, gk, row_ptr);
        else
            bcsr_count_kernel<uint16_t, false>
                <<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const uint16_t*>(dense), ld, bh, bw, gk, row_ptr);
        if (cudaGetLastError() != cudaSuccess) return SPMM_ERR_CUDA;
    } else if (nbr > 0) {
        if (cudaMemsetAsync(row_ptr, 0, sizeof(int32_t) * nbr, s) != cudaSuccess) return SPMM_ERR_CUDA;
    }
    if (cudaMemsetAsync(row_ptr + nbr, 0, sizeof(int32_t), s) != cudaSuccess) return SPMM_ERR_CUDA;
    exclusive_scan_kernel<<<1, 1024, 0, s>>>(row_ptr, nbr + 1);
    if (cudaGetLastError() != cudaSuccess) return SPMM_ERR_CUDA;
    int32_t total = 0;
    if (cudaMemcpyAsync(&total, row_ptr + nbr, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SPMM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPMM_ERR_CUDA;
    *nnzb = total;
    return SPMM_OK;
}

spmm_status run_bcsr_fill(const void* dense, int64_t M, int64_t K, int64_t ld, int bh, int bw, int32_t dtype,
                          const int32_t* row_ptr, int32_t* col_idx, void* vals, cudaStream_t s) {
    const int nbr = static_cast<int>(M / bh), gk = static_cast<int>(K / bw);
    const int smem = ((gk + 15) & ~15) + 4 * gk;
    if (nbr == 0 || gk == 0) return SPMM_OK;
    const bool vec = bcsr_vec(dense, ld, K, bh, bw, dtype == SPMM_I8 ? 1 : 2, vals);
    if (dtype == SPMM_I8 && vec)
        bcsr_fill_kernel<int8_t, true><<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const int8_t*>(dense), ld, bh, bw, gk,
                                                              row_ptr, col_idx, static_cast<int8_t*>(vals));
    else if (dtype == SPMM_I8)
        bcsr_fill_kernel<int8_t, false><<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const int8_t*>(dense), ld, bh, bw, gk,
                                                               row_ptr, col_idx, static_cast<int8_t*>(vals));
    else if (vec)
        bcsr_fill_kernel<uint16_t, true><<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const uint16_t*>(dense), ld, bh, bw,
                                                                gk, row_ptr, col_idx, static_cast<uint16_t*>(vals));
    else
        bcsr_fill_kernel<uint16_t, false><<<nbr, kBcsrBuildThreads, smem, s>>>(static_cast<const uint16_t*>(dense), ld, bh, bw,
                                                                 gk, row_ptr, col_idx, static_cast<uint16_t*>(vals));
    return cuda_status(cudaGetLastError());
}

spmm_status run_compress24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                           uint8_t* meta, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_build_mu);
    int* e = build_err_ptr();
    if (!e) return SPMM_ERR_CUDA;
    spmm_status st = build_begin(e, s);
    if (st != SPMM_OK) return st;
    const int64_t n = M * (K / 8);
    const int64_t es = dtype_bytes(dtype);  // 8 elements: 16 (or 8) bytes per access
    const int vec = (reinterpret_cast<uintptr_t>(dense) % (8 * es) == 0) && ((ld * es) % (8 * es) == 0) &&
                    (reinterpret_cast<uintptr_t>(vals) % (4 * es) == 0);
    const dim3 grid(static_cast<unsigned>((K / 8 + 255) / 256), static_cast<unsigned>(M < 65535 ? (M > 0 ? M : 1) : 65535));
    if (n > 0) {
        if (dtype == SPMM_I8)
            compress24_kernel<int8_t><<<grid, 256, 0, s>>>(
                static_cast<const int8_t*>(dense), M, K, ld, static_cast<int8_t*>(vals), meta, vec, e);
        else if (is_fp8(dtype))
            compress24_kernel<uint8_t><<<grid, 256, 0, s>>>(
                static_cast<const uint8_t*>(dense), M, K, ld, static_cast<uint8_t*>(vals), meta, vec, e);
        else
            compress24_kernel<uint16_t><<<grid, 256, 0, s>>>(
                static_cast<const uint16_t*>(dense), M, K, ld, static_cast<uint16_t*>(vals), meta, vec, e);
    }
    return build_end(e, s);
}

spmm_status run_prune24(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, void* vals,
                        uint8_t* meta, cudaStream_t s) {
    const int64_t n = M * (K / 8);
    const int64_t es = dtype_bytes(dtype);  // 8 elements: 16 (or 8) bytes per access
    const int vec = (reinterpret_cast<uintptr_t>(dense) % (8 * es) == 0) && ((ld * es) % (8 * es) == 0) &&
                    (reinterpret_cast<uintptr_t>(vals) % (4 * es) == 0);
    const dim3 grid(static_cast<unsigned>((K / 8 + 255) / 256), static_cast<unsigned>(M < 65535 ? (M > 0 ? M : 1) : 65535));
    if (n > 0) {
        trace_begin(SPMM_KERNEL_PRUNE, s);
        if (dtype == SPMM_I8)
            prune24_kernel<int8_t><<<grid, 256, 0, s>>>(
                static_cast<const int8_t*>(dense), M, K, ld, static_cast<int8_t*>(vals), meta, vec);
        else if (is_fp8(dtype))
            prune24_kernel<uint8_t><<<grid, 256, 0, s>>>(
                static_cast<const uint8_t*>(dense), M, K, ld, static_cast<uint8_t*>(vals), meta, vec);
        else
            prune24_kernel<uint16_t><<<grid, 256, 0, s>>>(
                static_cast<const uint16_t*>(dense), M, K, ld, static_cast<uint16_t*>(vals), meta, vec);
        trace_end(SPMM_KERNEL_PRUNE, s);
    }
    return cuda_status(cudaGetLastError());
}

spmm_status run_build_tvw(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t tile_rows,
                          const int32_t* tile_ptr, const int32_t* cols, int64_t n_tiles, int64_t Kp, void* vals,
                          uint8_t* meta, bool prune, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_build_mu);
    int* e = build_err_ptr();
    if (!e) return SPMM_ERR_CUDA;
    spmm_status st = build_begin(e, s);
    if (st != SPMM_OK) return st;
    if (n_tiles > 0)
        tvw_check_cols_kernel<<<static_cast<unsigned>(n_tiles), 256, 0, s>>>(tile_ptr, cols, n_tiles, K, e);
    if (M > 0) {
        auto run = [&](auto tag, const auto* d, auto* v) {
            using T = decltype(tag);
            if (prune)
                tvw_build_kernel<T, true><<<static_cast<unsigned>(M), 256, 0, s>>>(d, M, K, ld, tile_rows, tile_ptr,
                                                                                    cols, Kp, v, meta, e);
            else
                tvw_build_kernel<T, false><<<static_cast<unsigned>(M), 256, 0, s>>>(d, M, K, ld, tile_rows, tile_ptr,
                                                                                     cols, Kp, v, meta, e);
        };
        if (dtype == SPMM_I8)
            run(int8_t{}, static_cast<const int8_t*>(dense), static_cast<int8_t*>(vals));
        else
            run(uint16_t{}, static_cast<const uint16_t*>(dense), static_cast<uint16_t*>(vals));
    }
    return build_end(e, s);
}

spmm_status run_build_slide(const void* dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t n,
                            void* vals, uint8_t* meta, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_build_mu);
    int* e = build_err_ptr();
    if (!e) return SPMM_ERR_CUDA;
    spmm_status st = build_begin(e, s);
    if (st != SPMM_OK) return st;
    const int64_t G = K / (2 * n);
    const int64_t es = dtype == SPMM_I8 ? 1 : 2;
    const int vec = ((reinterpret_cast<uintptr_t>(dense) % (4 * es) == 0 && ld % 4 == 0) ? 1 : 0) |
                    (reinterpret_cast<uintptr_t>(vals) % (4 * es) == 0 ? 2 : 0);
    if (M > 0 && G > 0) {
        const dim3 grid(static_cast<unsigned>((G / 2 + 127) / 128), static_cast<unsigned>(M < 65535 ? M : 65535));
        auto run = [&](auto tag, const auto* d, auto* v) {
            using T = decltype(tag);
            switch (n) {
                case 2: slide_build_kernel<T, 2><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                case 3: slide_build_kernel<T, 3><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                case 4: slide_build_kernel<T, 4><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                case 5: slide_build_kernel<T, 5><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                case 6: slide_build_kernel<T, 6><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                case 7: slide_build_kernel<T, 7><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
                default: slide_build_kernel<T, 8><<<grid, 128, 0, s>>>(d, M, G, ld, v, meta, vec, e); break;
            }
        };
        if (dtype == SPMM_I8)
            run(int8_t{}, static_cast<const int8_t*>(dense), static_cast<int8_t*>(vals));
        else
            run(uint16_t{}, static_cast<const uint16_t*>(dense), static_cast<uint16_t*>(vals));
    }
    return build_end(e, s);
}

}  // namespace spmm
