// bcsr.cu -- C = A * B for A in block compressed sparse row form.
//
// The AsyncSparse BCSR kernel ("AsyncSparse", abstract; Fig. 3 timeline,
// Fig. 4 warp-specialised pipeline) overlaps TMA transfers of B tiles with
// tensor-core work on every nonzero block.  On sm_103a that becomes:
//
//   warp 0      TMA producer: per nonzero block j of a block row, the block
//               (bh x bw, K-major, swizzled) and the matching bw rows of B for a
//               128-column token tile, into a ring of shared-memory stages.
//   warp 1      one thread issues tcgen05.mma (kind::f16, fp32 accumulate) into a
//               TMEM accumulator, then tcgen05.commit frees the stage.
//   warps 2-5   epilogue: tcgen05.ld the accumulator into a double-buffered
//               shared-memory tile (64 rows x 128 tokens) and write it with TMA
//               tensor stores while the next work unit's MMAs run (accumulators
//               are multi-buffered).  Row-scattered 128-byte warp stores reached
//               only ~5 B/clk per SM; bulk tensor stores keep C at HBM speed.
//
// Orientation: the MMA computes C^T for one (token tile, block row) unit,
//   D[token][r] = sum_j sum_c B[col_idx[j]*bw + c][token] * vals[j][r][c],
// so M = 128 tokens sit on the TMEM lanes, N = bh block rows are the MMA N,
// and each stored block is one K = bw contraction (bw / 16 MMAs).  The B tile
// is MN-major (tokens contiguous, as B is row-major), the block K-major.
// Work units are ordered token-tile-major, so CTAs resident at the same time
// share one token slab of B in L2.
#include <cstring>

#include "internal.h"
#include "sm103.cuh"

namespace spmm {
namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kTokens = 128;

struct BcsrArgs {
    const int32_t* row_ptr;
    const int32_t* col_idx;
    float* C;
    int64_t ldc;
    int64_t N;
    int32_t n_brows;
    int32_t n_ntiles;
    int32_t bh, bw;
    int32_t stages;
    int32_t nacc;
    uint32_t tmem_cols;
    uint32_t x_bytes;  // per stage: B tile, two 64-token halves of bw rows x 128 B
    uint32_t cbuf_off; // offset of the two 32 KB C staging buffers (0: store C directly)
    uint32_t w_bytes;  // per stage: block tile (1024-aligned)
    uint32_t idesc;
    uint32_t w_swz;
    uint32_t w_sbo;
    int* err;
    uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
    bcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmC, const BcsrArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stage_bytes = a.x_bytes + a.w_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.stages * stage_bytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * a.stages + 2 * a.nacc + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t s0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    // barrier addresses: full[s], empty[s], acc_full[b], acc_empty[b], done
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (a.stages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * a.stages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * a.stages + a.nacc + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * a.stages + 2 * a.nacc);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < a.nacc; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);
        }
        mbar_init(done_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int64_t total = static_cast<int64_t>(a.n_brows) * a.n_ntiles;

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        // The warp reads a unit's block columns in one coalesced load and
        // prefetches the next unit's row_ptr pair, so index latency stays off the
        // issue path; lane 0 issues the copies.
        int s = 0;
        uint32_t ph = 0;
        int64_t issued = 0;
        bool ok = true;
        const uint32_t tx = a.x_bytes + static_cast<uint32_t>(a.bh * a.bw * 2);
        int64_t u = blockIdx.x;
        int j0 = 0, j1 = 0;
        if (u < total) {
            const int br = static_cast<int>(u % a.n_brows);
            j0 = __ldg(a.row_ptr + br);
            j1 = __ldg(a.row_ptr + br + 1);
        }
        for (; u < total && ok; u += gridDim.x) {
            const int ntile = static_cast<int>(u / a.n_brows);
            const int n0 = ntile * kTokens;
            const int cj0 = j0, cj1 = j1;
            const int64_t un = u + gridDim.x;
            if (un < total) {  // next unit's block range, in flight while this unit issues
                const int brn = static_cast<int>(un % a.n_brows);
                j0 = __ldg(a.row_ptr + brn);
                j1 = __ldg(a.row_ptr + brn + 1);
            }
            for (int jb = cj0; jb < cj1 && ok; jb += 32) {
                const int cidx = (jb + lane < cj1) ? __ldg(a.col_idx + jb + lane) : 0;
                const int nb = (cj1 - jb < 32) ? cj1 - jb : 32;
                for (int t = 0; t < nb; ++t) {
                    const int kc = __shfl_sync(0xffffffffu, cidx, t) * a.bw;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t xs = s0 + s * stage_bytes, ws = xs + a.x_bytes;
                        mbar_arrive_expect_tx(full_bar(s), tx);
                        tma_load_2d(ws, &tmW, full_bar(s), 0, (jb + t) * a.bh);
                        tma_load_2d(xs, &tmB, full_bar(s), n0, kc);
                        tma_load_2d(xs + a.x_bytes / 2, &tmB, full_bar(s), n0 + 64, kc);
                    }
                    ++issued;
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        // Leave no copy in flight: wait for the last phase armed on each slot.
        for (int i = 0; i < a.stages && i < issued; ++i) {
            const int slot = (s - 1 - i + 2 * a.stages) % a.stages;
            const uint32_t par = (slot < s) ? ph : (ph ^ 1u);
            mbar_wait(full_bar(slot), par, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            int s = 0;
            uint32_t ph = 0;
            int t = 0;
            bool ok = true;
            const int ksteps = a.bw / 16;
            auto blocks_of = [&](int64_t uu) {
                if (uu >= total) return 0;
                const int brr = static_cast<int>(uu % a.n_brows);
                return __ldg(a.row_ptr + brr + 1) - __ldg(a.row_ptr + brr);
            };
            int nblk_next = blocks_of(blockIdx.x);
            for (int64_t u = blockIdx.x; u < total && ok; u += gridDim.x, ++t) {
                const int b = t % a.nacc;
                const uint32_t aph = static_cast<uint32_t>(t / a.nacc) & 1u;
                const int nblk = nblk_next;
                nblk_next = blocks_of(u + gridDim.x);
                if (!mbar_wait(acce_bar(b), aph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(b * a.bh);
                for (int j = 0; j < nblk; ++j) {
                    if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = s0 + s * stage_bytes, ws = xs + a.x_bytes;
                    for (int kk = 0; kk < ksteps; ++kk) {
                        const uint64_t ad = smem_desc(xs + kk * 2048u, a.x_bytes / 2, 1024u, SWZ_128B);
                        const uint64_t bd = smem_desc(ws + kk * 32u, 16u, a.w_sbo, a.w_swz);
                        mma_f16(d, ad, bd, a.idesc, (j | kk) != 0);
                    }
                    mma_commit(empty_bar(s));
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit(accf_bar(b));
            }
            // Every MMA issued has completed before TMEM is released.
            mma_commit(done_bar);
            mbar_wait(done_bar, 0, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const bool elected = (warp == 2 && lane == 0);  // issues the bulk stores
        int t = 0, chunk = 0;
        auto blocks_of = [&](int64_t uu) {
            if (uu >= total) return 0;
            const int brr = static_cast<int>(uu % a.n_brows);
            return __ldg(a.row_ptr + brr + 1) - __ldg(a.row_ptr + brr);
        };
        int nblk_next = blocks_of(blockIdx.x);
        for (int64_t u = blockIdx.x; u < total; u += gridDim.x, ++t) {
            const int ntile = static_cast<int>(u / a.n_brows);
            const int br = static_cast<int>(u % a.n_brows);
            const int b = t % a.nacc;
            const uint32_t aph = static_cast<uint32_t>(t / a.nacc) & 1u;
            const int nblk = nblk_next;
            nblk_next = blocks_of(u + gridDim.x);
            if (!mbar_wait(accf_bar(b), aph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
            tc_fence_after();
            const int64_t n = static_cast<int64_t>(ntile) * kTokens + q * 32 + lane;
            const bool live = n < a.N;
            float* crow = a.C + static_cast<int64_t>(br) * a.bh * a.ldc + n;
            const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * a.bh);
            // 64 accumulator columns (C rows) per TMEM round trip
            for (int c0 = 0; c0 < a.bh; c0 += 64, ++chunk) {
                uint32_t v[4][16];
                const int nq = (a.bh - c0) >= 64 ? 4 : (a.bh - c0) / 16;
                if (nblk > 0) {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (g < nq) tmem_ld16(tl + c0 + 16 * g, v[g]);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[g][i] = 0u;
                }
                if (c0 + 64 >= a.bh) {  // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(b));
                }
                if (a.cbuf_off) {
                    // stage rows c0 .. c0+63 of the unit as [row][token] and bulk-store them
                    const uint32_t buf = static_cast<uint32_t>(chunk & 1);
                    float* st = reinterpret_cast<float*>(smem + a.cbuf_off + buf * 32768u);
                    if (elected) bulk_wait_read<1>();  // the store that last used `buf` has read it
                    named_barrier(1, 128);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (g < nq) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) st[(16 * g + i) * kTokens + q * 32 + lane] = __uint_as_float(v[g][i]);
                        }
                    fence_proxy_async_smem();
                    named_barrier(1, 128);
                    if (elected) {
                        tma_store_2d(&tmC, smem_u32(st), ntile * kTokens, br * a.bh + c0);
                        bulk_commit();
                    }
                } else if (live) {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (g < nq) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                __stcs(crow + static_cast<int64_t>(c0 + 16 * g + i) * a.ldc, __uint_as_float(v[g][i]));
                        }
                }
            }
        }
        if (elected) bulk_wait<0>();  // every bulk store has completed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

uint32_t pow2_at_least(uint32_t x) {
    uint32_t p = 32;
    while (p < x) p <<= 1;
    return p;
}

}  // namespace

spmm_status launch_bcsr(const spmm_bcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    if (A->nnzb == 0) {
        return cuda_status(cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(N) * 4,
                                             static_cast<size_t>(A->M), stream));
    }
    const int bh = A->bh, bw = A->bw;
    CUtensorMap tmB, tmW;
    if (!encode_tmap_2d(&tmB, half_type(A->dtype), B, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
                        static_cast<uint64_t>(ldb) * 2, 64, static_cast<uint32_t>(bw),
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return SPMM_ERR_CUDA;
    const CUtensorMapSwizzle wswz = bw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : bw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!encode_tmap_2d(&tmW, half_type(A->dtype), A->vals, static_cast<uint64_t>(bw),
                        static_cast<uint64_t>(A->nnzb) * bh, static_cast<uint64_t>(bw) * 2,
                        static_cast<uint32_t>(bw), static_cast<uint32_t>(bh), wswz))
        return SPMM_ERR_CUDA;

    BcsrArgs a{};
    a.row_ptr = A->row_ptr;
    a.col_idx = A->col_idx;
    a.C = C;
    a.ldc = ldc;
    a.N = N;
    a.n_brows = static_cast<int32_t>(A->M / bh);
    a.n_ntiles = static_cast<int32_t>((N + kTokens - 1) / kTokens);
    a.bh = bh;
    a.bw = bw;
    a.x_bytes = static_cast<uint32_t>(bw) * 256u;
    a.w_bytes = (static_cast<uint32_t>(bh * bw * 2) + 1023u) & ~1023u;
    a.nacc = bh <= 128 ? 4 : 2;
    a.tmem_cols = pow2_at_least(static_cast<uint32_t>(a.nacc * bh));
    a.idesc = idesc_f16(128, bh, A->dtype == SPMM_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false,
                        /*sparse=*/false);
    a.w_swz = bw == 64 ? SWZ_128B : bw == 32 ? SWZ_64B : SWZ_32B;
    a.w_sbo = 8u * static_cast<uint32_t>(bw) * 2u;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;

    // C through TMA stores when its rows are 16-byte aligned (box: 128 tokens x 64 rows)
    CUtensorMap tmC;
    const bool tma_c = (ldc % 4 == 0) && aligned16(C) && bh % 64 == 0 &&
                       encode_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N),
                                      static_cast<uint64_t>(A->M), static_cast<uint64_t>(ldc) * 4, kTokens, 64,
                                      CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!tma_c) std::memset(&tmC, 0, sizeof(tmC));
    const int max_smem = dev->max_smem_optin;
    const uint32_t stage_bytes = a.x_bytes + a.w_bytes;
    const int cbuf = tma_c ? 2 * 32768 : 0;
    const int fixed = 1024 + 8 * (2 * 8 + 2 * 4 + 1) + 16 + cbuf + (tma_c ? 1024 : 0);  // + staging alignment
    int stages = (max_smem - fixed) / static_cast<int>(stage_bytes);
    stages = stages > 8 ? 8 : stages;
    if (stages < 2) return SPMM_ERR_UNSUPPORTED;
    a.stages = stages;
    const int bar_bytes = 8 * (2 * stages + 2 * a.nacc + 1) + 16;
    a.cbuf_off = tma_c ? static_cast<uint32_t>((stages * stage_bytes + bar_bytes + 1023) & ~1023u) : 0u;
    const int smem = 1024 + (tma_c ? static_cast<int>(a.cbuf_off) + cbuf : stages * static_cast<int>(stage_bytes) + bar_bytes);
    if (!set_smem_attr_once(reinterpret_cast<const void*>(bcsr_spmm_kernel), max_smem, 0)) return SPMM_ERR_CUDA;
    const int64_t units = static_cast<int64_t>(a.n_brows) * a.n_ntiles;
    const int grid = static_cast<int>(units < dev->sms ? units : dev->sms);
    trace_begin(SPMM_KERNEL_BCSR, stream);
    bcsr_spmm_kernel<<<grid, kThreads, smem, stream>>>(tmB, tmW, tmC, a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_BCSR, stream);
    return cuda_status(e);
}

}  // namespace spmm
