// bcsr.cu -- C = A * B for A in block compressed sparse row form.
//
// The AsyncSparse BCSR kernel ("AsyncSparse", abstract; Fig. 3 timeline,
// Fig. 4 warp-specialised pipeline) overlaps TMA transfers of B tiles with
// tensor-core work on every nonzero block.  On sm_103a that becomes:
//
//   warps 0-1   TMA producers, taking alternate stages of one ring: per nonzero
//               block j of a block row, the block (bh x bw, K-major, swizzled)
//               and the matching bw rows of B for a 128-column token tile (one
//               3-D box holding both 64-token halves when N is a multiple of 64).
//               One issuing thread moves ~70 B/clk; two keep the ring full.
//   warp 2      one thread issues tcgen05.mma (kind::f16, fp32 accumulate) into a
//               TMEM accumulator, then tcgen05.commit frees the stage.  The shared
//               memory descriptors are built once; per MMA only the stage and K
//               offsets are added, which keeps the issue loop a few instructions
//               long (a single thread building two descriptors per MMA cost more
//               than the N = 64 MMA itself).
//   warps 3-6   epilogue: tcgen05.ld the accumulator into a double-buffered
//               shared-memory tile (64 rows x 128 tokens) and write it with TMA
//               tensor stores while the next work unit's MMAs run (accumulators
//               are multi-buffered).
//
// Orientation: the MMA computes C^T for one (token tile, block row) unit,
//   D[token][r] = sum_j sum_c B[col_idx[j]*bw + c][token] * vals[j][r][c],
// so M = 128 tokens sit on the TMEM lanes, N = bh block rows are the MMA N,
// and each stored block is one K = bw contraction (bw / 16 MMAs).  The B tile
// is MN-major (tokens contiguous, as B is row-major), the block K-major.
// Work units are ordered token-tile-major, so CTAs resident at the same time
// share one token slab of B in L2; every role walks its units with 32-bit
// increments (no division per unit).
#include <cstring>

#include "internal.h"
#include "sm103.cuh"

namespace spmm {
namespace {

using namespace ptx;

constexpr int kProducers = 2;
constexpr int kMmaWarp = kProducers;
constexpr int kEpiWarp0 = kProducers + 1;
constexpr int kThreads = 32 * (kEpiWarp0 + 4);
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
    int32_t stages;    // even: producer p owns the slots s with s % 2 == p
    int32_t nacc;
    int32_t x3d;       // B tile as one 3-D box (both halves) instead of two 2-D boxes
    uint32_t tmem_cols;
    uint32_t x_bytes;  // per stage: B tile, two 64-token halves of bw rows x 128 B
    uint32_t cbuf_off; // offset of the two 32 KB C staging buffers (0: store C directly)
    uint32_t w_bytes;  // per stage: block tile (1024-aligned)
    uint32_t idesc;
    uint32_t w_swz;
    uint32_t w_sbo;
    const int32_t* row_perm;  // wide kernel: C row row_perm[r] receives row r (nullptr: C row r)
    int* err;
    uint64_t timeout_ns;
};

// Units u = start, start + stride, ... as (token tile, block row) with
// u = nt * n_brows + br, advanced without division.
struct UnitWalk {
    int nt, br, step_nt, step_br, n_brows;
    __device__ __forceinline__ void init(int n_brows_, int start, int stride) {
        n_brows = n_brows_;
        nt = start / n_brows;
        br = start % n_brows;
        step_nt = stride / n_brows;
        step_br = stride % n_brows;
    }
    __device__ __forceinline__ void next() {
        br += step_br;
        nt += step_nt;
        if (br >= n_brows) {
            br -= n_brows;
            ++nt;
        }
    }
};

__device__ __forceinline__ int blocks_in_row(const BcsrArgs& a, int br) {
    return __ldg(a.row_ptr + br + 1) - __ldg(a.row_ptr + br);
}

template <int KSTEPS>
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
        if (a.cbuf_off) tma_prefetch_desc(&tmC);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tslot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp < kProducers) {
        // -------------------------------------------------------- TMA producers
        // Both warps walk every block of every unit; producer p issues the blocks
        // whose position in that sequence has parity p, into its own slots.  The
        // warp reads a unit's block columns in one coalesced load and prefetches
        // the next unit's row_ptr pair; lane 0 issues the copies.
        const int p = warp;
        const int own = a.stages / 2;
        int s = p;          // next own slot
        uint32_t ph = 0;    // its phase
        int armed = 0;      // own slots armed so far (saturates at `own`)
        bool mine = (p == 0);
        bool ok = true;
        const uint32_t tx = a.x_bytes + static_cast<uint32_t>(a.bh * a.bw * 2);
        UnitWalk w;
        w.init(a.n_brows, blockIdx.x, gridDim.x);
        int j0 = 0, j1 = 0;
        if (w.nt < a.n_ntiles) {
            j0 = __ldg(a.row_ptr + w.br);
            j1 = __ldg(a.row_ptr + w.br + 1);
        }
        while (w.nt < a.n_ntiles && ok) {
            const int n0 = w.nt * kTokens;
            const int cj0 = j0, cj1 = j1;
            UnitWalk wn = w;
            wn.next();
            if (wn.nt < a.n_ntiles) {  // next unit's block range, in flight while this unit issues
                j0 = __ldg(a.row_ptr + wn.br);
                j1 = __ldg(a.row_ptr + wn.br + 1);
            }
            for (int jb = cj0; jb < cj1 && ok; jb += 32) {
                const int cidx = (jb + lane < cj1) ? __ldg(a.col_idx + jb + lane) : 0;
                const int nb = (cj1 - jb < 32) ? cj1 - jb : 32;
                for (int t = 0; t < nb; ++t) {
                    const int kc = __shfl_sync(0xffffffffu, cidx, t) * a.bw;
                    if (mine) {
                        if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            const uint32_t xs = s0 + static_cast<uint32_t>(s) * stage_bytes, ws = xs + a.x_bytes;
                            mbar_arrive_expect_tx(full_bar(s), tx);
                            tma_load_2d(ws, &tmW, full_bar(s), 0, (jb + t) * a.bh);
                            if (a.x3d) {
                                tma_load_3d(xs, &tmB, full_bar(s), 0, kc, n0 / 64);
                            } else {
                                tma_load_2d(xs, &tmB, full_bar(s), n0, kc);
                                tma_load_2d(xs + a.x_bytes / 2, &tmB, full_bar(s), n0 + 64, kc);
                            }
                        }
                        if (armed < own) ++armed;
                        s += 2;
                        if (s >= a.stages) {
                            s -= a.stages;
                            ph ^= 1u;
                        }
                    }
                    mine = !mine;
                }
            }
            w = wn;
        }
        // Leave no copy in flight: wait for the last phase armed on each own slot.
        for (int i = 0; i < armed; ++i) {
            int idx = (s - p) / 2 - 1 - i;
            uint32_t par = ph;
            if (idx < 0) {
                idx += own;
                par ^= 1u;
            }
            mbar_wait(full_bar(2 * idx + p), par, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            // Descriptor of stage 0 at K offset 0; stage s and K step kk add
            // s * stage_bytes and kk * (16 rows x 128 B) (B tile) or kk * 32 B
            // (block), in 16-byte units, to the address field.
            const uint64_t adesc0 = smem_desc(s0, a.x_bytes / 2, 1024u, SWZ_128B);
            const uint64_t bdesc0 = smem_desc(s0 + a.x_bytes, 16u, a.w_sbo, a.w_swz);
            const uint32_t sdesc = stage_bytes >> 4;
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            UnitWalk w;
            w.init(a.n_brows, blockIdx.x, gridDim.x);
            int nblk_next = w.nt < a.n_ntiles ? blocks_in_row(a, w.br) : 0;
            while (w.nt < a.n_ntiles && ok) {
                UnitWalk wn = w;
                wn.next();
                const int nblk = nblk_next;
                nblk_next = wn.nt < a.n_ntiles ? blocks_in_row(a, wn.br) : 0;
                if (!mbar_wait(acce_bar(acc), aph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * a.bh);
                for (int j = 0; j < nblk; ++j) {
                    if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>(static_cast<uint32_t>(s) * sdesc);
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk)
                        mma_f16(d, adesc0 + so + 128u * kk, bdesc0 + so + 2u * kk, a.idesc, (j | kk) != 0 ? 1u : 0u);
                    mma_commit(empty_bar(s));
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit(accf_bar(acc));
                if (++acc == a.nacc) {
                    acc = 0;
                    aph ^= 1u;
                }
                w = wn;
            }
            // Every MMA issued has completed before TMEM is released.
            mma_commit(done_bar);
            mbar_wait(done_bar, 0, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const bool elected = (warp == kEpiWarp0 && lane == 0);  // issues the bulk stores
        int acc = 0, chunk = 0;
        uint32_t aph = 0;
        UnitWalk w;
        w.init(a.n_brows, blockIdx.x, gridDim.x);
        int nblk_next = w.nt < a.n_ntiles ? blocks_in_row(a, w.br) : 0;
        while (w.nt < a.n_ntiles) {
            UnitWalk wn = w;
            wn.next();
            const int nblk = nblk_next;
            nblk_next = wn.nt < a.n_ntiles ? blocks_in_row(a, wn.br) : 0;
            if (!mbar_wait(accf_bar(acc), aph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
            tc_fence_after();
            const int64_t n = static_cast<int64_t>(w.nt) * kTokens + q * 32 + lane;
            const bool live = n < a.N;
            float* crow = a.C + static_cast<int64_t>(w.br) * a.bh * a.ldc + n;
            const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * a.bh);
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
                    if (lane == 0) mbar_arrive(acce_bar(acc));
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
                        tma_store_2d(&tmC, smem_u32(st), w.nt * kTokens, w.br * a.bh + c0);
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
            if (++acc == a.nacc) {
                acc = 0;
                aph ^= 1u;
            }
            w = wn;
        }
        if (elected) bulk_wait<0>();  // every bulk store has completed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// ---------------------------------------------------------------------------
// 64-row blocks: the W block is the MMA's A operand (M = 64, K-major) and a
// 192-token tile of B its B operand (N = 192, MN-major), so one issued MMA does
// 1.5x the work of the M = 128 tokens x N = 64 orientation above, whose issue
// cost exceeds its tensor time.  An M = 64 accumulator keeps row m in TMEM lane
// 32 * (m / 16) + m % 16 (measured on the device), i.e. lanes 0-15 of each lane
// quarter.
//
// Roles (12 warps): warps 0-2 are TMA producers, producer p filling the stages
// s with s % 3 == p (a TMA copy of 128-byte rows moves ~25 B/clk per issuing
// thread, so a 32 KB stage needs several issuers to keep up with its ~420 clk
// of MMAs); warp 3 issues the MMAs; warps 4-11 are the epilogue, two per TMEM
// lane quarter.  The epilogue cuts a unit's 192 tokens into six 32-token boxes:
// warp e takes boxes (e / 4), (e / 4) + 2, ..., reads its 16 rows x 32 columns
// from TMEM, writes them 128-byte swizzled into its own double-buffered 2 KB
// staging tile and stores it with its own TMA store, so no epilogue warp waits
// for another.  192 tokens (not 256): a 32 KB stage leaves room for six stages
// beside the C staging tiles.
constexpr int kWideTokens = 192;
constexpr int kWideChunks = kWideTokens / 64;  // 64-token chunks per B tile (128-byte swizzle rows)
constexpr int kWideRows = 64;
constexpr int kWideProducers = 3;
constexpr int kWideMmaWarp = kWideProducers;
constexpr int kWideEpi0 = kWideProducers + 1;
constexpr int kWideEpiWarps = 8;
constexpr int kWideThreads = 32 * (kWideEpi0 + kWideEpiWarps);
constexpr int kWideBoxTokens = 32;                                  // one 128-byte swizzle row of fp32
constexpr int kWideBoxes = kWideTokens / kWideBoxTokens;            // per unit
constexpr uint32_t kWideBoxBytes = 16u * kWideBoxTokens * 4u;       // 16 rows x 32 fp32 = 2 KB
constexpr uint32_t kWideCStage = kWideEpiWarps * 2u * kWideBoxBytes;  // all epilogue warps, double-buffered
static_assert(kWideEpiWarps % 4 == 0 && kWideBoxes % (kWideEpiWarps / 4) == 0, "boxes split evenly over warp sets");

template <int KSTEPS>
__global__ void __launch_bounds__(kWideThreads, 1)
    bcsr_wide_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmC, const BcsrArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stage_bytes = a.x_bytes + a.w_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.stages * stage_bytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * a.stages + 2 * a.nacc + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t s0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
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
            mbar_init(acce_bar(b), kWideEpiWarps);
        }
        mbar_init(done_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmC);
    }
    if (warp == kWideMmaWarp) {
        tmem_alloc(smem_u32(tslot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp < kWideProducers) {
        // ------------------------------------------------ TMA producers
        // Every producer walks every block of every unit; producer p issues the
        // blocks whose position in that sequence is p modulo kWideProducers, into
        // its own slots s = p, p + kWideProducers, ... (stages is a multiple).
        const int p = warp;
        const int own = a.stages / kWideProducers;
        int s = p;
        uint32_t ph = 0;
        int armed = 0;
        int turn = 0;  // position of the next block in the sequence, modulo kWideProducers
        bool ok = true;
        const uint32_t tx = a.x_bytes + static_cast<uint32_t>(kWideRows * a.bw * 2);
        const uint64_t pol_keep = l2_policy_evict_last();
        UnitWalk w;
        w.init(a.n_brows, blockIdx.x, gridDim.x);
        int j0 = 0, j1 = 0;
        if (w.nt < a.n_ntiles) {
            j0 = __ldg(a.row_ptr + w.br);
            j1 = __ldg(a.row_ptr + w.br + 1);
        }
        while (w.nt < a.n_ntiles && ok) {
            const int n0 = w.nt * kWideTokens;
            const int cj0 = j0, cj1 = j1;
            UnitWalk wn = w;
            wn.next();
            if (wn.nt < a.n_ntiles) {
                j0 = __ldg(a.row_ptr + wn.br);
                j1 = __ldg(a.row_ptr + wn.br + 1);
            }
            for (int jb = cj0; jb < cj1 && ok; jb += 32) {
                const int cidx = (jb + lane < cj1) ? __ldg(a.col_idx + jb + lane) : 0;
                const int nb = (cj1 - jb < 32) ? cj1 - jb : 32;
                for (int t = 0; t < nb; ++t) {
                    const int kc = __shfl_sync(0xffffffffu, cidx, t) * a.bw;
                    if (turn == p) {
                        if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            const uint32_t xs = s0 + static_cast<uint32_t>(s) * stage_bytes, ws = xs + a.x_bytes;
                            mbar_arrive_expect_tx(full_bar(s), tx);
                            tma_load_2d(ws, &tmW, full_bar(s), 0, (jb + t) * kWideRows);
                            // B tiles are re-read by every block row with a block in this
                            // column while the C stream passes through L2: keep them there
                            if (a.x3d) {
                                tma_load_3d_hint(xs, &tmB, full_bar(s), 0, kc, n0 / 64, pol_keep);
                            } else {
#pragma unroll
                                for (int h = 0; h < kWideChunks; ++h)
                                    tma_load_2d_hint(xs + h * (a.x_bytes / kWideChunks), &tmB, full_bar(s), n0 + 64 * h,
                                                     kc, pol_keep);
                            }
                        }
                        if (armed < own) ++armed;
                        s += kWideProducers;
                        if (s >= a.stages) {
                            s -= a.stages;
                            ph ^= 1u;
                        }
                    }
                    turn = (turn + 1 == kWideProducers) ? 0 : turn + 1;
                }
            }
            w = wn;
        }
        // Leave no copy in flight: wait for the last phase armed on each own slot.
        for (int i = 0; i < armed; ++i) {
            int idx = (s - p) / kWideProducers - 1 - i;
            uint32_t par = ph;
            if (idx < 0) {
                idx += own;
                par ^= 1u;
            }
            mbar_wait(full_bar(kWideProducers * idx + p), par, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else if (warp == kWideMmaWarp) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            // A = block (K-major, +32 B per K step), B = token tile (MN-major,
            // 64-token chunks bw rows apart, +16 rows x 128 B per K step)
            const uint64_t bdesc0 = smem_desc(s0, a.x_bytes / kWideChunks, 1024u, SWZ_128B);
            const uint64_t adesc0 = smem_desc(s0 + a.x_bytes, 16u, a.w_sbo, a.w_swz);
            const uint32_t sdesc = stage_bytes >> 4;
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            UnitWalk w;
            w.init(a.n_brows, blockIdx.x, gridDim.x);
            int nblk_next = w.nt < a.n_ntiles ? blocks_in_row(a, w.br) : 0;
            while (w.nt < a.n_ntiles && ok) {
                UnitWalk wn = w;
                wn.next();
                const int nblk = nblk_next;
                nblk_next = wn.nt < a.n_ntiles ? blocks_in_row(a, wn.br) : 0;
                if (!mbar_wait(acce_bar(acc), aph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kWideTokens);
                for (int j = 0; j < nblk; ++j) {
                    if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>(static_cast<uint32_t>(s) * sdesc);
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk)
                        mma_f16(d, adesc0 + so + 2u * kk, bdesc0 + so + 128u * kk, a.idesc, (j | kk) != 0 ? 1u : 0u);
                    mma_commit(empty_bar(s));
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit(accf_bar(acc));
                if (++acc == a.nacc) {
                    acc = 0;
                    aph ^= 1u;
                }
                w = wn;
            }
            mma_commit(done_bar);
            mbar_wait(done_bar, 0, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else {
        // -------------------------------------------------------- epilogue
        // Warp e (0..7) reads TMEM lane quarter q = warp % 4, i.e. block rows
        // 16q .. 16q+15 in lanes 0-15, for the boxes e / 4, e / 4 + 2, ... of
        // every unit.  Empty units write zeros.
        const int e = warp - kWideEpi0;
        const int q = warp & 3;
        const int first_box = e >> 2;
        constexpr int kStep = kWideEpiWarps / 4;
        const uint32_t stage0 = s0 + a.cbuf_off + static_cast<uint32_t>(e) * 2u * kWideBoxBytes;
        int acc = 0, k = 0;
        uint32_t aph = 0;
        UnitWalk w;
        w.init(a.n_brows, blockIdx.x, gridDim.x);
        int nblk_next = w.nt < a.n_ntiles ? blocks_in_row(a, w.br) : 0;
        while (w.nt < a.n_ntiles) {
            UnitWalk wn = w;
            wn.next();
            const int nblk = nblk_next;
            nblk_next = wn.nt < a.n_ntiles ? blocks_in_row(a, wn.br) : 0;
            if (!mbar_wait(accf_bar(acc), aph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) break;
            tc_fence_after();
            const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kWideTokens);
            // all of this warp's boxes of the unit in one TMEM round trip
            constexpr int kMine = kWideBoxes / kStep;
            uint32_t v[kMine][2][16];
            if (nblk > 0) {
#pragma unroll
                for (int m = 0; m < kMine; ++m) {
                    tmem_ld16(tl + kWideBoxTokens * (first_box + kStep * m), v[m][0]);
                    tmem_ld16(tl + kWideBoxTokens * (first_box + kStep * m) + 16, v[m][1]);
                }
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int m = 0; m < kMine; ++m)
#pragma unroll
                    for (int g = 0; g < 2; ++g)
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[m][g][i] = 0u;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));  // this warp's share of the accumulator is read
#pragma unroll
            for (int m = 0; m < kMine; ++m, ++k) {
                const int bx = first_box + kStep * m;
                const uint32_t buf = stage0 + static_cast<uint32_t>(k & 1) * kWideBoxBytes;
                if (lane == 0) bulk_wait_read<1>();  // the store that last used `buf` has read it
                __syncwarp();
                if (lane < 16) {
                    // row `lane` of the box is 128 B, its 16-byte units XOR-swizzled by lane % 8
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t off = buf + static_cast<uint32_t>(lane) * 128u +
                                             (static_cast<uint32_t>(u ^ (lane & 7)) << 4);
                        const uint32_t* src = &v[m][u >> 2][4 * (u & 3)];
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(off), "r"(src[0]), "r"(src[1]),
                                     "r"(src[2]), "r"(src[3])
                                     : "memory");
                    }
                }
                if (a.row_perm == nullptr) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, w.nt * kWideTokens + kWideBoxTokens * bx, w.br * kWideRows + 16 * q);
                        bulk_commit();
                    }
                } else {
                    // rows scattered to C row row_perm[r]: the warp reads the staged box
                    // back four rows at a time (eight lanes x 16 B per row), so every
                    // row leaves as one contiguous 128-byte segment
                    __syncwarp();
                    const int64_t tok0 = static_cast<int64_t>(w.nt) * kWideTokens + kWideBoxTokens * bx;
                    const int u = lane & 7;
                    const int64_t col = tok0 + 4 * u;
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int r = 4 * it + (lane >> 3);
                        const int32_t dst = __ldg(a.row_perm + w.br * kWideRows + 16 * q + r);
                        uint32_t x0, x1, x2, x3;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                     : "r"(buf + static_cast<uint32_t>(r) * 128u +
                                           (static_cast<uint32_t>(u ^ (r & 7)) << 4))
                                     : "memory");
                        if (dst < 0 || dst >= a.n_brows * kWideRows) {
                            if (u == 0) atomicOr(a.err, SPMM_DEVERR_INDEX);
                            continue;
                        }
                        float* cp = a.C + static_cast<int64_t>(dst) * a.ldc + col;
                        const float4 f = make_float4(__uint_as_float(x0), __uint_as_float(x1), __uint_as_float(x2),
                                                     __uint_as_float(x3));
                        if (col + 4 <= a.N) {
                            __stcs(reinterpret_cast<float4*>(cp), f);
                        } else {
                            const float e4[4] = {f.x, f.y, f.z, f.w};
                            for (int t = 0; t < 4 && col + t < a.N; ++t) cp[t] = e4[t];
                        }
                    }
                    __syncwarp();  // the box is read before this buffer is written again
                }
            }
            if (++acc == a.nacc) {
                acc = 0;
                aph ^= 1u;
            }
            w = wn;
        }
        if (lane == 0) bulk_wait<0>();  // this warp's stores have completed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWideMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

uint32_t pow2_at_least(uint32_t x) {
    uint32_t p = 32;
    while (p < x) p <<= 1;
    return p;
}

spmm_status launch_bcsr_wide(const spmm_bcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                             cudaStream_t stream, const DeviceInfo* dev, const int32_t* row_perm) {
    const int bw = A->bw;
    const int64_t n_brows = A->M / kWideRows, n_ntiles = (N + kWideTokens - 1) / kWideTokens;
    if (n_brows * n_ntiles >= (int64_t(1) << 31) - dev->sms || n_ntiles * kWideTokens >= (int64_t(1) << 31) ||
        A->M >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    // B tile: one 3-D box {64 tokens, bw rows, 4 chunks} when whole 64-token
    // chunks tile N (a ragged chunk would read past the row), else four 2-D boxes.
    CUtensorMap tmB, tmW, tmC;
    bool x3d = false;
    if (N % 64 == 0) {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(A->K), static_cast<uint64_t>(N / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(ldb) * 2, 128};
        const uint32_t box[3] = {64, static_cast<uint32_t>(bw), kWideChunks};
        x3d = encode_tmap_3d(&tmB, half_type(A->dtype), B, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!x3d && !encode_tmap_2d(&tmB, half_type(A->dtype), B, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
                                static_cast<uint64_t>(ldb) * 2, 64, static_cast<uint32_t>(bw),
                                CU_TENSOR_MAP_SWIZZLE_128B))
        return SPMM_ERR_CUDA;
    const CUtensorMapSwizzle wswz = bw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : bw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!encode_tmap_2d(&tmW, half_type(A->dtype), A->vals, static_cast<uint64_t>(bw),
                        static_cast<uint64_t>(A->nnzb) * kWideRows, static_cast<uint64_t>(bw) * 2,
                        static_cast<uint32_t>(bw), kWideRows, wswz) ||
        !encode_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(A->M), static_cast<uint64_t>(ldc) * 4, kWideBoxTokens, 16,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return SPMM_ERR_CUDA;
    BcsrArgs a{};
    a.row_ptr = A->row_ptr;
    a.col_idx = A->col_idx;
    a.C = C;
    a.ldc = ldc;
    a.N = N;
    a.n_brows = static_cast<int32_t>(n_brows);
    a.n_ntiles = static_cast<int32_t>(n_ntiles);
    a.bh = kWideRows;
    a.bw = bw;
    a.x3d = x3d ? 1 : 0;
    a.x_bytes = static_cast<uint32_t>(bw) * 128u * kWideChunks;  // chunks of bw rows x 128 B
    a.w_bytes = (static_cast<uint32_t>(kWideRows * bw * 2) + 1023u) & ~1023u;
    a.nacc = 2;
    a.tmem_cols = pow2_at_least(2 * kWideTokens);
    a.row_perm = row_perm;
    a.idesc = idesc_f16(kWideRows, kWideTokens, A->dtype == SPMM_BF16, /*a_mn_major=*/false, /*b_mn_major=*/true,
                        /*sparse=*/false);
    a.w_swz = bw == 64 ? SWZ_128B : bw == 32 ? SWZ_64B : SWZ_32B;
    a.w_sbo = 8u * static_cast<uint32_t>(bw) * 2u;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;
    const int max_smem = dev->max_smem_optin;
    const uint32_t stage_bytes = a.x_bytes + a.w_bytes;
    const int cbuf = static_cast<int>(kWideCStage);
    const int fixed = 1024 + 8 * (2 * 9 + 2 * 2 + 1) + 16 + cbuf + 1024;  // + staging alignment
    int stages = (max_smem - fixed) / static_cast<int>(stage_bytes);
    stages = stages > 9 ? 9 : stages;
    stages -= stages % kWideProducers;  // every producer owns the same number of slots
    if (stages < kWideProducers) return SPMM_ERR_UNSUPPORTED;
    a.stages = stages;
    const int bar_bytes = 8 * (2 * stages + 2 * a.nacc + 1) + 16;
    a.cbuf_off = static_cast<uint32_t>((stages * stage_bytes + bar_bytes + 1023) & ~1023u);
    const int smem = 1024 + static_cast<int>(a.cbuf_off) + cbuf;
    const void* kern = bw == 64 ? reinterpret_cast<const void*>(bcsr_wide_kernel<4>)
                     : bw == 32 ? reinterpret_cast<const void*>(bcsr_wide_kernel<2>)
                                : reinterpret_cast<const void*>(bcsr_wide_kernel<1>);
    if (!set_smem_attr_once(kern, max_smem, bw == 64 ? 8 : bw == 32 ? 9 : 10)) return SPMM_ERR_CUDA;
    const int64_t units = n_brows * n_ntiles;
    const int grid = static_cast<int>(units < dev->sms ? units : dev->sms);
    trace_begin(SPMM_KERNEL_BCSR, stream);
    if (bw == 64)
        bcsr_wide_kernel<4><<<grid, kWideThreads, smem, stream>>>(tmB, tmW, tmC, a);
    else if (bw == 32)
        bcsr_wide_kernel<2><<<grid, kWideThreads, smem, stream>>>(tmB, tmW, tmC, a);
    else
        bcsr_wide_kernel<1><<<grid, kWideThreads, smem, stream>>>(tmB, tmW, tmC, a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_BCSR, stream);
    return cuda_status(e);
}

}  // namespace

spmm_status launch_bcsr(const spmm_bcsr_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                        cudaStream_t stream, const int32_t* row_perm) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    if (A->nnzb == 0) {
        return cuda_status(cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(N) * 4,
                                             static_cast<size_t>(A->M), stream));
    }
    const int bh = A->bh, bw = A->bw;
    const int64_t n_brows = A->M / bh, n_ntiles = (N + kTokens - 1) / kTokens;
    // unit indices and TMA coordinates (tokens, C rows) are 32-bit
    if (n_brows * n_ntiles >= (int64_t(1) << 31) - dev->sms || n_ntiles * kTokens >= (int64_t(1) << 31) ||
        A->M >= (int64_t(1) << 31))
        return SPMM_ERR_UNSUPPORTED;
    // B tile: one 3-D box {64 tokens, bw rows, 2 halves} when whole 64-token
    // halves tile N (a ragged half would read past the row), else two 2-D boxes.
    CUtensorMap tmB, tmW;
    bool x3d = false;
    if (N % 64 == 0) {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(A->K), static_cast<uint64_t>(N / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(ldb) * 2, 128};
        const uint32_t box[3] = {64, static_cast<uint32_t>(bw), 2};
        x3d = encode_tmap_3d(&tmB, half_type(A->dtype), B, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!x3d && !encode_tmap_2d(&tmB, half_type(A->dtype), B, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
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

    // 64-row blocks with TMA-storable C: the wide kernel (M = 64 block rows x N = 192 tokens)
    if (bh == kWideRows && (ldc % 4 == 0) && aligned16(C))
        return launch_bcsr_wide(A, B, ldb, C, ldc, N, stream, dev, row_perm);
    if (row_perm) return SPMM_ERR_UNSUPPORTED;  // scattered C rows: the wide kernel only

    BcsrArgs a{};
    a.row_ptr = A->row_ptr;
    a.col_idx = A->col_idx;
    a.C = C;
    a.ldc = ldc;
    a.N = N;
    a.n_brows = static_cast<int32_t>(n_brows);
    a.n_ntiles = static_cast<int32_t>(n_ntiles);
    a.bh = bh;
    a.bw = bw;
    a.x3d = x3d ? 1 : 0;
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
    stages &= ~1;  // the two producers own alternate slots
    if (stages < 2) return SPMM_ERR_UNSUPPORTED;
    a.stages = stages;
    const int bar_bytes = 8 * (2 * stages + 2 * a.nacc + 1) + 16;
    a.cbuf_off = tma_c ? static_cast<uint32_t>((stages * stage_bytes + bar_bytes + 1023) & ~1023u) : 0u;
    const int smem = 1024 + (tma_c ? static_cast<int>(a.cbuf_off) + cbuf : stages * static_cast<int>(stage_bytes) + bar_bytes);
    const void* kern = bw == 64 ? reinterpret_cast<const void*>(bcsr_spmm_kernel<4>)
                     : bw == 32 ? reinterpret_cast<const void*>(bcsr_spmm_kernel<2>)
                                : reinterpret_cast<const void*>(bcsr_spmm_kernel<1>);
    if (!set_smem_attr_once(kern, max_smem, bw == 64 ? 0 : bw == 32 ? 6 : 7)) return SPMM_ERR_CUDA;
    const int64_t units = n_brows * n_ntiles;
    const int grid = static_cast<int>(units < dev->sms ? units : dev->sms);
    trace_begin(SPMM_KERNEL_BCSR, stream);
    if (bw == 64)
        bcsr_spmm_kernel<4><<<grid, kThreads, smem, stream>>>(tmB, tmW, tmC, a);
    else if (bw == 32)
        bcsr_spmm_kernel<2><<<grid, kThreads, smem, stream>>>(tmB, tmW, tmC, a);
    else
        bcsr_spmm_kernel<1><<<grid, kThreads, smem, stream>>>(tmB, tmW, tmC, a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_BCSR, stream);
    return cuda_status(e);
}

}  // namespace spmm
