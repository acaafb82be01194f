// spmm24.cu -- C = A * B for A in 2:4 form (dense B) and in tile-vector-wise
// form (each 128-row tile gathers its kept rows of B), on the sparse tensor
// core: tcgen05.mma.sp, kind::f16, fp32 accumulation in TMEM.
//
// "Accelerating Sparse DNNs Based on Tiled GEMM" (abstract): tile-wise pruning
// is applied at the global-memory level (here: the kept rows of B are gathered
// into shared memory) and the 2:4 pattern executes inside the sparse tensor
// core (here: tcgen05.mma.sp with the 2-bit indices in TMEM).
//
// Roles (one CTA per SM, persistent over output tiles).  Described here for one
// 128-row tile per CTA (352 threads for 2:4, 608 for TVW); with two row tiles
// per CTA (see Tile: 256 x 128 output tiles) three producers own one stage
// each, the other roles move up one warp, the MMA issuer issues each stage's
// MMAs for both row tiles, and int8 uses sixteen epilogue warps (768 threads):
//   warps 0-1  producers, taking alternate stages of one ring: per 128-wide
//              dense-K step, TMA loads of the compressed A tile (128 x 64,
//              K-major, 128B swizzle), for TVW its metadata (128 x 16 B) and, for
//              2:4, the B tile (128 K-rows x 128 columns, MN-major, 128B swizzle;
//              one 3-D box for both 64-column halves when N is a multiple of 64).
//              A single issuing thread moves ~70 B/clk, less than a stage needs.
//   warp 2     MMA issuer: four sparse MMAs per stage (M=128, N=128, K=32 dense
//              each), then tcgen05.commit frees the stage.  Descriptors are built
//              once and only offset per stage and K step.
//   warps 3-6  metadata warps (one per TMEM lane quarter): they rewrite each
//              stage's stored metadata into the tensor core's order (below) and
//              tcgen05.st it to TMEM (one 8-column-aligned column per MMA).
//   TVW only, warps 7-14: gather the stage's kept B rows (16 rows each) with
//              16-byte cp.async copies into the swizzled tile, zero-filling rows
//              past the tile's kept count, as soon as the stage is released (far
//              more requests in flight than TMA gather4 of 4 x 128-byte rows gave;
//              copy issue, not bandwidth, bounds the gather, hence eight warps).
//   last four  epilogue: tcgen05.ld the accumulator and write C.
//
// Metadata order in TMEM (measured on the device for kind::f16, M = 128,
// selector 0): within each 16-row block, TMEM lane l (l < 8) holds in its low
// half the indices of row l for K columns 0-15 of the MMA and in its high half
// those of row l+8; lane l+8 holds the same for K columns 16-31.  The stored
// format keeps one little-endian 32-bit word per row and MMA, so the rewrite is
// a swap of 16-bit halves between rows l and l^8.  Each MMA reads its word from
// a TMEM column whose index is a multiple of 8.
//
// int8 operands: the tensor core on sm_103a has no integer MMA, so int8 values
// (exact in fp16) are multiplied as fp16 with fp32 accumulation: B is widened in
// the workspace on every call, the stored values too unless the operand carries
// them widened already (spmm_24_t.vals16).  Every product is an integer of magnitude at most 127*127; the
// accumulator is drained every 2048 dense K (1024 products, |partial| <=
// 16 516 096 < 2^24, so every partial sum is an exactly representable integer)
// and the chunks are summed in int32 by the epilogue, so C is exact.
#include <cuda_fp16.h>

#include <cstring>

#include "internal.h"
#include "sm103.cuh"

namespace spmm {
namespace {

using namespace ptx;

// Four metadata warps (one per TMEM lane quarter); TVW adds eight warps that
// gather the kept B rows.  The metadata warps do not gather: a gathering warp
// waits for the stage it fills to be released, and a metadata rewrite held up
// behind that wait left the MMAs waiting for their metadata.
constexpr int kMetaWarps = 4;
__host__ __device__ constexpr int gather_warps(bool gather) { return gather ? 8 : 0; }
constexpr int BM = 128, KS = 128;                           // KS: dense K per stage
constexpr uint32_t A_BYTES = BM * (KS / 2) * 2;             // 16 KB
constexpr uint32_t B_CHUNK = KS * 128;                      // 16 KB: 128 K rows of one 64-column chunk
constexpr uint32_t M_BYTES = BM * (KS / 8);                 // 2 KB
constexpr int NACC = 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t META_STRIDE = 8;                         // one aligned TMEM column per MMA
constexpr int INT_CHUNK_STEPS = 16;                         // 16 x 128 = 2048 dense K per int chunk
// 2:4: the metadata warps copy their rows' metadata with cp.async into a ring of
// META_RING tile steps, META_AHEAD steps ahead (the TMA unit moved 128 separate
// 16-byte rows per stage for it, ~6% of the kernel's time).
constexpr int META_RING = 8, META_AHEAD = 6;

// Output tile width.  BN = 128: four 50 KB stages, two producer warps (TVW, the
// int8 path, whose exact epilogue keeps BN int32 sums per thread, and N <= 128).
// BN = 192: N = 192 sparse MMAs, which do about a quarter more useful work per
// tensor-core cycle than N = 128 (measured), in three 66 KB stages with one
// producer warp per stage; fp16/bf16 2:4 where the count of tile waves favours
// it (wide_tile), and lifted operands with a single row tile (with more, two
// row tiles per CTA measured faster at the 6:8 shape).  Producer p fills
// the steps at positions t with t % PRODUCERS == p into slot t % STAGES, so each
// slot has one producer.
//
// F8: fp8 (E4M3 / E5M2) operands on kind::f8f6f4.  A stage then holds 256 dense
// K: the compressed A tile is still 128 rows x 128 bytes, the B tile one
// 128-byte-wide chunk of 256 K rows (32 KB), and each of the four K = 64 sparse
// MMAs reads 8 stored metadata bytes per row.  (No TVW gathers or lifted planes.)
//
// MT = 2: two 128-row tiles share each B stage (a 256 x 128 output tile per
// CTA).  Per 128-deep step the CTA moves 2 x 16 KB of A and 32 KB of B for 8
// MMAs instead of 16 + 32 KB for 4, so L2 -> SM bytes per MAC drop by a third
// and each of the three 64 KB stages buffers twice the MMA work.  TMEM then
// holds one accumulator per row tile (2 x 128 columns; the MMAs of the next
// tile wait for the epilogue to read the last one out) and 2 x 4 metadata
// columns per stage.  Plain 2:4 with fp16/bf16/fp8 operands.
template <int BN_, bool F8_ = false, int MT_ = 1>
struct Tile {
    static constexpr int BN = BN_;
    static constexpr int KSD = F8_ ? 2 * KS : KS;          // dense K per stage
    static constexpr int CHUNKS = F8_ ? 1 : BN_ / 64;       // 128-byte-wide B chunks (128-byte swizzle rows)
    static constexpr uint32_t B_BYTES = KSD * BN_ * (F8_ ? 1 : 2);
    static constexpr uint32_t MB = BM * (KSD / 8);          // stored metadata bytes per row tile and step
    // 1024-aligned; the per-stage metadata copy is used by TVW only
    static constexpr uint32_t STAGE_BYTES = MT_ * A_BYTES + B_BYTES + ((F8_ || MT_ > 1) ? 0 : M_BYTES);
    static constexpr int STAGES = MT_ > 1 ? 3 : (BN_ == 128 ? 4 : 3);
    static constexpr int PRODUCERS = MT_ > 1 ? 3 : (BN_ == 128 ? 2 : 3);
    static constexpr int NACC_T = MT_ > 1 ? 1 : NACC;       // accumulator buffers per row tile
    static constexpr int MRING = (MT_ > 1 && F8_) ? 4 : META_RING;    // metadata ring steps
    static constexpr int MAHEAD = (MT_ > 1 && F8_) ? 3 : META_AHEAD;  // metadata copies ahead of use
    static constexpr int MMA_WARP = PRODUCERS;
    static constexpr int META_WARP0 = PRODUCERS + 1;
    static constexpr uint32_t META_COL = NACC_T * MT_ * BN_;  // metadata columns after the accumulators
    static constexpr uint32_t RING_OFF = STAGES * STAGE_BYTES;
    static constexpr int SMEM = 1024 + RING_OFF + MRING * MT_ * MB + 8 * (3 * STAGES + 2 * NACC_T + 1) + 16;
    __host__ __device__ static constexpr int epi_warp0(bool gather) {
        return META_WARP0 + kMetaWarps + gather_warps(gather);
    }
    // Epilogue warps: four (one per TMEM lane quarter) draining every row tile, or,
    // for int8 with two row tiles, sixteen: one per (row tile, 64-column half,
    // lane quarter), so each thread keeps 64 exact int32 sums instead of 128.
    __host__ __device__ static constexpr int epi_warps(bool int_exact) { return (int_exact && MT_ > 1) ? 16 : 4; }
    __host__ __device__ static constexpr int threads(bool gather, bool int_exact = false) {
        return 32 * (epi_warp0(gather) + epi_warps(int_exact));
    }
};
static_assert(Tile<128>::STAGES % Tile<128>::PRODUCERS == 0 && Tile<192>::STAGES % Tile<192>::PRODUCERS == 0,
              "every slot belongs to one producer");
static_assert(Tile<192>::META_COL + META_STRIDE * 4 * Tile<192>::STAGES <= TMEM_COLS &&
                  Tile<128>::META_COL + META_STRIDE * 4 * Tile<128>::STAGES <= TMEM_COLS,
              "accumulators and metadata fit in TMEM");
static_assert(Tile<192>::SMEM <= 232448 && Tile<128>::SMEM <= 232448 && Tile<128, true>::SMEM <= 232448,
              "shared memory per block");
static_assert(Tile<128, true>::STAGE_BYTES % 1024 == 0, "swizzle alignment");
static_assert(Tile<128, false, 2>::STAGES % Tile<128, false, 2>::PRODUCERS == 0 &&
                  Tile<128, false, 2>::META_COL + META_STRIDE * 4 * 2 * Tile<128, false, 2>::STAGES <= TMEM_COLS &&
                  Tile<128, false, 2>::SMEM <= 232448 && Tile<128, true, 2>::SMEM <= 232448 &&
                  Tile<128, false, 2>::STAGE_BYTES % 1024 == 0 && Tile<128, true, 2>::STAGE_BYTES % 1024 == 0,
              "two row tiles per CTA: slots, TMEM, shared memory, swizzle alignment");
static_assert(Tile<192>::STAGE_BYTES % 1024 == 0 && Tile<128>::STAGE_BYTES % 1024 == 0, "swizzle alignment");

using T16 = uint16_t;  // B elements are moved as raw 16-bit patterns

// B's tensor maps.  2:4 and TVW use one.  A (2n-2):2n operand lifted into
// window planes ("SlideSparse", abstract: activations rearranged to match the
// windows) uses one per plane j: rows 2j + p + 2n g of B, viewed as the 4-D box
// {64 columns, 4 rows p, 32 groups g, 2 column halves}, so one load lands the
// 128 lifted rows of a K step (32 windows of one plane) in the same swizzled
// order as a plain 128-row tile, and TMA performs the lifting.
constexpr int kMaxPlanes = 7;  // (2n-2):2n with n <= 8
template <int P>
struct BMaps {
    CUtensorMap m[P];
};

struct SpArgs {
    const void* B;            // TVW: gathered with cp.async
    int64_t ldb;
    int64_t b_rows;           // TVW: rows of B (kept-column indices must be below it)
    int64_t M, N, K;          // K: dense depth of the 2:4 operand (multiple of 128)
    int32_t n_mtiles, n_ntiles;
    const int32_t* tile_ptr;  // TVW only
    const int32_t* cols;      // TVW only
    const uint8_t* meta;      // 2:4: stored metadata, ldm bytes per row
    int64_t ldm;
    void* C;
    int64_t ldc;
    uint32_t idesc;
    int32_t b3d;              // 2:4: B tile as one 3-D box (both halves); lifted: one 4-D box
    int32_t planes;           // B tensor maps in use (1, or n - 1 window planes)
    int32_t plane_groups;     // lifted: windows per plane (groups G, a multiple of 32)
    int32_t vec_ok;           // C rows 16-byte aligned
    int* err;
    uint64_t timeout_ns;
};

// Output tiles are visited in groups of kGroupN column tiles, row-tile major
// inside a group: the CTAs resident at one time share ~152 / kGroupN row tiles
// of A and the group's column slab of B, which stays in L2 while every row tile
// passes (A is streamed with an evict-first hint).  Visiting all column tiles of
// a row tile at once instead needs all of B per wave, and the C writes evict it.
// Tile indices fit in 32 bits (checked on the host).
constexpr int kGroupN = 16;
__device__ __forceinline__ void tile_of(const SpArgs& a, int u, int& mt, int& nt) {
    const int per_group = a.n_mtiles * kGroupN;
    const int g = u / per_group;
    const int r = u - g * per_group;
    const int rest = a.n_ntiles - g * kGroupN;
    const int gw = rest < kGroupN ? rest : kGroupN;  // the last group may be narrower
    mt = r / gw;
    nt = g * kGroupN + (r - (r / gw) * gw);
}

// K steps of row tile mt (ksd dense K per step).
__device__ __forceinline__ int tile_steps(const SpArgs& a, int mt, int& kb, int& kt, bool gather, int ksd = KS) {
    if (gather) {
        kb = __ldg(a.tile_ptr + mt);
        kt = __ldg(a.tile_ptr + mt + 1) - kb;
        return (kt + KS - 1) / KS;
    }
    kb = 0;
    kt = static_cast<int>(a.K);
    return static_cast<int>(a.K / ksd);
}

template <bool GATHER, bool INT_EXACT, int PLANES, int BNT, bool F8 = false, int MT = 1>
__global__ void __launch_bounds__(Tile<BNT, F8, MT>::threads(GATHER, INT_EXACT), 1)
    sparse_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmMeta,
                       const __grid_constant__ BMaps<PLANES> tmB, const SpArgs a) {
    using Cfg = Tile<BNT, F8, MT>;
    static_assert(MT == 1 || (!GATHER && BNT == 128 && !(F8 && INT_EXACT)),
                  "two row tiles per CTA: 2:4 and lifted operands, 128-column tiles");
    static_assert(!INT_EXACT || BNT == 128, "the int8 epilogue keeps 128 sums per thread");
    static_assert(!GATHER || BNT == 128, "TVW gathers two 64-column chunks");
    static_assert(!F8 || (BNT == 128 && !GATHER && !INT_EXACT && PLANES == 1), "fp8: plain 2:4, 128-column tiles");
    constexpr int BN = Cfg::BN, STAGES = Cfg::STAGES, kProducers = Cfg::PRODUCERS;
    constexpr int kMmaWarp = Cfg::MMA_WARP, kMetaWarp0 = Cfg::META_WARP0;
    constexpr uint32_t B_BYTES = Cfg::B_BYTES, STAGE_BYTES = Cfg::STAGE_BYTES, RING_OFF = Cfg::RING_OFF;
    constexpr uint32_t META_COL = Cfg::META_COL;
    constexpr int KSD = Cfg::KSD;
    constexpr uint32_t MB = Cfg::MB;
    constexpr int NAC = Cfg::NACC_T, MRING = Cfg::MRING, MAHEAD = Cfg::MAHEAD;
    constexpr int BMG = BM * MT;  // rows of A per output tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_OFF + MRING * MT * MB);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2 * NAC + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int kGatherWarps = gather_warps(GATHER);
    constexpr int kEpiWarp0 = Cfg::epi_warp0(GATHER);
    constexpr int kEpiWarps = Cfg::epi_warps(INT_EXACT);
    constexpr int kEpiTiles = kEpiWarps == 4 ? MT : 1;         // row tiles each epilogue warp drains
    constexpr int kEpiCols = kEpiWarps == 16 ? BN / 2 : BN;    // accumulator columns each epilogue warp drains
    constexpr int kRowsPerWarp = KS / (GATHER ? kGatherWarps : 1);  // TVW: kept rows each gathering warp copies per step
    const uint32_t s0 = smem_u32(smem), bar0 = smem_u32(bars);
    // stage s: [A of row tile 0 .. MT - 1 | B chunks 0 .. BN/64 - 1 | stored metadata (TVW)]
    auto a_s = [&](int s) { return s0 + s * STAGE_BYTES; };
    auto b_s = [&](int s) { return s0 + s * STAGE_BYTES + MT * A_BYTES; };
    auto mc_s = [&](int s) { return s0 + s * STAGE_BYTES + MT * A_BYTES + B_BYTES; };
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto mready_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + NAC + b); };
    const uint32_t done_bar = bar0 + 8u * (3 * STAGES + 2 * NAC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), GATHER ? 1 + 32 * kGatherWarps : 1);  // TVW: + one cp.async arrival per gathering lane
            mbar_init(mready_bar(s), 4);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NAC; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps);
        }
        mbar_init(done_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmMeta);
#pragma unroll
        for (int p = 0; p < PLANES; ++p)
            if (p < a.planes) tma_prefetch_desc(&tmB.m[p]);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tslot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int total = a.n_mtiles * a.n_ntiles;
    constexpr int CH = INT_EXACT ? INT_CHUNK_STEPS : (1 << 30);

    if (warp < kProducers) {
        // -------------------------------------------------------- producers
        // Every producer walks every (tile, K step); producer p issues the steps
        // at positions t of that sequence with t % kProducers == p, into slot
        // t % STAGES (STAGES is a multiple of kProducers, so the slot is its own).
        const int p = warp;
        constexpr int OWN = STAGES / kProducers;
        int t = 0, t_last = -1, armed = 0;
        const uint64_t pol_stream = l2_policy_evict_first();  // A is read once per column group
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            int mt, nt;
            tile_of(a, u, mt, nt);
            const int m0 = mt * BMG, n0 = nt * BN;
            int kb, kt;
            const int nk = tile_steps(a, mt, kb, kt, GATHER, KSD);
            // this producer's steps of the tile: t + ks = p (mod kProducers)
            for (int ks = (p - t % kProducers + kProducers) % kProducers; ks < nk; ks += kProducers) {
                const int tt = t + ks;
                const int s = tt % STAGES;
                const uint32_t ph = static_cast<uint32_t>(tt / STAGES) & 1u;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(s), GATHER ? A_BYTES + M_BYTES : MT * A_BYTES + B_BYTES);
                    // compressed A: 128 stored bytes per row and step for fp8, 64 elements for 16-bit;
                    // rows past M (a last row tile of a pair) arrive zero-filled
#pragma unroll
                    for (int r = 0; r < MT; ++r)
                        tma_load_2d_hint(a_s(s) + r * A_BYTES, &tmA, full_bar(s), ks * (F8 ? KSD / 2 : KS / 2),
                                         m0 + r * BM, pol_stream);
                    if (GATHER) tma_load_2d_hint(mc_s(s), &tmMeta, full_bar(s), ks * (KS / 8), m0, pol_stream);
                    if constexpr (!GATHER && PLANES > 1) {
                        // lifted rows ks KS .. ks KS + 127: windows w0 .. w0 + 31 of plane j
                        const int w0 = ks * (KS / 4);
                        int j = w0 / a.plane_groups;
                        j = j < PLANES ? j : PLANES - 1;
                        const int g0 = w0 - j * a.plane_groups;
                        const CUtensorMap* bm = &tmB.m[j];
                        if (a.b3d) {
                            tma_load_4d(b_s(s), bm, full_bar(s), 0, 0, g0, n0 / 64);
                        } else {
#pragma unroll
                            for (int h = 0; h < Cfg::CHUNKS; ++h)
                                tma_load_3d(b_s(s) + h * B_CHUNK, bm, full_bar(s), n0 + 64 * h, 0, g0);
                        }
                    } else if constexpr (F8) {
                        // one 128-byte-wide chunk of KSD rows (columns n0 .. n0 + 127)
                        tma_load_2d(b_s(s), &tmB.m[0], full_bar(s), n0, ks * KSD);
                    } else if constexpr (!GATHER) {
                        if (a.b3d) {
                            tma_load_3d(b_s(s), &tmB.m[0], full_bar(s), 0, ks * KS, n0 / 64);
                        } else {
#pragma unroll
                            for (int h = 0; h < Cfg::CHUNKS; ++h)
                                tma_load_2d(b_s(s) + h * B_CHUNK, &tmB.m[0], full_bar(s), n0 + 64 * h, ks * KS);
                        }
                    }
                }
                ++armed;
                t_last = tt;
            }
            t += nk;
        }
        // Leave no copy in flight: wait for the last phase armed on each own slot
        // (no other producer arms these slots, so their phases cannot run ahead).
        for (int i = 0; i < OWN && i < armed; ++i) {
            const int tt = t_last - i * kProducers;
            mbar_wait(full_bar(tt % STAGES), static_cast<uint32_t>(tt / STAGES) & 1u, a.timeout_ns, a.err,
                      SPMM_DEVERR_TIMEOUT);
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // stage 0 descriptors; stage s adds s * STAGE_BYTES, MMA i adds 32 B
            // (A: 16 stored K elements) or 4 KB (B: 32 K rows), in 16-byte units
            const uint64_t adesc0 = smem_desc(a_s(0), 16u, 1024u, SWZ_128B);
            const uint64_t bdesc0 = smem_desc(b_s(0), F8 ? B_BYTES : B_CHUNK, 1024u, SWZ_128B);
            int s = 0, acc_i = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                int mt, nt;
                tile_of(a, u, mt, nt);  // the MMA issuer needs only the row tile
                int kb, kt;
                const int nk = tile_steps(a, mt, kb, kt, GATHER, KSD);
                const int nch = nk > 0 ? (nk + CH - 1) / CH : 1;
                for (int c = 0; c < nch && ok; ++c, ++acc_i) {
                    const int b = acc_i % NAC;
                    const uint32_t aph = static_cast<uint32_t>(acc_i / NAC) & 1u;
                    if (!mbar_wait(acce_bar(b), aph ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(b * MT * BN);
                    const int k_lo = c * CH, k_hi = min(nk, k_lo + CH);
                    for (int ks = k_lo; ks < k_hi; ++ks) {
                        if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT) ||
                            !mbar_wait(mready_bar(s), ph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (GATHER) fence_proxy_async_smem();  // B rows arrived through cp.async
                        const uint32_t mcol = tmem + META_COL + META_STRIDE * 4u * MT * s;
                        const uint64_t so = static_cast<uint64_t>(static_cast<uint32_t>(s) * (STAGE_BYTES >> 4));
#pragma unroll
                        for (int r = 0; r < MT; ++r) {
                            // row tile r: its A tile, accumulator and metadata columns; the stage's B
                            const uint64_t ro = static_cast<uint64_t>(r) * (A_BYTES >> 4);
                            const uint32_t dr = d + static_cast<uint32_t>(r * BN);
                            const uint32_t mr = mcol + META_STRIDE * 4u * r;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                // MMA i: A +32 stored bytes; B +32 K rows (16-bit) or +64 K rows (fp8) of 128 B
                                if constexpr (F8)
                                    mma_sp_f8(dr, adesc0 + so + ro + 2u * i, bdesc0 + so + 512u * i,
                                              mr + META_STRIDE * i, a.idesc, (ks > k_lo || i > 0) ? 1u : 0u);
                                else
                                    mma_sp_f16(dr, adesc0 + so + ro + 2u * i, bdesc0 + so + 256u * i,
                                               mr + META_STRIDE * i, a.idesc, (ks > k_lo || i > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit(empty_bar(s));
                        if (++s == STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    mma_commit(accf_bar(b));
                }
            }
            mma_commit(done_bar);
            mbar_wait(done_bar, 0, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT);
        }
    } else if (warp < kEpiWarp0) {
        // -------------------------------------------------------- metadata warps
        const int q = warp & 3;  // TMEM lane quarter: rows 32q .. 32q+31 of the tile
        const int row = 32 * q + lane;
        const int gq = warp - kMetaWarp0 - kMetaWarps;  // TVW gathering warp: kept rows kRowsPerWarp * gq + [0, kRowsPerWarp)
        const bool writes_meta = gq < 0;                // one metadata warp per TMEM lane quarter
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16) + META_COL;
        bool ok = true;
        // Walk over the flat sequence of (tile, K step), skipping tiles without steps.
        struct Walk {
            int u, ks, nk, kb, kt, mt, nt;
        };
        auto seek = [&](Walk& w, int u0) {
            w.u = u0;
            w.ks = 0;
            while (w.u < total) {
                tile_of(a, w.u, w.mt, w.nt);
                w.nk = tile_steps(a, w.mt, w.kb, w.kt, GATHER, KSD);
                if (w.nk > 0) break;
                w.u += gridDim.x;
            }
        };
        auto advance = [&](Walk& w) {
            if (++w.ks >= w.nk) seek(w, w.u + gridDim.x);
        };
        Walk m;
        seek(m, blockIdx.x);
        int s = 0;
        uint32_t ph = 0;
        // Rewrite the stored metadata of walker m's step into the tensor core's
        // order and place it in TMEM (one 8-aligned column per MMA).
        // 2:4: walker f runs META_AHEAD steps ahead of m and copies this thread's
        // row of metadata for its step into ring slot (step % META_RING); the
        // thread later reads back only what it copied itself.
        Walk f = m;
        int f_step = 0;
        auto meta_copy = [&]() {
#pragma unroll
            for (int r = 0; r < MT; ++r) {
                const int64_t grow = static_cast<int64_t>(f.mt) * BMG + r * BM + row;
                const bool live = f.u < total && grow < a.M;
                const uint8_t* src = live ? a.meta + grow * a.ldm + static_cast<int64_t>(f.ks) * (KSD / 8) : a.meta;
                const uint32_t dst = s0 + RING_OFF + static_cast<uint32_t>(f_step % MRING) * (MT * MB) + r * MB +
                                     (MB / BM) * row;
                cp_async16(dst, src, live ? 16u : 0u);
                if constexpr (F8) cp_async16(dst + 16u, live ? src + 16 : src, live ? 16u : 0u);
            }
            cp_async_commit();
            ++f_step;
            if (f.u < total) advance(f);
        };
        int m_step = 0;
        if (!GATHER)
            for (int i = 0; i < MAHEAD; ++i) meta_copy();
        auto meta_step = [&]() -> bool {
            const int cmt = m.mt;
            const int slot = s;
            const uint32_t par = ph;
            advance(m);
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
            uint4 wr[MT];
            uint4 w2r[F8 ? MT : 1];
            if (GATHER) {
                if (!mbar_wait(full_bar(slot), par, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) return false;
                const uint8_t* mc = smem + slot * STAGE_BYTES + A_BYTES + B_BYTES;  // TVW: one row tile
                wr[0] = *reinterpret_cast<const uint4*>(mc + 16 * row);
            } else {
                cp_async_wait<MAHEAD - 1>();  // this thread's copies for this step have landed
                const uint8_t* mine = smem + RING_OFF + (m_step % MRING) * (MT * MB) + (MB / BM) * row;
#pragma unroll
                for (int r = 0; r < MT; ++r) {
                    wr[r] = *reinterpret_cast<const uint4*>(mine + r * MB);
                    if constexpr (F8) w2r[r] = *reinterpret_cast<const uint4*>(mine + r * MB + 16);
                }
                ++m_step;
                meta_copy();
                // the MMAs that read this slot's metadata columns last time are done
                if (!mbar_wait(empty_bar(slot), par ^ 1u, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) return false;
            }
#pragma unroll
            for (int r = 0; r < MT; ++r) {
                // rows past M arrive zero-filled; give them the valid (0, 1) pattern
                const bool row_live = static_cast<int64_t>(cmt) * BMG + r * BM + row < a.M;
                uint4 w = wr[r];
                const uint32_t tb = tl + META_STRIDE * (4u * MT * slot + 4u * r);
                if constexpr (F8) {
                    // kind::f8f6f4 reads row r's 64 bits of one MMA from TMEM lane r, two
                    // consecutive columns, in stored order (measured): copy them as they are
                    uint4 w2 = w2r[r];
                    if (!row_live) {
                        w = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);
                        w2 = w;
                    }
                    tmem_st2(tb, w.x, w.y);
                    tmem_st2(tb + META_STRIDE, w.z, w.w);
                    tmem_st2(tb + 2 * META_STRIDE, w2.x, w2.y);
                    tmem_st2(tb + 3 * META_STRIDE, w2.z, w2.w);
                } else {
                    if (!row_live) w = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);
                    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t p = __shfl_xor_sync(0xffffffffu, in[i], 8);
                        const uint32_t o = (lane & 8) ? __byte_perm(p, in[i], 0x7632) : __byte_perm(in[i], p, 0x5410);
                        tmem_st1(tb + META_STRIDE * i, o);
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(mready_bar(slot));
            return true;
        };
        if constexpr (GATHER) {
            // TVW: eight warps gather the kept rows of B into each stage's swizzled
            // MN-major tile with 16-byte cp.async copies, as soon as the stage is
            // released; the metadata warps rewrite a step once its copies (and the
            // A tile) have landed.  This lane's kept-row index for walker g's step is
            // loaded one step ahead of its use.
            const T16* Bp = static_cast<const T16*>(a.B);
            const int gi = lane & 7;                 // 16-byte piece within a 128-byte chunk row
            const int hi = lane >> 4;                // row parity within an iteration's pair of rows
            const uint32_t hoff = ((lane >> 3) & 1) * B_CHUNK;
            Walk g = m;
            int sg = 0;
            uint32_t phg = 0;
            auto kept_row = [&](const Walk& w) {
                const int k = w.ks * KS + kRowsPerWarp * gq + lane;
                return (w.u < total && lane < kRowsPerWarp && k < w.kt) ? __ldg(a.cols + w.kb + k) : -1;
            };
            int32_t rnext = kept_row(g);
            auto gather_step = [&]() -> bool {
                const int32_t rcur = rnext;
                const int64_t n0 = static_cast<int64_t>(g.nt) * BN;
                const int slot = sg;
                const uint32_t par = phg ^ 1u;
                advance(g);
                rnext = kept_row(g);
                if (++sg == STAGES) {
                    sg = 0;
                    phg ^= 1u;
                }
                if (!mbar_wait(empty_bar(slot), par, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) return false;
                const bool in_b = rcur >= 0 && rcur < a.b_rows;
                if (rcur >= 0 && !in_b) atomicOr(a.err, SPMM_DEVERR_INDEX);
                const int32_t myrow = in_b ? rcur : -1;
                const int64_t col = n0 + 64 * ((lane >> 3) & 1) + 8 * gi;  // this lane's first column
                const int64_t left = a.N - col;
                const uint32_t nb_full = left >= 8 ? 16u : (left > 0 ? static_cast<uint32_t>(left) * 2u : 0u);
                const uint32_t dst0 = b_s(slot) + hoff;
#pragma unroll
                for (int it = 0; it < kRowsPerWarp / 2; ++it) {
                    const int lr = 2 * it + hi;  // row within the warp's kept rows
                    const int32_t brow = __shfl_sync(0xffffffffu, myrow, lr);
                    const int k = kRowsPerWarp * gq + lr;
                    const uint32_t nbytes = brow < 0 ? 0u : nb_full;
                    const T16* src = nbytes ? Bp + static_cast<int64_t>(brow) * a.ldb + col : Bp;
                    cp_async16(dst0 + k * 128u + (static_cast<uint32_t>(gi ^ (k & 7)) << 4), src, nbytes);
                }
                cp_async_arrive_noinc(full_bar(slot));
                return true;
            };
            if (writes_meta) {
                while (ok && m.u < total) ok = meta_step();
            } else {
                while (ok && g.u < total) ok = gather_step();
            }
        } else {
            while (ok && m.u < total) ok = meta_step();
            cp_async_wait<0>();  // no copy into shared memory outstanding at exit
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;                // TMEM lane quarter this warp may read
        const int e = warp - kEpiWarp0;        // groups of four consecutive warps cover the four quarters
        const int r0 = kEpiWarps == 4 ? 0 : e / 8;                           // first row tile this warp drains
        const int c0 = kEpiWarps == 16 ? ((e / 4) & 1) * kEpiCols : 0;      // first accumulator column
        int acc_i = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            int mt, nt;
            tile_of(a, u, mt, nt);
            int kb, kt;
            const int nk = tile_steps(a, mt, kb, kt, GATHER, KSD);
            const int nch = nk > 0 ? (nk + CH - 1) / CH : 1;
            const int64_t n0 = static_cast<int64_t>(nt) * BN + c0;           // this warp's first output column
            const bool full_n = n0 + kEpiCols <= a.N && a.vec_ok;
            const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0);
            int32_t run[INT_EXACT ? kEpiCols : 1];
#pragma unroll
            for (int i = 0; i < (INT_EXACT ? kEpiCols : 1); ++i) run[i] = 0;
            bool ok = true;
            for (int c = 0; c < nch; ++c, ++acc_i) {
                const int b = acc_i % NAC;
                const uint32_t aph = static_cast<uint32_t>(acc_i / NAC) & 1u;
                if (!mbar_wait(accf_bar(b), aph, a.timeout_ns, a.err, SPMM_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int r = r0; r < r0 + kEpiTiles; ++r) {
                    // row tile r of the output tile: this thread's row, its accumulator
                    const int64_t row = static_cast<int64_t>(mt) * BMG + r * BM + q * 32 + lane;
                    const bool row_live = row < a.M;
                    const uint32_t tb = tl + static_cast<uint32_t>((b * MT + r) * BN);
#pragma unroll
                    for (int j = 0; j < kEpiCols / 16; ++j) {
                        uint32_t v[16];
                        if (nk > 0) {
                            tmem_ld16(tb + 16 * j, v);
                            tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0u;
                        }
                        if constexpr (INT_EXACT) {
                            // every chunk partial is an integer of magnitude below 2^24, exact in
                            // fp32; round-to-nearest conversion returns it unchanged
#pragma unroll
                            for (int i = 0; i < 16; ++i) run[16 * j + i] += __float2int_rn(__uint_as_float(v[i]));
                        } else if (row_live) {
                            float* cp = static_cast<float*>(a.C) + row * a.ldc + n0 + 16 * j;
                            if (full_n) {
#pragma unroll
                                for (int i = 0; i < 16; i += 4)
                                    __stcs(reinterpret_cast<float4*>(cp + i),
                                           make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                       __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])));
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (n0 + 16 * j + i < a.N) cp[i] = __uint_as_float(v[i]);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar(b));
            }
            if (!ok) break;
            if constexpr (INT_EXACT) {
                const int64_t row = static_cast<int64_t>(mt) * BMG + r0 * BM + q * 32 + lane;  // one row tile
                if (row < a.M) {
                    int32_t* cp = static_cast<int32_t*>(a.C) + row * a.ldc + n0;
                    if (full_n) {
#pragma unroll
                        for (int i = 0; i < kEpiCols; i += 4)
                            __stcs(reinterpret_cast<int4*>(cp + i),
                                   make_int4(run[i], run[i + 1], run[i + 2], run[i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < kEpiCols; ++i)
                            if (n0 + i < a.N) cp[i] = run[i];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// int8 -> fp16, exact.  Four bytes become four halves without a conversion
// instruction: flipping the sign bit gives v + 128 in [0, 255]; placed under
// the fp16 exponent of 1024 (high byte 0x64) each half reads 1024 + v + 128,
// and subtracting 1152 leaves v.  Every step is exact in fp16 (integers below
// 2048 are representable).
__device__ __forceinline__ uint2 widen4(uint32_t w) {
    const uint32_t b = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(b, 0x64646464u, 0x4150);  // halves 0x64 b0, 0x64 b1
    const uint32_t hi = __byte_perm(b, 0x64646464u, 0x4352);  // halves 0x64 b2, 0x64 b3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
    const __half2 l = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&l), *reinterpret_cast<const uint32_t*>(&h));
}

// One row-major int8 matrix to widen: rows of `cols` elements, leading
// dimensions lds (source) and ldd (destination, columns [cols, ldd) zeroed).
struct WidenJob {
    const int8_t* src;
    int64_t lds;
    __half* dst;
    int64_t ldd;
    int64_t rows, cols;
    int64_t per_row;   // threads per row: ceil(ldd / 16)
    int64_t threads;   // rows * per_row
};

// Both operands in one launch; 16 elements (one 16-byte load) per thread.
__global__ void widen_i8_kernel(const WidenJob j0, const WidenJob j1) {
    int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool first = id < j0.threads;
    const WidenJob& j = first ? j0 : j1;
    if (!first) id -= j0.threads;
    if (id >= j.threads) return;
    const int64_t r = id / j.per_row, c = (id - r * j.per_row) * 16;
    const int8_t* sp = j.src + r * j.lds + c;
    __half* dp = j.dst + r * j.ldd + c;
    if (c + 16 <= j.cols && (reinterpret_cast<uintptr_t>(sp) & 15) == 0 && (reinterpret_cast<uintptr_t>(dp) & 15) == 0) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(sp));
        const uint2 a = widen4(w.x), b = widen4(w.y), e = widen4(w.z), f = widen4(w.w);
        reinterpret_cast<uint4*>(dp)[0] = make_uint4(a.x, a.y, b.x, b.y);
        reinterpret_cast<uint4*>(dp)[1] = make_uint4(e.x, e.y, f.x, f.y);
    } else {
        for (int i = 0; i < 16 && c + i < j.ldd; ++i)
            dp[i] = c + i < j.cols ? __int2half_rn(sp[i]) : __float2half(0.f);
    }
}

template <bool GATHER, bool INT_EXACT, int PLANES, int BNT, bool F8 = false, int MT = 1>
spmm_status launch_sparse(const CUtensorMap& tmA, const CUtensorMap& tmM, const BMaps<PLANES>& tmB, const SpArgs& a,
                          cudaStream_t stream, int slot) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    constexpr int kSmem = Tile<BNT, F8, MT>::SMEM;
    if (dev->max_smem_optin < kSmem) return SPMM_ERR_UNSUPPORTED;
    auto kern = sparse_spmm_kernel<GATHER, INT_EXACT, PLANES, BNT, F8, MT>;
    if (!set_smem_attr_once(reinterpret_cast<const void*>(kern), kSmem, slot)) return SPMM_ERR_CUDA;
    const int64_t units = static_cast<int64_t>(a.n_mtiles) * a.n_ntiles;
    if (units >= (int64_t(1) << 31) - dev->sms) return SPMM_ERR_UNSUPPORTED;  // 32-bit tile indices
    const int grid = static_cast<int>(units < dev->sms ? units : dev->sms);
    trace_begin(SPMM_KERNEL_SPARSE, stream);
    kern<<<grid, Tile<BNT, F8, MT>::threads(GATHER, INT_EXACT), kSmem, stream>>>(tmA, tmM, tmB, a);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_SPARSE, stream);
    return cuda_status(e);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// int8 operands: the stored values (rows x kv) and B (kb rows x N) widened to
// fp16 in the workspace, B with pitch np = N rounded up to 8.  With values
// widened beforehand (have_a16) only B is.
size_t widen_bytes(int64_t rows, int64_t kv, int64_t kb, int64_t N, bool have_a16 = false) {
    const int64_t np = (N + 7) / 8 * 8;
    return (have_a16 ? 0 : align256(static_cast<size_t>(rows) * kv * 2)) + align256(static_cast<size_t>(kb) * np * 2);
}

WidenJob widen_job(const void* src, int64_t lds, __half* dst, int64_t ldd, int64_t r, int64_t cols) {
    WidenJob j{static_cast<const int8_t*>(src), lds, dst, ldd, r, cols, (ldd + 15) / 16, 0};
    j.threads = r * j.per_row;
    return j;
}

// vals16: the values already widened (the workspace then holds only B), or null.
spmm_status widen_operands(const void* vals, int64_t rows, int64_t kv, const void* B, int64_t ldb, int64_t kb,
                           int64_t N, void* ws, cudaStream_t stream, const void** vals16, const void** b16,
                           int64_t* ld16, const void* a16 = nullptr) {
    __half* wa = a16 ? nullptr : static_cast<__half*>(ws);
    __half* wb = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) +
                                           (a16 ? 0 : align256(static_cast<size_t>(rows) * kv * 2)));
    const int64_t np = (N + 7) / 8 * 8;
    const WidenJob ja = a16 ? widen_job(vals, kv, nullptr, kv, 0, kv) : widen_job(vals, kv, wa, kv, rows, kv);
    const WidenJob jb = widen_job(B, ldb, wb, np, kb, N);
    const int64_t threads = ja.threads + jb.threads;
    trace_begin(SPMM_KERNEL_WIDEN, stream);
    widen_i8_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(ja, jb);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WIDEN, stream);
    if (e != cudaSuccess) return SPMM_ERR_CUDA;
    *vals16 = a16 ? a16 : wa;
    *b16 = wb;
    *ld16 = np;
    return SPMM_OK;
}

// Maps of the stored values (M x K/2, 128 x 64 boxes) and metadata (M x K/8)
// of a 2:4 operand of dense depth K.
bool encode_a_maps(CUtensorMapDataType t, const void* vals, const uint8_t* meta, int64_t M, int64_t K,
                   CUtensorMap* tmA, CUtensorMap* tmM) {
    return encode_tmap_2d(tmA, t, vals, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M),
                          static_cast<uint64_t>(K), 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tmap_2d(tmM, CU_TENSOR_MAP_DATA_TYPE_UINT8, meta, static_cast<uint64_t>(K / 8),
                          static_cast<uint64_t>(M), static_cast<uint64_t>(K / 8), 16, 128,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 192-column tiles for fp16/bf16 operands when they take fewer tile-times
// than 128-column ones.  Persistent CTAs run ceil(tiles / SMs) waves, and a
// 192-column tile costs about 1.44 times a 128-column one (measured: the
// three-stage ring, not the wider MMA, sets its pace), so the count of waves
// decides.  int8 keeps 128 (its exact epilogue holds 128 int32 sums per thread).
bool wide_tile(bool i8, int64_t M, int64_t N, int sms) {
    if (i8 || N <= 128) return false;
    const int64_t mt = (M + BM - 1) / BM;
    const int64_t w128 = (mt * ((N + 127) / 128) + sms - 1) / sms;
    const int64_t w192 = (mt * ((N + 191) / 192) + sms - 1) / sms;
    return w192 * 144 < w128 * 100;
}

// Two 128-row tiles per CTA whenever A has more than one row tile: they share
// each B stage (see Tile).  For int8 this is measured 2% faster per call than
// one row tile (359 us against 366 us at 8192^2 x 4096, widening included): the
// four exact-chunk drains per tile stall the MMAs on the single accumulator.
constexpr bool kPairInt8 = true;
bool pair_tiles(bool i8, int64_t M) { return M > BM && (!i8 || kPairInt8); }

SpArgs dense_b_args(const DeviceInfo* dev, int64_t M, int64_t K, int64_t N, int32_t dtype, const uint8_t* meta,
                    void* C, int64_t ldc, int bn, int mt = 1) {
    SpArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.n_mtiles = static_cast<int32_t>((M + BM * mt - 1) / (BM * mt));  // output tiles of mt row tiles
    a.n_ntiles = static_cast<int32_t>((N + bn - 1) / bn);
    a.C = C;
    a.ldc = ldc;
    a.idesc = idesc_f16(128, bn, dtype == SPMM_BF16, false, true, true, 0);
    a.vec_ok = (ldc % 4 == 0) && aligned16(C);
    a.meta = meta;
    a.ldm = K / 8;
    a.planes = 1;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;
    return a;
}

}  // namespace

size_t spmm24_workspace_bytes(const spmm_24_t* A, int64_t N) {
    return A->dtype == SPMM_I8 ? widen_bytes(A->M, A->K / 2, A->K, N, A->vals16 != nullptr) : 0;
}

spmm_status widen_values_24(const void* vals, int64_t rows, int64_t kv, void* dst, cudaStream_t stream) {
    const WidenJob ja = widen_job(vals, kv, static_cast<__half*>(dst), kv, rows, kv);
    const WidenJob jb = widen_job(vals, kv, nullptr, kv, 0, kv);
    trace_begin(SPMM_KERNEL_WIDEN, stream);
    widen_i8_kernel<<<static_cast<unsigned>((ja.threads + 255) / 256), 256, 0, stream>>>(ja, jb);
    const cudaError_t e = cudaGetLastError();
    trace_end(SPMM_KERNEL_WIDEN, stream);
    return cuda_status(e);
}

// fp8 operands (kind::f8f6f4): A's stored bytes in 128 x 128-byte boxes, B in
// 256-row x 128-byte boxes (128 columns), both 128-byte swizzled.
spmm_status launch_spmm24_f8(const DeviceInfo* dev, const spmm_24_t* A, const void* B, int64_t ldb, void* C,
                             int64_t ldc, int64_t N, cudaStream_t stream) {
    CUtensorMap tmA, tmM;
    BMaps<1> tmB;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!encode_tmap_2d(&tmA, u8, A->vals, static_cast<uint64_t>(A->K / 2), static_cast<uint64_t>(A->M),
                        static_cast<uint64_t>(A->K / 2), 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tmM, u8, A->meta, static_cast<uint64_t>(A->K / 8), static_cast<uint64_t>(A->M),
                        static_cast<uint64_t>(A->K / 8), 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&tmB.m[0], u8, B, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
                        static_cast<uint64_t>(ldb), 128, 256, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPMM_ERR_CUDA;
    const bool pair = pair_tiles(false, A->M);
    SpArgs a = dense_b_args(dev, A->M, A->K, N, A->dtype, A->meta, C, ldc, 128, pair ? 2 : 1);
    a.idesc = idesc_f8(128, 128, A->dtype == SPMM_E5M2, false, true, true);
    if (pair) return launch_sparse<false, false, 1, 128, true, 2>(tmA, tmM, tmB, a, stream, 17);
    return launch_sparse<false, false, 1, 128, true>(tmA, tmM, tmB, a, stream, 15);
}

spmm_status launch_spmm24(const spmm_24_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                          void* ws, cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    if (A->dtype == SPMM_E4M3 || A->dtype == SPMM_E5M2) return launch_spmm24_f8(dev, A, B, ldb, C, ldc, N, stream);
    const bool i8 = A->dtype == SPMM_I8;
    const void* vals = A->vals;
    const void* bsrc = B;
    int64_t bld = ldb;
    const CUtensorMapDataType t = i8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : half_type(A->dtype);
    if (i8) {
        const spmm_status st =
            widen_operands(A->vals, A->M, A->K / 2, B, ldb, A->K, N, ws, stream, &vals, &bsrc, &bld, A->vals16);
        if (st != SPMM_OK) return st;
    }
    CUtensorMap tmA, tmM;
    BMaps<1> tmB;
    const int bn = wide_tile(i8, A->M, N, dev->sms) ? 192 : 128;
    // B tile: one 3-D box {64 columns, 128 K rows, bn / 64 chunks} when whole
    // 64-column chunks tile N (a ragged chunk would read past the row), else one
    // 2-D box per chunk.
    bool b3d = false;
    if (N % 64 == 0) {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(A->K), static_cast<uint64_t>(N / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(bld) * 2, 128};
        const uint32_t box[3] = {64, 128, static_cast<uint32_t>(bn / 64)};
        b3d = encode_tmap_3d(&tmB.m[0], t, bsrc, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!encode_a_maps(t, vals, A->meta, A->M, A->K, &tmA, &tmM) ||
        (!b3d && !encode_tmap_2d(&tmB.m[0], t, bsrc, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
                                 static_cast<uint64_t>(bld) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)))
        return SPMM_ERR_CUDA;
    const bool pair = bn == 128 && pair_tiles(i8, A->M);
    SpArgs a = dense_b_args(dev, A->M, A->K, N, A->dtype, A->meta, C, ldc, bn, pair ? 2 : 1);
    a.b3d = b3d ? 1 : 0;
    if (i8 && pair) return launch_sparse<false, true, 1, 128, false, 2>(tmA, tmM, tmB, a, stream, 20);
    if (i8) return launch_sparse<false, true, 1, 128>(tmA, tmM, tmB, a, stream, 2);
    if (bn == 192) return launch_sparse<false, false, 1, 192>(tmA, tmM, tmB, a, stream, 13);
    if (pair) return launch_sparse<false, false, 1, 128, false, 2>(tmA, tmM, tmB, a, stream, 18);
    return launch_sparse<false, false, 1, 128>(tmA, tmM, tmB, a, stream, 1);
}

size_t slide_workspace_bytes(const spmm_slide_t* A, int64_t N) {
    const int64_t Kl = 4 * (A->n - 1) * (A->K / (2 * A->n));
    return A->dtype == SPMM_I8 ? widen_bytes(A->M, Kl / 2, A->K, N) : 0;
}

spmm_status launch_slide(const spmm_slide_t* A, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t N,
                         void* ws, cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    const int n = A->n;
    const int64_t G = A->K / (2 * n), Kl = 4 * (n - 1) * G;
    const bool i8 = A->dtype == SPMM_I8;
    const void* vals = A->vals;
    const void* bsrc = B;
    int64_t bld = ldb;
    const CUtensorMapDataType t = i8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : half_type(A->dtype);
    if (i8) {
        const spmm_status st = widen_operands(A->vals, A->M, Kl / 2, B, ldb, A->K, N, ws, stream, &vals, &bsrc, &bld);
        if (st != SPMM_OK) return st;
    }
    CUtensorMap tmA, tmM;
    BMaps<kMaxPlanes> tmB;
    std::memset(&tmB, 0, sizeof(tmB));
    // Plane j: rows 2j + p + 2n g of B (p < 4, g < G).  Whole 64-column chunks:
    // one 4-D box {64, 4, 32, bn / 64}; otherwise one 3-D box {64, 4, 32} per chunk.
    // fp16/bf16 with more than one row tile: two row tiles per CTA at 128 columns.
    const bool pair = !i8 && pair_tiles(i8, A->M);  // int8 lifted operands keep one row tile
    const int bn = !pair && wide_tile(i8, A->M, N, dev->sms) ? 192 : 128;
    const bool b4d = N % 64 == 0;
    const uint64_t row = static_cast<uint64_t>(bld) * 2;
    for (int j = 0; j < n - 1; ++j) {
        const void* base = static_cast<const uint8_t*>(bsrc) + 2 * j * row;
        bool ok;
        if (b4d) {
            const uint64_t dims[4] = {64, 4, static_cast<uint64_t>(G), static_cast<uint64_t>(N / 64)};
            const uint64_t strides[3] = {row, 2 * n * row, 128};
            const uint32_t box[4] = {64, 4, 32, static_cast<uint32_t>(bn / 64)};
            ok = encode_tmap_4d(&tmB.m[j], t, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            const uint64_t dims[3] = {static_cast<uint64_t>(N), 4, static_cast<uint64_t>(G)};
            const uint64_t strides[2] = {row, 2 * n * row};
            const uint32_t box[3] = {64, 4, 32};
            ok = encode_tmap_3d(&tmB.m[j], t, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return SPMM_ERR_CUDA;
    }
    if (!encode_a_maps(t, vals, A->meta, A->M, Kl, &tmA, &tmM)) return SPMM_ERR_CUDA;
    SpArgs a = dense_b_args(dev, A->M, Kl, N, A->dtype, A->meta, C, ldc, bn, pair ? 2 : 1);
    a.b3d = b4d ? 1 : 0;
    a.planes = n - 1;
    a.plane_groups = static_cast<int32_t>(G);
    if (i8) return launch_sparse<false, true, kMaxPlanes, 128>(tmA, tmM, tmB, a, stream, 12);
    if (pair) return launch_sparse<false, false, kMaxPlanes, 128, false, 2>(tmA, tmM, tmB, a, stream, 19);
    if (bn == 192) return launch_sparse<false, false, kMaxPlanes, 192>(tmA, tmM, tmB, a, stream, 14);
    return launch_sparse<false, false, kMaxPlanes, 128>(tmA, tmM, tmB, a, stream, 11);
}

spmm_status launch_tvw(const spmm_tvw_t* A, const void* B, int64_t ldb, float* C, int64_t ldc, int64_t N,
                       cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return SPMM_ERR_CUDA;
    if (A->M == 0 || N == 0) return SPMM_OK;
    const CUtensorMapDataType t = half_type(A->dtype);
    CUtensorMap tmA, tmM;
    BMaps<1> tmB;
    if (!encode_a_maps(t, A->vals, A->meta, A->M, A->Kp, &tmA, &tmM) ||
        !encode_tmap_2d(&tmB.m[0], t, B, static_cast<uint64_t>(N), static_cast<uint64_t>(A->K),
                        static_cast<uint64_t>(ldb) * 2, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPMM_ERR_CUDA;
    SpArgs a{};
    a.B = B;
    a.ldb = ldb;
    a.b_rows = A->K;
    a.M = A->M;
    a.N = N;
    a.K = A->Kp;
    a.n_mtiles = static_cast<int32_t>(A->n_tiles);
    a.n_ntiles = static_cast<int32_t>((N + 127) / 128);
    a.tile_ptr = A->tile_ptr;
    a.cols = A->cols;
    a.C = C;
    a.ldc = ldc;
    a.idesc = idesc_f16(128, 128, A->dtype == SPMM_BF16, false, true, true, 0);
    a.vec_ok = (ldc % 4 == 0) && aligned16(C);
    a.planes = 1;
    a.err = dev->err;
    a.timeout_ns = kWaitTimeoutNs;
    return launch_sparse<true, false, 1, 128>(tmA, tmM, tmB, a, stream, 3);
}

}  // namespace spmm
