/*
 * spmm_gb300.h -- C ABI of the GB300 (sm_103a) sparse x dense matrix multiply
 * library:  C = A_sparse * B_dense.
 *
 * A is stored in one of four formats:
 *   BCSR  block compressed sparse row       ("AsyncSparse", abstract, Fig. 2)
 *   WCSR  CSR regrouped into row windows     ("AsyncSparse", abstract, Fig. 2)
 *   2:4   semi-structured, 2 of every 4      ("Accelerating Sparse DNNs Based on
 *         consecutive K entries kept           Tiled GEMM", abstract)
 *   TVW   tile-vector-wise: per row tile a   ("Accelerating Sparse DNNs Based on
 *         kept column set, 2:4 inside it       Tiled GEMM", abstract)
 * and two routes onto them: (2n-2):2n lifted into overlapping 2:4 windows
 * ("SlideSparse", abstract) and a Reverse Cuthill-McKee permutation before
 * BCSR ("SMaT", abstract).  SDDMM samples a dense product at a CSR pattern.
 *
 * Conventions shared by every entry point
 *   - All matrix pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory.  Scratch space, where an
 *     operation needs it, is a caller-provided workspace whose size a
 *     *_workspace_size() query returns.
 *   - B is K x N row-major with leading dimension ldb (elements); C is M x N
 *     row-major with leading dimension ldc.  Every element of C[0:M, 0:N] is
 *     written (rows without stored entries get 0).  When M or N is 0 there is
 *     nothing to write: B and C may then be null and the call returns SPMM_OK
 *     without launching.
 *   - Floating-point inputs are bf16 or fp16 (2:4 also fp8) with fp32
 *     accumulation and fp32 C; int8 2:4 accumulates exactly and writes int32 C.
 *   - Every call validates its scalar arguments on the host first and returns a
 *     status without launching anything when they are invalid.  SpMM calls are
 *     asynchronous on `stream`; builders that must report sizes or
 *     data-dependent format errors synchronise `stream` (stated per call).
 *   - Kernels never wait without bound: a pipeline wait that exceeds its limit
 *     (about 2 s) records SPMM_DEVERR_TIMEOUT in a sticky per-device error word
 *     and the kernel returns; spmm_last_device_error() reads and clears it.
 *   - Alignment: B, C, format value arrays and 2:4 metadata must be 16-byte
 *     aligned, and ldb must make a row 16-byte aligned (TMA requirement).
 *     Violations return SPMM_ERR_SHAPE.
 */
#ifndef SPMM_GB300_H
#define SPMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPMM_API __attribute__((visibility("default")))
#else
#define SPMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *spmm_stream_t;

typedef enum {
    SPMM_OK = 0,
    SPMM_ERR_NULL = 1,        /* a required pointer is NULL                          */
    SPMM_ERR_SHAPE = 2,       /* bad dimension, leading dimension or alignment       */
    SPMM_ERR_DTYPE = 3,       /* dtype not supported by this call                    */
    SPMM_ERR_FORMAT = 4,      /* format data invalid (builders detect it on device)  */
    SPMM_ERR_WORKSPACE = 5,   /* workspace NULL or too small                         */
    SPMM_ERR_TIMEOUT = 6,     /* a device pipeline wait exceeded its bound           */
    SPMM_ERR_CUDA = 7,        /* CUDA runtime / driver error                         */
    SPMM_ERR_UNSUPPORTED = 8  /* valid request outside what the kernels implement    */
} spmm_status;

/* SPMM_E4M3 / SPMM_E5M2: 8-bit floats in the two encodings of the OCP 8-bit
 * floating-point specification (E4M3: exponent bias 7, no infinities, max 448;
 * E5M2: exponent bias 15, IEEE-style infinities and NaN), the FP8 that the
 * pages pair with 2:4 sparse tensor cores ("Spense", abstract, on the "sparse
 * FP4 GEMM" search page: B200 with FP8 precision). */
typedef enum { SPMM_BF16 = 0, SPMM_F16 = 1, SPMM_I8 = 2, SPMM_E4M3 = 3, SPMM_E5M2 = 4 } spmm_dtype;

/* Bits of the sticky device error word. */
#define SPMM_DEVERR_TIMEOUT 1 /* a bounded pipeline wait gave up                        */
#define SPMM_DEVERR_INDEX 2   /* an out-of-range index was skipped                      */
#define SPMM_DEVERR_FORMAT 4  /* a builder found invalid data                           */

/* ---------------------------------------------------------------- formats */

/* Block compressed sparse row ("AsyncSparse", abstract and Fig. 2).
 * A (M x K) is cut into bh x bw blocks; a block is stored iff one entry is
 * nonzero (IEEE compare: -0.0 is zero, NaN is not).  Block rows ascending,
 * block columns ascending inside a block row.
 *   row_ptr[M/bh + 1]   first stored block of each block row
 *   col_idx[nnzb]       block-column index (element column / bw)
 *   vals[nnzb][bh][bw]  block values, row-major inside a block
 * GPU SpMM supports bh in {16, 32, ..., 256} (multiple of 16), bw in {16, 32, 64}. */
typedef struct {
    int64_t M, K;
    int32_t bh, bw;
    int64_t nnzb;
    int32_t dtype; /* SPMM_BF16 or SPMM_F16 */
    int32_t *row_ptr;
    int32_t *col_idx;
    void *vals;
} spmm_bcsr_t;

/* Plain CSR (input of the row-window builder): row_ptr[M+1], col[nnz]
 * strictly ascending inside a row, val[nnz]. */
typedef struct {
    int64_t M, K, nnz;
    int32_t dtype; /* SPMM_F16 or SPMM_BF16; SPMM_I8 as the pattern of an int8 spmm_sddmm */
    int32_t *row_ptr;
    int32_t *col;
    void *val;
} spmm_csr_t;

/* Row-window CSR ("AsyncSparse", abstract: sparse operand loaded per row
 * window, long windows split across thread blocks).  Rows are grouped into
 * windows of h rows (the last may be shorter).  Per window w:
 *   wcols[wcol_ptr[w] .. wcol_ptr[w+1])  distinct columns, ascending (T_w of them)
 *   units unit_ptr[w] .. unit_ptr[w+1]-1: U_w = max(1, ceil(T_w / (16 S)))
 *     work units; unit u of the window covers column slots [16 S u, 16 S (u+1)).
 * Per nonzero (window-major; inside a window unit-major, then row, then
 * column): lrow (row - h w), slot (index into the window's wcols), val.
 * wnz_ptr[w] is the window's first nonzero, unit_win[u] the window of unit u,
 * unit_nz_ptr[u] the unit's first nonzero (unit_nz_ptr[n_units] = nnz). */
typedef struct {
    int64_t M, K, nnz;
    int32_t h, S;
    int32_t dtype; /* SPMM_F16 or SPMM_BF16 */
    int64_t n_windows, n_wcols, n_units;
    int32_t *wcol_ptr;    /* [n_windows + 1] */
    int32_t *wcols;       /* [n_wcols]       */
    int32_t *wnz_ptr;     /* [n_windows + 1] */
    int32_t *unit_ptr;    /* [n_windows + 1] */
    int32_t *unit_win;    /* [n_units]       */
    int32_t *unit_nz_ptr; /* [n_units + 1]   */
    uint8_t *lrow;        /* [nnz]           */
    int32_t *slot;        /* [nnz]           */
    void *val;            /* [nnz]           */
} spmm_wcsr_t;

/* 2:4 semi-structured ("Accelerating Sparse DNNs Based on Tiled GEMM",
 * abstract).  In every group of 4 consecutive K entries two positions are
 * stored: vals[M][K/2] (group g's entries at 2g, 2g+1), meta[M][K/8] with
 * group g's nibble idx0 | idx1 << 2 (idx0 < idx1) in byte g/2, low nibble for
 * even g.  A group with fewer than two nonzeros stores its nonzero positions
 * plus the lowest-index zero positions.  The SpMM hands meta to the tensor
 * core as stored: every nibble must have idx0 < idx1, as every builder here
 * writes; other nibbles lie outside the format. */
typedef struct {
    int64_t M, K;
    int32_t dtype; /* SPMM_I8 (-> int32 C); SPMM_F16, SPMM_BF16, SPMM_E4M3 or SPMM_E5M2 (-> fp32 C) */
    void *vals;
    uint8_t *meta;
    /* Optional, int8 only: vals widened to fp16 once (vals16[M][K/2], device
     * memory, 16-byte aligned, written by spmm_widen_24 and owned by the caller).
     * When set, spmm_24 multiplies with it instead of widening vals on every
     * call (only B is widened per call).  NULL for every other dtype (else
     * SPMM_ERR_DTYPE). */
    void *vals16;
} spmm_24_t;

/* (2n-2):2n sparsity run as 2:4 ("SlideSparse", abstract: sliding window
 * decomposition of a (2n-2):2n block into n-1 overlapping 2:4 windows, with
 * the activations lifted to match).  Group g of a row is columns
 * 2n g .. 2n g + 2n - 1; its window j (j < n - 1) covers the group's columns
 * 2j .. 2j + 3.  With G = K / 2n groups the lifted depth is K' = 4 (n-1) G, and
 * window j of group g is 2:4 group j G + g of the lifted row ("window
 * planes"), so lifted column 4 (j G + g) + p is original column
 * 2n g + 2j + p.  vals[M][K'/2] and meta[M][K'/8] store the lifted rows in the
 * layout of spmm_24_t.  2 <= n <= 8; K is the original depth. */
typedef struct {
    int64_t M, K;
    int32_t n;
    int32_t dtype; /* SPMM_I8 (-> int32 C), SPMM_F16 or SPMM_BF16 (-> fp32 C) */
    void *vals;
    uint8_t *meta;
} spmm_slide_t;

/* Tile-vector-wise ("Accelerating Sparse DNNs Based on Tiled GEMM",
 * abstract).  Rows form tiles of tile_rows rows; tile t keeps the ascending
 * columns cols[tile_ptr[t] .. tile_ptr[t+1]) (Kt entries, Kt % 4 == 0); each
 * row is 2:4 over its tile's kept columns in that order.  vals[M][Kp/2] and
 * meta[M][Kp/8] use the common pitch Kp >= max Kt; entries past a tile's Kt
 * hold value 0 and nibble (0, 1).  The GPU SpMM needs tile_rows == 128 and
 * Kp % 128 == 0. */
typedef struct {
    int64_t M, K;
    int32_t tile_rows;
    int32_t dtype; /* SPMM_F16 or SPMM_BF16 */
    int64_t n_tiles, Kp;
    int32_t *tile_ptr; /* [n_tiles + 1] */
    int32_t *cols;     /* [tile_ptr[n_tiles]] */
    void *vals;
    uint8_t *meta;
} spmm_tvw_t;

/* ---------------------------------------------------------------- utilities */

SPMM_API const char *spmm_status_string(spmm_status s);
/* Library version (major * 100 + minor). */
SPMM_API int spmm_version(void);
/* Reads and clears the sticky device error word of the current device
 * (SPMM_DEVERR_* bits).  Synchronises the device. */
SPMM_API spmm_status spmm_last_device_error(int32_t *bits);
/* Tests the bounded-wait path: launches one CTA that waits on an mbarrier no
 * one arrives on, with the given limit; the kernel gives up, records
 * SPMM_DEVERR_TIMEOUT and returns.  Synchronises `stream`. */
SPMM_API spmm_status spmm_selftest_timeout(uint64_t timeout_ns, spmm_stream_t stream);

/* Kernel-level tracing.  While enabled, the library records a pair of CUDA
 * events on the launch stream around every kernel it launches; the reads below
 * return how many launches of one kernel kind were traced and their summed
 * device time.  Used by the benchmark to time the dominant kernel alone. */
#define SPMM_KERNEL_BCSR 1    /* tcgen05 BCSR SpMM                                 */
#define SPMM_KERNEL_SPARSE 2  /* tcgen05.mma.sp SpMM (2:4 and tile-vector-wise)    */
#define SPMM_KERNEL_WIDEN 3   /* int8 -> fp16 operand widening (int8 2:4)          */
#define SPMM_KERNEL_WCSR 4    /* row-window SpMM                                   */
#define SPMM_KERNEL_PRUNE 5   /* dense -> 2:4 magnitude pruning                    */
#define SPMM_KERNEL_PERMUTE 6 /* row gather / scatter (permuted BCSR product)      */
#define SPMM_KERNEL_SDDMM 7   /* sampled dense-dense product                       */
/* Turns tracing on (clearing earlier records) or off. */
SPMM_API spmm_status spmm_trace_enable(int32_t on);
/* Synchronises the traced events and reports launches and total milliseconds
 * of `kernel` (an SPMM_KERNEL_* id) since tracing was enabled. */
SPMM_API spmm_status spmm_trace_read(int32_t kernel, int64_t *launches, double *total_ms);

/* ---------------------------------------------------------------- SpMM */

/* C = A * B with A in BCSR ("AsyncSparse": warp-specialised TMA -> tensor core
 * pipeline over nonzero blocks).  bf16/fp16 in, fp32 C. */
SPMM_API spmm_status spmm_bcsr(const spmm_bcsr_t *A, const void *B, int64_t ldb, float *C, int64_t ldc, int64_t N,
                               spmm_stream_t stream);

/* Workspace bytes spmm_wcsr needs for this operand and N: a work counter, one
 * arrival counter per (window, 128-column slab), and the partial tiles of
 * split windows (n_units x h x N fp32). */
SPMM_API spmm_status spmm_wcsr_workspace_size(const spmm_wcsr_t *A, int64_t N, size_t *bytes);
/* C = A * B with A in row-window CSR ("AsyncSparse", abstract and Fig. 2:
 * the sparse operand loaded per row window, long windows split across thread
 * blocks).  Where windows reuse their columns (at least 4 nonzeros per
 * distinct window column and 384 per work unit) each window's product runs on
 * the tensor core: for every 16 of its column slots, D (128 output columns x h
 * rows) += (the 16 gathered B rows)^T x (the window's h x 16 value tile)^T with
 * fp32 accumulation in TMEM (windows of <= 16 rows with S <= 32 in a streaming
 * kernel whose gathers run ahead of the MMAs, taller windows per item);
 * otherwise each nonzero's B row is gathered and multiplied on CUDA cores.
 * Split windows are summed in split order by the last unit to finish, so
 * results are run-to-run identical.  The workspace needs no clearing: its
 * counters carry a per-call tag, so a call that stopped early (a timed-out
 * wait) does not affect later ones; calls sharing one workspace must not
 * overlap on the GPU.  h <= 64.  fp16/bf16 in, fp32 C.  B (K x N, row pitch
 * ldb elements) must start on a 16-byte boundary with ldb a multiple of 8,
 * else SPMM_ERR_SHAPE. */
SPMM_API spmm_status spmm_wcsr(const spmm_wcsr_t *A, const void *B, int64_t ldb, float *C, int64_t ldc, int64_t N,
                               void *workspace, size_t workspace_bytes, spmm_stream_t stream);

/* Workspace bytes spmm_24 needs (int8 operands are widened to fp16 for the
 * tensor core; 0 for fp16/bf16). */
SPMM_API spmm_status spmm_24_workspace_size(const spmm_24_t *A, int64_t N, size_t *bytes);
/* int8 2:4 operand: write its values widened to fp16 (exactly: every int8 is an
 * fp16 integer) into vals16[M][K/2] (caller-allocated device memory, 16-byte
 * aligned), for spmm_24_t.vals16.  A->vals16 is not read.  A dtype other than
 * SPMM_I8 -> SPMM_ERR_DTYPE.  Asynchronous on `stream`. */
SPMM_API spmm_status spmm_widen_24(const spmm_24_t *A, void *vals16, spmm_stream_t stream);
/* C = A * B with A 2:4 ("Accelerating Sparse DNNs Based on Tiled GEMM": 2:4
 * executed inside the sparse tensor core).  int8: C is int32 and exact (the
 * kernel accumulates 2048-wide K chunks in fp32, every partial an integer of
 * magnitude below 2^24, and sums the chunks in int32).  fp16/bf16: C is fp32.
 * fp8 (E4M3 / E5M2, "Spense", abstract: 2:4 sparse tensor cores in FP8): B is
 * K x N of the same 8-bit type (row pitch ldb bytes, a multiple of 16), C is
 * fp32; products are exact and summed in fp32 by the tensor core.  Needs
 * K % 128 == 0 (K % 256 == 0 for fp8), else SPMM_ERR_SHAPE. */
SPMM_API spmm_status spmm_24(const spmm_24_t *A, const void *B, int64_t ldb, void *C, int64_t ldc, int64_t N,
                             void *workspace, size_t workspace_bytes, spmm_stream_t stream);

/* spmm_24 without a workspace argument, for callers that cannot allocate
 * device memory: for example code running inside another runtime that is
 * handed only its input and output buffers, a service that reserves all
 * device memory at start-up and forbids allocation afterwards, or a
 * latency-critical path that cannot afford cudaMalloc's implicit
 * synchronisation.  (The papers have no counterpart; this is a library
 * convenience.)  The scratch that int8 operands need (the same amount
 * spmm_24_workspace_size reports) comes from a fixed 32 MiB array inside the
 * library's device image, which every GPU that loads the library holds until
 * the process exits.  A call whose scratch would exceed 32 MiB returns
 * SPMM_ERR_WORKSPACE without launching; fp16/bf16 operands need no scratch.
 * The call allocates nothing.  Its first call on a device looks up the array's
 * device address for that device and keeps it for the life of the process;
 * make that first call before any stream capture, and do not keep using the
 * library on a device after cudaDeviceReset (the kept address then belongs to
 * the old context).  fp8 and 16-bit operands use no scratch at all.  All calls share the one array, and each call rewrites every byte
 * it later reads, so nothing has to be cleared between calls; calls that can
 * overlap on the GPU (different streams, or different host threads) race on
 * the array and must be serialised by the caller. */
SPMM_API spmm_status spmm_24_noalloc(const spmm_24_t *A, const void *B, int64_t ldb, void *C, int64_t ldc,
                                     int64_t N, spmm_stream_t stream);

/* Workspace bytes spmm_slide needs (int8: the lifted values and B widened to
 * fp16; 0 for fp16/bf16). */
SPMM_API spmm_status spmm_slide_workspace_size(const spmm_slide_t *A, int64_t N, size_t *bytes);
/* C = A * B with A a lifted (2n-2):2n operand ("SlideSparse", abstract): the
 * 2:4 sparse tensor-core SpMM over the lifted depth K', B (K x N, the original
 * rows) read through window-plane tensor maps, so that B is lifted on its way
 * into shared memory and never written out.  Arithmetic, C types and the int8
 * exactness are those of spmm_24.  Needs K % (64 n) == 0 (each 128-deep lifted
 * K step within one window plane), else SPMM_ERR_SHAPE; n outside [2, 8] ->
 * SPMM_ERR_SHAPE. */
SPMM_API spmm_status spmm_slide(const spmm_slide_t *A, const void *B, int64_t ldb, void *C, int64_t ldc, int64_t N,
                                void *workspace, size_t workspace_bytes, spmm_stream_t stream);

/* C = A * B with A tile-vector-wise ("Accelerating Sparse DNNs Based on Tiled
 * GEMM": tile-wise column selection at global-memory level, 2:4 in the sparse
 * tensor core).  Each tile gathers its kept rows of B.  fp32 C. */
SPMM_API spmm_status spmm_tvw(const spmm_tvw_t *A, const void *B, int64_t ldb, float *C, int64_t ldc, int64_t N,
                              spmm_stream_t stream);

/* ---------------------------------------------------------------- builders */

/* dense (M x K, leading dim ld) -> BCSR, phase 1: row_ptr[M/bh + 1] on the
 * device and the block count in *nnzb.  Synchronises `stream`. */
SPMM_API spmm_status spmm_build_bcsr_count(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t bh,
                                           int32_t bw, int32_t dtype, int32_t *row_ptr, int64_t *nnzb,
                                           spmm_stream_t stream);
/* Phase 2: col_idx[nnzb] and vals[nnzb][bh][bw] (values copied bit for bit). */
SPMM_API spmm_status spmm_build_bcsr_fill(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t bh,
                                          int32_t bw, int32_t dtype, const int32_t *row_ptr, int32_t *col_idx,
                                          void *vals, spmm_stream_t stream);

/* CSR -> row windows.  Workspace for both phases (must be the same buffer,
 * untouched between them). */
SPMM_API spmm_status spmm_build_wcsr_workspace_size(const spmm_csr_t *A, int32_t h, size_t *bytes);
/* Phase 1: validates the CSR (row_ptr monotone, columns strictly ascending
 * and in range: SPMM_ERR_FORMAT otherwise), and returns the total number of
 * window columns and of work units.  Synchronises `stream`. */
SPMM_API spmm_status spmm_build_wcsr_count(const spmm_csr_t *A, int32_t h, int32_t S, void *workspace,
                                           size_t workspace_bytes, int64_t *n_wcols, int64_t *n_units,
                                           spmm_stream_t stream);
/* Phase 2: fills every array of *out (allocated by the caller from the
 * counts; out->M/K/nnz/h/S/dtype/n_* are set by this call).  Bit-exact with
 * the layout described at spmm_wcsr_t. */
SPMM_API spmm_status spmm_build_wcsr_fill(const spmm_csr_t *A, int32_t h, int32_t S, void *workspace,
                                          size_t workspace_bytes, spmm_wcsr_t *out, spmm_stream_t stream);

/* dense (M x K) -> 2:4 vals[M][K/2] + meta[M][K/8].  K % 8 == 0.  More than
 * two nonzeros in a group -> SPMM_ERR_FORMAT.  Any 2:4 dtype (fp8: an entry is
 * zero iff its bits without the sign are 0; values copied bit for bit).
 * Synchronises `stream`. */
SPMM_API spmm_status spmm_compress_24(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t dtype,
                                      void *vals, uint8_t *meta, spmm_stream_t stream);

/* Magnitude pruning into 2:4 ("Accelerating Sparse DNNs Based on Tiled GEMM",
 * abstract: pruning into the 2:4 pattern of the sparse tensor core): dense
 * (M x K, row pitch ld elements, device memory) -> vals[M][K/2] + meta[M][K/8]
 * in the layout of spmm_compress_24 (caller-allocated device arrays).  In every
 * group of 4 consecutive K entries the two of largest magnitude are kept, ties
 * going to the lower index; magnitude is |v| for int8 and the bit pattern
 * without its sign for bf16/fp16/fp8 (so NaN ranks above every number).  The result
 * equals spmm_compress_24 of the matrix with the other two entries zeroed.
 * K % 8 == 0 (else SPMM_ERR_SHAPE); never fails on data.  Asynchronous on
 * `stream`. */
SPMM_API spmm_status spmm_prune_24(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t dtype,
                                   void *vals, uint8_t *meta, spmm_stream_t stream);

/* dense (M x K) + kept columns -> TVW vals[M][Kp/2] + meta[M][Kp/8].
 * tile_ptr/cols are device arrays (tile_ptr has n_tiles + 1 entries).  Kept
 * columns not ascending or out of range, a nonzero outside the kept set, or
 * more than two nonzeros in a group -> SPMM_ERR_FORMAT.  Synchronises
 * `stream`. */
SPMM_API spmm_status spmm_build_tvw(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t dtype,
                                    int32_t tile_rows, const int32_t *tile_ptr, const int32_t *cols,
                                    int64_t n_tiles, int64_t Kp, void *vals, uint8_t *meta, spmm_stream_t stream);

/* Magnitude pruning into TVW ("Accelerating Sparse DNNs Based on Tiled GEMM",
 * abstract: tile-wise pattern with 2:4 inside): arguments, layout and output
 * as spmm_build_tvw, but entries outside a tile's kept columns are dropped and
 * each group of 4 consecutive kept columns keeps its two largest magnitudes
 * (ties to the lower index; magnitude as for spmm_prune_24).  The kept columns
 * are still checked (ascending, inside [0, K)) -> SPMM_ERR_FORMAT; the matrix
 * values never cause an error.  Synchronises `stream`. */
SPMM_API spmm_status spmm_prune_tvw(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t dtype,
                                    int32_t tile_rows, const int32_t *tile_ptr, const int32_t *cols, int64_t n_tiles,
                                    int64_t Kp, void *vals, uint8_t *meta, spmm_stream_t stream);

/* dense (M x K, row pitch ld elements, device memory, at most 2n-2 nonzeros in
 * every group of 2n consecutive K entries) -> the lifted operand of
 * spmm_slide_t ("SlideSparse", abstract): vals[M][K'/2] + meta[M][K'/8] in
 * caller-allocated device arrays, K' = 2 K (n-1) / n.  Windows of a group are
 * filled in order j = 0, 1, ...: each first takes the nonzeros of its lower pair
 * that the previous window left (no later window covers them), then those of
 * its upper pair in ascending order while it holds fewer than two.  This places
 * every nonzero of a group with at most 2n-2 of them in exactly one window; a
 * window with fewer than two nonzeros is padded with its lowest other
 * positions, value +0.  Values are copied bit for bit.  2 <= n <= 8 and
 * K % (4 n) == 0 (else SPMM_ERR_SHAPE); a group with more than 2n-2 nonzeros ->
 * SPMM_ERR_FORMAT.  Synchronises `stream`. */
SPMM_API spmm_status spmm_build_slide(const void *dense, int64_t M, int64_t K, int64_t ld, int32_t dtype, int32_t n,
                                      void *vals, uint8_t *meta, spmm_stream_t stream);

/* ---------------------------------------------------------------- SDDMM
 * The sampled dense-dense product, the second sparse operation of "Magicube"
 * (abstract: SpMM and SDDMM on low-precision, quantized integers).  out[e] =
 * sum_k A[i][k] * Bt[j][k] for every stored entry e = (i, j) of the CSR
 * pattern S, i.e. (A B) at the pattern's positions with B given transposed as
 * Bt.  S->M rows, S->K columns (= rows of Bt), S->nnz entries; S->val is not
 * read.  S->dtype is the type of A and Bt:
 *   SPMM_F16 / SPMM_BF16: out is fp32, products summed in fp32; K, lda and
 *     ldbt multiples of 8;
 *   SPMM_I8: out is int32 and exact (products of signed bytes summed in int32;
 *     K * 16384 < 2^31, so no sum can overflow); K, lda and ldbt multiples of 16.
 * A is S->M x K (row pitch lda elements), Bt is S->K x K (row pitch ldbt), both
 * device arrays, 16-byte aligned; out[S->nnz] in pattern order, device memory,
 * owned by the caller.  A bad shape, pitch or alignment -> SPMM_ERR_SHAPE, any
 * other dtype -> SPMM_ERR_DTYPE.  A column outside [0, S->K) sets
 * SPMM_DEVERR_INDEX and writes 0; row_ptr is read within [0, S->M].
 * Asynchronous on `stream`. */
SPMM_API spmm_status spmm_sddmm(const spmm_csr_t *S, int64_t K, const void *A, int64_t lda, const void *Bt,
                                int64_t ldbt, void *out, spmm_stream_t stream);

/* ---------------------------------------------------------------- permutation
 * Permuting a square sparse matrix to cut its nonzero blocks before the
 * block-sparse multiply ("SMaT", abstract).  The permutation is Reverse
 * Cuthill-McKee (Cuthill and McKee, "Reducing the bandwidth of sparse
 * symmetric matrices", cited by that page), applied to rows and columns alike:
 * A' = P A P^T with A'[i][j] = A[perm[i]][perm[j]], and C = A B = P^T A' (P B). */

/* Reverse Cuthill-McKee order of an n x n CSR pattern, on the HOST: row_ptr
 * [n + 1], col [row_ptr[n]] and perm [n] are host arrays (values are not
 * needed).  The graph is the pattern of A + A^T without the diagonal.  While
 * nodes remain unvisited, a breadth-first search starts at the unvisited node
 * of least degree (lowest index on ties) and every dequeued node appends its
 * unvisited neighbours in ascending (degree, index) order; perm is the
 * visiting order reversed (perm[i] = original index at position i).  Column
 * order within a row and duplicate entries do not matter.  row_ptr not
 * starting at 0 or decreasing, or a column outside [0, n) -> SPMM_ERR_FORMAT.
 * Runs on the host because each step of the search depends on the order of
 * every earlier one; O(nnz log nnz), once per matrix. */
SPMM_API spmm_status spmm_rcm_order(int64_t n, const int32_t *row_ptr, const int32_t *col, int32_t *perm);

/* out[i][j] = dense[perm[i]][perm[j]] for an n x n dense matrix (device
 * arrays; row pitches ld and ldo elements; any dtype).  perm must be a
 * permutation of [0, n); an entry outside the range sets SPMM_DEVERR_INDEX and
 * writes 0.  Asynchronous on `stream`. */
SPMM_API spmm_status spmm_permute_sym(const void *dense, int64_t n, int64_t ld, int32_t dtype, const int32_t *perm,
                                      void *out, int64_t ldo, spmm_stream_t stream);

/* Row permutation of a rows x cols matrix of elem_bytes-byte elements (1, 2
 * or 4; device arrays, pitches lds / ldd in elements): gather (scatter = 0)
 * dst row i <- src row perm[i]; scatter (scatter = 1) dst row perm[i] <- src
 * row i.  perm entries outside [0, rows) set SPMM_DEVERR_INDEX and that row is
 * skipped.  src and dst must not overlap.  Asynchronous on `stream`. */
SPMM_API spmm_status spmm_permute_rows(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t rows,
                                       int64_t cols, int32_t elem_bytes, const int32_t *perm, int32_t scatter,
                                       spmm_stream_t stream);

/* Workspace bytes spmm_bcsr_permuted needs: B' (K x N, pitch N rounded up to
 * 8) and C' (M x N fp32, pitch N rounded up to 4). */
SPMM_API spmm_status spmm_bcsr_permuted_workspace_size(const spmm_bcsr_t *A, int64_t N, size_t *bytes);
/* C = A B for A given as the BCSR A' of P A P^T (square, M == K) and its
 * permutation perm (device, n entries): B' = P B (row gather), C' = A' B'
 * (spmm_bcsr), C = P^T C' (row scatter).  Arguments and types as spmm_bcsr;
 * M != K -> SPMM_ERR_SHAPE. */
SPMM_API spmm_status spmm_bcsr_permuted(const spmm_bcsr_t *A, const int32_t *perm, const void *B, int64_t ldb,
                                        float *C, int64_t ldc, int64_t N, void *workspace, size_t workspace_bytes,
                                        spmm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPMM_GB300_H */
