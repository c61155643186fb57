/*
 * evocg.h -- C ABI of the GB300 tile-wise mixed-precision CG library (libevocg.so).
 *
 * The method is the one of "EvoCG: Self-Evolving Precision Control for Faster Conjugate
 * Gradient" (arXiv 2611.04469): a sparse matrix cut into square tiles, each tile holding
 * its values in FP64, FP32 and BF16 and read in the precision a per-tile map selects
 * (§3.3 EvoSpMV, Fig. 4), inside a CG / Jacobi-PCG loop (§2.1 Fig. 1, §4.6) whose map is
 * rewritten in-loop by a controller (§3.2 Eq. 8-10, §4.7), run on the device without a
 * host round trip per iteration (§3.4 EvoRun, Fig. 5).
 *
 * Conventions for every call:
 *  - Return value: an evocg_status; EVOCG_OK (0) on success. No call throws, aborts or
 *    prints. evocg_last_error() gives a message for the calling thread's last failure.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Device work is queued
 *    on it; a call that must hand back a host-visible result synchronises that stream.
 *  - Vector arguments marked "host or device" may point to either; the library checks
 *    with cudaPointerGetAttributes and stages host data through its own device buffers.
 *  - Indices are 0-based. Matrices are square, n x n, n < 2^31.
 *  - The caller owns every pointer it passes; the library owns the tile structure and
 *    its workspaces, which evocg_tiles_free releases. A handle may be used from one
 *    thread at a time.
 */
#ifndef EVOCG_H
#define EVOCG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct evocg_tiles *evocg_tiles_t;

typedef enum {
    EVOCG_OK = 0,
    EVOCG_EINVAL = 1,      /* bad argument or input (message says which) */
    EVOCG_ENOMEM = 2,      /* a device or host allocation failed */
    EVOCG_ECUDA = 3,       /* a CUDA runtime call failed */
    EVOCG_ENOTCONV = 4,    /* CG stopped at maxit; iterations and history are filled */
    EVOCG_EBREAKDOWN = 5,  /* p.Ap <= 0 or not finite: the operator is not SPD */
    EVOCG_ETIMEOUT = 6,    /* a bounded device wait ran out */
    EVOCG_EDEVICE = 7      /* no usable CUDA device, or not an sm_103 device */
} evocg_status;

/* Precision codes of EvoCG Eq. 9. */
enum { EVOCG_FP64 = 0, EVOCG_FP32 = 1, EVOCG_BF16 = 2 };

/* Map layouts for evocg_set_tile_precision. */
enum {
    EVOCG_MAP_PER_TILE = 0,     /* one code per nonempty tile, in tile order */
    EVOCG_MAP_PER_COLBLOCK = 1  /* one code per column block (EvoCG Eq. 10), every tile of
                                   column block i takes code i */
};

/* Controllers (EvoCG §3.2, §4.7). */
enum {
    EVOCG_CTRL_STATIC = 0,     /* the matrix's current map is used for every iteration */
    EVOCG_CTRL_THRESHOLD = 1,  /* residual-threshold rule on m_i = max |p_i| */
    EVOCG_CTRL_MLP = 2         /* policy MLP on phi(p_i) = p_i / max(||p_i||, delta) */
};

typedef struct {
    int64_t n;            /* matrix order */
    int64_t nrb;          /* row blocks = column blocks = ceil(n / tile_size) */
    int64_t ntiles;       /* nonempty tiles */
    int64_t nnz;          /* stored entries */
    int32_t tile_size;    /* T: tiles are T x T */
    int32_t map_kind;     /* which map the SpMV reads (EVOCG_MAP_*) */
    int64_t bytes_index;  /* tileRowPtr + tileColIdx + tileNnzOff + rowMask + tileWidth + colIdx */
    int64_t bytes_v64, bytes_v32, bytes_v16, bytes_colexp;   /* per value stream (slots) */
    int64_t nslots;       /* slots of the value streams: entries plus row padding */
} evocg_tiles_desc;

typedef struct {
    int kind;              /* EVOCG_CTRL_* */
    int kstar;             /* the controller runs on iterations k with k % kstar == 0 (EvoCG
                              §3.4 interval reuse); values < 1 mean 1 */
    double eps;            /* THRESHOLD: BF16 if m_i < 0.1 eps, FP32 if m_i < eps, else FP64 */
    int hidden1, hidden2;  /* MLP hidden widths (EvoCG §4.1: 64, 64); at most 64 each */
    const float *weights;  /* MLP: host pointer to W1 (hidden1 x T), b1, W2 (hidden2 x
                              hidden1), b2, W3 (3 x hidden2), b3, packed in that order, each
                              W row-major (out, in), FP32 */
    double delta;          /* MLP: the floor of the segment norm in phi (EvoCG Eq. 8) */
    uint8_t *map_log;      /* NULL, or a HOST or DEVICE buffer of map_log_rows x nrb bytes: row k
                              receives the column-block map the SpMV of iteration k used, for the
                              iterations of the controlled phase (k < map_log_rows; rows past
                              the last such iteration are left as they were). The profiling run
                              of EvoCG §3.4 interval reuse: log with kstar = 1, then choose the
                              interval with evocg_kstar_select. Ignored for EVOCG_CTRL_STATIC */
    int64_t map_log_rows;
    int eps_relative;      /* THRESHOLD: 0 (the default) applies eps as an absolute bound, as
                              EvoCG §4.7 states the rule; 1 scales both cut points by
                              ||r_0||_inf = ||b||_inf (x0 = 0), an option beside the paper's
                              rule. Ignored by evocg_ctrl_decide */
} evocg_ctrl;

typedef struct {
    int status;            /* same value the solve returns */
    int iters;             /* SpMVs performed in the loop, restarts included */
    int iters_recursive;   /* iterations at the first recursive convergence, or -1 */
    int restarts;          /* FP64-finish restarts taken */
    double rel_res;        /* last recursively updated ||r_k|| / ||r_0|| */
    double true_res;       /* ||b - A x|| / ||b|| recomputed in FP64 (all tiles FP64), or -1 */
    int64_t prec_nnz[3];   /* stored entries (pads not counted) processed per precision,
                              summed over SpMVs */
    int64_t ctrl_calls;    /* controller invocations */
} evocg_solve_info;

/*
 * Build the tile structure (EvoCG §3.3.1 Fig. 4(a) and §3.3.2): row blocks of
 * tile_size rows, the nonempty tile_size x tile_size tiles of each row block listed in
 * ascending column block (tileRowPtr / tileColIdx). Inside a tile: rowMask (bit r: local
 * row r has entries in the tile), tileWidth w (its longest row) and w x h slots, h =
 * popcount(rowMask), in slot-major order: slot (k, j) at tileNnzOff[t] + k*h + j holds the
 * k-th entry (ascending column) of the j-th nonempty row, or a pad (local column T,
 * value +0) when that row has k or fewer entries. One local column byte per slot
 * (colIdx) and three value streams over the same slots: FP64 a_ij, FP32 and BF16 of
 * a_ij / s_j, where s_j = 2^e_j is the per-column factor of §3.3.2 with
 * e_j = floor(log2 max_i |a_ij|) clamped to [-100, 100] (0 for an empty column). FP32 and
 * BF16 values are rounded once from FP64, to nearest with ties to even.
 *   n, row_ptr (n+1, int64), col_idx (row_ptr[n], int32, strictly ascending per row,
 *   0 <= col < n), vals (FP64, finite): HOST pointers, read only.
 *   tile_size: 16, 32 or 64.
 *   *out receives the handle; the map starts all-FP64 (per tile).
 * Errors: EINVAL (bad sizes, unsorted or out-of-range columns, non-finite values),
 * ENOMEM, ECUDA, EDEVICE.
 */
int evocg_tile_build(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                     const double *vals, int tile_size, evocg_tiles_t *out);

/* Release the handle and all device memory it owns (synchronises the device first).
 * NULL is accepted. */
int evocg_tiles_free(evocg_tiles_t A);

/* Sizes of the structure. d: host pointer. */
int evocg_tiles_info(evocg_tiles_t A, evocg_tiles_desc *d);

/*
 * Copy the structure back to HOST arrays, for bit-exact layout checks. Sizes:
 * tileRowPtr nrb+1, tileColIdx ntiles, tileNnzOff ntiles+1, rowMask ntiles,
 * tileWidth ntiles, colIdx / v64 / v32 / v16 nslots, colExp n. Any pointer may be NULL to
 * skip that array. Synchronises the device.
 */
int evocg_tiles_export(evocg_tiles_t A, int64_t *tileRowPtr, int32_t *tileColIdx,
                       int64_t *tileNnzOff, uint64_t *rowMask, uint8_t *tileWidth,
                       uint8_t *colIdx, double *v64, float *v32, uint16_t *v16,
                       int8_t *colExp);

/*
 * The tile layout of evocg_tile_build (EvoCG §3.3.1 Fig. 4(a), §3.3.2, with the slot-major
 * tile interior described there) computed on the HOST only, without a GPU: the same
 * builder, its arrays written to caller buffers (sizes as in evocg_tiles_export: tileRowPtr
 * nrb+1, tileColIdx / tileNnzOff(+1) / rowMask / tileWidth ntiles, colIdx / v64 / v32 / v16
 * nslots, colExp n), for inspecting a layout or checking it where no device is present.
 *   n, row_ptr, col_idx, vals, tile_size: as evocg_tile_build (HOST arrays).
 *   ntiles, nslots: receive the sizes (either may be NULL). Every array pointer may be NULL;
 *   a call with all of them NULL only sizes the layout (the builder runs on every call).
 * Errors: as evocg_tile_build (EINVAL, ENOMEM); no device is touched.
 */
int evocg_tile_layout_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                           const double *vals, int tile_size, int64_t *ntiles, int64_t *nslots,
                           int64_t *tileRowPtr, int32_t *tileColIdx, int64_t *tileNnzOff,
                           uint64_t *rowMask, uint8_t *tileWidth, uint8_t *colIdx, double *v64,
                           float *v32, uint16_t *v16, int8_t *colExp);

/*
 * The Tile-CSC layout of EvoCG §3.3.1 Fig. 4(a) and §3.3.2 Fig. 4(b), written from this
 * library's tile builder on the HOST (no GPU): the inter-tile CSR over row blocks
 * (tileRowPtr nrb+1, tileColIdx ntiles: tiles of a row block in ascending column block) and
 * inside every tile a CSC. Tile t's entries start at tileNnzOff[t] (ntiles+1 entries) in the
 * padded streams; colPtr[t*(T+1) + c] .. colPtr[t*(T+1) + c + 1] is the range of local column
 * c relative to that start (colPtr: ntiles x (T+1), uint16); a column's entries are in
 * ascending row and rowIdx (nnz_p bytes) holds each entry's row relative to the row block's
 * first row. With pad = 2 (the paper's padding of every column to a multiple of two) a
 * column with an odd number of entries ends with one sentinel-marked zero: rowIdx = T (the
 * row index "R" of Fig. 4(b)) and +0 in the three value streams; pad = 1 stores no sentinel.
 * v64 / v32 / v16 (nnz_p each): a_ij, and a_ij / s_j rounded once to FP32 / BF16 (s_j =
 * 2^colExp[j], colExp: n bytes), the same bits the SpMV reads.
 *   n, row_ptr, col_idx, vals, tile_size: as evocg_tile_build (HOST arrays).
 *   ntiles, nnz_p: receive the sizes (either may be NULL). Every array pointer may be NULL; a
 *   call with all of them NULL only sizes the layout.
 * Errors: as evocg_tile_build; EINVAL for pad other than 1 or 2. No device is touched.
 */
int evocg_tile_csc_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                        const double *vals, int tile_size, int pad, int64_t *ntiles,
                        int64_t *nnz_p, int64_t *tileRowPtr, int32_t *tileColIdx,
                        int64_t *tileNnzOff, uint16_t *colPtr, uint8_t *rowIdx, double *v64,
                        float *v32, uint16_t *v16, int8_t *colExp);

/*
 * The same Tile-CSC arrays as evocg_tile_csc_host, written from the DEVICE-resident
 * structure of a handle: the arrays the SpMV kernels read are copied back and rewritten as
 * Tile-CSC on the host, so a bit-exact comparison checks what the GPU computes with. Sizes
 * as in evocg_tile_csc_host (ntiles from evocg_tiles_info); *nnz_p receives the padded
 * length (may be NULL); every array pointer may be NULL. Synchronises the device.
 * Errors: EINVAL (NULL handle, pad other than 1 or 2), ENOMEM, ECUDA.
 */
int evocg_tiles_export_csc(evocg_tiles_t A, int pad, int64_t *nnz_p, int64_t *tileRowPtr,
                           int32_t *tileColIdx, int64_t *tileNnzOff, uint16_t *colPtr,
                           uint8_t *rowIdx, double *v64, float *v32, uint16_t *v16,
                           int8_t *colExp);

/*
 * The panel SpMV's batch plan for a matrix, computed on the HOST only (no GPU), for inspection.
 * The paper has no counterpart: the plan belongs to this library's SpMV kernel. The same
 * builder and planner evocg_tile_build runs cut every 32-row panel's tiles into batches that
 * fit a shared-memory stage of stage_bytes (each tile sized for FP64), for `warps` warps
 * walking contiguous panel ranges.
 *   *nbatches receives the number of batches; *valid 1 when the plan passes the checks the
 *   library applies before using it (every record matching the tile structure, tile slices
 *   16-byte aligned inside the streams, every batch inside its stage), 0 when the library would
 *   run the direct kernel instead (the reason is in evocg_last_error). Either may be NULL.
 * Errors: as evocg_tile_build; EINVAL for warps < 1 or stage_bytes < 1.
 */
int evocg_panel_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                          const double *vals, int tile_size, int64_t warps, int stage_bytes,
                          int64_t *nbatches, int *valid);

/*
 * The row-block SpMV's plan for a matrix (tiles of 32), computed on the HOST only (no GPU),
 * for inspection. The paper has no counterpart: the plan belongs to this library's SpMV
 * kernel. Every tile of two or more slots gets a 16-byte descriptor; the single-entry tiles
 * of each row block are gathered into a row-owned ELL block (rows with such tiles x the
 * largest count of them in one row, shorter rows padded).
 *   *ndesc receives the descriptor count, *nsingle_slots the ELL slots (pads included),
 *   *valid 1 when the plan passes the checks the library applies before using it (every
 *   descriptor and single matching the tile structure, tile slices 16-slot aligned), 0 when
 *   the library would run another kernel (tiles other than 32, a size limit; the reason is
 *   in evocg_last_error). Each pointer may be NULL.
 * Errors: as evocg_tile_build.
 */
int evocg_rowblock_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                             const double *vals, int tile_size, int64_t *ndesc,
                             int64_t *nsingle_slots, int *valid);

/*
 * The row-ELL SpMV's plan for a matrix, computed on the HOST only (no GPU), for inspection.
 * The paper has no counterpart. It exists for tiles of 64 holding at most 1.5 entries per
 * nonempty tile row (random banded matrices): each row block's entries laid out by row, an
 * ELL block of width = its longest row, every slot with its absolute column, its tile and
 * the tile slot's three values.
 *   *nslots receives the ELL slots (pads included), *valid 1 when the plan exists and passes
 *   the checks the library applies before using it (every row's entries, in column order,
 *   with their tiles and values), 0 otherwise (the reason is in evocg_last_error). Each
 *   pointer may be NULL.
 * Errors: as evocg_tile_build.
 */
int evocg_rowell_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                           const double *vals, int tile_size, int64_t *nslots, int *valid);

/*
 * Set the precision map (EvoCG Eq. 9-10): codes EVOCG_FP64/FP32/BF16.
 *   map: host or device, len = ntiles (PER_TILE) or nrb (PER_COLBLOCK).
 * The SpMV and static-map solves read the map set last. With the row-ELL kernel (tiles of
 * 64 holding about one entry per row) a PER_TILE map also reorders every row's entries by
 * (precision, column) on the device, which changes the order of a row's sum but not its
 * terms; the order is a function of the map alone (all-FP64: column order). Synchronises
 * the stream. Errors: EINVAL on a wrong length or a code above 2 (the map is checked on the
 * host; a device map is copied there).
 */
int evocg_set_tile_precision(evocg_tiles_t A, const uint8_t *map, int64_t len,
                             int map_kind, void *stream);

/* Copy the current per-tile map (the per-column-block map broadcast to tiles when that
 * kind is set) to a HOST array of ntiles entries. Synchronises the stream. */
int evocg_get_tile_precision(evocg_tiles_t A, uint8_t *map_out, int64_t len, void *stream);

/*
 * Mixed-precision SpMV y = (A + E(map)) x (EvoCG Eq. 2 / Eq. 5 and §3.3.2): a tile in
 * FP64 multiplies its FP64 values by x; a tile in FP32 or BF16 multiplies its FP32/BF16
 * values by the x entries rounded to the same format and scaled by s_j. Every product is
 * exact or, for FP64 tiles, rounded once; each row is summed in FP64 (FP32/BF16 products
 * through an error-free FP32 pair). x, y: host or device, n FP64 each, not overlapping.
 * Asynchronous on `stream` for device pointers; with a host pointer the call returns once
 * y is written.
 */
int evocg_spmv(evocg_tiles_t A, const double *x, double *y, void *stream);

/* Flags of evocg_spmv_ex. */
enum {
    EVOCG_SPMV_REUSE_XCOPIES = 1, /* skip rounding x: reuse the FP32/BF16 copies of x made by
                                     the previous evocg_spmv / evocg_spmv_ex call on this
                                     handle; x must hold the same values as in that call */
    EVOCG_SPMV_DIRECT = 2,        /* run the direct kernel: a warp per row block, every operand
                                     loaded by the lanes from global memory, one tile after
                                     the other (the kernel for tiles of 64). At most one of
                                     DIRECT, PANEL, ROWBLOCK, ROWELL may be set */
    EVOCG_SPMV_PANEL = 8,         /* run the panel kernel (the default for tiles of 16):
                                     a warp streams batches of tiles of consecutive row blocks
                                     through two shared-memory stages, every tile's own lane
                                     issuing its bulk copies; single-entry tiles take one lane
                                     each */
    EVOCG_SPMV_TEST_LOST_WAIT = 16, /* test hook of the panel kernel: one warp withholds its first
                                     stage arrival and waits 2 ms instead of 2 s, so that the
                                     path of a lost stage wait runs; the call must then return
                                     EVOCG_ETIMEOUT (host pointers) and the handle's error word
                                     is cleared by that report */
    EVOCG_SPMV_ROWELL = 64,        /* run the row-ELL kernel (the default for tiles of 64 that
                                     hold at most 1.5 entries per nonempty tile row): each row
                                     block's entries laid out by row, lanes owning rows */
    EVOCG_SPMV_ROWBLOCK = 32       /* run the row-block kernel (the default for tiles of 32): a
                                     warp per row block, lane l owning row l; regular tiles from
                                     16-byte descriptors, the single-entry tiles of the row block
                                     from a row-owned ELL block; the next row block's tile
                                     slices prefetched into L2 */
};

/*
 * evocg_spmv with flags (EVOCG_SPMV_*). With EVOCG_SPMV_REUSE_XCOPIES the call is exactly
 * one SpMV kernel launch, which repeated products with one x and kernel timing use.
 * x, y: DEVICE pointers when EVOCG_SPMV_REUSE_XCOPIES is set (EINVAL otherwise, and also
 * when no earlier call on the handle made the copies); otherwise as evocg_spmv.
 */
int evocg_spmv_ex(evocg_tiles_t A, const double *x, double *y, int flags, void *stream);

/*
 * evocg_spmv without any memory allocation. The EvoCG paper has no counterpart: this entry
 * point exists for callers that must not have the library allocate at call time (device
 * allocation can synchronise the whole GPU, is not allowed while a stream is being captured
 * into a graph, and is off limits to programs that hand out all device memory from their
 * own pool or run under a fixed budget). It computes the same product as evocg_spmv, with
 * the rounded copies of x kept in a fixed 8 MiB array that is part of the loaded library
 * (reserved on every GPU that loads it, until the process exits) instead of library-owned
 * buffers.
 *   x, y: DEVICE pointers, n FP64 each, not overlapping. n must be at most 1,048,576
 *   (EINVAL otherwise, with a message naming the limit).
 * The first call on a device looks up that array's device address (cudaGetSymbolAddress),
 * once per device and CUDA context (again after a cudaDeviceReset, which loads the library's
 * module anew); make that first call before any stream capture. Every call shares the
 * one array and overwrites all of it that it reads, so no state carries over between calls,
 * but calls that may overlap on the GPU (concurrent streams, or several handles at once)
 * race on it: order them. It runs only SpMV kernels without device-side waits (the
 * row-block kernel for tiles of 32, the direct kernel for the other sizes), so no stage
 * wait can run out unreported. Asynchronous on `stream`.
 */
int evocg_spmv_noalloc(evocg_tiles_t A, const double *x, double *y, void *stream);

/*
 * CG (jacobi = 0) or Jacobi-preconditioned CG (jacobi = 1) for A x = b from x0 = 0, in
 * the order of EvoCG Algorithm 1 (the solver lines) and §4.6:
 *   controller on p_k when k % kstar == 0; q = A~ p; sigma = p.q (breakdown unless
 *   finite and > 0); alpha = rho / sigma; x += alpha p; r -= alpha q;
 *   res_hist[k+1] = ||r|| / ||r_0||; stop when <= rtol (the recursively updated residual,
 *   §4.1); z = D^-1 r (or r); rho' = r.z; beta = rho'/rho; p = z + beta p.
 * All vector arithmetic is FP64; only the SpMV follows the precision map. The whole loop
 * runs on the device as one CUDA graph with a conditional while node: no host round trip
 * per iteration.
 *   b: host or device, n FP64. x: host or device, n FP64 (output; x0 = 0).
 *   rtol > 0 or 0 (run maxit iterations); maxit >= 0.
 *   ctrl: NULL = static map (the map set last); otherwise a controller.
 *   finish_fp64: after a recursive convergence, recompute ||b - A x|| in FP64; if above
 *   rtol, continue from r = b - A x with every tile in FP64 (up to 8 restarts).
 *   res_hist: host or device, maxit+1 FP64 entries, or NULL; entries past iters are
 *   left untouched.
 *   info: host pointer or NULL.
 * Returns OK on convergence, ENOTCONV at maxit, EBREAKDOWN, or an error. Synchronises
 * `stream` before returning. Jacobi needs every diagonal entry present and > 0 (EINVAL).
 */
int evocg_cg_solve(evocg_tiles_t A, const double *b, double *x, double rtol, int maxit,
                   int jacobi, const evocg_ctrl *ctrl, int finish_fp64, double *res_hist,
                   evocg_solve_info *info, void *stream);

/*
 * One controller decision (EvoCG Eq. 8-10, §4.7) on a given vector p, for controller
 * parity checks: cb_prec[i] for each column block i of A. p: host or device, n FP64.
 * cb_prec: host or device, nrb bytes. logits: NULL or host/device 3*nrb FP32 (MLP only).
 * Synchronises the stream for host outputs.
 */
int evocg_ctrl_decide(evocg_tiles_t A, const evocg_ctrl *ctrl, const double *p,
                      uint8_t *cb_prec, float *logits, void *stream);

/*
 * Choose the reuse interval K* of EvoCG §3.4 (interval reuse scheduling) from a per-iteration
 * log of column-block decisions (rows x ncb bytes, HOST, codes 0/1/2, row k = the map of
 * iteration k, as evocg_ctrl.map_log records it with kstar = 1). An upward transition is a
 * block whose code drops from row k-1 to row k (a higher precision). Reusing the decisions
 * of every K-th iteration puts row K*floor(k/K) in force at iteration k; the transition is
 * delayed when that row's code for the block is above row k's. For K = 1, 2, 4, ... up to
 * the largest power of two <= rows, fractions[i] receives (delayed upward transitions) /
 * (upward transitions), 0 when there are none; *kstar receives the largest K whose fraction
 * is below `limit` (the paper: 0.1); K = 1 always qualifies.
 *   fractions: NULL or room for max_candidates doubles; *ncand (may be NULL) receives the
 *   number of candidates examined. A host-only computation: no GPU is needed.
 * Errors: EINVAL (NULL log or kstar with rows > 0, ncb < 1, rows < 0, a code above 2).
 */
int evocg_kstar_select(const uint8_t *map_log, int64_t rows, int64_t ncb, double limit,
                       int *kstar, double *fractions, int max_candidates, int *ncand);

/*
 * The device's FP64 -> FP32 and FP64 -> BF16 rounding (integer-pipe, round to nearest
 * even, one rounding from FP64), exposed for rounding checks. x: host or device, n FP64;
 * out32 (FP32) / out16 (BF16 bit patterns): host or device, may be NULL.
 */
int evocg_round(const double *x, int64_t n, float *out32, uint16_t *out16, void *stream);

/* Message for the calling thread's last failed call ("" if none). */
const char *evocg_last_error(void);

/* Library ABI version (increases on incompatible changes). */
int evocg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EVOCG_H */
