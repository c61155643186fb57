// evocg_internal.h -- structures shared by the host driver and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "evocg.h"

namespace evocg {

constexpr int kMaxBlocks = 2048;      // upper bound of any grid here (partials buffers)
constexpr int kMaxPq = 16384;         // p.q partials of one SpMV (grid x warps at most)
constexpr int kVecThreads = 256;      // threads per block of the vector kernels
constexpr int kUpdMinBlocks = 3;      // resident blocks per SM of the CG update and p-update kernels (their grid)
constexpr int kSpmvThreads = 256;     // threads per block of the SpMV
constexpr int kSpmvMinBlocks = 4;     // resident blocks per SM the SpMV registers are budgeted for
constexpr int kMlpHiddenMax = 64;
constexpr int kSlack = 16;            // bytes past the end of every device array (16-byte copies)
constexpr int kPanelThreads = 128;    // threads per block of the panel SpMV
constexpr int kPanelVariants = 4;     // (tiles issued together, blocks per SM) variants built
constexpr int kRbThreads = 256;       // threads per block of the row-block SpMV
constexpr int kElThreads = 256;       // threads per block of the row-ELL SpMV

// Device-resident solver state; one per handle. Written by the last block of each
// reducing kernel, read by every block of the next kernel.
struct DevState {
    double rho;        // r.z of the current iterate
    double alpha, beta, sigma;
    double nr0;        // ||r_0|| = ||b||
    double rr;         // ||r_k||^2
    double rtol;
    double eps_lo, eps_hi;  // threshold rule cut points (0.1 eps, eps)
    double tr_num, tr_den;  // true-residual check
    int k;             // iterations done
    int maxit;
    int kstar;
    int done;          // 1: the loop stops
    int status;        // EVOCG_OK / ENOTCONV / EBREAKDOWN while running or done
    int converged;
    int xstep;         // 1: the last update formed a valid alpha, so x += alpha p is due
    unsigned int tickets[8];
    unsigned long long census[3];
    unsigned long long ctrl_calls;
};

// ticket slots
enum { TK_SPMV = 0, TK_UPDATE = 1, TK_INIT = 2, TK_TRUE = 3, TK_SCALE = 4 };

// Everything the SpMV reads from the tile structure.
struct TilesView {
    int64_t n, nrb, ntiles, nslots;
    int T;
    const int64_t *tileRowPtr;
    const int32_t *tileColIdx;
    const int64_t *tileNnzOff;  // first slot of every tile (ntiles + 1)
    const int32_t *tileRowIdx;  // row block of each tile (device-side helper, not exported)
    const uint64_t *rowMask;    // nonempty local rows of every tile
    const uint8_t *tileWidth;   // slots per nonempty row of every tile
    const uint8_t *colIdx;      // local column of every slot (T: a pad)
    const double *v64;
    const float *v32;
    const uint16_t *v16;
    const int8_t *colExp;
    int *err;          // error word: a panel-kernel stage wait that ran out sets it
    int spmv_kind;     // kernel launch_spmv runs by default (SPMV_KIND_*)
    // panel SpMV: batch stream (panel_plan.cpp), the first batch record of every warp's
    // contiguous range (warps + 1) and of every panel (nrb + 1), and the grid the plan was made
    // for (0: no plan)
    const uint4 *pdesc;
    const int64_t *warpRec;
    const int64_t *panelRec;
    const uint8_t *recPrec;   // a per-tile precision map in record order (0 at headers)
    int64_t nrec;             // records of the stream before its 32 closing records
    int panel_grid;
    int panel_variant;
    // row-block SpMV (tiles of 32): meta words (nrb + 1), regular-tile descriptors and the
    // single-entry tiles' ELL blocks (rowblock_plan.cpp); rb_grid 0: no plan
    const uint4 *rbMeta;
    const uint4 *rgDesc;
    const int32_t *sgCol;
    const int32_t *sgTile;
    const double *sgV64;
    const float *sgV32;
    const uint16_t *sgV16;
    int rb_grid;
    // row-ELL SpMV (tiles of 64 with about one entry per row): block bases (nrb + 1) and the
    // slots' columns, per-slot precision codes and values (rowell_plan.cpp); el_grid 0: no plan
    const int64_t *elBase;
    const int32_t *elCol;
    const uint8_t *elPrec;
    const double *elV64;
    const float *elV32;
    const uint16_t *elV16;
    int el_grid;
    int mlp_grid;             // grid of the policy kernel: its resident blocks on every SM
};

// SpMV kernels: the row-block kernel (spmv_rowblock.cu; tiles of 32), the row-ELL kernel
// (spmv_rowell.cu; tiles of 64 holding about one entry per row), the panel kernel
// (spmv_panel.cu; tiles of 16 and 32) and the direct kernel (spmv.cu: warp per row block,
// plain loads; any tile size). AUTO: the row-block or row-ELL kernel where its plan exists,
// else the panel kernel where its plan exists, else the direct one.
enum { SPMV_KIND_AUTO = 0, SPMV_KIND_DIRECT = 1, SPMV_KIND_PANEL = 3, SPMV_KIND_ROWBLOCK = 4, SPMV_KIND_ROWELL = 5 };

struct SolveWS {
    int64_t cap_n = 0, cap_ncb = 0;
    int cap_hist = 0;
    double *b = nullptr, *x = nullptr, *r = nullptr, *p = nullptr, *q = nullptr, *z = nullptr;
    double *hist = nullptr;
    double *partials = nullptr;       // 2 * kMaxBlocks
    double *pq = nullptr;             // kMaxPq p.q partials of the SpMV (per warp or per block)
    uint8_t *cbPrec = nullptr;        // controller decisions per column block
    uint8_t *logbuf = nullptr;        // device copy of a host decision log
    int64_t cap_log = 0;
    float *mlpW = nullptr;            // packed MLP weights on the device
    int64_t cap_mlp = 0;
    DevState *st = nullptr;
    DevState *st_host = nullptr;      // pinned mirror
    // cached graphs
    cudaGraphExec_t exec = nullptr;
    cudaGraph_t graph = nullptr;
    uint64_t exec_key = 0;
    cudaGraphExec_t exec_rs = nullptr;
    cudaGraph_t graph_rs = nullptr;
    uint64_t exec_rs_key = 0;
};

}  // namespace evocg

struct evocg_tiles {
    int device = 0;
    int sms = 0;
    int64_t n = 0, nrb = 0, ntiles = 0, nnz = 0, nslots = 0;
    int T = 0;
    int64_t *tileRowPtr = nullptr;
    int32_t *tileColIdx = nullptr;
    int64_t *tileNnzOff = nullptr;
    int32_t *tileRowIdx = nullptr;
    uint64_t *rowMask = nullptr;
    uint8_t *tileWidth = nullptr;
    uint8_t *colIdx = nullptr;
    double *v64 = nullptr;
    float *v32 = nullptr;
    uint16_t *v16 = nullptr;
    int8_t *colExp = nullptr;
    uint4 *pdesc = nullptr;        // panel SpMV plan (see TilesView)
    int64_t *warpRec = nullptr;
    int64_t *panelRec = nullptr;
    uint8_t *recPrec = nullptr;
    int64_t nrec = 0;
    std::vector<int32_t> tileRec;  // host: the record of every tile (for recPrec)
    int panel_grid = 0;
    int panel_variant = 0;
    uint4 *rbMeta = nullptr;       // row-block SpMV plan (see TilesView)
    uint4 *rgDesc = nullptr;
    int32_t *sgCol = nullptr;
    int32_t *sgTile = nullptr;
    double *sgV64 = nullptr;
    float *sgV32 = nullptr;
    uint16_t *sgV16 = nullptr;
    int rb_grid = 0;
    int64_t *elBase = nullptr;     // row-ELL SpMV plan (see TilesView)
    int32_t *elCol = nullptr;
    int32_t *elTile = nullptr;     // the tile of every slot (for the per-slot precision copy)
    uint8_t *elPrec = nullptr;
    double *elV64 = nullptr;
    float *elV32 = nullptr;
    uint16_t *elV16 = nullptr;
    int64_t el_slots = 0;
    int el_grid = 0;
    int mlp_grid = 0;
    int *errw = nullptr;           // device error word (a lost stage wait)
    int spmv_kind = 0;             // default SpMV kernel (SPMV_KIND_*)
    uint8_t *tilePrec = nullptr;   // per-tile map
    uint8_t *cbPrec = nullptr;     // per-column-block map
    int map_kind = EVOCG_MAP_PER_TILE;
    int map_all64 = 1;   // every code of the map set last is FP64: the FP64 kernel variants run
    double *dinv = nullptr;        // 1 / a_ii (Jacobi)
    int diag_ok = 0;               // every diagonal entry present and > 0
    // SpMV scratch: rounded x copies and host staging
    float *x32 = nullptr;
    float *x16f = nullptr;          // BF16 roundings held in FP32 containers
    double *xstage = nullptr, *ystage = nullptr;
    int xcopies_valid = 0;          // x32/x16f hold the copies of the last SpMV's x
    int spmv_grid = 0, vec_grid = 0;
    evocg::SolveWS ws;

    evocg::TilesView view() const
    {
        return evocg::TilesView{n, nrb, ntiles, nslots, T, tileRowPtr, tileColIdx, tileNnzOff,
                                tileRowIdx, rowMask, tileWidth, colIdx, v64, v32, v16, colExp,
                                errw, spmv_kind, pdesc, warpRec, panelRec, recPrec, nrec, panel_grid, panel_variant,
                                rbMeta, rgDesc, sgCol, sgTile, sgV64, sgV32, sgV16, rb_grid,
                                elBase, elCol, elPrec, elV64, elV32, elV16, el_grid, mlp_grid};
    }
};

namespace evocg {

// ---- host helpers (api.cpp) ----
void set_error(const std::string &msg);
int fail(int code, const std::string &msg);
int cuda_fail(cudaError_t e, const char *what);

// ---- tile builder (tile_build.cpp) ----
struct HostTiles {
    int64_t n = 0, nrb = 0, ntiles = 0, nnz = 0, nslots = 0;
    int T = 0;
    int64_t *tileRowPtr = nullptr;
    int32_t *tileColIdx = nullptr;
    int64_t *tileNnzOff = nullptr;
    int32_t *tileRowIdx = nullptr;
    uint64_t *rowMask = nullptr;
    uint8_t *tileWidth = nullptr;
    uint8_t *colIdx = nullptr;
    double *v64 = nullptr;
    float *v32 = nullptr;
    uint16_t *v16 = nullptr;
    int8_t *colExp = nullptr;
    double *dinv = nullptr;
    int diag_ok = 0;
    void release();
};
int build_host_tiles(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
                     HostTiles *out, std::string *err);

// ---- kernels (spmv.cu, cg.cu, ctrl.cu) ----
struct SpmvLaunch {
    TilesView A;
    const double *x64;
    const float *x32;
    const float *x16f;
    double *y;
    const uint8_t *prec;   // tilePrec (map_kind 0) or cbPrec (map_kind 1); ignored if force64
    int map_kind;
    int force64;
    // p.q for CG (dot != 0): the sum over rows of x_i y_i, as spmv_dot_partials() partials in
    // pq (one per warp, or one per block for the row-block and row-ELL kernels); the update kernel sums
    // them in order
    int dot;
    double *pq;
    double *partials;
    DevState *st;
    int census;            // accumulate per-precision stored-entry counts (pads excluded) into st->census
    int gate;              // return at once when st->done is set (a stopped solve)
    int grid;              // grid of the direct kernel
    int direct;            // 1: the direct kernel whatever the default
    int kind;              // SPMV_KIND_*: a kernel other than the matrix's default (0: default)
    int test_lost_wait;    // test hook of the panel kernel: one warp withholds its first stage
                           // arrival and waits 2 ms, so that the lost-wait path runs
};
// Kernel choice: L.direct, else L.kind, else the matrix's default; the panel kernel only when
// the view has its plan (else the direct one).
cudaError_t launch_spmv(const SpmvLaunch &L, cudaStream_t s);
// The kernel an SpMV with these flags runs on this matrix (SPMV_KIND_*).
int spmv_kind_for(const TilesView &A, int direct, int kind);
cudaError_t launch_spmv_direct(const SpmvLaunch &L, cudaStream_t s);
int spmv_dot_partials(const SpmvLaunch &L);   // warps that write a p.q partial
cudaError_t launch_spmv_panel(const SpmvLaunch &L, cudaStream_t s);
int panel_grid_for(int T, int sms, int variant);   // 0 if no panel kernel exists for T
int panel_stage_bytes(int variant);                // shared-memory stage of one warp
struct PanelPlan {
    std::vector<uint4> desc;        // the batch stream
    std::vector<int64_t> warpRec;   // warps + 1
    std::vector<int64_t> panelRec;  // nrb + 1
    uint32_t batches = 0;
};
bool panel_plan(const HostTiles &H, int64_t warps, int stage_bytes, PanelPlan *out, std::string *why);
bool panel_plan_ok(const HostTiles &H, int64_t warps, int stage_bytes, const PanelPlan &pl, std::string *why);
cudaError_t launch_spmv_rowblock(const SpmvLaunch &L, cudaStream_t s);
int rowblock_grid_for(int sms);
struct RowBlockPlan {
    std::vector<uint4> meta;      // nrb + 1: {first descriptor, first single slot, rows mask, width}
    std::vector<uint4> desc;      // regular tiles: {first slot, column block | width << 26, rows, tile}
    std::vector<int32_t> sgCol;   // single-entry tiles, row-owned ELL per row block (-1: pad)
    std::vector<int32_t> sgTile;
    std::vector<double> sgV64;
    std::vector<float> sgV32;
    std::vector<uint16_t> sgV16;
};
bool rowblock_plan(const HostTiles &H, RowBlockPlan *out, std::string *why);
bool rowblock_plan_ok(const HostTiles &H, const RowBlockPlan &P, std::string *why);
cudaError_t launch_spmv_rowell(const SpmvLaunch &L, cudaStream_t s);
int rowell_grid_for(int sms);
cudaError_t launch_elprec(int64_t ns, const int32_t *tile, const uint8_t *tilePrec, uint8_t *out, cudaStream_t s);
// Every row of the row-ELL blocks put in (precision, column) order (spmv_rowell.cu).
cudaError_t launch_elsort(int64_t nrb, const int64_t *base, int32_t *col, int32_t *tile, double *v64,
                          float *v32, uint16_t *v16, uint8_t *prec, cudaStream_t s);
struct RowEllPlan {
    std::vector<int64_t> base;    // nrb + 1: first slot of every row block's ELL block
    std::vector<int32_t> col;     // absolute column (-1: pad), slot (k, r) at base + k*T + r
    std::vector<int32_t> tile;
    std::vector<double> v64;
    std::vector<float> v32;
    std::vector<uint16_t> v16;
};
bool rowell_wanted(const HostTiles &H);   // tiles of 64 with at most 1.5 entries per nonempty tile row
bool rowell_plan(const HostTiles &H, RowEllPlan *out, std::string *why);
bool rowell_plan_ok(const HostTiles &H, const RowEllPlan &P, std::string *why);

cudaError_t launch_xcopies(const TilesView &A, const double *x, float *x32, float *x16f,
                           int grid, cudaStream_t s);
cudaError_t launch_round(const double *x, int64_t n, float *o32, uint16_t *o16, cudaStream_t s);
int spmv_grid_for(int T, int sms);   // also raises the kernels' shared-memory limit

struct CgLaunch {
    TilesView A;
    int64_t n;
    int T;
    int jacobi;
    int ctrl;              // EVOCG_CTRL_*
    int eps_relative;      // threshold cut points scaled by ||b||_inf before the first decision
    const double *dinv;
    double *b, *x, *r, *p, *q, *z;
    float *x32;
    float *x16f;
    double *hist;
    double *partials;
    double *pq;            // the SpMV's p.q partials (per warp or per block)
    uint8_t *cbPrec;       // controller output (map_kind 1 for the SpMV)
    const uint8_t *prec;   // static map
    int map_kind;
    const float *mlpW;
    int H1, H2;
    double delta;
    DevState *st;
    int vec_grid, spmv_grid;
    int upd_grid;          // grid of the update and p-update kernels (kUpdMinBlocks per SM)
    uint8_t *map_log;      // device decision log (NULL: none), map_log_rows x ncb
    int64_t map_log_rows;
    cudaGraphConditionalHandle cond;
    int use_cond;          // 1 inside the solve graph: the kernels drive its while node
};
cudaError_t launch_cg_init(const CgLaunch &L, int restart, cudaStream_t s);
cudaError_t launch_threshold_scale(const CgLaunch &L, cudaStream_t s);
cudaError_t launch_cg_body(const CgLaunch &L, int force64, cudaStream_t s);
cudaError_t launch_true_residual(const CgLaunch &L, cudaStream_t s);
cudaError_t launch_ctrl_threshold(const TilesView &A, const double *p, double eps_lo,
                                  double eps_hi, uint8_t *cbPrec, cudaStream_t s);
int mlp_grid_for(int T, int sms);   // resident policy-kernel blocks on every SM (0: none)
// The policy weights in the layout the kernel stages (W1 and W2 transposed, zero-padded to
// 64 outputs): mlp_staged_words(T) floats, written by mlp_stage_weights from the packed
// layout of evocg_ctrl.weights.
int64_t mlp_staged_words(int T);
void mlp_stage_weights(const float *packed, int T, int H1, int H2, float *out);
cudaError_t launch_ctrl_mlp(const TilesView &A, const double *p, const float *W, int H1,
                            int H2, double delta, uint8_t *cbPrec, float *logits,
                            const DevState *gate, cudaStream_t s);
cudaError_t launch_broadcast_map(const TilesView &A, const uint8_t *cbPrec, uint8_t *tilePrec,
                                 cudaStream_t s);

}  // namespace evocg
