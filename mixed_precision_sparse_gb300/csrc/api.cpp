// api.cpp -- the C ABI of libevocg.so (declared in include/evocg.h): argument checks,
// device memory, host<->device staging, and the CUDA-graph loop driver of the CG solve
// (EvoCG, "Self-Evolving Precision Control for Faster Conjugate Gradient", §3.4: the
// SpMV and the fused step replayed as a graph; here the whole loop is one graph with a
// conditional while node, so no host round trip happens per iteration).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "evocg_internal.h"

using namespace evocg;

namespace evocg {

static thread_local std::string g_err;

void set_error(const std::string &msg) { g_err = msg; }

int fail(int code, const std::string &msg)
{
    g_err = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    g_err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return e == cudaErrorMemoryAllocation ? EVOCG_ENOMEM : EVOCG_ECUDA;
}

}  // namespace evocg

#define CK(call, what)                                       \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
    } while (0)

namespace {

bool is_device_ptr(const void *p)
{
    if (!p) return false;
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

template <class T>
cudaError_t dalloc(T **p, int64_t count)
{
    *p = nullptr;
    if (count <= 0) count = 1;
    // kSlack bytes past the end: the SpMV stages arrays in 16-byte granules
    return cudaMalloc((void **)p, sizeof(T) * (size_t)count + kSlack);
}

template <class T>
void dfree(T *&p)
{
    if (p) cudaFree((void *)p);
    p = nullptr;
}

int check_device(int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail(e, "no usable CUDA device (cudaGetDevice)");
        return EVOCG_EDEVICE;
    }
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(EVOCG_EDEVICE, "this library is built for sm_103a (GB300); device is sm_" +
                                       std::to_string(prop.major) + std::to_string(prop.minor));
    *sms = prop.multiProcessorCount;
    return EVOCG_OK;
}

void release_graphs(SolveWS &w)
{
    if (w.exec) cudaGraphExecDestroy(w.exec);
    if (w.graph) cudaGraphDestroy(w.graph);
    if (w.exec_rs) cudaGraphExecDestroy(w.exec_rs);
    if (w.graph_rs) cudaGraphDestroy(w.graph_rs);
    w.exec = nullptr; w.graph = nullptr; w.exec_rs = nullptr; w.graph_rs = nullptr;
}

void release_ws(SolveWS &w)
{
    release_graphs(w);
    dfree(w.b); dfree(w.x); dfree(w.r); dfree(w.p); dfree(w.q); dfree(w.z); dfree(w.hist);
    dfree(w.partials); dfree(w.pq); dfree(w.cbPrec); dfree(w.mlpW); dfree(w.st); dfree(w.logbuf);
    if (w.st_host) cudaFreeHost(w.st_host);
    w.st_host = nullptr;
    w.cap_n = 0; w.cap_hist = 0; w.cap_ncb = 0; w.cap_mlp = 0; w.cap_log = 0;
}

int ensure_ws(evocg_tiles *A, int maxit)
{
    SolveWS &w = A->ws;
    if (w.cap_n < A->n || w.cap_ncb < A->nrb || w.st == nullptr) {
        release_ws(w);
        const int64_t n = A->n;
        CK(dalloc(&w.b, n), "cudaMalloc b");
        CK(dalloc(&w.x, n), "cudaMalloc x");
        CK(dalloc(&w.r, n), "cudaMalloc r");
        CK(dalloc(&w.p, n), "cudaMalloc p");
        CK(dalloc(&w.q, n), "cudaMalloc q");
        CK(dalloc(&w.z, n), "cudaMalloc z");
        CK(dalloc(&w.partials, 2 * kMaxBlocks), "cudaMalloc partials");
        CK(dalloc(&w.pq, kMaxPq), "cudaMalloc p.q partials");
        CK(dalloc(&w.cbPrec, A->nrb), "cudaMalloc cbPrec");
        CK(dalloc(&w.st, 1), "cudaMalloc state");
        CK(cudaMemset(w.st, 0, sizeof(DevState)), "cudaMemset state");
        CK(cudaMallocHost((void **)&w.st_host, sizeof(DevState)), "cudaMallocHost state");
        w.cap_n = n;
        w.cap_ncb = A->nrb;
        w.cap_hist = 0;
        w.cap_mlp = 0;
    }
    if (w.cap_hist < maxit + 1) {
        release_graphs(w);
        dfree(w.hist);
        int cap = maxit + 1 < 1024 ? 1024 : maxit + 1;
        CK(dalloc(&w.hist, cap), "cudaMalloc history");
        w.cap_hist = cap;
    }
    return EVOCG_OK;
}

int upload_mlp(evocg_tiles *A, const evocg_ctrl *c, int *H1, int *H2)
{
    if (!c->weights) return fail(EVOCG_EINVAL, "MLP controller needs weights");
    if (c->hidden1 < 1 || c->hidden1 > kMlpHiddenMax || c->hidden2 < 1 || c->hidden2 > kMlpHiddenMax)
        return fail(EVOCG_EINVAL, "MLP hidden widths must be in [1, 64]");
    if (!(c->delta >= 0.0)) return fail(EVOCG_EINVAL, "MLP delta must be >= 0");
    const int64_t T = A->T, h1 = c->hidden1, h2 = c->hidden2;
    const int64_t words = mlp_staged_words((int)T);   // the kernel's staged layout
    if (words <= 0) return fail(EVOCG_EINVAL, "MLP controller needs tiles of 16, 32 or 64");
    std::vector<float> staged;
    try {
        staged.resize((size_t)words);
    } catch (const std::bad_alloc &) {
        return fail(EVOCG_ENOMEM, "host allocation for the mlp weights");
    }
    mlp_stage_weights(c->weights, (int)T, (int)h1, (int)h2, staged.data());
    SolveWS &w = A->ws;
    if (w.cap_mlp < words) {
        release_graphs(w);  // the graphs hold the weight pointer
        dfree(w.mlpW);
        CK(dalloc(&w.mlpW, words), "cudaMalloc mlp weights");
        w.cap_mlp = words;
    }
    CK(cudaMemcpy(w.mlpW, staged.data(), sizeof(float) * (size_t)words, cudaMemcpyHostToDevice),
       "copy mlp weights");
    *H1 = (int)h1;
    *H2 = (int)h2;
    return EVOCG_OK;
}

// force64: the loop's SpMV runs its all-FP64 variant (the FP64 finish, or a static map whose
// codes are all FP64: the same products without reading a precision code)
int build_graph(CgLaunch L, int restart, int force64, cudaGraph_t *graph_out, cudaGraphExec_t *exec_out)
{
    cudaStream_t cs = nullptr;
    CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking), "cudaStreamCreate (capture)");
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ex = nullptr;
    int rc = EVOCG_OK;
    cudaError_t e = cudaGraphCreate(&g, 0);
    cudaGraphConditionalHandle h = 0;
    if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&h, g, 1u, cudaGraphCondAssignDefault);
    if (e == cudaSuccess) {
        L.cond = h;
        L.use_cond = 1;
        e = cudaStreamBeginCaptureToGraph(cs, g, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    }
    bool capturing = (e == cudaSuccess);
    if (e == cudaSuccess && restart) {
        // q = A x with every tile in FP64, for r = b - A x
        SpmvLaunch S{};
        S.A = L.A; S.x64 = L.x; S.y = L.q; S.force64 = 1; S.dot = 0; S.st = L.st;
        S.census = 0; S.grid = L.spmv_grid;
        e = launch_spmv(S, cs);
    }
    if (e == cudaSuccess && !restart && L.ctrl == EVOCG_CTRL_THRESHOLD && L.eps_relative)
        e = launch_threshold_scale(L, cs);
    if (e == cudaSuccess) e = launch_cg_init(L, restart, cs);
    // cudaGraphNodeParams has no default constructor in C++ (a union member has one);
    // zeroed storage is its documented initial state.
    alignas(cudaGraphNodeParams) unsigned char np_storage[sizeof(cudaGraphNodeParams)];
    std::memset(np_storage, 0, sizeof(np_storage));
    cudaGraphNodeParams &np = *reinterpret_cast<cudaGraphNodeParams *>(np_storage);
    if (e == cudaSuccess) {
        cudaStreamCaptureStatus cst;
        const cudaGraphNode_t *deps = nullptr;
        size_t ndeps = 0;
        e = cudaStreamGetCaptureInfo(cs, &cst, nullptr, nullptr, &deps, nullptr, &ndeps);
        if (e == cudaSuccess) {
            np.type = cudaGraphNodeTypeConditional;
            np.conditional.handle = h;
            np.conditional.type = cudaGraphCondTypeWhile;
            np.conditional.size = 1;
            cudaGraphNode_t wn;
            e = cudaGraphAddNode(&wn, g, deps, nullptr, ndeps, &np);
            if (e == cudaSuccess)
                e = cudaStreamUpdateCaptureDependencies(cs, &wn, nullptr, 1,
                                                        cudaStreamSetCaptureDependencies);
        }
    }
    if (capturing) {
        cudaGraph_t gg = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(cs, &gg);
        if (e == cudaSuccess) e = e2;
    }
    if (e == cudaSuccess) {
        cudaGraph_t body = np.conditional.phGraph_out[0];
        e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
        if (e == cudaSuccess) {
            cudaError_t e1 = launch_cg_body(L, force64, cs);
            cudaGraph_t bb = nullptr;
            cudaError_t e2 = cudaStreamEndCapture(cs, &bb);
            e = (e1 != cudaSuccess) ? e1 : e2;
        }
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&ex, g, 0);
    if (e != cudaSuccess) {
        rc = cuda_fail(e, "building the CG graph");
        if (ex) cudaGraphExecDestroy(ex);
        if (g) cudaGraphDestroy(g);
        ex = nullptr;
        g = nullptr;
    }
    cudaStreamDestroy(cs);
    *graph_out = g;
    *exec_out = ex;
    return rc;
}

// The same kernels as the graph, launched one by one, with the stop flag read back every
// kPlainBatch iterations (kernels queued after the stop return at once). Selected with
// EVOCG_GRAPH=0 in the environment; profilers that cannot see inside graphs with
// conditional nodes list every kernel of the solve this way.
constexpr int kPlainBatch = 32;

int run_plain(evocg_tiles *A, CgLaunch L, int restart, int force64, cudaStream_t s)
{
    SolveWS &w = A->ws;
    L.use_cond = 0;
    L.cond = 0;
    if (restart) {
        SpmvLaunch S{};
        S.A = L.A; S.x64 = L.x; S.y = L.q; S.force64 = 1; S.dot = 0; S.st = L.st;
        S.census = 0; S.grid = L.spmv_grid;
        CK(launch_spmv(S, s), "spmv (restart)");
    }
    if (!restart && L.ctrl == EVOCG_CTRL_THRESHOLD && L.eps_relative)
        CK(launch_threshold_scale(L, s), "threshold scale");
    CK(launch_cg_init(L, restart, s), "cg init");
    for (;;) {
        CK(cudaMemcpyAsync(w.st_host, w.st, sizeof(DevState), cudaMemcpyDeviceToHost, s), "read state");
        CK(cudaStreamSynchronize(s), "synchronise");
        if (w.st_host->done) break;
        for (int i = 0; i < kPlainBatch; ++i) CK(launch_cg_body(L, force64, s), "cg body");
    }
    return EVOCG_OK;
}

bool graphs_enabled()
{
    const char *v = std::getenv("EVOCG_GRAPH");
    return !(v && v[0] == '0');
}

}  // namespace

// --------------------------------------------------------------------------------------

extern "C" int evocg_version(void) { return 2; }

extern "C" const char *evocg_last_error(void) { return g_err.c_str(); }

extern "C" int evocg_tile_build(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                const double *vals, int tile_size, evocg_tiles_t *out)
{
    g_err.clear();
    if (!out) return fail(EVOCG_EINVAL, "out is NULL");
    *out = nullptr;
    int sms = 0;
    int rc = check_device(&sms);
    if (rc) return rc;
    if (is_device_ptr(row_ptr) || is_device_ptr(col_idx) || is_device_ptr(vals))
        return fail(EVOCG_EINVAL, "evocg_tile_build takes host CSR arrays");
    HostTiles H;
    std::string err;
    rc = build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return fail(rc, err);
    evocg_tiles *A = new (std::nothrow) evocg_tiles();
    if (!A) { H.release(); return fail(EVOCG_ENOMEM, "host allocation"); }
    cudaGetDevice(&A->device);
    A->sms = sms;
    A->n = H.n; A->nrb = H.nrb; A->ntiles = H.ntiles; A->nnz = H.nnz; A->nslots = H.nslots; A->T = H.T;
    A->diag_ok = H.diag_ok;
    cudaError_t e = cudaSuccess;
    auto up = [&](auto **dst, const auto *src, int64_t count) {
        if (e != cudaSuccess) return;
        e = dalloc(dst, count);
        if (e == cudaSuccess && count > 0)
            e = cudaMemcpy(*dst, src, sizeof(**dst) * (size_t)count, cudaMemcpyHostToDevice);
    };
    up(&A->tileRowPtr, H.tileRowPtr, H.nrb + 1);
    up(&A->tileColIdx, H.tileColIdx, H.ntiles);
    up(&A->tileNnzOff, H.tileNnzOff, H.ntiles + 1);
    up(&A->tileRowIdx, H.tileRowIdx, H.ntiles);
    up(&A->rowMask, H.rowMask, H.ntiles);
    up(&A->tileWidth, H.tileWidth, H.ntiles);
    up(&A->colIdx, H.colIdx, H.nslots);
    up(&A->v64, H.v64, H.nslots);
    up(&A->v32, H.v32, H.nslots);
    up(&A->v16, H.v16, H.nslots);
    up(&A->colExp, H.colExp, H.n);
    up(&A->dinv, H.dinv, H.n);
    // panel SpMV plan (tiles of 16 or 32)
    if (e == cudaSuccess && H.nrb > 0) {
        int variant = 0;
        if (const char *v = std::getenv("EVOCG_PANEL_VARIANT")) variant = std::atoi(v);
        if (variant < 0 || variant >= kPanelVariants) variant = 0;
        const int pg = panel_grid_for(H.T, sms, variant);
        if (pg > 0) {
            PanelPlan pl;
            std::string why;
            const int64_t warps = (int64_t)pg * (kPanelThreads / 32);
            const int sb = panel_stage_bytes(variant);
            if (panel_plan(H, warps, sb, &pl, &why) && panel_plan_ok(H, warps, sb, pl, &why) &&
                pl.panelRec.back() < INT32_MAX) {
                A->panel_variant = variant;
                A->nrec = pl.panelRec.back();
                try {   // every tile's record, for the record-ordered precision map
                    A->tileRec.assign((size_t)std::max<int64_t>(H.ntiles, 1), 0);
                    int64_t t = 0;
                    for (int64_t r = 0; r < A->nrec;) {
                        const int64_t nt = pl.desc[(size_t)r].x & 0xFFu;
                        for (int64_t i = 1; i <= nt; ++i) A->tileRec[(size_t)t++] = (int32_t)(r + i);
                        r += 1 + nt;
                    }
                } catch (const std::bad_alloc &) {
                    e = cudaErrorMemoryAllocation;
                }
                up(&A->pdesc, pl.desc.data(), (int64_t)pl.desc.size());
                up(&A->warpRec, pl.warpRec.data(), (int64_t)pl.warpRec.size());
                up(&A->panelRec, pl.panelRec.data(), (int64_t)pl.panelRec.size());
                if (e == cudaSuccess) e = dalloc(&A->recPrec, A->nrec + 32);
                if (e == cudaSuccess) e = cudaMemset(A->recPrec, 0, (size_t)(A->nrec + 32));
                A->panel_grid = pg;
            }
        }
    }
    // row-block SpMV plan (tiles of 32)
    if (e == cudaSuccess && H.nrb > 0 && H.T == 32) {
        RowBlockPlan P;
        std::string why;
        if (rowblock_plan(H, &P, &why) && rowblock_plan_ok(H, P, &why)) {
            up(&A->rbMeta, P.meta.data(), (int64_t)P.meta.size());
            up(&A->rgDesc, P.desc.data(), (int64_t)P.desc.size());
            up(&A->sgCol, P.sgCol.data(), (int64_t)P.sgCol.size());
            up(&A->sgTile, P.sgTile.data(), (int64_t)P.sgTile.size());
            up(&A->sgV64, P.sgV64.data(), (int64_t)P.sgV64.size());
            up(&A->sgV32, P.sgV32.data(), (int64_t)P.sgV32.size());
            up(&A->sgV16, P.sgV16.data(), (int64_t)P.sgV16.size());
            if (e == cudaSuccess) A->rb_grid = rowblock_grid_for(sms);
        }
    }
    // row-ELL SpMV plan (tiles of 64 holding about one entry per row)
    if (e == cudaSuccess && H.nrb > 0 && rowell_wanted(H)) {
        RowEllPlan P;
        std::string why;
        if (rowell_plan(H, &P, &why) && rowell_plan_ok(H, P, &why)) {
            A->el_slots = P.base.back();
            up(&A->elBase, P.base.data(), (int64_t)P.base.size());
            up(&A->elCol, P.col.data(), (int64_t)P.col.size());
            up(&A->elTile, P.tile.data(), (int64_t)P.tile.size());
            up(&A->elV64, P.v64.data(), (int64_t)P.v64.size());
            up(&A->elV32, P.v32.data(), (int64_t)P.v32.size());
            up(&A->elV16, P.v16.data(), (int64_t)P.v16.size());
            if (e == cudaSuccess) e = dalloc(&A->elPrec, A->el_slots);
            if (e == cudaSuccess) e = cudaMemset(A->elPrec, 0, (size_t)(A->el_slots > 0 ? A->el_slots : 1));
            if (e == cudaSuccess) A->el_grid = rowell_grid_for(sms);
        }
    }
    if (e == cudaSuccess) e = dalloc(&A->errw, 1);
    if (e == cudaSuccess) e = cudaMemset(A->errw, 0, sizeof(int));
    H.release();
    if (e == cudaSuccess) e = dalloc(&A->tilePrec, A->ntiles);
    if (e == cudaSuccess) e = cudaMemset(A->tilePrec, 0, (size_t)(A->ntiles > 0 ? A->ntiles : 1));
    if (e == cudaSuccess) e = dalloc(&A->cbPrec, A->nrb);
    if (e == cudaSuccess) e = cudaMemset(A->cbPrec, 0, (size_t)(A->nrb > 0 ? A->nrb : 1));
    if (e == cudaSuccess) e = dalloc(&A->x32, A->n);
    if (e == cudaSuccess) e = dalloc(&A->x16f, A->n);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        int code = cuda_fail(e, "uploading the tile structure");
        evocg_tiles_free(A);
        return code;
    }
    A->spmv_grid = spmv_grid_for(A->T, sms);
    // Default kernel: the row-block kernel where its plan exists, else the panel kernel where
    // its plan exists, else the direct one; EVOCG_SPMV_KERNEL=direct|panel|rowblock selects
    // another for every SpMV of the matrices built afterwards (where its plan exists).
    A->spmv_kind = SPMV_KIND_AUTO;
    if (const char *k = std::getenv("EVOCG_SPMV_KERNEL")) {
        if (!std::strcmp(k, "direct")) A->spmv_kind = SPMV_KIND_DIRECT;
        else if (!std::strcmp(k, "panel")) A->spmv_kind = SPMV_KIND_PANEL;
        else if (!std::strcmp(k, "rowblock")) A->spmv_kind = SPMV_KIND_ROWBLOCK;
        else if (!std::strcmp(k, "rowell")) A->spmv_kind = SPMV_KIND_ROWELL;
    }
    A->vec_grid = sms * 4 > kMaxBlocks ? kMaxBlocks : sms * 4;
    A->mlp_grid = mlp_grid_for(A->T, sms);
    *out = A;
    return EVOCG_OK;
}

extern "C" int evocg_tiles_free(evocg_tiles_t A)
{
    if (!A) return EVOCG_OK;
    cudaDeviceSynchronize();
    release_ws(A->ws);
    dfree(A->tileRowPtr); dfree(A->tileColIdx); dfree(A->tileNnzOff); dfree(A->tileRowIdx);
    dfree(A->rowMask); dfree(A->tileWidth);
    dfree(A->errw); dfree(A->pdesc); dfree(A->warpRec); dfree(A->panelRec); dfree(A->recPrec);
    dfree(A->rbMeta); dfree(A->rgDesc); dfree(A->sgCol); dfree(A->sgTile); dfree(A->sgV64);
    dfree(A->sgV32); dfree(A->sgV16);
    dfree(A->elBase); dfree(A->elCol); dfree(A->elTile); dfree(A->elPrec); dfree(A->elV64);
    dfree(A->elV32); dfree(A->elV16);
    dfree(A->colIdx); dfree(A->v64); dfree(A->v32); dfree(A->v16); dfree(A->colExp);
    dfree(A->tilePrec); dfree(A->cbPrec); dfree(A->dinv); dfree(A->x32); dfree(A->x16f);
    dfree(A->xstage); dfree(A->ystage);
    delete A;
    return EVOCG_OK;
}

extern "C" int evocg_tiles_info(evocg_tiles_t A, evocg_tiles_desc *d)
{
    if (!A || !d) return fail(EVOCG_EINVAL, "NULL argument");
    d->n = A->n; d->nrb = A->nrb; d->ntiles = A->ntiles; d->nnz = A->nnz; d->tile_size = A->T;
    d->map_kind = A->map_kind;
    d->nslots = A->nslots;
    d->bytes_index = 8 * (A->nrb + 1) + 4 * A->ntiles + 8 * (A->ntiles + 1) + 9 * A->ntiles +
                     A->nslots;
    d->bytes_v64 = 8 * A->nslots;
    d->bytes_v32 = 4 * A->nslots;
    d->bytes_v16 = 2 * A->nslots;
    d->bytes_colexp = A->n;
    return EVOCG_OK;
}

extern "C" int evocg_tiles_export(evocg_tiles_t A, int64_t *tileRowPtr, int32_t *tileColIdx,
                                  int64_t *tileNnzOff, uint64_t *rowMask, uint8_t *tileWidth,
                                  uint8_t *colIdx, double *v64, float *v32, uint16_t *v16,
                                  int8_t *colExp)
{
    if (!A) return fail(EVOCG_EINVAL, "NULL handle");
    CK(cudaDeviceSynchronize(), "synchronise");
    auto dn = [&](auto *dst, const auto *src, int64_t count) -> cudaError_t {
        if (!dst || count <= 0) return cudaSuccess;
        return cudaMemcpy(dst, src, sizeof(*dst) * (size_t)count, cudaMemcpyDeviceToHost);
    };
    CK(dn(tileRowPtr, A->tileRowPtr, A->nrb + 1), "export tileRowPtr");
    CK(dn(tileColIdx, A->tileColIdx, A->ntiles), "export tileColIdx");
    CK(dn(tileNnzOff, A->tileNnzOff, A->ntiles + 1), "export tileNnzOff");
    CK(dn(rowMask, A->rowMask, A->ntiles), "export rowMask");
    CK(dn(tileWidth, A->tileWidth, A->ntiles), "export tileWidth");
    CK(dn(colIdx, A->colIdx, A->nslots), "export colIdx");
    CK(dn(v64, A->v64, A->nslots), "export v64");
    CK(dn(v32, A->v32, A->nslots), "export v32");
    CK(dn(v16, A->v16, A->nslots), "export v16");
    CK(dn(colExp, A->colExp, A->n), "export colExp");
    return EVOCG_OK;
}

extern "C" int evocg_set_tile_precision(evocg_tiles_t A, const uint8_t *map, int64_t len,
                                        int map_kind, void *stream)
{
    g_err.clear();
    if (!A || (!map && len > 0)) return fail(EVOCG_EINVAL, "NULL argument");
    cudaStream_t s = (cudaStream_t)stream;
    int64_t want;
    if (map_kind == EVOCG_MAP_PER_TILE) want = A->ntiles;
    else if (map_kind == EVOCG_MAP_PER_COLBLOCK) want = A->nrb;
    else return fail(EVOCG_EINVAL, "unknown map kind");
    if (len != want)
        return fail(EVOCG_EINVAL, "map length " + std::to_string(len) + " != " + std::to_string(want));
    std::vector<uint8_t> h((size_t)(len > 0 ? len : 1));
    if (len > 0) {
        if (is_device_ptr(map)) {
            CK(cudaMemcpyAsync(h.data(), map, (size_t)len, cudaMemcpyDeviceToHost, s), "copy map");
            CK(cudaStreamSynchronize(s), "synchronise");
        } else {
            std::memcpy(h.data(), map, (size_t)len);
        }
        for (int64_t i = 0; i < len; ++i)
            if (h[(size_t)i] > 2)
                return fail(EVOCG_EINVAL, "precision code " + std::to_string(h[(size_t)i]) +
                                              " at " + std::to_string(i) + " (codes are 0, 1, 2)");
        uint8_t *dst = (map_kind == EVOCG_MAP_PER_TILE) ? A->tilePrec : A->cbPrec;
        CK(cudaMemcpyAsync(dst, h.data(), (size_t)len, cudaMemcpyHostToDevice, s), "upload map");
        std::vector<uint8_t> rp;
        if (map_kind == EVOCG_MAP_PER_TILE && A->recPrec) {   // the same map in record order
            rp.assign((size_t)(A->nrec + 32), 0);
            for (int64_t t = 0; t < len; ++t) rp[(size_t)A->tileRec[(size_t)t]] = h[(size_t)t];
            CK(cudaMemcpyAsync(A->recPrec, rp.data(), rp.size(), cudaMemcpyHostToDevice, s), "upload map");
        }
        if (map_kind == EVOCG_MAP_PER_TILE && A->elTile) {   // the per-slot copy of the row-ELL plan,
            // and its rows reordered by precision
            CK(launch_elprec(A->el_slots, A->elTile, A->tilePrec, A->elPrec, s), "per-slot map");
            CK(launch_elsort(A->nrb, A->elBase, A->elCol, A->elTile, A->elV64, A->elV32, A->elV16,
                             A->elPrec, s), "order row-ELL rows by precision");
        }
        CK(cudaStreamSynchronize(s), "synchronise");
    }
    A->map_kind = map_kind;
    A->map_all64 = 1;
    for (int64_t i = 0; i < len; ++i)
        if (h[(size_t)i] != EVOCG_FP64) { A->map_all64 = 0; break; }
    return EVOCG_OK;
}

extern "C" int evocg_get_tile_precision(evocg_tiles_t A, uint8_t *map_out, int64_t len, void *stream)
{
    if (!A || !map_out) return fail(EVOCG_EINVAL, "NULL argument");
    if (len != A->ntiles) return fail(EVOCG_EINVAL, "map length must be ntiles");
    cudaStream_t s = (cudaStream_t)stream;
    if (len == 0) return EVOCG_OK;
    if (A->map_kind == EVOCG_MAP_PER_COLBLOCK) {
        uint8_t *tmp = nullptr;
        CK(dalloc(&tmp, len), "cudaMalloc map");
        cudaError_t e = launch_broadcast_map(A->view(), A->cbPrec, tmp, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(map_out, tmp, (size_t)len, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        cudaFree(tmp);
        if (e != cudaSuccess) return cuda_fail(e, "broadcast map");
        return EVOCG_OK;
    }
    CK(cudaMemcpyAsync(map_out, A->tilePrec, (size_t)len, cudaMemcpyDeviceToHost, s), "copy map");
    CK(cudaStreamSynchronize(s), "synchronise");
    return EVOCG_OK;
}

extern "C" int evocg_spmv_ex(evocg_tiles_t A, const double *x, double *y, int flags, void *stream)
{
    g_err.clear();
    if (!A || (A->n > 0 && (!x || !y))) return fail(EVOCG_EINVAL, "NULL argument");
    const int kflags = flags & (EVOCG_SPMV_DIRECT | EVOCG_SPMV_PANEL | EVOCG_SPMV_ROWBLOCK | EVOCG_SPMV_ROWELL);
    if (flags & ~(EVOCG_SPMV_REUSE_XCOPIES | EVOCG_SPMV_DIRECT | EVOCG_SPMV_PANEL | EVOCG_SPMV_TEST_LOST_WAIT |
                  EVOCG_SPMV_ROWBLOCK | EVOCG_SPMV_ROWELL))
        return fail(EVOCG_EINVAL, "unknown flags");
    if (kflags & (kflags - 1)) return fail(EVOCG_EINVAL, "at most one kernel flag");
    if (A->n == 0) return EVOCG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const bool reuse = (flags & EVOCG_SPMV_REUSE_XCOPIES) != 0;
    const bool xdev = is_device_ptr(x), ydev = is_device_ptr(y);
    if (reuse && (!xdev || !ydev))
        return fail(EVOCG_EINVAL, "EVOCG_SPMV_REUSE_XCOPIES needs device x and y");
    const int kdirect = (flags & EVOCG_SPMV_DIRECT) ? 1 : 0;
    const int kkind = (flags & EVOCG_SPMV_PANEL) ? SPMV_KIND_PANEL : (flags & EVOCG_SPMV_ROWBLOCK) ? SPMV_KIND_ROWBLOCK
                      : (flags & EVOCG_SPMV_ROWELL) ? SPMV_KIND_ROWELL : 0;
    if (reuse && !A->xcopies_valid)
        return fail(EVOCG_EINVAL, "EVOCG_SPMV_REUSE_XCOPIES: no earlier SpMV made the copies");
    const size_t bytes = sizeof(double) * (size_t)A->n;
    const double *xd = x;
    double *yd = y;
    if (!xdev || !ydev) {
        if (!A->xstage) CK(dalloc(&A->xstage, A->n), "cudaMalloc staging");
        if (!A->ystage) CK(dalloc(&A->ystage, A->n), "cudaMalloc staging");
    }
    if (!xdev) {
        CK(cudaMemcpyAsync(A->xstage, x, bytes, cudaMemcpyHostToDevice, s), "copy x");
        xd = A->xstage;
    }
    if (!ydev) yd = A->ystage;
    if (!reuse) {
        CK(launch_xcopies(A->view(), xd, A->x32, A->x16f, A->vec_grid, s), "launch x copies");
        A->xcopies_valid = 1;
    }
    SpmvLaunch S{};
    S.A = A->view();
    S.x64 = xd; S.x32 = A->x32; S.x16f = A->x16f; S.y = yd;
    S.prec = (A->map_kind == EVOCG_MAP_PER_TILE) ? A->tilePrec : A->cbPrec;
    S.map_kind = A->map_kind;
    S.force64 = A->map_all64;   // an all-FP64 map: the same products without reading codes
    S.dot = 0; S.st = nullptr; S.census = 0; S.grid = A->spmv_grid;
    S.direct = kdirect;
    S.kind = kkind;
    S.test_lost_wait = (flags & EVOCG_SPMV_TEST_LOST_WAIT) ? 1 : 0;
    CK(launch_spmv(S, s), "launch spmv");
    if (!ydev) {
        int lost = 0;
        CK(cudaMemcpyAsync(y, yd, bytes, cudaMemcpyDeviceToHost, s), "copy y");
        CK(cudaMemcpyAsync(&lost, A->errw, sizeof(int), cudaMemcpyDeviceToHost, s), "read error word");
        CK(cudaStreamSynchronize(s), "synchronise");
        if (lost) {
            cudaMemsetAsync(A->errw, 0, sizeof(int), s);
            cudaStreamSynchronize(s);
            return fail(EVOCG_ETIMEOUT, "an SpMV stage wait ran out (its bulk copies did not complete)");
        }
    }
    return EVOCG_OK;
}

extern "C" int evocg_spmv(evocg_tiles_t A, const double *x, double *y, void *stream)
{
    return evocg_spmv_ex(A, x, y, 0, stream);
}

extern "C" int evocg_round(const double *x, int64_t n, float *out32, uint16_t *out16, void *stream)
{
    g_err.clear();
    if (n < 0 || (n > 0 && !x)) return fail(EVOCG_EINVAL, "bad arguments");
    if (n == 0) return EVOCG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    double *xd = nullptr;
    float *o32 = nullptr;
    uint16_t *o16 = nullptr;
    cudaError_t e = dalloc(&xd, n);
    if (e == cudaSuccess) e = dalloc(&o32, n);
    if (e == cudaSuccess) e = dalloc(&o16, n);
    if (e == cudaSuccess) e = cudaMemcpyAsync(xd, x, sizeof(double) * (size_t)n, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = launch_round(xd, n, o32, o16, s);
    if (e == cudaSuccess && out32) e = cudaMemcpyAsync(out32, o32, 4 * (size_t)n, cudaMemcpyDefault, s);
    if (e == cudaSuccess && out16) e = cudaMemcpyAsync(out16, o16, 2 * (size_t)n, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(xd); cudaFree(o32); cudaFree(o16);
    if (e != cudaSuccess) return cuda_fail(e, "evocg_round");
    return EVOCG_OK;
}

extern "C" int evocg_ctrl_decide(evocg_tiles_t A, const evocg_ctrl *ctrl, const double *p,
                                 uint8_t *cb_prec, float *logits, void *stream)
{
    g_err.clear();
    if (!A || !ctrl || (A->n > 0 && (!p || !cb_prec))) return fail(EVOCG_EINVAL, "NULL argument");
    if (A->n == 0) return EVOCG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    int rc = ensure_ws(A, 1);
    if (rc) return rc;
    SolveWS &w = A->ws;
    const size_t bytes = sizeof(double) * (size_t)A->n;
    CK(cudaMemcpyAsync(w.p, p, bytes, cudaMemcpyDefault, s), "copy p");
    float *dlog = nullptr;
    if (ctrl->kind == EVOCG_CTRL_THRESHOLD) {
        if (!(ctrl->eps >= 0.0)) return fail(EVOCG_EINVAL, "threshold eps must be >= 0");
        CK(launch_ctrl_threshold(A->view(), w.p, 0.1 * ctrl->eps, ctrl->eps, w.cbPrec, s), "threshold");
    } else if (ctrl->kind == EVOCG_CTRL_MLP) {
        int H1 = 0, H2 = 0;
        rc = upload_mlp(A, ctrl, &H1, &H2);
        if (rc) return rc;
        if (logits) CK(dalloc(&dlog, 3 * A->nrb), "cudaMalloc logits");
        cudaError_t e = launch_ctrl_mlp(A->view(), w.p, w.mlpW, H1, H2, ctrl->delta, w.cbPrec, dlog, nullptr, s);
        if (e != cudaSuccess) { cudaFree(dlog); return cuda_fail(e, "mlp"); }
    } else {
        return fail(EVOCG_EINVAL, "evocg_ctrl_decide needs a THRESHOLD or MLP controller");
    }
    cudaError_t e = cudaMemcpyAsync(cb_prec, w.cbPrec, (size_t)A->nrb, cudaMemcpyDefault, s);
    if (e == cudaSuccess && logits)
        e = cudaMemcpyAsync(logits, dlog, sizeof(float) * 3 * (size_t)A->nrb, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(dlog);
    if (e != cudaSuccess) return cuda_fail(e, "controller outputs");
    return EVOCG_OK;
}

extern "C" int evocg_cg_solve(evocg_tiles_t A, const double *b, double *x, double rtol, int maxit,
                              int jacobi, const evocg_ctrl *ctrl, int finish_fp64, double *res_hist,
                              evocg_solve_info *info, void *stream)
{
    g_err.clear();
    if (!A || (A->n > 0 && (!b || !x))) return fail(EVOCG_EINVAL, "NULL argument");
    if (!(rtol >= 0.0) || maxit < 0) return fail(EVOCG_EINVAL, "rtol must be >= 0 and maxit >= 0");
    if (jacobi && !A->diag_ok)
        return fail(EVOCG_EINVAL, "Jacobi needs every diagonal entry present and > 0");
    cudaStream_t s = (cudaStream_t)stream;
    const int kind = ctrl ? ctrl->kind : EVOCG_CTRL_STATIC;
    if (kind != EVOCG_CTRL_STATIC && kind != EVOCG_CTRL_THRESHOLD && kind != EVOCG_CTRL_MLP)
        return fail(EVOCG_EINVAL, "unknown controller kind");
    if (kind == EVOCG_CTRL_THRESHOLD && !(ctrl->eps >= 0.0))
        return fail(EVOCG_EINVAL, "threshold eps must be >= 0");
    const bool logging = kind != EVOCG_CTRL_STATIC && ctrl->map_log && ctrl->map_log_rows > 0 && A->nrb > 0;
    if (kind != EVOCG_CTRL_STATIC && ctrl->map_log_rows < 0)
        return fail(EVOCG_EINVAL, "map_log_rows must be >= 0");
    int rc = ensure_ws(A, maxit);
    if (rc) return rc;
    SolveWS &w = A->ws;
    // decision log: written on the device; a host log goes through a library buffer
    uint8_t *dlog = nullptr;
    const bool host_log = logging && !is_device_ptr(ctrl->map_log);
    const int64_t log_bytes = logging ? ctrl->map_log_rows * A->nrb : 0;
    if (logging) {
        if (host_log) {
            if (w.cap_log < log_bytes) {
                release_graphs(w);   // the graphs hold the buffer's address
                dfree(w.logbuf);
                CK(dalloc(&w.logbuf, log_bytes), "cudaMalloc decision log");
                w.cap_log = log_bytes;
            }
            CK(cudaMemcpy(w.logbuf, ctrl->map_log, (size_t)log_bytes, cudaMemcpyHostToDevice),
               "copy decision log");   // rows the solve does not reach keep their contents
            dlog = w.logbuf;
        } else {
            dlog = ctrl->map_log;
        }
    }
    int H1 = 0, H2 = 0;
    if (kind == EVOCG_CTRL_MLP) {
        rc = upload_mlp(A, ctrl, &H1, &H2);
        if (rc) return rc;
    }
    const int64_t n = A->n;
    const size_t bytes = sizeof(double) * (size_t)(n > 0 ? n : 0);

    CgLaunch L{};
    L.A = A->view();
    L.n = n; L.T = A->T; L.jacobi = jacobi ? 1 : 0; L.ctrl = kind; L.dinv = A->dinv;
    L.eps_relative = (kind == EVOCG_CTRL_THRESHOLD && ctrl->eps_relative) ? 1 : 0;
    L.b = w.b; L.x = w.x; L.r = w.r; L.p = w.p; L.q = w.q; L.z = w.z;
    L.x32 = A->x32; L.x16f = A->x16f; L.hist = w.hist; L.partials = w.partials; L.pq = w.pq;
    L.cbPrec = w.cbPrec;
    L.prec = (A->map_kind == EVOCG_MAP_PER_TILE) ? A->tilePrec : A->cbPrec;
    L.map_kind = A->map_kind;
    L.mlpW = w.mlpW; L.H1 = H1; L.H2 = H2; L.delta = (kind == EVOCG_CTRL_MLP) ? ctrl->delta : 0.0;
    L.st = w.st; L.vec_grid = A->vec_grid; L.spmv_grid = A->spmv_grid;
    L.upd_grid = A->sms * kUpdMinBlocks > kMaxBlocks ? kMaxBlocks : A->sms * kUpdMinBlocks;
    L.map_log = dlog;
    L.map_log_rows = logging ? ctrl->map_log_rows : 0;
    L.cond = 0;

    // a static map whose codes are all FP64 runs the SpMV's all-FP64 variant (same products)
    const int f64 = (kind == EVOCG_CTRL_STATIC && A->map_all64) ? 1 : 0;
    // graph cache: the key is every launch parameter (the handle aside) and the variant
    uint64_t key = 1469598103934665603ull;
    {
        const unsigned char *pb = reinterpret_cast<const unsigned char *>(&L);
        for (size_t i = 0; i < sizeof(L); ++i) key = (key ^ pb[i]) * 1099511628211ull;
        key = (key ^ (uint64_t)f64) * 1099511628211ull;
    }
    const bool use_graph = graphs_enabled();
    if (use_graph && (!w.exec || w.exec_key != key)) {
        if (w.exec) { cudaGraphExecDestroy(w.exec); w.exec = nullptr; }
        if (w.graph) { cudaGraphDestroy(w.graph); w.graph = nullptr; }
        rc = build_graph(L, 0, f64, &w.graph, &w.exec);
        if (rc) return rc;
        w.exec_key = key;
    }
    // state for this solve
    DevState &H = *w.st_host;
    std::memset(&H, 0, sizeof(DevState));
    H.rtol = rtol;
    H.maxit = maxit;
    H.kstar = (ctrl && ctrl->kstar > 1) ? ctrl->kstar : 1;
    H.eps_lo = (kind == EVOCG_CTRL_THRESHOLD) ? 0.1 * ctrl->eps : 0.0;
    H.eps_hi = (kind == EVOCG_CTRL_THRESHOLD) ? ctrl->eps : 0.0;
    CK(cudaMemcpyAsync(w.st, &H, sizeof(DevState), cudaMemcpyHostToDevice, s), "upload state");
    if (n > 0) CK(cudaMemcpyAsync(w.b, b, bytes, cudaMemcpyDefault, s), "copy b");
    A->xcopies_valid = 0;  // the solve reuses the copy buffers for p
    if (use_graph) {
        CK(cudaGraphLaunch(w.exec, s), "cudaGraphLaunch");
    } else {
        rc = run_plain(A, L, 0, f64, s);
        if (rc) return rc;
    }
    CK(cudaMemcpyAsync(w.st_host, w.st, sizeof(DevState), cudaMemcpyDeviceToHost, s), "read state");
    CK(cudaStreamSynchronize(s), "synchronise solve");

    int iters_rec = (H.converged) ? H.k : -1;
    int restarts = 0;
    double true_res = -1.0;
    if (finish_fp64 && n > 0) {
        for (;;) {
            CK(launch_true_residual(L, s), "true residual");
            CK(cudaMemcpyAsync(w.st_host, w.st, sizeof(DevState), cudaMemcpyDeviceToHost, s), "read state");
            CK(cudaStreamSynchronize(s), "synchronise true residual");
            true_res = H.tr_den > 0.0 ? std::sqrt(H.tr_num) / std::sqrt(H.tr_den) : std::sqrt(H.tr_num);
            if (!H.converged || true_res <= rtol || H.k >= maxit || restarts >= 8) break;
            // continue from the true residual with every tile in FP64
            CgLaunch R = L;
            R.ctrl = EVOCG_CTRL_STATIC;
            R.map_log = nullptr;   // the FP64 finish is not the controlled phase
            R.map_log_rows = 0;
            uint64_t rkey = key ^ 0x9E3779B97F4A7C15ull;
            if (use_graph && (!w.exec_rs || w.exec_rs_key != rkey)) {
                if (w.exec_rs) { cudaGraphExecDestroy(w.exec_rs); w.exec_rs = nullptr; }
                if (w.graph_rs) { cudaGraphDestroy(w.graph_rs); w.graph_rs = nullptr; }
                rc = build_graph(R, 1, 1, &w.graph_rs, &w.exec_rs);
                if (rc) return rc;
                w.exec_rs_key = rkey;
            }
            restarts++;
            if (use_graph) {
                CK(cudaGraphLaunch(w.exec_rs, s), "cudaGraphLaunch (restart)");
            } else {
                rc = run_plain(A, R, 1, 1, s);
                if (rc) return rc;
            }
            CK(cudaMemcpyAsync(w.st_host, w.st, sizeof(DevState), cudaMemcpyDeviceToHost, s), "read state");
            CK(cudaStreamSynchronize(s), "synchronise restart");
        }
        if (H.converged && true_res > rtol && H.status == EVOCG_OK) H.status = EVOCG_ENOTCONV;
    }
    const int k = H.k;
    int lost = 0;
    CK(cudaMemcpyAsync(&lost, A->errw, sizeof(int), cudaMemcpyDeviceToHost, s), "read error word");
    if (n > 0) CK(cudaMemcpyAsync(x, w.x, bytes, cudaMemcpyDefault, s), "copy x");
    if (res_hist) CK(cudaMemcpyAsync(res_hist, w.hist, sizeof(double) * (size_t)(k + 1), cudaMemcpyDefault, s), "copy history");
    if (host_log)
        CK(cudaMemcpyAsync(ctrl->map_log, dlog, (size_t)log_bytes, cudaMemcpyDeviceToHost, s), "copy decision log");
    CK(cudaStreamSynchronize(s), "synchronise outputs");
    if (info) {
        info->status = H.status;
        info->iters = k;
        info->iters_recursive = iters_rec;
        info->restarts = restarts;
        info->rel_res = (H.nr0 > 0.0) ? std::sqrt(H.rr) / H.nr0 : 0.0;
        info->true_res = true_res;
        info->prec_nnz[0] = (int64_t)H.census[0];
        info->prec_nnz[1] = (int64_t)H.census[1];
        info->prec_nnz[2] = (int64_t)H.census[2];
        info->ctrl_calls = (int64_t)H.ctrl_calls;
    }
    if (lost) {
        cudaMemsetAsync(A->errw, 0, sizeof(int), s);
        cudaStreamSynchronize(s);
        return fail(EVOCG_ETIMEOUT, "an SpMV stage wait ran out (bulk copies did not complete); "
                                    "the solve's results are not valid");
    }
    if (H.status == EVOCG_ENOTCONV) set_error("CG did not reach rtol within maxit");
    if (H.status == EVOCG_EBREAKDOWN) set_error("CG breakdown: p.Ap <= 0 or not finite");
    return H.status;
}
