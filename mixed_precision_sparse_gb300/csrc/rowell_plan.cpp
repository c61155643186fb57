// rowell_plan.cpp -- host plan of the row-ELL SpMV (spmv_rowell.cu), tiles of 64 holding about
// one entry per row.
//
// On GB300 the FP64 unit takes a warp instruction per 64 cycles of a sub-partition, so an
// SpMV whose lanes own rows must keep every lane busy in every FP64 instruction. With tiles
// that hold about one entry per nonempty row (a random banded matrix in 64 x 64 tiles: ~8
// entries per tile in ~8 rows), walking tile after tile leaves ~56 of a warp's 64 rows idle in
// each instruction. For such matrices the plan lays each row block's entries out by row
// instead: an ELL block of width W (the longest row of the row block), slot (k, r) at
// base + k*T + r holding row r's k-th entry in column order (its absolute column, its tile's
// index, and copies of the tile slot's three values), shorter rows padded with column -1.
// The tiles, their precision map and the Tile-CSC export are unchanged: a slot's precision is
// its tile's.
//
// elBase (nrb + 1): the first slot of every row block's block (W_rb * T slots each).
#include <algorithm>
#include <thread>

#include "evocg_internal.h"

namespace evocg {

namespace {

template <class F>
void parallel_blocks(int64_t count, F &&fn)
{
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 4, 64));
    nt = std::min<int64_t>(nt, std::max<int64_t>(1, count / 1024));
    if (nt <= 1) { fn(0, count); return; }
    std::vector<std::thread> th;
    th.reserve((size_t)nt);
    for (int64_t t = 0; t < nt; ++t) {
        const int64_t a = count * t / nt, b = count * (t + 1) / nt;
        th.emplace_back([&fn, a, b] { fn(a, b); });
    }
    for (auto &x : th) x.join();
}

// Entries per row of one row block, from its tiles' row masks and widths (an upper bound per
// row: w levels per row present; exact counts come from the pads).
void row_counts(const HostTiles &H, int64_t rb, int *cnt)
{
    const int T = H.T;
    for (int r = 0; r < T; ++r) cnt[r] = 0;
    for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {
        const uint64_t m = H.rowMask[t];
        const int h = __builtin_popcountll(m), w = H.tileWidth[t];
        const int64_t off = H.tileNnzOff[t];
        int j = 0;
        for (int r = 0; r < T; ++r) {
            if (!((m >> r) & 1ull)) continue;
            for (int k = 0; k < w; ++k)
                if (H.colIdx[off + (int64_t)k * h + j] < T) ++cnt[r];
            ++j;
        }
    }
}

}  // namespace

bool rowell_wanted(const HostTiles &H)
{
    if (H.T != 64 || H.ntiles == 0) return false;
    int64_t pairs = 0;   // nonempty (tile, row) pairs
    for (int64_t t = 0; t < H.ntiles; ++t) pairs += __builtin_popcountll(H.rowMask[t]);
    return pairs > 0 && (double)H.nnz <= 1.5 * (double)pairs;
}

bool rowell_plan(const HostTiles &H, RowEllPlan *out, std::string *why)
{
    if (H.T != 64) { *why = "row-ELL plan: tiles of 64 only"; return false; }
    const int T = H.T;
    const int64_t nrb = H.nrb;
    RowEllPlan P;
    try {
        std::vector<int64_t> width((size_t)nrb, 0);
        parallel_blocks(nrb, [&](int64_t a, int64_t b) {
            int cnt[64];
            for (int64_t rb = a; rb < b; ++rb) {
                row_counts(H, rb, cnt);
                int w = 0;
                for (int r = 0; r < T; ++r) w = std::max(w, cnt[r]);
                width[(size_t)rb] = w;
            }
        });
        P.base.assign((size_t)nrb + 1, 0);
        for (int64_t rb = 0; rb < nrb; ++rb) P.base[(size_t)rb + 1] = P.base[(size_t)rb] + width[(size_t)rb] * T;
        const int64_t ns = P.base[(size_t)nrb];
        if (ns >= ((int64_t)1 << 31)) { *why = "row-ELL plan: 2^31 slots or more"; return false; }
        if (H.n >= ((int64_t)1 << 29)) { *why = "row-ELL plan: n of 2^29 or more"; return false; }
        P.col.assign((size_t)ns, -1);
        P.tile.assign((size_t)ns, -1);
        P.v64.assign((size_t)ns, 0.0);
        P.v32.assign((size_t)ns, 0.0f);
        P.v16.assign((size_t)ns, 0);
        parallel_blocks(nrb, [&](int64_t a, int64_t b) {
            int k[64];
            for (int64_t rb = a; rb < b; ++rb) {
                for (int r = 0; r < T; ++r) k[r] = 0;
                const int64_t base = P.base[(size_t)rb];
                for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {   // ascending column blocks
                    const uint64_t m = H.rowMask[t];
                    const int h = __builtin_popcountll(m), w = H.tileWidth[t];
                    const int64_t off = H.tileNnzOff[t], cb = H.tileColIdx[t];
                    int j = 0;
                    for (int r = 0; r < T; ++r) {
                        if (!((m >> r) & 1ull)) continue;
                        for (int kk = 0; kk < w; ++kk) {   // ascending columns within the tile row
                            const int64_t s = off + (int64_t)kk * h + j;
                            if (H.colIdx[s] >= T) continue;
                            const size_t e = (size_t)(base + (int64_t)k[r]++ * T + r);
                            P.col[e] = (int32_t)(cb * T + H.colIdx[s]);
                            P.tile[e] = (int32_t)t;
                            P.v64[e] = H.v64[s];
                            P.v32[e] = H.v32[s];
                            P.v16[e] = H.v16[s];
                        }
                        ++j;
                    }
                }
            }
        });
    } catch (const std::bad_alloc &) {
        *why = "row-ELL plan: host allocation";
        return false;
    }
    *out = std::move(P);
    return true;
}

// Independent check against the tile structure: per row, the plan's entries are the row's
// stored entries of the tiles, in ascending column order, with their tiles and values; the
// rest of the row's slots are pads.
bool rowell_plan_ok(const HostTiles &H, const RowEllPlan &P, std::string *why)
{
    auto bad = [&](const std::string &m) { *why = "row-ELL plan: " + m; return false; };
    const int T = H.T;
    if (P.base.size() != (size_t)H.nrb + 1 || P.base[0] != 0) return bad("base");
    for (int64_t rb = 0; rb < H.nrb; ++rb) {
        const int64_t b0 = P.base[(size_t)rb], b1 = P.base[(size_t)rb + 1];
        if (b1 < b0 || (b1 - b0) % T) return bad("width of row block " + std::to_string(rb));
        const int64_t W = (b1 - b0) / T;
        std::vector<std::vector<int64_t>> rows((size_t)T);   // (column, tile, slot) per row
        std::vector<std::vector<int64_t>> slots((size_t)T);
        for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {
            const uint64_t m = H.rowMask[t];
            const int h = __builtin_popcountll(m), w = H.tileWidth[t];
            int j = 0;
            for (int r = 0; r < T; ++r) {
                if (!((m >> r) & 1ull)) continue;
                for (int kk = 0; kk < w; ++kk) {
                    const int64_t s = H.tileNnzOff[t] + (int64_t)kk * h + j;
                    if (H.colIdx[s] < T) { rows[(size_t)r].push_back(t); slots[(size_t)r].push_back(s); }
                }
                ++j;
            }
        }
        for (int r = 0; r < T; ++r) {
            const auto &tl = rows[(size_t)r];
            if ((int64_t)tl.size() > W) return bad("row " + std::to_string(rb * T + r) + " longer than its block");
            int64_t prev = -1;
            for (int64_t k = 0; k < W; ++k) {
                const size_t e = (size_t)(b0 + k * T + r);
                if (k >= (int64_t)tl.size()) {
                    if (P.col[e] != -1 || P.v64[e] != 0.0) return bad("pad of row " + std::to_string(rb * T + r));
                    continue;
                }
                const int64_t t = tl[(size_t)k], s = slots[(size_t)r][(size_t)k];
                const int64_t c = (int64_t)H.tileColIdx[t] * T + H.colIdx[s];
                if (P.col[e] != c || P.tile[e] != t || P.v64[e] != H.v64[s] || P.v32[e] != H.v32[s] ||
                    P.v16[e] != H.v16[s] || c <= prev)
                    return bad("entry " + std::to_string(k) + " of row " + std::to_string(rb * T + r));
                prev = c;
            }
        }
    }
    return true;
}

}  // namespace evocg

// Host-only: builds the tile structure and, when its tiles hold about one entry per row
// (tiles of 64), the row-ELL plan, and checks it. *valid = 1 when the plan exists and passes.
extern "C" int evocg_rowell_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                      const double *vals, int tile_size, int64_t *nslots,
                                      int *valid)
{
    evocg::set_error("");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    evocg::RowEllPlan P;
    std::string why = "row-ELL plan: the tiles are not sparse enough (more than 1.5 entries per tile row)";
    const bool ok = evocg::rowell_wanted(H) && evocg::rowell_plan(H, &P, &why) && evocg::rowell_plan_ok(H, P, &why);
    if (nslots) *nslots = ok ? P.base.back() : 0;
    if (valid) *valid = ok ? 1 : 0;
    if (!ok) evocg::set_error(why);
    H.release();
    return EVOCG_OK;
}
