// rowblock_plan.cpp -- host plan of the row-block SpMV (spmv_rowblock.cu), tiles of 32.
//
// The kernel gives one warp a row block at a time, lane l owning local row l, and reads
// two kinds of work from this plan:
//
//   regular tiles (two or more slots): one 16-byte descriptor each, in the row block's tile
//     order, {first slot, column block | width << 26, row mask, tile index}; the slots
//     themselves stay where the builder put them (16-slot aligned, a multiple of 16 long),
//     so that a tile's slices of the value streams and of the column bytes are copied
//     whole in 16-byte pieces;
//   single-entry tiles: on stencil matrices most tiles of a row block hold one entry (the
//     neighbour across a column-block edge: six of the nine tiles of a 9-point row block,
//     eighteen of the twenty-seven of a 27-point one), and a warp pass per such tile
//     would cost far more than its one entry. The plan gathers them per row block into a
//     small ELL block owned by the rows: the rows that have single-entry tiles (mask hs,
//     hc of them), each with up to ws of them in column order; slot (k, j) at
//     first + k*hc + j holds the k-th single of the j-th such row, with its absolute
//     column, its tile index and its value in the three streams (copies of the tile's
//     slot); shorter rows are padded with column -1.
//
// meta[rb] = {first descriptor, first single slot, hs, ws}; meta[nrb] closes both lists.
#include <algorithm>
#include <thread>

#include "evocg_internal.h"

namespace evocg {

namespace {

constexpr unsigned kCbBits = 26;

template <class F>
void parallel_rb(int64_t count, F &&fn)
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

bool single(const HostTiles &H, int64_t t)
{
    return H.tileWidth[t] == 1 && __builtin_popcountll(H.rowMask[t]) == 1;
}

// Singles geometry of one row block: per-row counts, the row mask and the width.
void singles_geo(const HostTiles &H, int64_t rb, unsigned *hs, unsigned *ws, int64_t *nreg)
{
    int cnt[32] = {0};
    *hs = 0; *ws = 0; *nreg = 0;
    for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {
        if (!single(H, t)) { ++*nreg; continue; }
        const int r = __builtin_ctzll(H.rowMask[t]);
        *hs |= 1u << r;
        *ws = std::max(*ws, (unsigned)++cnt[r]);
    }
}

}  // namespace

bool rowblock_plan(const HostTiles &H, RowBlockPlan *out, std::string *why)
{
    if (H.T != 32) { *why = "row-block plan: tiles of 32 only"; return false; }
    if (H.nslots >= ((int64_t)1 << 30) || H.ntiles >= ((int64_t)1 << 31) ||
        H.nrb >= ((int64_t)1 << kCbBits)) {
        *why = "row-block plan: 2^30 slots, 2^31 tiles or 2^26 row blocks or more";
        return false;
    }
    const int64_t nrb = H.nrb;
    RowBlockPlan P;
    try {
        std::vector<int64_t> nreg((size_t)nrb + 1, 0), nsg((size_t)nrb + 1, 0);
        std::vector<unsigned> hs((size_t)nrb, 0), ws((size_t)nrb, 0);
        parallel_rb(nrb, [&](int64_t a, int64_t b) {
            for (int64_t rb = a; rb < b; ++rb) {
                singles_geo(H, rb, &hs[(size_t)rb], &ws[(size_t)rb], &nreg[(size_t)rb]);
                nsg[(size_t)rb] = (int64_t)ws[(size_t)rb] * __builtin_popcount(hs[(size_t)rb]);
            }
        });
        std::vector<int64_t> reg0((size_t)nrb + 1, 0), sg0((size_t)nrb + 1, 0);
        for (int64_t rb = 0; rb < nrb; ++rb) {
            reg0[(size_t)rb + 1] = reg0[(size_t)rb] + nreg[(size_t)rb];
            sg0[(size_t)rb + 1] = sg0[(size_t)rb] + nsg[(size_t)rb];
        }
        if (reg0[(size_t)nrb] >= ((int64_t)1 << 32) || sg0[(size_t)nrb] >= ((int64_t)1 << 32)) {
            *why = "row-block plan: 2^32 descriptors or singles or more";
            return false;
        }
        const size_t nd = (size_t)reg0[(size_t)nrb], ns = (size_t)sg0[(size_t)nrb];
        P.meta.resize((size_t)nrb + 1);
        P.desc.resize(nd);
        P.sgCol.assign(ns, -1);
        P.sgTile.assign(ns, -1);
        P.sgV64.assign(ns, 0.0);
        P.sgV32.assign(ns, 0.0f);
        P.sgV16.assign(ns, 0);
        for (int64_t rb = 0; rb <= nrb; ++rb) {
            const bool last = rb == nrb;
            P.meta[(size_t)rb] = make_uint4((unsigned)reg0[(size_t)rb], (unsigned)sg0[(size_t)rb],
                                            last ? 0u : hs[(size_t)rb], last ? 0u : ws[(size_t)rb]);
        }
        parallel_rb(nrb, [&](int64_t a, int64_t b) {
            for (int64_t rb = a; rb < b; ++rb) {
                const unsigned h = hs[(size_t)rb];
                const int64_t hc = __builtin_popcount(h);
                int k[32] = {0};
                int64_t d = reg0[(size_t)rb];
                for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {
                    const int64_t s = H.tileNnzOff[t];
                    const uint32_t cb = (uint32_t)H.tileColIdx[t];
                    if (!single(H, t)) {
                        P.desc[(size_t)d++] = make_uint4((unsigned)s, cb | ((unsigned)H.tileWidth[t] << kCbBits),
                                                         (unsigned)H.rowMask[t], (unsigned)t);
                        continue;
                    }
                    const int r = __builtin_ctzll(H.rowMask[t]);
                    const int64_t j = __builtin_popcount(h & ((1u << r) - 1u));
                    const size_t e = (size_t)(sg0[(size_t)rb] + (int64_t)k[r]++ * hc + j);
                    P.sgCol[e] = (int32_t)((int64_t)cb * 32 + H.colIdx[s]);
                    P.sgTile[e] = (int32_t)t;
                    P.sgV64[e] = H.v64[s];
                    P.sgV32[e] = H.v32[s];
                    P.sgV16[e] = H.v16[s];
                }
            }
        });
    } catch (const std::bad_alloc &) {
        *why = "row-block plan: host allocation";
        return false;
    }
    *out = std::move(P);
    return true;
}

// Independent check of a plan against the tile structure: every tile of every row block is
// either the next regular descriptor (same slot, column block, width, mask and index) or a
// single at its ELL position with its column, index and values; every other single slot
// is a pad; the meta words close both lists.
bool rowblock_plan_ok(const HostTiles &H, const RowBlockPlan &P, std::string *why)
{
    auto bad = [&](const std::string &m) { *why = "row-block plan: " + m; return false; };
    if (P.meta.size() != (size_t)H.nrb + 1) return bad("meta size");
    if (P.meta.back().x != P.desc.size() || P.meta.back().y != P.sgCol.size()) return bad("closing meta");
    for (int64_t rb = 0; rb < H.nrb; ++rb) {
        const uint4 m = P.meta[(size_t)rb], m1 = P.meta[(size_t)rb + 1];
        const unsigned hc = (unsigned)__builtin_popcount(m.z);
        if (m1.y - m.y != hc * m.w || m1.x < m.x) return bad("lists of row block " + std::to_string(rb));
        std::vector<char> seen((size_t)(hc * m.w), 0);
        unsigned d = m.x;
        int cnt[32] = {0};
        for (int64_t t = H.tileRowPtr[rb]; t < H.tileRowPtr[rb + 1]; ++t) {
            const unsigned w = H.tileWidth[t];
            const int h = __builtin_popcountll(H.rowMask[t]);
            if (w * h >= 2) {
                if (d >= m1.x) return bad("descriptor count of row block " + std::to_string(rb));
                const uint4 q = P.desc[d++];
                if (q.x != (unsigned)H.tileNnzOff[t] || (q.y & ((1u << kCbBits) - 1)) != (unsigned)H.tileColIdx[t] ||
                    (q.y >> kCbBits) != w || q.z != (unsigned)H.rowMask[t] || q.w != (unsigned)t)
                    return bad("descriptor of tile " + std::to_string(t));
                if ((q.x & 15u) != 0) return bad("alignment of tile " + std::to_string(t));
                continue;
            }
            const int r = __builtin_ctzll(H.rowMask[t]);
            if (!((m.z >> r) & 1u)) return bad("row of single tile " + std::to_string(t));
            const unsigned j = (unsigned)__builtin_popcount(m.z & ((1u << r) - 1u));
            const unsigned k = (unsigned)cnt[r]++;
            if (k >= m.w) return bad("width of row block " + std::to_string(rb));
            const size_t e = (size_t)m.y + k * hc + j;
            seen[k * hc + j] = 1;
            const int64_t s = H.tileNnzOff[t];
            if (P.sgCol[e] != (int64_t)H.tileColIdx[t] * 32 + H.colIdx[s] || P.sgTile[e] != t ||
                P.sgV64[e] != H.v64[s] || P.sgV32[e] != H.v32[s] || P.sgV16[e] != H.v16[s] ||
                H.colIdx[s] >= 32)
                return bad("single tile " + std::to_string(t));
        }
        if (d != m1.x) return bad("descriptors of row block " + std::to_string(rb));
        for (size_t i = 0; i < seen.size(); ++i)
            if (!seen[i] && (P.sgCol[(size_t)m.y + i] != -1 || P.sgV64[(size_t)m.y + i] != 0.0))
                return bad("pad of row block " + std::to_string(rb));
    }
    return true;
}

}  // namespace evocg

// Host-only: builds the tile structure and the row-block plan for a CSR matrix and checks
// the plan. Returns EVOCG_OK with *valid = 1 (plan built and consistent) or 0 (no plan for
// this matrix: tiles other than 32, or a size limit).
extern "C" int evocg_rowblock_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                        const double *vals, int tile_size, int64_t *ndesc,
                                        int64_t *nsingle_slots, int *valid)
{
    evocg::set_error("");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    evocg::RowBlockPlan P;
    std::string why;
    const bool ok = evocg::rowblock_plan(H, &P, &why) && evocg::rowblock_plan_ok(H, P, &why);
    if (ndesc) *ndesc = ok ? (int64_t)P.desc.size() : 0;
    if (nsingle_slots) *nsingle_slots = ok ? (int64_t)P.sgCol.size() : 0;
    if (valid) *valid = ok ? 1 : 0;
    if (!ok) evocg::set_error(why);
    H.release();
    return EVOCG_OK;
}
