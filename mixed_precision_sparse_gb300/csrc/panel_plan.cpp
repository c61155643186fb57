// panel_plan.cpp -- the descriptor stream and the warp plan of the panel SpMV (spmv_panel.cu),
// made once per tile structure on the host.
//
// Stream: for every panel, in panel order, one header record {tiles in the panel, panel
// index, first slot (low, high 32 bits)} followed by one record per tile {slot offset from
// the panel's first slot, width w | (local column of a single-entry tile) << 8, column
// block, row mask}; the top 16 bits of the second word hold the tile's stored entries (at most
// 32 x 32). 32 zero records close the stream so that a warp's 32-record window
// never reads past it. Record r of panel p's tile i is at p + tileRowPtr[p] + 1 + i, so the
// kernel finds a tile's index (for a per-tile precision map) as r - p - 1.
//
// Plan: warps take consecutive panels, split where the running cost (one per slot, 16 per
// tile, 32 per panel) crosses multiples of total / warps.
#include <algorithm>

#include "evocg_internal.h"

namespace evocg {

bool panel_plan(const HostTiles &H, int64_t warps, std::vector<uint4> *desc,
                std::vector<int64_t> *warpRec, std::vector<int32_t> *warpPanel, std::string *why)
{
    if (H.T > 32) { *why = "panel plan: tiles wider than 32 are not planned here"; return false; }
    if (warps < 1) { *why = "panel plan: no warps"; return false; }
    const int64_t P = H.nrb;   // panels = row blocks for T <= 32
    if (H.ntiles + P >= ((int64_t)1 << 40)) { *why = "panel plan: too many tiles"; return false; }
    desc->assign((size_t)(P + H.ntiles + 32), make_uint4(0u, 0u, 0u, 0u));
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        const int64_t r = p + t0;
        const int64_t sbase = H.tileNnzOff[t0];
        (*desc)[(size_t)r] = make_uint4((unsigned)(t1 - t0), (unsigned)p, (unsigned)(uint64_t)sbase,
                                        (unsigned)((uint64_t)sbase >> 32));
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t off = H.tileNnzOff[t] - sbase;
            if (off >= ((int64_t)1 << 32)) { *why = "panel plan: a panel holds 2^32 slots or more"; return false; }
            const uint64_t m = H.rowMask[t];
            const unsigned w = H.tileWidth[t];
            const bool single = (w == 1u) && m && !(m & (m - 1u));
            const unsigned cs = single ? (unsigned)H.colIdx[H.tileNnzOff[t]] : 0u;
            unsigned nnz = 0;   // stored entries (slots that are not pads)
            for (int64_t s = H.tileNnzOff[t]; s < H.tileNnzOff[t + 1]; ++s) nnz += H.colIdx[s] < H.T;
            (*desc)[(size_t)(r + 1 + (t - t0))] =
                make_uint4((unsigned)off, w | (cs << 8) | (nnz << 16), (unsigned)H.tileColIdx[t],
                           (unsigned)m);
        }
    }
    // balanced contiguous panel ranges
    std::vector<int64_t> pre((size_t)P + 1, 0);
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        pre[(size_t)p + 1] = pre[(size_t)p] + (H.tileNnzOff[t1] - H.tileNnzOff[t0]) + 16 * (t1 - t0) + 32;
    }
    const int64_t total = pre[(size_t)P];
    warpPanel->assign((size_t)warps + 1, 0);
    warpRec->assign((size_t)warps + 1, 0);
    int64_t p = 0;
    for (int64_t w = 1; w < warps; ++w) {
        const int64_t target = (int64_t)((__int128)total * w / warps);
        while (p < P && pre[(size_t)p] < target) ++p;
        (*warpPanel)[(size_t)w] = (int32_t)p;
    }
    (*warpPanel)[(size_t)warps] = (int32_t)P;
    for (int64_t w = 0; w <= warps; ++w) {
        const int64_t q = (*warpPanel)[(size_t)w];
        (*warpRec)[(size_t)w] = q + H.tileRowPtr[q];
    }
    return true;
}

// What the panel kernel assumes of a plan, checked before it is uploaded: every record the
// kernel reads lies in the stream, headers and tile records match the tile structure, every
// slot a record names lies inside its tile's slots, single-entry columns are real entries,
// and the warp ranges tile the panels in order. A plan that fails is not used.
bool panel_plan_ok(const HostTiles &H, int64_t warps, const std::vector<uint4> &desc,
                   const std::vector<int64_t> &warpRec, const std::vector<int32_t> &warpPanel,
                   std::string *why)
{
    const int64_t P = H.nrb, T = H.T, R = T < 32 ? T : 32;
    auto bad = [&](const std::string &m) { *why = "panel plan check: " + m; return false; };
    if ((int64_t)desc.size() < P + H.ntiles + 32) return bad("stream too short");
    if ((int64_t)warpRec.size() != warps + 1 || (int64_t)warpPanel.size() != warps + 1)
        return bad("warp tables");
    if (warpPanel[0] != 0 || warpPanel[(size_t)warps] != P) return bad("warp ranges do not cover the panels");
    for (int64_t w = 0; w < warps; ++w) {
        const int64_t a = warpPanel[(size_t)w], b = warpPanel[(size_t)w + 1];
        if (b < a || a < 0 || b > P) return bad("warp ranges out of order");
        if (warpRec[(size_t)w] != a + H.tileRowPtr[a]) return bad("warp record index");
    }
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        const uint4 h = desc[(size_t)(p + t0)];
        const int64_t sbase = (int64_t)(((uint64_t)h.w << 32) | h.z);
        if ((int64_t)h.x != t1 - t0 || (int64_t)h.y != p || sbase != H.tileNnzOff[t0])
            return bad("header of panel " + std::to_string(p));
        for (int64_t t = t0; t < t1; ++t) {
            const uint4 d = desc[(size_t)(p + 1 + t)];
            const int64_t off = sbase + d.x;
            const unsigned w = d.y & 0xFFu, cs = (d.y >> 8) & 0xFFu, nnz = d.y >> 16;
            const unsigned m = d.w;
            const int64_t h_rows = __builtin_popcount(m);
            if (off != H.tileNnzOff[t] || w < 1 || m == 0u || (R < 32 && (m >> R)) ||
                off + (int64_t)w * h_rows != H.tileNnzOff[t + 1] || off + (int64_t)w * h_rows > H.nslots)
                return bad("slots of tile " + std::to_string(t));
            if ((int64_t)d.z != H.tileColIdx[t] || (int64_t)d.z < 0 || (int64_t)d.z >= H.nrb)
                return bad("column block of tile " + std::to_string(t));
            if (w == 1u && h_rows == 1 &&
                (cs >= (unsigned)T || H.colIdx[off] != cs || (int64_t)d.z * T + cs >= H.n))
                return bad("single-entry column of tile " + std::to_string(t));
            if (nnz > (unsigned)(w * h_rows)) return bad("entry count of tile " + std::to_string(t));
        }
    }
    return true;
}

}  // namespace evocg

