// panel_plan.cpp -- the batch stream and the warp plan of the panel SpMV (spmv_panel.cu), made
// once per tile structure on the host.
//
// A panel is a row block (T <= 32). Its tiles are cut into batches, in order: a batch holds at
// most 31 tiles whose stage areas fit one shared-memory stage (every tile sized for FP64, the
// widest stream, so the plan holds for every precision map); a tile too large for a stage on
// its own is a batch by itself, computed from global memory ("direct"). A panel without tiles
// is one empty batch, so that its rows are written.
//
// Stream: for every batch, in panel order, one header record and one record per tile:
//   header  x: tiles in the batch (bits 0-7) | first batch of its panel (bit 8) | last batch of
//              its panel (bit 9) | a direct tile (bit 10)
//           y: panel index
//           z: the batch's ordinal B in the stream (tile i of the batch, i = 1..tiles, is the
//              tile of index rec - B - 1 + i, rec = the header's record index)
//           w: 0
//   tile    x: first slot of the tile (absolute; the stream has fewer than 2^32 slots)
//           y: w (bits 0-7) | stage offset in 16-byte units (bits 8-19) | local column of a
//              single-entry tile (bits 20-25) | single-entry tile (bit 26)
//           z: column block
//           w: row mask
// 32 zero records close the stream so that a 32-record window never reads past it.
//
// Stage: 16 bytes for its mbarrier, 32 single-entry slots of 16 bytes (value, x entry), then at
// each tile's stage offset its values (8 bytes per slot), its column bytes (1 per slot) and its
// x segment (8 bytes per entry); a tile's slots are a multiple of 16.
//
// Warps: each warp walks either a contiguous range of panels (warpRec: its first batch record;
// the range ends at the next warp's) or every nwarps-th panel (panelRec: each panel's first
// batch record), which the kernel variant chooses.
#include <algorithm>

#include "evocg_internal.h"

namespace evocg {

namespace {

constexpr unsigned kSingleBit = 1u << 26;
constexpr unsigned kFirstBit = 1u << 8, kLastBit = 1u << 9, kDirectBit = 1u << 10;
constexpr int kStageHead = 16 + 32 * 16;
constexpr int kMaxBatchTiles = 31;

bool is_single(const HostTiles &H, int64_t t)
{
    const uint64_t m = H.rowMask[t];
    return H.tileWidth[t] == 1 && m && !(m & (m - 1u));
}

int64_t slots16(const HostTiles &H, int64_t t)
{
    return ((int64_t)H.tileWidth[t] * __builtin_popcountll(H.rowMask[t]) + 15) & ~(int64_t)15;
}

// Stage bytes of a tile with m16 slots (a multiple of 16): values sized for FP64, column bytes,
// x segment sized for FP64.
int64_t tile_stage_bytes(int64_t m16, int T) { return 9 * m16 + 8 * T; }

}  // namespace

bool panel_plan(const HostTiles &H, int64_t warps, int stage_bytes, PanelPlan *out, std::string *why)
{
    if (H.T > 32) { *why = "panel plan: tiles wider than 32 are not planned here"; return false; }
    if (warps < 1) { *why = "panel plan: no warps"; return false; }
    if (stage_bytes <= kStageHead || stage_bytes > 16 * 4095) { *why = "panel plan: stage size"; return false; }
    if (H.nslots >= ((int64_t)1 << 32)) { *why = "panel plan: 2^32 slots or more"; return false; }
    const int64_t P = H.nrb;
    std::vector<uint4> &d = out->desc;
    d.clear();
    d.reserve((size_t)(H.ntiles + 2 * P + 32));
    out->panelRec.assign((size_t)P + 1, 0);
    uint32_t B = 0;   // batch ordinal
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        out->panelRec[(size_t)p] = (int64_t)d.size();
        int64_t t = t0;
        bool first = true;
        do {
            // one batch: tiles [t, e)
            int64_t e = t, used = kStageHead;
            bool direct = false;
            while (e < t1 && e - t < kMaxBatchTiles) {
                if (is_single(H, e)) { ++e; continue; }
                const int64_t need = tile_stage_bytes(slots16(H, e), H.T);
                if (kStageHead + need > stage_bytes) {   // alone, from global memory
                    if (e == t) { direct = true; ++e; }
                    break;
                }
                if (used + need > stage_bytes) break;
                used += need;
                ++e;
            }
            const bool last = e >= t1;
            d.push_back(make_uint4((unsigned)(e - t) | (first ? kFirstBit : 0u) | (last ? kLastBit : 0u) |
                                       (direct ? kDirectBit : 0u),
                                   (unsigned)p, B, 0u));
            int64_t off = kStageHead;
            for (int64_t u = t; u < e; ++u) {
                unsigned y = H.tileWidth[u];
                if (is_single(H, u)) {
                    y |= kSingleBit | ((unsigned)H.colIdx[H.tileNnzOff[u]] << 20);
                } else if (!direct) {
                    y |= (unsigned)(off / 16) << 8;
                    off += tile_stage_bytes(slots16(H, u), H.T);
                }
                d.push_back(make_uint4((unsigned)H.tileNnzOff[u], y, (unsigned)H.tileColIdx[u],
                                       (unsigned)H.rowMask[u]));
            }
            ++B;
            first = false;
            t = e;
        } while (t < t1);
    }
    out->panelRec[(size_t)P] = (int64_t)d.size();
    out->batches = B;
    d.resize(d.size() + 32, make_uint4(0u, 0u, 0u, 0u));
    // balanced contiguous panel ranges
    std::vector<int64_t> pre((size_t)P + 1, 0);
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        pre[(size_t)p + 1] = pre[(size_t)p] + (H.tileNnzOff[t1] - H.tileNnzOff[t0]) + 16 * (t1 - t0) + 32;
    }
    const int64_t total = pre[(size_t)P];
    out->warpRec.assign((size_t)warps + 1, 0);
    int64_t p = 0;
    for (int64_t w = 1; w < warps; ++w) {
        const int64_t target = (int64_t)((__int128)total * w / warps);
        while (p < P && pre[(size_t)p] < target) ++p;
        out->warpRec[(size_t)w] = out->panelRec[(size_t)p];
    }
    out->warpRec[0] = 0;
    out->warpRec[(size_t)warps] = out->panelRec[(size_t)P];
    return true;
}

// What the panel kernel assumes of a plan, checked before it is uploaded: the stream walks the
// panels in order with one or more batches each (first and last flags, ordinals counting up,
// at most 31 tiles a batch); every tile record matches the tile structure; a tile with more than
// one slot starts on a multiple of 16 slots and its 16-slot-rounded slice lies inside the slot
// streams; single-entry columns are real entries; a direct batch holds one tile; the tiles of a
// batch sit at increasing, non-overlapping stage offsets past the stage head and inside the
// stage; panelRec and warpRec point at batch headers in order, and the 32 closing records are
// zero. A plan that fails is not used.
bool panel_plan_ok(const HostTiles &H, int64_t warps, int stage_bytes, const PanelPlan &pl, std::string *why)
{
    const int64_t P = H.nrb, T = H.T, R = T < 32 ? T : 32;
    auto bad = [&](const std::string &m) { *why = "panel plan check: " + m; return false; };
    const std::vector<uint4> &d = pl.desc;
    if ((int64_t)pl.panelRec.size() != P + 1 || (int64_t)pl.warpRec.size() != warps + 1) return bad("tables");
    const int64_t end = pl.panelRec[(size_t)P];
    if ((int64_t)d.size() != end + 32) return bad("stream length");
    for (int64_t r = end; r < end + 32; ++r)
        if (d[(size_t)r].x | d[(size_t)r].y | d[(size_t)r].z | d[(size_t)r].w) return bad("closing records");
    int64_t rec = 0, t = 0;
    uint32_t B = 0;
    for (int64_t p = 0; p < P; ++p) {
        if (pl.panelRec[(size_t)p] != rec) return bad("panel record of panel " + std::to_string(p));
        const int64_t t1 = H.tileRowPtr[p + 1];
        bool first = true;
        for (;;) {
            if (rec >= end) return bad("stream ends inside panel " + std::to_string(p));
            const uint4 h = d[(size_t)rec];
            const int64_t nt = h.x & 0xFFu;
            const bool bfirst = h.x & kFirstBit, blast = h.x & kLastBit, direct = h.x & kDirectBit;
            if (h.y != (unsigned)p || h.z != B || bfirst != first || nt > kMaxBatchTiles || (direct && nt != 1) ||
                t + nt > t1 || (blast != (t + nt == t1)) || (!blast && nt == 0) || (h.x >> 11))
                return bad("batch header at record " + std::to_string(rec));
            int64_t sused = kStageHead;
            for (int64_t i = 1; i <= nt; ++i, ++t) {
                const uint4 r = d[(size_t)(rec + i)];
                const unsigned w = r.y & 0xFFu, so16 = (r.y >> 8) & 0xFFFu, cs = (r.y >> 20) & 0x3Fu;
                const bool single = r.y & kSingleBit;
                const int64_t hr = __builtin_popcount(r.w);
                if ((int64_t)r.x != H.tileNnzOff[t] || w != H.tileWidth[t] || r.w != (unsigned)H.rowMask[t] ||
                    r.w == 0u || (R < 32 && (r.w >> R)) || (int64_t)r.z != H.tileColIdx[t] || (int64_t)r.z >= H.nrb ||
                    (int64_t)r.x + (int64_t)w * hr > H.tileNnzOff[t + 1])
                    return bad("tile record of tile " + std::to_string(t));
                if (single != (w == 1 && hr == 1)) return bad("single flag of tile " + std::to_string(t));
                if (single) {
                    if (cs >= (unsigned)T || H.colIdx[r.x] != cs || (int64_t)r.z * T + cs >= H.n)
                        return bad("single-entry column of tile " + std::to_string(t));
                    continue;
                }
                const int64_t m16 = ((int64_t)w * hr + 15) & ~(int64_t)15;
                if ((r.x & 15u) || (int64_t)r.x + m16 > H.nslots) return bad("alignment of tile " + std::to_string(t));
                if (direct) continue;
                if ((int64_t)so16 * 16 < sused) return bad("stage overlap at tile " + std::to_string(t));
                sused = (int64_t)so16 * 16 + tile_stage_bytes(m16, (int)T);
                if (sused > stage_bytes) return bad("stage overflow at tile " + std::to_string(t));
            }
            rec += 1 + nt;
            ++B;
            first = false;
            if (blast) break;
        }
    }
    if (rec != end || t != H.ntiles || B != pl.batches) return bad("stream does not end with the tiles");
    if (pl.warpRec[0] != 0 || pl.warpRec[(size_t)warps] != end) return bad("warp ranges");
    for (int64_t w = 0; w < warps; ++w) {
        if (pl.warpRec[(size_t)w + 1] < pl.warpRec[(size_t)w]) return bad("warp ranges out of order");
        if (!std::binary_search(pl.panelRec.begin(), pl.panelRec.end(), pl.warpRec[(size_t)w]))
            return bad("a warp range that does not start a panel");
    }
    return true;
}

}  // namespace evocg

extern "C" int evocg_panel_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                     const double *vals, int tile_size, int64_t warps,
                                     int stage_bytes, int64_t *nbatches, int *valid)
{
    evocg::set_error("");
    if (warps < 1 || stage_bytes < 1) return evocg::fail(EVOCG_EINVAL, "warps and stage_bytes must be >= 1");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    int out = EVOCG_OK;
    try {
        evocg::PanelPlan pl;
        std::string why;
        const bool ok = evocg::panel_plan(H, warps, stage_bytes, &pl, &why) &&
                        evocg::panel_plan_ok(H, warps, stage_bytes, pl, &why);
        if (nbatches) *nbatches = ok ? (int64_t)pl.batches : 0;
        if (valid) *valid = ok ? 1 : 0;
        if (!ok) evocg::set_error(why);
    } catch (const std::bad_alloc &) {
        out = evocg::fail(EVOCG_ENOMEM, "host allocation failed while planning");
    }
    H.release();
    return out;
}
