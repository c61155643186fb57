// panel_plan.cpp -- the descriptor stream and the warp plan of the panel SpMV (spmv_panel.cu),
// made once per tile structure on the host.
//
// Stream: for every panel, in panel order, one header record {tiles in the panel, panel
// index, first slot (low, high 32 bits)} followed by one record per tile:
//   x: slot offset from the panel's first slot
//   y: w (bits 0-7) | stage offset of the tile in 16-byte units (bits 8-19) | local column
//      of a single-entry tile (bits 20-25) | single (bit 26) | batch start (bit 27) | direct
//      (bit 28: too large for the stage, computed from global memory)
//   z: column block
//   w: row mask
// 32 zero records close the stream so that a 32-record window never reads past it. Record r
// of panel p's tile i is at p + tileRowPtr[p] + 1 + i, so a tile's index is r - p - 1.
//
// Batches. A warp stages a batch of consecutive tiles of one panel in its shared-memory stage,
// computes it and moves on. The stage holds 32 single-entry slots of 16 bytes, then, for every
// other tile of the batch at its stage offset, its values (sized for FP64, the widest stream,
// so the plan holds for every precision map), its local-column bytes (rounded up to 16) and
// its x segment (T entries, sized for FP64). A batch never crosses a 32-record window of the
// panel (tiles 0..30, 31..62, ...), so the kernel finds every tile of a batch in the window
// it holds.
//
// Warp plan: warps take consecutive panels, split where the running cost (one per slot, 16
// per tile, 32 per panel) crosses multiples of total / warps (the interleaved kernel variants
// ignore it).
#include <algorithm>

#include "evocg_internal.h"

namespace evocg {

namespace {

constexpr unsigned kSingleBit = 1u << 26, kBatchBit = 1u << 27, kDirectBit = 1u << 28;
constexpr int kSingleArea = 32 * 16;

bool is_single(const HostTiles &H, int64_t t)
{
    const uint64_t m = H.rowMask[t];
    return H.tileWidth[t] == 1 && m && !(m & (m - 1u));
}

// Stage bytes of a tile with more than one slot: FP64 values of its slots (a multiple of 8),
// its column bytes rounded up to 16, its FP64 x segment.
int64_t tile_stage_bytes(int64_t m8, int T) { return 8 * m8 + ((m8 + 15) & ~(int64_t)15) + 8 * T; }

}  // namespace

bool panel_plan(const HostTiles &H, int64_t warps, int stage_bytes, std::vector<uint4> *desc,
                std::vector<int64_t> *warpRec, std::vector<int32_t> *warpPanel, std::string *why)
{
    if (H.T > 32) { *why = "panel plan: tiles wider than 32 are not planned here"; return false; }
    if (warps < 1) { *why = "panel plan: no warps"; return false; }
    if (stage_bytes <= kSingleArea || stage_bytes > 16 * 4095) { *why = "panel plan: stage size"; return false; }
    const int64_t P = H.nrb;   // panels = row blocks for T <= 32
    desc->assign((size_t)(P + H.ntiles + 32), make_uint4(0u, 0u, 0u, 0u));
    for (int64_t p = 0; p < P; ++p) {
        const int64_t t0 = H.tileRowPtr[p], t1 = H.tileRowPtr[p + 1];
        const int64_t r = p + t0;
        const int64_t sbase = H.tileNnzOff[t0];
        (*desc)[(size_t)r] = make_uint4((unsigned)(t1 - t0), (unsigned)p, (unsigned)(uint64_t)sbase,
                                        (unsigned)((uint64_t)sbase >> 32));
        int64_t used = kSingleArea;
        bool open = false;   // a batch is open in the current window
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t i = t - t0;
            const int64_t off = H.tileNnzOff[t] - sbase;
            if (off >= ((int64_t)1 << 32)) { *why = "panel plan: a panel holds 2^32 slots or more"; return false; }
            if ((i + 1) % 32 == 0) open = false;   // tile i starts a new 32-record window
            const uint64_t m = H.rowMask[t];
            const unsigned w = H.tileWidth[t];
            unsigned y = w;
            if (is_single(H, t)) {
                y |= kSingleBit | ((unsigned)H.colIdx[H.tileNnzOff[t]] << 20);
                if (!open) { y |= kBatchBit; open = true; used = kSingleArea; }
            } else {
                const int64_t m8 = ((int64_t)w * __builtin_popcountll(m) + 7) & ~(int64_t)7;
                const int64_t need = tile_stage_bytes(m8, H.T);
                if (kSingleArea + need > stage_bytes) {   // alone in a batch, from global memory
                    y |= kDirectBit | kBatchBit;
                    open = false;
                } else {
                    if (!open || used + need > stage_bytes) { y |= kBatchBit; open = true; used = kSingleArea; }
                    y |= (unsigned)(used / 16) << 8;
                    used += need;
                }
            }
            (*desc)[(size_t)(r + 1 + i)] = make_uint4((unsigned)off, y, (unsigned)H.tileColIdx[t], (unsigned)m);
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
// kernel reads lies in the stream; headers and tile records match the tile structure; every
// tile with more than one slot starts on a multiple of 8 slots and its 8-slot-rounded slice
// lies inside the slot streams (plus their slack); single-entry columns are real entries;
// every window starts a batch; the tiles of a batch sit at increasing, non-overlapping stage
// offsets past the single-entry area and inside the stage; and the warp ranges tile the
// panels in order. A plan that fails is not used.
bool panel_plan_ok(const HostTiles &H, int64_t warps, int stage_bytes, const std::vector<uint4> &desc,
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
        if ((int64_t)h.x != t1 - t0 || (int64_t)h.y != p || sbase != H.tileNnzOff[t0] || (sbase & 15))
            return bad("header of panel " + std::to_string(p));
        int64_t end = 0;   // end of the last stage area of the open batch
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t i = t - t0;
            const uint4 d = desc[(size_t)(p + 1 + t)];
            const int64_t off = sbase + d.x;
            const unsigned w = d.y & 0xFFu, so16 = (d.y >> 8) & 0xFFFu, cs = (d.y >> 20) & 0x3Fu;
            const bool single = d.y & kSingleBit, bstart = d.y & kBatchBit, direct = d.y & kDirectBit;
            const unsigned m = d.w;
            const int64_t hr = __builtin_popcount(m);
            if (off != H.tileNnzOff[t] || w < 1 || w != H.tileWidth[t] || m == 0u || m != (unsigned)H.rowMask[t] ||
                (R < 32 && (m >> R)) || off + (int64_t)w * hr > H.tileNnzOff[t + 1])
                return bad("slots of tile " + std::to_string(t));
            if ((int64_t)d.z != H.tileColIdx[t] || (int64_t)d.z < 0 || (int64_t)d.z >= H.nrb)
                return bad("column block of tile " + std::to_string(t));
            if (single != (w == 1 && hr == 1)) return bad("single flag of tile " + std::to_string(t));
            if (((i + 1) % 32 == 0 || i == 0) && !bstart)
                return bad("a window without a batch start at tile " + std::to_string(t));
            if (single) {
                if (cs >= (unsigned)T || H.colIdx[off] != cs || (int64_t)d.z * T + cs >= H.n)
                    return bad("single-entry column of tile " + std::to_string(t));
                if (bstart) end = kSingleArea;
                continue;
            }
            const int64_t m8 = ((int64_t)w * hr + 7) & ~(int64_t)7;
            if ((off & 7) || off + m8 > H.nslots) return bad("alignment of tile " + std::to_string(t));
            if (direct) {
                if (!bstart) return bad("direct tile inside a batch");
                end = stage_bytes;   // nothing may follow it in its batch
                continue;
            }
            if (bstart) end = kSingleArea;
            if ((int64_t)so16 * 16 < end) return bad("stage overlap at tile " + std::to_string(t));
            end = (int64_t)so16 * 16 + tile_stage_bytes(m8, (int)T);
            if (end > stage_bytes) return bad("stage overflow at tile " + std::to_string(t));
        }
    }
    return true;
}

}  // namespace evocg
