// staged_plan.cpp -- the static work plan of the staged SpMV, made once per tile structure.
//
// Warps get consecutive row blocks, split where the running cost (32 per tile + 1 per entry
// + 32 per row block) crosses multiples of total / warps. Each warp's tiles are cut into
// batches of at most `nb` tiles whose worst-case stage bytes fit one stage: the 16-byte
// cover of the value slice in FP64 (every precision's cover fits in it) plus the FP64 x
// segment, and the local-column bytes. Because the slots are sized for FP64, the plan does
// not depend on the precision map: the kernel reads it as is whatever map is set.
#include <algorithm>

#include "evocg_internal.h"

namespace evocg {

void staged_plan(const HostTiles &H, int64_t warps, const StagedLimits &lim,
                 std::vector<int32_t> *warpRb, std::vector<int32_t> *warpBatch,
                 std::vector<int64_t> *batchTile, std::vector<uint16_t> *tileSlot)
{
    const int64_t nrb = H.nrb, T = H.T;
    std::vector<int64_t> pre((size_t)nrb + 1, 0);
    for (int64_t rb = 0; rb < nrb; ++rb) {
        const int64_t t0 = H.tileRowPtr[rb], t1 = H.tileRowPtr[rb + 1];
        pre[(size_t)rb + 1] = pre[(size_t)rb] + 32 * (t1 - t0) + (H.tileNnzOff[t1] - H.tileNnzOff[t0]) + 32;
    }
    const int64_t total = pre[(size_t)nrb];
    warpRb->assign((size_t)warps + 1, 0);
    int64_t rb = 0;
    for (int64_t w = 1; w < warps; ++w) {
        const int64_t target = (int64_t)((__int128)total * w / warps);
        while (rb < nrb && pre[(size_t)rb] < target) ++rb;
        (*warpRb)[(size_t)w] = (int32_t)rb;
    }
    (*warpRb)[(size_t)warps] = (int32_t)nrb;

    tileSlot->assign((size_t)std::max<int64_t>(H.ntiles, 1), 0);
    batchTile->clear();
    warpBatch->assign((size_t)warps + 1, 0);
    for (int64_t w = 0; w < warps; ++w) {
        (*warpBatch)[(size_t)w] = (int32_t)batchTile->size();
        int64_t t = H.tileRowPtr[(*warpRb)[(size_t)w]];
        const int64_t te = H.tileRowPtr[(*warpRb)[(size_t)w + 1]];
        while (t < te) {
            batchTile->push_back(t);
            int nb = 0, used = 0;
            int64_t usedm = 0;
            while (t + nb < te && nb < lim.nb) {
                const int64_t m = H.tileNnzOff[t + nb + 1] - H.tileNnzOff[t + nb];
                const int need = staged_slot_bytes(m, (int)T);
                if (nb == 0 && (need > lim.data_bytes || m + 32 > lim.col_bytes)) {
                    (*tileSlot)[(size_t)t] = kDirectSlot;  // computed from global memory
                    nb = 1;
                    break;
                }
                if (used + need > lim.data_bytes || usedm + m + 32 > lim.col_bytes) break;
                (*tileSlot)[(size_t)(t + nb)] = (uint16_t)used;
                used += need;
                usedm += m;
                ++nb;
            }
            t += nb;
        }
    }
    (*warpBatch)[(size_t)warps] = (int32_t)batchTile->size();
    batchTile->push_back(H.ntiles);
}

}  // namespace evocg

namespace evocg {

// Check a plan against what the staged kernel assumes of it: warp row-block ranges that
// tile [0, nrb); per warp, batches that cover its tiles in order; at most nb tiles per
// batch; a tile too large for a stage alone in its batch; slots packed from 0 in tile
// order, each sized for FP64 values plus an FP64 x segment, all inside the stage's data
// area; local-column bytes (with the slack the producer's 16-byte covers need) inside the
// column area. A plan that fails is not used (the direct kernel runs instead).
bool staged_plan_ok(const HostTiles &H, int64_t warps, const StagedLimits &lim,
                    const std::vector<int32_t> &wr, const std::vector<int32_t> &wbt,
                    const std::vector<int64_t> &bt, const std::vector<uint16_t> &slot)
{
    const int T = H.T;
    if ((int64_t)wr.size() != warps + 1 || (int64_t)wbt.size() != warps + 1 || bt.empty()) return false;
    if (wr[0] != 0 || wr[(size_t)warps] != H.nrb || wbt[0] != 0) return false;
    if (wbt[(size_t)warps] != (int64_t)bt.size() - 1 || bt.back() != H.ntiles) return false;
    if ((int64_t)slot.size() < H.ntiles) return false;
    for (int64_t w = 0; w < warps; ++w) {
        if (wr[(size_t)w + 1] < wr[(size_t)w] || wbt[(size_t)w + 1] < wbt[(size_t)w]) return false;
        const int64_t t0 = H.tileRowPtr[wr[(size_t)w]], t1 = H.tileRowPtr[wr[(size_t)w + 1]];
        const int64_t b0 = wbt[(size_t)w], b1 = wbt[(size_t)w + 1];
        if (b0 == b1) {
            if (t0 != t1) return false;
            continue;
        }
        if (bt[(size_t)b0] != t0 || bt[(size_t)b1] != t1) return false;
        for (int64_t b = b0; b < b1; ++b) {
            const int64_t tb = bt[(size_t)b], te = bt[(size_t)b + 1];
            if (te <= tb || te - tb > lim.nb) return false;
            if (slot[(size_t)tb] == kDirectSlot) {
                if (te - tb != 1) return false;
                continue;
            }
            int64_t used = 0, usedm = 0;
            for (int64_t t = tb; t < te; ++t) {
                const int64_t m = H.tileNnzOff[t + 1] - H.tileNnzOff[t];
                if (slot[(size_t)t] != used) return false;
                used += staged_slot_bytes(m, T);
                usedm += m;
            }
            if (used > lim.data_bytes || usedm + 32 > lim.col_bytes) return false;
        }
    }
    return true;
}

}  // namespace evocg

extern "C" int evocg_staged_plan_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                      const double *vals, int tile_size, int64_t warps,
                                      int64_t *nbatches, int *valid)
{
    evocg::set_error("");
    if (warps < 1) return evocg::fail(EVOCG_EINVAL, "warps must be >= 1");
    evocg::StagedLimits lim;
    if (!evocg::staged_limits(tile_size, &lim))
        return evocg::fail(EVOCG_EINVAL, "no staged kernel for this tile size");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    std::vector<int32_t> wr, wbt;
    std::vector<int64_t> bt;
    std::vector<uint16_t> slot;
    evocg::staged_plan(H, warps, lim, &wr, &wbt, &bt, &slot);
    const bool ok = evocg::staged_plan_ok(H, warps, lim, wr, wbt, bt, slot);
    if (nbatches) *nbatches = (int64_t)bt.size() - 1;
    if (valid) *valid = ok ? 1 : 0;
    H.release();
    return EVOCG_OK;
}
