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
