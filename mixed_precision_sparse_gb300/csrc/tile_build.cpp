// tile_build.cpp -- host construction of the tile structure, multi-threaded over row
// blocks.
//
// Layout (EvoCG, "Self-Evolving Precision Control for Faster Conjugate Gradient",
// §3.3.1 Fig. 4(a) and §3.3.2): CSR over row blocks of nonempty T x T tiles. Inside a
// tile: a mask of its nonempty local rows (rowMask), its width w = the longest row
// (tileWidth), and w x h slots (h = nonempty rows) in slot-major order: slot (k, j) at
// tileNnzOff[t] + k*h + j holds the k-th entry of the j-th nonempty row, or a pad
// (local column T, value +0) when that row is shorter. One local column byte per slot
// (colIdx) and three value streams over the same slots (FP64 a_ij; FP32 and BF16 of
// a_ij / 2^e_j with the per-column exponent e_j = floor(log2 max_i |a_ij|) clamped to
// [-100, 100]).
//
// The SpMV gives each row to one lane and accumulates it in registers (no cross-lane
// FP64 reduction, which GB300's FP64 rate would make the bottleneck); with slots in this
// order the lanes of a warp read consecutive slots at every k, and the position of a
// lane's slot is a popcount of the mask: no per-row offset table.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

void HostTiles::release()
{
    delete[] tileRowPtr; delete[] tileColIdx; delete[] tileNnzOff; delete[] tileRowIdx; delete[] rowMask;
    delete[] tileWidth; delete[] colIdx; delete[] v64; delete[] v32; delete[] v16; delete[] colExp;
    delete[] dinv;
    tileRowPtr = nullptr; tileColIdx = nullptr; tileNnzOff = nullptr; tileRowIdx = nullptr; rowMask = nullptr;
    tileWidth = nullptr;
    colIdx = nullptr; v64 = nullptr; v32 = nullptr; v16 = nullptr; colExp = nullptr;
    dinv = nullptr;
}

namespace {

template <class F>
void parallel_for(int64_t count, F &&fn)
{
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 4, 64));
    nt = std::min<int64_t>(nt, std::max<int64_t>(1, count / 256));
    if (nt <= 1) { fn(0, count); return; }
    std::vector<std::thread> th;
    th.reserve((size_t)nt);
    for (int64_t t = 0; t < nt; ++t) {
        int64_t a = count * t / nt, b = count * (t + 1) / nt;
        th.emplace_back([&fn, a, b] { fn(a, b); });
    }
    for (auto &x : th) x.join();
}

// floor(log2 |v|) for a finite nonzero v
int ilog2_abs(double v)
{
    uint64_t u;
    std::memcpy(&u, &v, 8);
    int ef = (int)((u >> 52) & 0x7FF);
    if (ef != 0) return ef - 1023;
    int e2;
    std::frexp(v, &e2);  // FP64 subnormal
    return e2 - 1;
}

}  // namespace

// Slot placement inside a row block (the SpMV moves a tile's slots with bulk copies, which
// need 16-byte aligned addresses and sizes): a tile with more than one slot starts on a
// multiple of 16 slots and occupies a multiple of 16 slots (its w x h slots, then pads), so
// its slice of every value stream and of the column bytes starts and ends on a 16-byte
// boundary; a single-entry tile takes one slot wherever it falls; a row block's slots are a
// multiple of 16 (its base stays 16-slot aligned). Returns where a tile of m slots starts
// when the row block's slots so far end at pos, and sets *end to where it ends.
int64_t place_tile(int64_t pos, int64_t m, int64_t *end)
{
    if (m <= 1) {
        *end = pos + m;
        return pos;
    }
    const int64_t s = (pos + 15) & ~(int64_t)15;
    *end = s + ((m + 15) & ~(int64_t)15);
    return s;
}

int build_host_tiles(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
                     HostTiles *out, std::string *err)
{
    if (n < 0 || n >= (int64_t)INT32_MAX) { *err = "n out of range"; return EVOCG_EINVAL; }
    if (T != 16 && T != 32 && T != 64) { *err = "tile_size must be 16, 32 or 64"; return EVOCG_EINVAL; }
    if (!rp || (n > 0 && (!ci || !v)) || rp[0] != 0) { *err = "bad CSR pointers"; return EVOCG_EINVAL; }
    const int64_t nnz = rp[n];
    // --- validate rows
    std::atomic<int64_t> bad_row{-1};
    parallel_for(n, [&](int64_t a, int64_t b) {
        for (int64_t i = a; i < b; ++i) {
            if (rp[i + 1] < rp[i] || rp[i + 1] > nnz) { bad_row = i; return; }
            for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
                if (ci[k] < 0 || ci[k] >= n || (k > rp[i] && ci[k] <= ci[k - 1]) ||
                    !std::isfinite(v[k])) { bad_row = i; return; }
            }
        }
    });
    if (bad_row.load() >= 0) {
        *err = "invalid CSR at row " + std::to_string(bad_row.load()) +
               " (row pointers must be monotone, columns in [0,n) strictly ascending, values finite)";
        return EVOCG_EINVAL;
    }
    HostTiles H;
    H.n = n; H.T = T; H.nnz = nnz; H.nrb = (n + T - 1) / T;
    const int64_t nrb = H.nrb;
    try {
        // --- per-column exponent (max over the column of floor(log2 |a_ij|))
        std::vector<std::atomic<int>> emax((size_t)std::max<int64_t>(n, 1));
        for (auto &e : emax) e.store(INT_MIN, std::memory_order_relaxed);
        parallel_for(n, [&](int64_t a, int64_t b) {
            for (int64_t i = a; i < b; ++i)
                for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
                    if (v[k] == 0.0) continue;
                    int e = ilog2_abs(v[k]);
                    std::atomic<int> &slot = emax[(size_t)ci[k]];
                    int cur = slot.load(std::memory_order_relaxed);
                    while (e > cur && !slot.compare_exchange_weak(cur, e, std::memory_order_relaxed)) {}
                }
        });
        H.colExp = new int8_t[(size_t)std::max<int64_t>(n, 1)];
        for (int64_t j = 0; j < n; ++j) {
            int e = emax[(size_t)j].load(std::memory_order_relaxed);
            e = (e == INT_MIN) ? 0 : std::min(100, std::max(-100, e));
            H.colExp[j] = (int8_t)e;
        }
        // --- diagonal
        H.dinv = new double[(size_t)std::max<int64_t>(n, 1)];
        std::atomic<int> diag_bad{0};
        parallel_for(n, [&](int64_t a, int64_t b) {
            for (int64_t i = a; i < b; ++i) {
                const int32_t *lo = ci + rp[i], *hi = ci + rp[i + 1];
                const int32_t *f = std::lower_bound(lo, hi, (int32_t)i);
                double d = (f != hi && *f == i) ? v[rp[i] + (f - lo)] : 0.0;
                if (!(d > 0.0)) { diag_bad = 1; H.dinv[i] = 0.0; }
                else H.dinv[i] = 1.0 / d;
            }
        });
        H.diag_ok = diag_bad.load() ? 0 : 1;
        // --- pass 1: tiles and slots per row block. The entries of one tile row are a
        // contiguous run of the CSR row (columns ascend), so a row block is walked once
        // per tile with one cursor per row.
        std::vector<int64_t> ntile_rb((size_t)nrb + 1, 0), nslot_rb((size_t)nrb + 1, 0);
        auto walk = [&](int64_t rb, auto &&on_tile) {
            const int64_t r0 = rb * T, r1 = std::min<int64_t>(n, r0 + T);
            const int nr = (int)(r1 - r0);
            int64_t cur[64], k1[64];
            for (int r = 0; r < nr; ++r) cur[r] = rp[r0 + r];
            for (;;) {
                int32_t cb = INT32_MAX;  // smallest column block left in the row block
                for (int r = 0; r < nr; ++r)
                    if (cur[r] < rp[r0 + r + 1]) cb = std::min(cb, ci[cur[r]] / T);
                if (cb == INT32_MAX) break;
                uint64_t mask = 0;
                int w = 0;
                for (int r = 0; r < nr; ++r) {
                    int64_t k = cur[r];
                    while (k < rp[r0 + r + 1] && ci[k] / T == cb) ++k;
                    k1[r] = k;
                    if (k > cur[r]) mask |= 1ull << r;
                    w = std::max(w, (int)(k - cur[r]));
                }
                on_tile(cb, mask, w, nr, cur, k1);
                for (int r = 0; r < nr; ++r) cur[r] = k1[r];
            }
        };
        parallel_for(nrb, [&](int64_t a, int64_t b) {
            for (int64_t rb = a; rb < b; ++rb) {
                int64_t nt = 0, ns = 0;
                walk(rb, [&](int32_t, uint64_t mask, int w, int, const int64_t *, const int64_t *) {
                    ++nt;
                    place_tile(ns, (int64_t)w * __builtin_popcountll(mask), &ns);
                });
                ntile_rb[(size_t)rb] = nt;
                nslot_rb[(size_t)rb] = (ns + 15) & ~(int64_t)15;
            }
        });
        H.tileRowPtr = new int64_t[(size_t)nrb + 1];
        std::vector<int64_t> slot0((size_t)nrb + 1, 0);
        H.tileRowPtr[0] = 0;
        for (int64_t rb = 0; rb < nrb; ++rb) {
            H.tileRowPtr[rb + 1] = H.tileRowPtr[rb] + ntile_rb[(size_t)rb];
            slot0[(size_t)rb + 1] = slot0[(size_t)rb] + nslot_rb[(size_t)rb];
        }
        H.ntiles = H.tileRowPtr[nrb];
        H.nslots = slot0[(size_t)nrb];
        const int64_t nt = H.ntiles, ns = H.nslots;
        H.tileColIdx = new int32_t[(size_t)std::max<int64_t>(nt, 1)];
        H.tileNnzOff = new int64_t[(size_t)nt + 1];
        H.tileRowIdx = new int32_t[(size_t)std::max<int64_t>(nt, 1)];
        H.rowMask = new uint64_t[(size_t)std::max<int64_t>(nt, 1)];
        H.tileWidth = new uint8_t[(size_t)std::max<int64_t>(nt, 1)];
        H.colIdx = new uint8_t[(size_t)std::max<int64_t>(ns, 1)];
        H.v64 = new double[(size_t)std::max<int64_t>(ns, 1)];
        H.v32 = new float[(size_t)std::max<int64_t>(ns, 1)];
        H.v16 = new uint16_t[(size_t)std::max<int64_t>(ns, 1)];
        H.tileNnzOff[nt] = ns;
        // slots between tiles (alignment) and after a tile's w x h rectangle: pads
        std::memset(H.colIdx, T, (size_t)std::max<int64_t>(ns, 1));
        std::memset(H.v64, 0, sizeof(double) * (size_t)std::max<int64_t>(ns, 1));
        std::memset(H.v32, 0, sizeof(float) * (size_t)std::max<int64_t>(ns, 1));
        std::memset(H.v16, 0, sizeof(uint16_t) * (size_t)std::max<int64_t>(ns, 1));
        // --- pass 2: fill the slots of every tile
        parallel_for(nrb, [&](int64_t a, int64_t b) {
            for (int64_t rb = a; rb < b; ++rb) {
                int64_t t = H.tileRowPtr[rb], pos = slot0[(size_t)rb];
                walk(rb, [&](int32_t cb, uint64_t mask, int w, int nr, const int64_t *k0,
                             const int64_t *k1) {
                    const int h = __builtin_popcountll(mask);
                    int64_t tile_end = 0;
                    pos = place_tile(pos, (int64_t)w * h, &tile_end);
                    H.tileColIdx[t] = cb;
                    H.tileNnzOff[t] = pos;
                    H.tileRowIdx[t] = (int32_t)rb;
                    H.rowMask[t] = mask;
                    H.tileWidth[t] = (uint8_t)w;
                    int j = 0;
                    for (int r = 0; r < nr; ++r) {
                        if (!((mask >> r) & 1)) continue;
                        for (int k = 0; k < w; ++k) {
                            const int64_t s = pos + (int64_t)k * h + j;
                            const int64_t e = k0[r] + k;
                            if (e < k1[r]) {
                                const int32_t c = ci[e];
                                const double sc = std::ldexp(v[e], -(int)H.colExp[c]);
                                uint64_t sb;
                                std::memcpy(&sb, &sc, 8);
                                H.colIdx[s] = (uint8_t)(c - cb * T);
                                H.v64[s] = v[e];
                                const uint32_t b32 = rne_bits_from_f64<23>(sb);
                                std::memcpy(&H.v32[s], &b32, 4);
                                H.v16[s] = (uint16_t)rne_bits_from_f64<7>(sb);
                            } else {  // pad: column T, +0 in every stream
                                H.colIdx[s] = (uint8_t)T;
                                H.v64[s] = 0.0;
                                H.v32[s] = 0.0f;
                                H.v16[s] = 0;
                            }
                        }
                        ++j;
                    }
                    pos = tile_end;
                    ++t;
                });
            }
        });
    } catch (const std::bad_alloc &) {
        H.release();
        *err = "host allocation failed while building tiles";
        return EVOCG_ENOMEM;
    }
    *out = H;
    return EVOCG_OK;
}

}  // namespace evocg

extern "C" int evocg_tile_layout_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                      const double *vals, int tile_size, int64_t *ntiles,
                                      int64_t *nslots, int64_t *tileRowPtr, int32_t *tileColIdx,
                                      int64_t *tileNnzOff, uint64_t *rowMask, uint8_t *tileWidth,
                                      uint8_t *colIdx, double *v64, float *v32, uint16_t *v16,
                                      int8_t *colExp)
{
    evocg::set_error("");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    if (ntiles) *ntiles = H.ntiles;
    if (nslots) *nslots = H.nslots;
    auto put = [](auto *dst, const auto *src, int64_t count) {
        if (dst && count > 0) std::memcpy(dst, src, sizeof(*dst) * (size_t)count);
    };
    put(tileRowPtr, H.tileRowPtr, H.nrb + 1);
    put(tileColIdx, H.tileColIdx, H.ntiles);
    put(tileNnzOff, H.tileNnzOff, H.ntiles + 1);
    put(rowMask, H.rowMask, H.ntiles);
    put(tileWidth, H.tileWidth, H.ntiles);
    put(colIdx, H.colIdx, H.nslots);
    put(v64, H.v64, H.nslots);
    put(v32, H.v32, H.nslots);
    put(v16, H.v16, H.nslots);
    put(colExp, H.colExp, H.n);
    H.release();
    return EVOCG_OK;
}
