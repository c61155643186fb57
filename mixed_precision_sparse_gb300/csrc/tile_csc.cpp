// tile_csc.cpp -- the Tile-CSC layout of EvoCG ("Self-Evolving Precision Control for Faster
// Conjugate Gradient", §3.3.1 Fig. 4(a) and §3.3.2 Fig. 4(b)) produced from this library's
// own tile structure, for export and for bit-exact checks against an independent builder.
//
// The SpMV kernels read a slot-major interior (a row mask, a width and w x h slots per tile:
// lanes own rows). The paper stores every tile as CSC instead: colPtr (T + 1 offsets from the
// tile's first entry), rowIdx (row relative to the row block's first row), entries of a
// column in ascending row, and, in the paper, every column padded to even length with a
// sentinel row index R (here T) and zero values. The two hold the same entries with the same
// value bits; this file rewrites one into the other, tile by tile, so that the structure the
// kernels read is checked against the paper's.
#include <cuda_runtime.h>

#include <cstring>
#include <string>
#include <vector>

#include "evocg_internal.h"

namespace evocg {

namespace {

struct CscArrays {
    int64_t *tileNnzOff;
    uint16_t *colPtr;
    uint8_t *rowIdx;
    double *v64;
    float *v32;
    uint16_t *v16;
};

// Entries of the padded streams (stored entries plus sentinels) of every tile, or the
// arrays themselves when out is given. Columns of a tile are visited through its slots:
// rows in ascending order, each row's slots in ascending column, so every column's
// bucket receives its rows in ascending order.
int64_t slots_to_csc(const HostTiles &H, int pad, const CscArrays *out)
{
    const int T = H.T;
    int64_t pos = 0;
    std::vector<int64_t> cnt((size_t)T + 1), fill((size_t)T);
    for (int64_t t = 0; t < H.ntiles; ++t) {
        const uint64_t m = H.rowMask[t];
        const int64_t w = H.tileWidth[t], h = __builtin_popcountll(m);
        const int64_t off = H.tileNnzOff[t];
        std::fill(cnt.begin(), cnt.end(), 0);
        for (int64_t s = off; s < off + w * h; ++s)
            if (H.colIdx[s] < T) ++cnt[H.colIdx[s]];
        // colPtr: running padded counts
        int64_t local = 0;
        for (int c = 0; c < T; ++c) {
            if (out) {
                out->colPtr[t * (T + 1) + c] = (uint16_t)local;
                fill[(size_t)c] = local;
            }
            local += (cnt[(size_t)c] + pad - 1) / pad * pad;
        }
        if (out) {
            out->colPtr[t * (T + 1) + T] = (uint16_t)local;
            out->tileNnzOff[t] = pos;
            int j = 0;
            for (int r = 0; r < T; ++r) {
                if (!((m >> r) & 1ull)) continue;
                for (int64_t k = 0; k < w; ++k) {
                    const int64_t s = off + k * h + j;
                    const int c = H.colIdx[s];
                    if (c >= T) continue;
                    const int64_t e = pos + fill[(size_t)c]++;
                    out->rowIdx[e] = (uint8_t)r;
                    out->v64[e] = H.v64[s];
                    out->v32[e] = H.v32[s];
                    out->v16[e] = H.v16[s];
                }
                ++j;
            }
            for (int c = 0; c < T; ++c) {   // sentinel-marked zeros of padded columns
                const int64_t end = out->colPtr[t * (T + 1) + c + 1];
                for (int64_t e = fill[(size_t)c]; e < end; ++e) {
                    out->rowIdx[pos + e] = (uint8_t)T;
                    out->v64[pos + e] = 0.0;
                    out->v32[pos + e] = 0.0f;
                    out->v16[pos + e] = 0;
                }
            }
        }
        pos += local;
    }
    if (out) out->tileNnzOff[H.ntiles] = pos;
    return pos;
}

// Caller buffers (any may be NULL) receive the Tile-CSC arrays of H.
int write_csc(const HostTiles &H, int pad, int64_t *ntiles, int64_t *nnz_p, int64_t *tileRowPtr,
              int32_t *tileColIdx, int64_t *tileNnzOff, uint16_t *colPtr, uint8_t *rowIdx,
              double *v64, float *v32, uint16_t *v16, int8_t *colExp)
{
    const int64_t np_ = slots_to_csc(H, pad, nullptr);
    if (ntiles) *ntiles = H.ntiles;
    if (nnz_p) *nnz_p = np_;
    auto put = [](auto *dst, const auto *src, int64_t count) {
        if (dst && count > 0) std::memcpy(dst, src, sizeof(*dst) * (size_t)count);
    };
    put(tileRowPtr, H.tileRowPtr, H.nrb + 1);
    put(tileColIdx, H.tileColIdx, H.ntiles);
    put(colExp, H.colExp, H.n);
    if (tileNnzOff || colPtr || rowIdx || v64 || v32 || v16) {
        std::vector<int64_t> a((size_t)H.ntiles + 1);
        std::vector<uint16_t> b((size_t)(H.ntiles * (H.T + 1) + 1));
        std::vector<uint8_t> c((size_t)np_ + 1);
        std::vector<double> d((size_t)np_ + 1);
        std::vector<float> e((size_t)np_ + 1);
        std::vector<uint16_t> f((size_t)np_ + 1);
        CscArrays o{a.data(), b.data(), c.data(), d.data(), e.data(), f.data()};
        slots_to_csc(H, pad, &o);
        put(tileNnzOff, a.data(), H.ntiles + 1);
        put(colPtr, b.data(), H.ntiles * (H.T + 1));
        put(rowIdx, c.data(), np_);
        put(v64, d.data(), np_);
        put(v32, e.data(), np_);
        put(v16, f.data(), np_);
    }
    return EVOCG_OK;
}

}  // namespace

}  // namespace evocg

extern "C" int evocg_tile_csc_host(int64_t n, const int64_t *row_ptr, const int32_t *col_idx,
                                   const double *vals, int tile_size, int pad, int64_t *ntiles,
                                   int64_t *nnz_p, int64_t *tileRowPtr, int32_t *tileColIdx,
                                   int64_t *tileNnzOff, uint16_t *colPtr, uint8_t *rowIdx,
                                   double *v64, float *v32, uint16_t *v16, int8_t *colExp)
{
    evocg::set_error("");
    if (pad != 1 && pad != 2) return evocg::fail(EVOCG_EINVAL, "pad must be 1 or 2");
    evocg::HostTiles H;
    std::string err;
    const int rc = evocg::build_host_tiles(n, row_ptr, col_idx, vals, tile_size, &H, &err);
    if (rc) return evocg::fail(rc, err);
    int out = EVOCG_OK;
    try {
        out = evocg::write_csc(H, pad, ntiles, nnz_p, tileRowPtr, tileColIdx, tileNnzOff, colPtr,
                               rowIdx, v64, v32, v16, colExp);
    } catch (const std::bad_alloc &) {
        out = evocg::fail(EVOCG_ENOMEM, "host allocation failed while writing the Tile-CSC layout");
    }
    H.release();
    return out;
}

extern "C" int evocg_tiles_export_csc(evocg_tiles_t A, int pad, int64_t *nnz_p, int64_t *tileRowPtr,
                                      int32_t *tileColIdx, int64_t *tileNnzOff, uint16_t *colPtr,
                                      uint8_t *rowIdx, double *v64, float *v32, uint16_t *v16,
                                      int8_t *colExp)
{
    evocg::set_error("");
    if (!A) return evocg::fail(EVOCG_EINVAL, "NULL handle");
    if (pad != 1 && pad != 2) return evocg::fail(EVOCG_EINVAL, "pad must be 1 or 2");
    evocg::HostTiles H;
    H.n = A->n; H.T = A->T; H.nrb = A->nrb; H.ntiles = A->ntiles; H.nnz = A->nnz; H.nslots = A->nslots;
    int out = EVOCG_OK;
    try {
        H.tileRowPtr = new int64_t[(size_t)H.nrb + 1];
        H.tileColIdx = new int32_t[(size_t)H.ntiles + 1];
        H.tileNnzOff = new int64_t[(size_t)H.ntiles + 1];
        H.rowMask = new uint64_t[(size_t)H.ntiles + 1];
        H.tileWidth = new uint8_t[(size_t)H.ntiles + 1];
        H.colIdx = new uint8_t[(size_t)H.nslots + 1];
        H.v64 = new double[(size_t)H.nslots + 1];
        H.v32 = new float[(size_t)H.nslots + 1];
        H.v16 = new uint16_t[(size_t)H.nslots + 1];
        H.colExp = new int8_t[(size_t)H.n + 1];
    } catch (const std::bad_alloc &) {
        H.release();
        return evocg::fail(EVOCG_ENOMEM, "host allocation failed while exporting the layout");
    }
    // the device-resident structure, copied back as the kernels read it
    cudaError_t e = cudaDeviceSynchronize();
    auto dn = [&](auto *dst, const auto *src, int64_t count) {
        if (e == cudaSuccess && count > 0)
            e = cudaMemcpy(dst, src, sizeof(*dst) * (size_t)count, cudaMemcpyDeviceToHost);
    };
    dn(H.tileRowPtr, A->tileRowPtr, H.nrb + 1);
    dn(H.tileColIdx, A->tileColIdx, H.ntiles);
    dn(H.tileNnzOff, A->tileNnzOff, H.ntiles + 1);
    dn(H.rowMask, A->rowMask, H.ntiles);
    dn(H.tileWidth, A->tileWidth, H.ntiles);
    dn(H.colIdx, A->colIdx, H.nslots);
    dn(H.v64, A->v64, H.nslots);
    dn(H.v32, A->v32, H.nslots);
    dn(H.v16, A->v16, H.nslots);
    dn(H.colExp, A->colExp, H.n);
    if (e != cudaSuccess) {
        H.release();
        return evocg::cuda_fail(e, "copying the tile structure back");
    }
    try {
        out = evocg::write_csc(H, pad, nullptr, nnz_p, tileRowPtr, tileColIdx, tileNnzOff, colPtr,
                               rowIdx, v64, v32, v16, colExp);
    } catch (const std::bad_alloc &) {
        out = evocg::fail(EVOCG_ENOMEM, "host allocation failed while writing the Tile-CSC layout");
    }
    H.release();
    return out;
}
