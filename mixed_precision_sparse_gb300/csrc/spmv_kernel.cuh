// spmv_kernel.cuh -- the tile-wise mixed-precision SpMV (EvoCG, "Self-Evolving Precision
// Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 / Eq. 5) for sm_103a.
//
// Work mapping. Each warp owns a contiguous range of row blocks and walks their tiles as
// one stream, in tile order (row block, then ascending column block), so every row is
// summed in column order. Lane l owns local row l (T = 32), rows l and l+32 (T = 64), or
// row l & 15 (T = 16; the upper half-warp mirrors the lower one). A row's sum stays in
// the lane's registers across the whole row block: no cross-lane reduction.
//
// Latency. The SpMV streams the matrix once, so it is bound by memory-level parallelism:
// a naive walk pays three dependent round trips per tile (descriptor, then the row's
// entries, then x). Here the descriptors of up to 32 tiles are loaded by the 32 lanes in
// one go and handed out by shuffle; the tile's x segment is loaded by lane (coalesced, it
// depends only on the descriptor) and gathered by shuffle; and a two-stage software
// pipeline issues the row ends of tile u+2 and the first entries of tile u+1 before it
// computes tile u.
//
// Arithmetic. An FP64 tile costs one FP64 fused multiply-add per entry. FP32 and BF16
// tiles never touch the FP64 unit: their products are exact in an FP32 pair, summed
// error-free (TwoSum) into an FP32 hi/lo pair, merged into the FP64 row sum once per
// row. GB300 issues FP64 at about 1/58 of the FP32 rate.
#pragma once
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

template <int T>
struct Geo {
    static constexpr int G = T < 32 ? T : 32;  // lanes that own rows (and shuffle width)
    static constexpr int RPL = T / G;          // rows per lane
    static constexpr int J = (T == 64) ? 2 : 4;  // entries per row fetched ahead per tile
};

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// One tile's inputs for the lane: its descriptor, its rows' entry ranges, the first J
// entries of each row (local column bytes packed into one word, raw value bits), and the
// lane's entries of the tile's x segment (raw bits in the tile's format).
template <int T>
struct TileStage {
    using Gm = Geo<T>;
    int valid;
    int prec;
    int cb;
    int drb;
    int64_t off;
    int s[Gm::RPL], e[Gm::RPL];
    uint32_t cip[Gm::RPL];
    uint64_t vp[Gm::RPL][Gm::J];
    uint64_t xr[Gm::RPL];
};

template <int T>
struct RowEnds {
    int s[Geo<T>::RPL], e[Geo<T>::RPL];
};

// Row ranges of tile (tbase + u) for this lane's rows.
template <int T>
__device__ __forceinline__ void load_rowends(const TilesView &A, int64_t tbase, int u, int nt,
                                             RowEnds<T> &R)
{
    using Gm = Geo<T>;
    const int gl = (int)(lane_id() % Gm::G);
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) {
        R.s[rr] = 0;
        R.e[rr] = 0;
        if (u < nt) {
            const uint16_t *re = A.rowEnd + (tbase + u) * T;
            const int r = gl + rr * Gm::G;
            R.e[rr] = __ldcs(re + r);
            R.s[rr] = r ? (int)__ldcs(re + r - 1) : 0;
        }
    }
}

// Descriptor of tile u of the chunk, handed out from lane u.
__device__ __forceinline__ void chunk_desc(uint32_t dw0, uint32_t dw1, int u, int64_t offbase,
                                           int &cb, int &prec, int64_t &off, int &drb)
{
    const uint32_t w0 = __shfl_sync(0xffffffffu, dw0, u & 31);
    const uint32_t w1 = __shfl_sync(0xffffffffu, dw1, u & 31);
    cb = (int)(w0 & 0x0FFFFFFFu);
    prec = (int)(w0 >> 28);
    off = offbase + (int64_t)(w1 & 0x00FFFFFFu);
    drb = (int)(w1 >> 24);
}

template <int T>
__device__ __forceinline__ void load_stage(const TilesView &A, const SpmvLaunch &L, uint32_t dw0,
                                           uint32_t dw1, int64_t offbase, int u, int nt,
                                           const RowEnds<T> &R, TileStage<T> &S)
{
    using Gm = Geo<T>;
    const int gl = (int)(lane_id() % Gm::G);
    chunk_desc(dw0, dw1, u, offbase, S.cb, S.prec, S.off, S.drb);
    S.valid = (u < nt);
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) {
        S.s[rr] = R.s[rr];
        S.e[rr] = R.e[rr];
        S.cip[rr] = 0u;
        S.xr[rr] = 0ull;
#pragma unroll
        for (int j = 0; j < Gm::J; ++j) S.vp[rr][j] = 0ull;
    }
    if (!S.valid) return;
    const int64_t xb = (int64_t)S.cb * T;
    const uint8_t *ci = A.colIdx + S.off;
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) {
        const int64_t xc = xb + gl + rr * Gm::G;
        const bool xin = xc < A.n;
#pragma unroll
        for (int j = 0; j < Gm::J; ++j) {
            const int k = S.s[rr] + j;
            if (k < S.e[rr]) S.cip[rr] |= (uint32_t)__ldcs(ci + k) << (8 * j);
        }
        if (S.prec == EVOCG_FP64) {
            if (xin) S.xr[rr] = __ldg(reinterpret_cast<const unsigned long long *>(L.x64) + xc);
            const unsigned long long *vv = reinterpret_cast<const unsigned long long *>(A.v64) + S.off;
#pragma unroll
            for (int j = 0; j < Gm::J; ++j)
                if (S.s[rr] + j < S.e[rr]) S.vp[rr][j] = __ldcs(vv + S.s[rr] + j);
        } else if (S.prec == EVOCG_FP32) {
            if (xin) S.xr[rr] = __ldg(reinterpret_cast<const unsigned *>(L.x32) + xc);
            const unsigned *vv = reinterpret_cast<const unsigned *>(A.v32) + S.off;
#pragma unroll
            for (int j = 0; j < Gm::J; ++j)
                if (S.s[rr] + j < S.e[rr]) S.vp[rr][j] = __ldcs(vv + S.s[rr] + j);
        } else {
            if (xin) S.xr[rr] = __ldg(L.x16 + xc);
            const unsigned short *vv = A.v16 + S.off;
#pragma unroll
            for (int j = 0; j < Gm::J; ++j)
                if (S.s[rr] + j < S.e[rr]) S.vp[rr][j] = __ldcs(vv + S.s[rr] + j);
        }
    }
}

// x entry `col` of the tile's segment, from the lane that holds it (all lanes call).
template <int T>
__device__ __forceinline__ uint64_t gather64(const uint64_t (&xr)[Geo<T>::RPL], int col)
{
    using Gm = Geo<T>;
    const int src = col % Gm::G;
    uint64_t v = 0;
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) {
        const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)xr[rr], src, Gm::G);
        const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(xr[rr] >> 32), src, Gm::G);
        if (col / Gm::G == rr) v = ((uint64_t)hi << 32) | lo;
    }
    return v;
}

template <int T>
__device__ __forceinline__ uint32_t gather32(const uint64_t (&xr)[Geo<T>::RPL], int col)
{
    using Gm = Geo<T>;
    const int src = col % Gm::G;
    uint32_t v = 0;
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) {
        const uint32_t w = __shfl_sync(0xffffffffu, (uint32_t)xr[rr], src, Gm::G);
        if (col / Gm::G == rr) v = w;
    }
    return v;
}

// Accumulate one tile into the lane's row sums. Every lane of the warp calls this with
// the same tile (the branch on the precision is warp-uniform).
template <int T>
__device__ __forceinline__ void compute_stage(const TilesView &A, const SpmvLaunch &L,
                                              const TileStage<T> &S, double (&acc)[Geo<T>::RPL],
                                              F32Pair (&pr)[Geo<T>::RPL])
{
    using Gm = Geo<T>;
    constexpr int J = Gm::J;
    int rem = 0;
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) rem = max(rem, S.e[rr] - S.s[rr] - J);
    const int more = (int)__reduce_max_sync(0xffffffffu, (unsigned)max(rem, 0));
    const uint8_t *ci = A.colIdx + S.off;
    if (S.prec == EVOCG_FP64) {
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int col = (int)((S.cip[rr] >> (8 * j)) & 0xFFu);
                const uint64_t xb = gather64<T>(S.xr, col);
                if (S.s[rr] + j < S.e[rr])
                    acc[rr] = fma(__longlong_as_double((long long)S.vp[rr][j]),
                                  __longlong_as_double((long long)xb), acc[rr]);
            }
        const double *vv = A.v64 + S.off;
        for (int jj = 0; jj < more; ++jj)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int k = S.s[rr] + J + jj;
                const bool have = k < S.e[rr];
                const int col = have ? (int)__ldcs(ci + k) : 0;
                const double v = have ? __ldcs(vv + k) : 0.0;
                const uint64_t xb = gather64<T>(S.xr, col);
                if (have) acc[rr] = fma(v, __longlong_as_double((long long)xb), acc[rr]);
            }
    } else if (S.prec == EVOCG_FP32) {
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int col = (int)((S.cip[rr] >> (8 * j)) & 0xFFu);
                const uint32_t xb = gather32<T>(S.xr, col);
                if (S.s[rr] + j < S.e[rr])
                    pr[rr].add_prod(__uint_as_float((uint32_t)S.vp[rr][j]), __uint_as_float(xb));
            }
        const float *vv = A.v32 + S.off;
        for (int jj = 0; jj < more; ++jj)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int k = S.s[rr] + J + jj;
                const bool have = k < S.e[rr];
                const int col = have ? (int)__ldcs(ci + k) : 0;
                const float v = have ? __ldcs(vv + k) : 0.f;
                const uint32_t xb = gather32<T>(S.xr, col);
                if (have) pr[rr].add_prod(v, __uint_as_float(xb));
            }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int col = (int)((S.cip[rr] >> (8 * j)) & 0xFFu);
                const uint32_t xb = gather32<T>(S.xr, col);
                if (S.s[rr] + j < S.e[rr])  // BF16 x BF16 is exact in FP32
                    pr[rr].add(__fmul_rn(f32_from_bf16((uint16_t)S.vp[rr][j]),
                                         f32_from_bf16((uint16_t)xb)));
            }
        const unsigned short *vv = A.v16 + S.off;
        for (int jj = 0; jj < more; ++jj)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int k = S.s[rr] + J + jj;
                const bool have = k < S.e[rr];
                const int col = have ? (int)__ldcs(ci + k) : 0;
                const uint16_t v = have ? __ldcs(vv + k) : (unsigned short)0;
                const uint32_t xb = gather32<T>(S.xr, col);
                if (have) pr[rr].add(__fmul_rn(f32_from_bf16(v), f32_from_bf16((uint16_t)xb)));
            }
    }
}

}  // namespace evocg
