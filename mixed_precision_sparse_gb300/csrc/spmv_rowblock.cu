// spmv_rowblock.cu -- the row-block tile-wise mixed-precision SpMV for tiles of 32 (EvoCG,
// "Self-Evolving Precision Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 /
// Eq. 5) on sm_103a.
//
// Work mapping. A warp takes row blocks in a grid stride; lane l owns local row l and keeps
// its FP64 sum and its FP32 pair in registers for the whole row block (no cross-lane FP64
// reduction). The row block's work comes from its plan (rowblock_plan.cpp): the regular
// tiles' descriptors and the row-owned ELL block of its single-entry tiles.
//
// Latency. Every load a panel needs is issued ahead of it: a warp keeps three row blocks in
// flight -- the meta words of the one after next, the descriptors of the next one (lane i
// holding tile i) and, once their precisions are known, a bulk L2 prefetch of each of the
// next row block's tile slices in the value stream that tile will be read in, plus its
// column bytes (cp.async.bulk.prefetch.L2: no registers, no completion to wait for). The
// current row block's loads then hit L2, and they are issued together per tile (up to four
// levels at once), never one dependent load per entry.
//
// x. A tile's 32 x entries (its column block) are one coalesced load, one per lane, in the
// tile's format (FP64 x, or the scaled FP32 / BF16 copies); a slot takes its entry with a
// shuffle from the lane its local column names.
//
// Arithmetic (as the direct kernel): one FP64 fused multiply-add per FP64 entry; FP32 and
// BF16 products exact in FP32 pairs, summed error-free (TwoSum) into a hi/lo pair; the pair
// joins the FP64 sum once per row, and only in row blocks that have low-precision entries.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr unsigned kCbMask = (1u << 26) - 1u;
constexpr int kRbMinBlocks = 4;   // resident blocks of kRbThreads per SM the registers are sized for
constexpr int kSgUnroll = 2;      // single-entry tiles of a row loaded together

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Prefetch [p, p + bytes) into L2; p and bytes are multiples of 16 and the range lies inside
// one allocation.
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int PR> struct Fmt;
template <> struct Fmt<EVOCG_FP64> {
    using V = double;
    using X = double;
    static __device__ __forceinline__ const V *vals(const TilesView &A) { return A.v64; }
};
template <> struct Fmt<EVOCG_FP32> {
    using V = float;
    using X = float;
    static __device__ __forceinline__ const V *vals(const TilesView &A) { return A.v32; }
};
template <> struct Fmt<EVOCG_BF16> {
    using V = uint16_t;
    using X = float;
    static __device__ __forceinline__ const V *vals(const TilesView &A) { return A.v16; }
};

// Levels k .. k + W - 1 of one tile: the slots of the lanes whose row is in the tile are at
// s + u*h (s already holds the lane's slot column); the other lanes keep column 32, which
// selects nothing. The loads of all W levels are issued before the first product.
template <int PR, int W>
__device__ __forceinline__ void levels(const TilesView &A, unsigned s, unsigned h, bool mine,
                                       typename Fmt<PR>::X xs, double &acc, F32Pair &lp, unsigned &cnt)
{
    unsigned c[W];
    typename Fmt<PR>::V v[W];
#pragma unroll
    for (int u = 0; u < W; ++u) {
        c[u] = 32u;
        v[u] = 0;
        if (mine) {
            const unsigned q = s + (unsigned)u * h;
            c[u] = __ldcs(A.colIdx + q);
            v[u] = __ldcs(Fmt<PR>::vals(A) + q);
        }
    }
#pragma unroll
    for (int u = 0; u < W; ++u) {
        const typename Fmt<PR>::X xv = __shfl_sync(kAll, xs, (int)(c[u] & 31u));
        if (c[u] < 32u) {
            if constexpr (PR == EVOCG_FP64) acc = fma(v[u], xv, acc);
            else if constexpr (PR == EVOCG_FP32) lp.add_prod(v[u], xv);
            else lp.add(__fmul_rn(f32_from_bf16(v[u]), xv));   // BF16 x BF16: exact in FP32
            ++cnt;
        }
    }
}

template <int PR>
__device__ __forceinline__ void tile_levels(const TilesView &A, unsigned s, unsigned h, int w, bool mine,
                                            typename Fmt<PR>::X xs, double &acc, F32Pair &lp, unsigned &cnt)
{
    int k = 0;
    for (; k + 4 <= w; k += 4) levels<PR, 4>(A, s + (unsigned)k * h, h, mine, xs, acc, lp, cnt);
    const unsigned q = s + (unsigned)k * h;
    switch (w - k) {
    case 3: levels<PR, 3>(A, q, h, mine, xs, acc, lp, cnt); break;
    case 2: levels<PR, 2>(A, q, h, mine, xs, acc, lp, cnt); break;
    case 1: levels<PR, 1>(A, q, h, mine, xs, acc, lp, cnt); break;
    default: break;
    }
}

// Precision of the tile a lane's descriptor names (FP64 for lanes without one).
template <bool FORCE64>
__device__ __forceinline__ int desc_prec(const SpmvLaunch &L, const uint4 &d, bool have)
{
    if (FORCE64 || !have) return EVOCG_FP64;
    return (int)__ldg(L.prec + (L.map_kind ? (d.y & kCbMask) : d.w));
}

// The nt regular tiles whose descriptors the lanes hold (lane i: tile i).
template <bool FORCE64>
__device__ __forceinline__ void run_tiles(const SpmvLaunch &L, const uint4 &d, int pr, int nt, int lane,
                                          unsigned ltm, double &acc, F32Pair &lp, unsigned (&cnt)[3])
{
    const TilesView &A = L.A;
    for (int i = 0; i < nt; ++i) {
        const unsigned slot = __shfl_sync(kAll, d.x, i);
        const unsigned cbw = __shfl_sync(kAll, d.y, i);
        const unsigned mask = __shfl_sync(kAll, d.z, i);
        const int prec = FORCE64 ? EVOCG_FP64 : __shfl_sync(kAll, pr, i);
        const unsigned xi = (cbw & kCbMask) * 32u + (unsigned)lane;   // n < 2^31
        const bool xin = (int64_t)xi < A.n;
        const int w = (int)(cbw >> 26);
        const bool mine = (mask >> lane) & 1u;
        const unsigned h = __popc(mask);
        const unsigned s = slot + __popc(mask & ltm);   // slots < 2^32
        if (prec == EVOCG_FP64) {
            const double xs = xin ? __ldg(L.x64 + xi) : 0.0;
            tile_levels<EVOCG_FP64>(A, s, h, w, mine, xs, acc, lp, cnt[0]);
        } else if (prec == EVOCG_FP32) {
            const float xs = xin ? __ldg(L.x32 + xi) : 0.f;
            tile_levels<EVOCG_FP32>(A, s, h, w, mine, xs, acc, lp, cnt[1]);
        } else {
            const float xs = xin ? __ldg(L.x16f + xi) : 0.f;
            tile_levels<EVOCG_BF16>(A, s, h, w, mine, xs, acc, lp, cnt[2]);
        }
    }
}

// The row block's single-entry tiles: a lane whose row has some walks its ELL row, kSgUnroll
// entries at a time (columns and tile indices first, then precisions, then values and x).
template <bool FORCE64>
__device__ __forceinline__ void run_singles(const SpmvLaunch &L, unsigned sg0, unsigned hs, unsigned ws,
                                            int lane, unsigned ltm, double &acc, F32Pair &lp,
                                            unsigned (&cnt)[3])
{
    if (!((hs >> lane) & 1u)) return;
    const TilesView &A = L.A;
    const unsigned hc = __popc(hs);
    const size_t e0 = (size_t)sg0 + __popc(hs & ltm);
    for (unsigned k0 = 0; k0 < ws; k0 += kSgUnroll) {
        int col[kSgUnroll], prec[kSgUnroll];
        double av[kSgUnroll], xv[kSgUnroll];   // FP64 operands, or the FP32 ones in the low word
#pragma unroll
        for (int u = 0; u < kSgUnroll; ++u) {
            col[u] = -1;
            prec[u] = EVOCG_FP64;
            if (k0 + u < ws) {
                const size_t e = e0 + (size_t)(k0 + u) * hc;
                col[u] = __ldcs(A.sgCol + e);
                if (!FORCE64 && !L.map_kind) prec[u] = __ldcs(A.sgTile + e);   // tile index for now
            }
        }
#pragma unroll
        for (int u = 0; u < kSgUnroll; ++u)
            if (!FORCE64 && col[u] >= 0)
                prec[u] = (int)__ldg(L.prec + (L.map_kind ? (col[u] >> 5) : prec[u]));
#pragma unroll
        for (int u = 0; u < kSgUnroll; ++u) {
            av[u] = 0.0;
            xv[u] = 0.0;
            if (col[u] < 0) continue;
            const size_t e = e0 + (size_t)(k0 + u) * hc;
            if (prec[u] == EVOCG_FP64) {
                av[u] = __ldcs(A.sgV64 + e);
                xv[u] = __ldg(L.x64 + col[u]);
            } else if (prec[u] == EVOCG_FP32) {
                av[u] = __longlong_as_double((long long)__float_as_uint(__ldcs(A.sgV32 + e)));
                xv[u] = __longlong_as_double((long long)__float_as_uint(__ldg(L.x32 + col[u])));
            } else {
                av[u] = __longlong_as_double((long long)((unsigned)__ldcs(A.sgV16 + e) << 16));
                xv[u] = __longlong_as_double((long long)__float_as_uint(__ldg(L.x16f + col[u])));
            }
        }
#pragma unroll
        for (int u = 0; u < kSgUnroll; ++u) {
            if (col[u] < 0) continue;
            const float a = __uint_as_float((unsigned)__double_as_longlong(av[u]));
            const float x = __uint_as_float((unsigned)__double_as_longlong(xv[u]));
            if (prec[u] == EVOCG_FP64) { acc = fma(av[u], xv[u], acc); ++cnt[0]; }
            else if (prec[u] == EVOCG_FP32) { lp.add_prod(a, x); ++cnt[1]; }
            else { lp.add(__fmul_rn(a, x)); ++cnt[2]; }
        }
    }
}

template <bool FORCE64, bool DOT>
__global__ void __launch_bounds__(kRbThreads, kRbMinBlocks) spmv_rowblock_kernel(SpmvLaunch L)
{
    if ((DOT || L.gate) && L.st->done) return;  // a stopped solve: nothing to compute or count
    const TilesView &A = L.A;
    const int lane = threadIdx.x & 31;
    const unsigned ltm = lanemask_lt();
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nw = (int64_t)gridDim.x * wpb;
    const int64_t wid = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t nrb = A.nrb;
    double dotp = 0.0;
    unsigned cnt[3] = {0u, 0u, 0u};

    // meta words of a row block, one per lane: lanes 0-3 hold meta[rb] (first descriptor,
    // first single slot, single rows, singles per row), lane 4 meta[rb + 1]'s first descriptor
    auto meta = [&](int64_t rb) {
        unsigned m = 0u;
        if (rb < nrb && lane < 5) m = __ldg(reinterpret_cast<const unsigned *>(A.rbMeta + rb) + lane);
        return m;
    };
    auto ntiles = [&](unsigned m) { return __shfl_sync(kAll, m, 4) - __shfl_sync(kAll, m, 0); };
    // descriptors of a row block's first 32 regular tiles, lane i holding tile i
    auto descs = [&](int64_t rb, unsigned m) {
        const unsigned r0 = __shfl_sync(kAll, m, 0), nt = ntiles(m);
        uint4 d = make_uint4(0u, 0u, 0u, 0u);
        if (rb < nrb && (unsigned)lane < nt) d = __ldcs(A.rgDesc + r0 + lane);
        return d;
    };
    auto prefetch = [&](int64_t rb, unsigned m, const uint4 &d, int pr) {
        const unsigned nt = ntiles(m);
        if (rb >= nrb || (unsigned)lane >= nt) return;
        const unsigned m16 = ((d.y >> 26) * (unsigned)__popc(d.z) + 15u) & ~15u;
        if (pr == EVOCG_FP64) prefetch_l2(A.v64 + d.x, m16 * 8u);
        else if (pr == EVOCG_FP32) prefetch_l2(A.v32 + d.x, m16 * 4u);
        else prefetch_l2(A.v16 + d.x, m16 * 2u);
        prefetch_l2(A.colIdx + d.x, m16);
    };

    int64_t rb = wid;
    unsigned m0 = meta(rb);
    uint4 d0 = descs(rb, m0);
    int p0 = desc_prec<FORCE64>(L, d0, rb < nrb && (unsigned)lane < ntiles(m0));
    unsigned m1 = meta(rb + nw);
    unsigned m2 = meta(rb + 2 * nw);
    uint4 d1 = descs(rb + nw, m1);
    while (rb < nrb) {
        const int p1 = desc_prec<FORCE64>(L, d1, rb + nw < nrb && (unsigned)lane < ntiles(m1));
        double acc = 0.0;
        F32Pair lp;
        const unsigned nt = ntiles(m0);
        run_singles<FORCE64>(L, __shfl_sync(kAll, m0, 1), __shfl_sync(kAll, m0, 2),
                             __shfl_sync(kAll, m0, 3), lane, ltm, acc, lp, cnt);
        prefetch(rb + nw, m1, d1, p1);
        run_tiles<FORCE64>(L, d0, p0, nt < 32u ? (int)nt : 32, lane, ltm, acc, lp, cnt);
        for (unsigned c0 = 32; c0 < nt; c0 += 32) {   // a row block of more than 32 regular tiles
            const unsigned r0 = __shfl_sync(kAll, m0, 0);
            const bool have = (unsigned)lane < nt - c0;
            const uint4 d = have ? __ldcs(A.rgDesc + r0 + c0 + lane) : make_uint4(0u, 0u, 0u, 0u);
            run_tiles<FORCE64>(L, d, desc_prec<FORCE64>(L, d, have), nt - c0 < 32u ? (int)(nt - c0) : 32,
                               lane, ltm, acc, lp, cnt);
        }
        const bool low = !FORCE64 && __any_sync(kAll, lp.hi != 0.f || lp.lo != 0.f);
        const int64_t row = rb * 32 + lane;
        if (row < A.n) {
            double y = acc;
            if (low) y = acc + (f64_from_f32(lp.hi) + f64_from_f32(lp.lo));
            L.y[row] = y;
            if (DOT) dotp = fma(__ldg(L.x64 + row), y, dotp);
        }
        rb += nw;
        m0 = m1;
        d0 = d1;
        p0 = p1;
        m1 = m2;
        d1 = descs(rb + nw, m1);
        m2 = meta(rb + 2 * nw);
    }
    if (L.census) {
        for (int o = 16; o; o >>= 1) {
            cnt[0] += __shfl_xor_sync(kAll, cnt[0], o);
            cnt[1] += __shfl_xor_sync(kAll, cnt[1], o);
            cnt[2] += __shfl_xor_sync(kAll, cnt[2], o);
        }
        if (lane == 0) {
            if (cnt[0]) atomicAdd(&L.st->census[0], (unsigned long long)cnt[0]);
            if (cnt[1]) atomicAdd(&L.st->census[1], (unsigned long long)cnt[1]);
            if (cnt[2]) atomicAdd(&L.st->census[2], (unsigned long long)cnt[2]);
        }
    }
    if (DOT) {   // this warp's p.q partial (lanes summed in a fixed tree)
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(kAll, dotp, o);
        if (lane == 0) L.pq[wid] = dotp;
    }
}

}  // namespace

int rowblock_grid_for(int sms)
{
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_rowblock_kernel<false, true>, kRbThreads, 0) !=
            cudaSuccess || per < 1)
        per = 1;
    cudaGetLastError();
    const int g = sms * per;
    return g > kMaxBlocks ? kMaxBlocks : g;
}

cudaError_t launch_spmv_rowblock(const SpmvLaunch &L, cudaStream_t s)
{
    const int g = L.A.rb_grid;
    if (g <= 0 || !L.A.rbMeta) return cudaErrorInvalidValue;
    if (L.force64) {
        if (L.dot) spmv_rowblock_kernel<true, true><<<g, kRbThreads, 0, s>>>(L);
        else spmv_rowblock_kernel<true, false><<<g, kRbThreads, 0, s>>>(L);
    } else {
        if (L.dot) spmv_rowblock_kernel<false, true><<<g, kRbThreads, 0, s>>>(L);
        else spmv_rowblock_kernel<false, false><<<g, kRbThreads, 0, s>>>(L);
    }
    return cudaGetLastError();
}

}  // namespace evocg
