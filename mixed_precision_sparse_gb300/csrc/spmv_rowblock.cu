// spmv_rowblock.cu -- the row-block tile-wise mixed-precision SpMV for tiles of 32 (EvoCG,
// "Self-Evolving Precision Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 /
// Eq. 5) on sm_103a.
//
// Work mapping. A warp takes row blocks in a grid stride; lane l owns local row l and keeps
// its FP64 sum and its FP32 pair in registers for the whole row block (no cross-lane FP64
// reduction). The row block's work comes from its plan (rowblock_plan.cpp): the regular
// tiles' descriptors and the row-owned ELL block of its single-entry tiles.
//
// Latency. A row block's descriptors and precisions are loaded lane-parallel one row block
// ahead (lane i holding tile i), and a tile's loads are issued together (up to four levels at
// once) before its first product. Single-entry tiles are the exception the plan isolates:
// each needs its own column before its precision, value and x entry can be fetched, a chain
// of dependent loads per entry. So a warp stages the next row block's single-entry operands in
// shared memory with per-lane asynchronous copies (cp.async: both values, the x entry in all
// three formats and the 4-byte word holding its precision code), from columns loaded two row
// blocks ahead; the owner lanes then read them from shared memory. Completion is the copies'
// own group count (cp.async.wait_group): no device-side wait.
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
constexpr int kSgUnroll = 2;      // single-entry tiles of a row loaded together (unstaged path)
constexpr unsigned kSgMax = 32;   // ELL slots of a row block staged in shared memory (more: unstaged)

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Asynchronous global -> shared copies of 4 and 8 bytes; completion by group count.
__device__ __forceinline__ void cp4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ unsigned lds_u32(uint32_t a)
{
    unsigned v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ double lds_f64(uint32_t a)
{
    double v;
    asm volatile("ld.shared.f64 %0, [%1];" : "=d"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_u32(uint32_t a, unsigned v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Staged single-entry operands of one row block (ELL slot e < kSgMax), as arrays: FP64 value
// and x at 8e and 256 + 8e, FP32 value and x at 512 + 4e and 640 + 4e, the 4-byte words
// holding the BF16 value and the precision code at 768 + 4e and 1024 + 4e, the BF16 x at
// 896 + 4e, and the slot's code word at 1152 + 4e (bit 0: an entry; bit 1: the BF16 half;
// bits 2-3: the precision's byte in its word).
constexpr unsigned kSgBuf = 1280;

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

// The row block's single-entry tiles read from global memory (a row block with more ELL slots
// than a buffer holds): a lane whose row has some walks its ELL row, kSgUnroll entries at a
// time (columns and tile indices first, then precisions, then values and x).
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

// The staged single-entry tiles of a row block: owner lanes walk their ELL row in the buffer.
template <bool FORCE64>
__device__ __forceinline__ void staged_singles(uint32_t sb, unsigned hs, unsigned ws, int lane, unsigned ltm,
                                               double &acc, F32Pair &lp, unsigned (&cnt)[3])
{
    if (!((hs >> lane) & 1u)) return;
    const unsigned hc = __popc(hs), j = __popc(hs & ltm);
    for (unsigned k = 0; k < ws; ++k) {
        const unsigned e = k * hc + j;
        const unsigned code = lds_u32(sb + 1152u + 4u * e);
        if (!(code & 1u)) continue;   // a pad
        const int prec = FORCE64 ? EVOCG_FP64
                                 : (int)((lds_u32(sb + 1024u + 4u * e) >> (8u * ((code >> 2) & 3u))) & 0xFFu);
        if (prec == EVOCG_FP64) {
            acc = fma(lds_f64(sb + 8u * e), lds_f64(sb + 256u + 8u * e), acc);
            ++cnt[0];
        } else if (prec == EVOCG_FP32) {
            lp.add_prod(__uint_as_float(lds_u32(sb + 512u + 4u * e)), __uint_as_float(lds_u32(sb + 640u + 4u * e)));
            ++cnt[1];
        } else {
            const unsigned w = lds_u32(sb + 768u + 4u * e);
            const float a = f32_from_bf16((uint16_t)((code & 2u) ? (w >> 16) : (w & 0xFFFFu)));
            lp.add(__fmul_rn(a, __uint_as_float(lds_u32(sb + 896u + 4u * e))));
            ++cnt[2];
        }
    }
}

template <bool FORCE64, bool DOT>
__global__ void __launch_bounds__(kRbThreads, kRbMinBlocks) spmv_rowblock_kernel(SpmvLaunch L)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
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
    const uint32_t sgbuf = smem_u32(smem_raw) + (uint32_t)(threadIdx.x >> 5) * 2u * kSgBuf;

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
    auto nslots = [&](unsigned m) { return __popc(__shfl_sync(kAll, m, 2)) * __shfl_sync(kAll, m, 3); };
    // a row block's single-entry columns and tiles, lane e holding ELL slot e (when it has at
    // most kSgMax slots: those are staged)
    auto sgload = [&](int64_t rb, unsigned m, int &col, int &tile) {
        const unsigned sg0 = __shfl_sync(kAll, m, 1), ns = nslots(m);
        col = -1;
        tile = 0;
        if (rb < nrb && ns <= kSgMax && (unsigned)lane < ns) {
            col = __ldg(A.sgCol + sg0 + lane);
            if (!FORCE64 && !L.map_kind) tile = __ldg(A.sgTile + sg0 + lane);
        }
    };
    // issue the copies of a row block's single-entry operands into buffer sb (one group)
    auto stage = [&](int64_t rb, unsigned m, int col, int tile, uint32_t sb) {
        const unsigned sg0 = __shfl_sync(kAll, m, 1), ns = nslots(m);
        if (rb < nrb && ns <= kSgMax && (unsigned)lane < ns) {
            const unsigned e = (unsigned)lane, g = sg0 + e;
            unsigned code = 0u;
            if (col >= 0) {
                cp8(sb + 8u * e, A.sgV64 + g);
                cp8(sb + 256u + 8u * e, L.x64 + col);
                unsigned key = 0u;
                if (!FORCE64) {   // an all-FP64 product reads no low-precision operand (x32 and
                                  // x16f may not exist for it)
                    cp4(sb + 512u + 4u * e, A.sgV32 + g);
                    cp4(sb + 640u + 4u * e, L.x32 + col);
                    cp4(sb + 768u + 4u * e, A.sgV16 + (g & ~1u));
                    cp4(sb + 896u + 4u * e, L.x16f + col);
                    key = L.map_kind ? ((unsigned)col >> 5) : (unsigned)tile;
                    cp4(sb + 1024u + 4u * e, L.prec + (key & ~3u));
                }
                code = 1u | ((g & 1u) << 1) | ((key & 3u) << 2);
            }
            sts_u32(sb + 1152u + 4u * e, code);
        }
        cp_commit();
    };

    int64_t rb = wid;
    unsigned m0 = meta(rb);
    uint4 d0 = descs(rb, m0);
    int p0 = desc_prec<FORCE64>(L, d0, rb < nrb && (unsigned)lane < ntiles(m0));
    unsigned m1 = meta(rb + nw);
    unsigned m2 = meta(rb + 2 * nw);
    uint4 d1 = descs(rb + nw, m1);
    int sc, st;   // single-entry columns and tiles of the row block after the next one
    sgload(rb, m0, sc, st);
    stage(rb, m0, sc, st, sgbuf);
    sgload(rb + nw, m1, sc, st);
    unsigned buf = 0u;
    while (rb < nrb) {
        const int p1 = desc_prec<FORCE64>(L, d1, rb + nw < nrb && (unsigned)lane < ntiles(m1));
        stage(rb + nw, m1, sc, st, sgbuf + (buf ^ 1u) * kSgBuf);   // the next row block's singles
        sgload(rb + 2 * nw, m2, sc, st);
        double acc = 0.0;
        F32Pair lp;
        const unsigned nt = ntiles(m0);
        const unsigned hs = __shfl_sync(kAll, m0, 2), ws = __shfl_sync(kAll, m0, 3);
        if (__popc(hs) * ws <= kSgMax) {
            cp_wait1();   // this row block's copies (the older group) have landed
            __syncwarp();
            staged_singles<FORCE64>(sgbuf + buf * kSgBuf, hs, ws, lane, ltm, acc, lp, cnt);
        } else {
            run_singles<FORCE64>(L, __shfl_sync(kAll, m0, 1), hs, ws, lane, ltm, acc, lp, cnt);
        }
        __syncwarp();   // the buffer is refilled two row blocks later
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
        buf ^= 1u;
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
    if (DOT) {   // this block's p.q partial: lanes in a fixed tree, then the warps in order
        __shared__ double s_pq[kRbThreads / 32];
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(kAll, dotp, o);
        if (lane == 0) s_pq[threadIdx.x >> 5] = dotp;
        __syncthreads();
        if (threadIdx.x == 0) {
            double v = 0.0;
            for (int i = 0; i < kRbThreads / 32; ++i) v += s_pq[i];
            L.pq[blockIdx.x] = v;
        }
    }
}

constexpr size_t kRbSmem = (size_t)(kRbThreads / 32) * 2u * kSgBuf;

}  // namespace

int rowblock_grid_for(int sms)
{
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_rowblock_kernel<false, true>, kRbThreads,
                                                      kRbSmem) != cudaSuccess || per < 1)
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
        if (L.dot) spmv_rowblock_kernel<true, true><<<g, kRbThreads, kRbSmem, s>>>(L);
        else spmv_rowblock_kernel<true, false><<<g, kRbThreads, kRbSmem, s>>>(L);
    } else {
        if (L.dot) spmv_rowblock_kernel<false, true><<<g, kRbThreads, kRbSmem, s>>>(L);
        else spmv_rowblock_kernel<false, false><<<g, kRbThreads, kRbSmem, s>>>(L);
    }
    return cudaGetLastError();
}

}  // namespace evocg
