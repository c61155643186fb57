// spmv_panel.cu -- the tile-wise mixed-precision SpMV (EvoCG, "Self-Evolving Precision Control
// for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 / Eq. 5) as a panel-streaming kernel for
// sm_103a.
//
// Work mapping. A panel is R consecutive rows (R = 32, or 16 for 16 x 16 tiles). Every warp
// owns a contiguous range of panels (a static plan balanced by slots) and streams their tile
// descriptors in order: one 16-byte record per panel (its tile count and first slot) followed
// by one per tile (slot offset, width, column block, row mask). Lane l owns row l of the
// current panel and keeps its sums in registers: no cross-lane reduction of any row.
//
// Staging. Each warp owns one shared-memory stage with its own mbarrier. A panel's tiles come
// in batches planned on the host (panel_plan.cpp: every tile sized for FP64, so the plan holds
// for any precision map), each tile with a fixed stage offset. For a batch every lane that
// holds a tile issues that tile's copies itself, all lanes at once, as bulk asynchronous
// copies (cp.async.bulk) completing on the stage's mbarrier: the tile's value slice in the
// stream its precision selects, its local-column bytes and its x segment in that precision
// (the builder aligns every tile with more than one slot to 16 slots and pads it to a multiple
// of 16, so every slice is a whole number of 16-byte units). Single-entry tiles (one row,
// width one: the panel-edge tiles of stencils, most of a stencil's tiles by count) copy just
// their value and x entry (cp.async, 4 or 8 bytes). The warp then waits for the mbarrier's
// phase (bounded in time: a wait that runs out sets the handle's error word and the warp
// stops) and computes the batch from shared memory. The next panel's descriptors and their
// precisions are loaded while the current panel is in flight. A tile too large for the stage
// on its own is computed from global memory level by level.
//
// Arithmetic. On GB300 the FP64 unit issues about two operations per clock per SM, so FP64
// instructions go only where the data is FP64: one fused multiply-add per FP64 entry. FP32
// and BF16 entries never touch it: their products are exact in an FP32 pair (BF16 x BF16
// fits in FP32; an FP32 x FP32 product is split by one fused multiply-add), summed
// error-free (TwoSum) into an FP32 pair per row, and merged into the FP64 row sum with two
// FP64 adds per row. Each row is thus the FP64 sum of the exactly rounded-operand products
// of EvoCG's error model, to about 1e-15 of the row's absolute sum.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

namespace {

constexpr unsigned kAll = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Small asynchronous global -> shared copies (a single entry's value or x entry); completion is
// awaited with cp_wait_all by the same threads.
__device__ __forceinline__ void cp8(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Bulk global -> shared copy completing on an mbarrier: dst, src 16-byte aligned, bytes a
// positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
// One bounded test of the phase: the thread may be suspended until the phase completes or
// about suspend_ns have passed (a suspended warp issues nothing while its copies are in flight).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(suspend_ns) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the mbarrier phase with the given parity, for at most about limit_ns of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    constexpr uint32_t kSuspendNs = 100000;   // one test sleeps up to 0.1 ms
    if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    const uint64_t t0 = global_ns();
    do {
        if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    } while (global_ns() - t0 < limit_ns);
    return false;
}

// Error-free FP32 accumulation: s + c carries the running sum, the rounding of each add kept
// in c (Knuth's TwoSum).
__device__ __forceinline__ void acc_low(float &s, float &c, float p)
{
    const float t = __fadd_rn(s, p);
    const float bp = __fsub_rn(t, s);
    c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp)));
    s = t;
}

// a * b added exactly (as p + e, e from one fused multiply-add) to the pair (s, c).
__device__ __forceinline__ void acc_prod(float &s, float &c, float a, float b)
{
    const float p = __fmul_rn(a, b);
    const float e = __fmaf_rn(a, b, -p);
    acc_low(s, c, p);
    c = __fadd_rn(c, e);
}

// One row's entries of a full tile (all 32 rows present, so the lane's slots are lane, lane + 32,
// ...) with W levels known at compile time: constant offsets in the stage, no row mapping.
// tb: the tile's stage area (values from tb, column bytes from tb + 8 m16, x from tb + 9 m16).
template <int PR, int W, int C, bool DOT>
__device__ __forceinline__ void full_tile(const unsigned char *tb, unsigned m16, int lane, double &acc,
                                          float &ls, float &lc, unsigned &cnt)
{
    const unsigned char *cs = tb + 8u * m16 + lane;
    if (PR == EVOCG_FP64) {
        const double *vs = reinterpret_cast<const double *>(tb) + lane;
        const double *xs = reinterpret_cast<const double *>(tb + 9u * m16);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const unsigned c = cs[32 * k];
            const double a = vs[32 * k], xv = xs[c & (C - 1)];
            if (c < (unsigned)C) { acc = fma(a, xv, acc); if (DOT) ++cnt; }
        }
    } else if (PR == EVOCG_FP32) {
        const float *vs = reinterpret_cast<const float *>(tb) + lane;
        const float *xs = reinterpret_cast<const float *>(tb + 9u * m16);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const unsigned c = cs[32 * k];
            const float a = vs[32 * k], xv = xs[c & (C - 1)];
            if (c < (unsigned)C) { acc_prod(ls, lc, a, xv); if (DOT) ++cnt; }
        }
    } else {
        const unsigned short *vs = reinterpret_cast<const unsigned short *>(tb) + lane;
        const float *xs = reinterpret_cast<const float *>(tb + 9u * m16);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const unsigned c = cs[32 * k];
            const float a = __uint_as_float((unsigned)vs[32 * k] << 16), xv = xs[c & (C - 1)];
            if (c < (unsigned)C) { acc_low(ls, lc, __fmul_rn(a, xv)); if (DOT) ++cnt; }   // exact
        }
    }
}

// Any tile's rows: lane's slots are j, j + h, ... (j = the lane's rank among the tile's rows).
template <int PR, int C, bool DOT>
__device__ __forceinline__ void any_tile(const unsigned char *tb, unsigned m16, unsigned wi, unsigned hi,
                                         unsigned j, double &acc, float &ls, float &lc, unsigned &cnt)
{
    const unsigned char *cs = tb + 8u * m16 + j;
    for (unsigned k = 0; k < wi; ++k) {
        const unsigned c = cs[k * hi];
        if (PR == EVOCG_FP64) {
            const double a = reinterpret_cast<const double *>(tb)[j + k * hi];
            const double xv = reinterpret_cast<const double *>(tb + 9u * m16)[c & (C - 1)];
            if (c < (unsigned)C) { acc = fma(a, xv, acc); if (DOT) ++cnt; }
        } else if (PR == EVOCG_FP32) {
            const float a = reinterpret_cast<const float *>(tb)[j + k * hi];
            const float xv = reinterpret_cast<const float *>(tb + 9u * m16)[c & (C - 1)];
            if (c < (unsigned)C) { acc_prod(ls, lc, a, xv); if (DOT) ++cnt; }
        } else {
            const float a = __uint_as_float((unsigned)reinterpret_cast<const unsigned short *>(tb)[j + k * hi] << 16);
            const float xv = reinterpret_cast<const float *>(tb + 9u * m16)[c & (C - 1)];
            if (c < (unsigned)C) { acc_low(ls, lc, __fmul_rn(a, xv)); if (DOT) ++cnt; }
        }
    }
}

template <int PR, int C, bool DOT>
__device__ __forceinline__ void tile_rows(const unsigned char *tb, unsigned m16, unsigned wi, unsigned mi,
                                          int lane, unsigned ltm, double &acc, float &ls, float &lc,
                                          unsigned &cnt)
{
    if (mi == 0xFFFFFFFFu) {   // every row of a 32-row panel: the stencil case
        switch (wi) {
        case 1: full_tile<PR, 1, C, DOT>(tb, m16, lane, acc, ls, lc, cnt); return;
        case 2: full_tile<PR, 2, C, DOT>(tb, m16, lane, acc, ls, lc, cnt); return;
        case 3: full_tile<PR, 3, C, DOT>(tb, m16, lane, acc, ls, lc, cnt); return;
        default: any_tile<PR, C, DOT>(tb, m16, wi, 32u, (unsigned)lane, acc, ls, lc, cnt); return;
        }
    }
    if ((mi >> lane) & 1u)
        any_tile<PR, C, DOT>(tb, m16, wi, (unsigned)__popc(mi), (unsigned)__popc(mi & ltm), acc, ls, lc, cnt);
}

// Record flags (panel_plan.cpp).
constexpr unsigned kSingleBit = 1u << 26;
constexpr unsigned kFirstBit = 1u << 8, kLastBit = 1u << 9, kDirectBit = 1u << 10;
constexpr uint64_t kWaitNs = 2000000000ull;   // a stage wait longer than 2 s is declared lost
constexpr uint64_t kTestWaitNs = 2000000ull;  // the limit under the lost-wait test hook (2 ms)
constexpr uint32_t kSingleSlots = 16;         // stage offset of the single-entry slots

// Everything a batch needs on its way through the pipeline: its record window (lane 0: the
// header, lanes 1..tiles: the tiles), the lane's tile precision, and its record index.
struct Batch {
    uint4 w;
    int prec;
    int64_t rec;
};

// Precision of lane's tile: a per-tile map is read in record order (the library keeps it so),
// which needs only the record index; a per-column-block map needs the tile's column block.
// Every lane of the warp must call it (the tile count comes from lane 0 by shuffle); only lanes
// 1..tiles read a map.
template <bool FORCE64>
__device__ __forceinline__ int batch_prec(const SpmvLaunch &L, const Batch &b, int lane)
{
    const unsigned nt = __shfl_sync(kAll, b.w.x, 0) & 0xFFu;
    if (FORCE64 || lane == 0 || lane > (int)nt) return 0;
    if (!L.map_kind) return (int)__ldcs(L.A.recPrec + b.rec + lane);
    return (int)__ldg(L.prec + (int)b.w.z);
}

// Record layout and batches: panel_plan.cpp. SB: bytes of one of the warp's two stages; MB:
// blocks per SM the registers are sized for.
template <int R, int C, bool FORCE64, bool DOT, int SB, int MB, bool IL>
__global__ void __launch_bounds__(kPanelThreads, MB) spmv_panel_kernel(SpmvLaunch L)
{
    static_assert(R == 16 || R == 32, "panel rows");
    static_assert(C == R, "this kernel reads tiles as wide as the panel is tall");
    static_assert(!IL, "batches are streamed over contiguous panel ranges");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    if ((DOT || L.gate) && L.st->done) return;
    const TilesView &A = L.A;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
    unsigned char *const stages = smem_raw + (size_t)wib * 2 * SB;
    const uint32_t sbase = smem_addr(stages);
    const unsigned ltm = lanemask_lt();
    const uint64_t wait_ns = L.test_lost_wait ? kTestWaitNs : kWaitNs;
    if (lane == 0) {   // one mbarrier at the head of each stage, 32 arrivals a phase
        mbar_init(sbase, 32u);
        mbar_init(sbase + SB, 32u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // x segments go as bulk copies when x's base is 16-byte aligned (the library's own copies
    // always are); a misaligned FP64 x is copied entry by entry
    const bool x64al = (reinterpret_cast<uintptr_t>(L.x64) & 15u) == 0;
    const int64_t rec_end = A.warpRec[wid + 1];
    double dotp = 0.0;
    unsigned cnt0 = 0, cnt1 = 0, cnt2 = 0;
    unsigned phases = 0u;          // bit s: parity of stage s's next phase
    bool lost = false;

    // ---- issue a batch's copies into stage s (returns whether the stage was armed)
    auto issue = [&](const Batch &b, int s) -> bool {
        const unsigned hx = __shfl_sync(kAll, b.w.x, 0);
        if (hx & kDirectBit) return false;                 // computed from global memory
        const unsigned nt = hx & 0xFFu;
        const uint32_t st = sbase + (uint32_t)s * SB;
        unsigned char *const stp = stages + (size_t)s * SB;
        const bool mine = lane >= 1 && lane <= (int)nt;
        const bool single = mine && (b.w.y & kSingleBit);
        const bool reg = mine && !single;
        const int prec = b.prec;
        const unsigned m16 = (((b.w.y & 0xFFu) * (unsigned)__popc(b.w.w)) + 15u) & ~15u;
        const unsigned sz = 8u >> prec;   // 8, 4, 2 bytes
        const uint32_t tst = st + ((b.w.y >> 8) & 0xFFFu) * 16u;
        const int64_t xj0 = (int64_t)(int)b.w.z * C;
        const bool xbulk = reg && (prec != EVOCG_FP64 || x64al) && xj0 + C <= A.n;
        uint32_t bytes = 0;
        if (reg) bytes = m16 * sz + m16 + (xbulk ? (uint32_t)C * (prec == EVOCG_FP64 ? 8u : 4u) : 0u);
        const bool withhold = L.test_lost_wait && lane == 0 && b.rec == A.warpRec[wid];
        if (!withhold) {
            if (bytes) mbar_arrive_expect_tx(st, bytes);
            else mbar_arrive(st);
        }
        if (reg) {
            const unsigned char *vs =
                prec == EVOCG_FP64 ? reinterpret_cast<const unsigned char *>(A.v64)
                : prec == EVOCG_FP32 ? reinterpret_cast<const unsigned char *>(A.v32)
                                     : reinterpret_cast<const unsigned char *>(A.v16);
            bulk_g2s(tst, vs + (size_t)b.w.x * sz, m16 * sz, st);
            bulk_g2s(tst + 8u * m16, A.colIdx + b.w.x, m16, st);
            if (xbulk) {
                if (prec == EVOCG_FP64) bulk_g2s(tst + 9u * m16, L.x64 + xj0, 8u * C, st);
                else bulk_g2s(tst + 9u * m16, (prec == EVOCG_FP32 ? L.x32 : L.x16f) + xj0, 4u * C, st);
            }
        }
        // x segments that cannot go in bulk (a misaligned FP64 x, the last column block of a
        // matrix whose order is not a multiple of T): entry by entry
        unsigned xs = __ballot_sync(kAll, reg && !xbulk);
        while (xs) {
            const int i = __ffs(xs) - 1;
            xs &= xs - 1u;
            const int pi = __shfl_sync(kAll, prec, i);
            const int64_t xj = (int64_t)__shfl_sync(kAll, (int)b.w.z, i) * C + lane;
            const uint32_t xst = __shfl_sync(kAll, tst, i) + 9u * __shfl_sync(kAll, m16, i);
            if (lane < C && xj < A.n) {
                if (pi == EVOCG_FP64) cp8(xst + 8u * lane, L.x64 + xj);
                else cp4(xst + 4u * lane, (pi == EVOCG_FP32 ? L.x32 : L.x16f) + xj);
            }
        }
        // single-entry tiles: their value and x entry into the lane's own 16-byte slot
        if (single) {
            const uint32_t sd = st + kSingleSlots + (uint32_t)lane * 16u;
            const int64_t xj = xj0 + (int64_t)((b.w.y >> 20) & 0x3Fu);
            if (prec == EVOCG_FP64) {
                cp8(sd, A.v64 + b.w.x);
                cp8(sd + 8u, L.x64 + xj);
            } else if (prec == EVOCG_FP32) {
                cp4(sd, A.v32 + b.w.x);
                cp4(sd + 8u, L.x32 + xj);
            } else {
                cp4(sd, A.v16 + (b.w.x & ~1u));   // the aligned pair holding it
                cp4(sd + 8u, L.x16f + xj);
            }
        }
        (void)stp;
        asm volatile("cp.async.commit_group;" ::: "memory");
        return true;
    };

    // ---- wait for stage s, then compute batch b from it (or from global memory when direct)
    auto compute = [&](const Batch &b, int s, bool armed, bool newest, double &acc, float &ls,
                       float &lc) -> bool {
        const unsigned hx = __shfl_sync(kAll, b.w.x, 0);
        const unsigned nt = hx & 0xFFu;
        const bool mine = lane >= 1 && lane <= (int)nt;
        const int prec = b.prec;
        if (hx & kDirectBit) {   // one tile larger than a stage: level by level from global memory
            const int pi = __shfl_sync(kAll, prec, 1);
            const unsigned so = __shfl_sync(kAll, b.w.x, 1);
            const int cbi = __shfl_sync(kAll, (int)b.w.z, 1);
            const unsigned mi = __shfl_sync(kAll, b.w.w, 1);
            const int wi = (int)(__shfl_sync(kAll, b.w.y, 1) & 0xFFu), hi = __popc(mi);
            const bool has = lane < R && ((mi >> lane) & 1u);
            const unsigned s0 = so + (unsigned)__popc(mi & ltm);
            for (int k = 0; has && k < wi; ++k) {
                const unsigned sl = s0 + (unsigned)(k * hi);
                const unsigned c = A.colIdx[sl];
                if (c >= (unsigned)C) continue;
                const int64_t xj = (int64_t)cbi * C + c;
                if (pi == EVOCG_FP64) {
                    acc = fma(__ldcs(A.v64 + sl), __ldg(L.x64 + xj), acc);
                    if (DOT) ++cnt0;
                } else if (pi == EVOCG_FP32) {
                    acc_prod(ls, lc, __ldcs(A.v32 + sl), __ldg(L.x32 + xj));
                    if (DOT) ++cnt1;
                } else {
                    const unsigned bb = __ldcs(reinterpret_cast<const unsigned short *>(A.v16) + sl);
                    acc_low(ls, lc, __fmul_rn(__uint_as_float(bb << 16), __ldg(L.x16f + xj)));
                    if (DOT) ++cnt2;
                }
            }
            return true;
        }
        if (armed) {
            // this batch's small copies (not the newest group when another batch is in flight)
            if (newest) asm volatile("cp.async.wait_group 0;" ::: "memory");
            else asm volatile("cp.async.wait_group 1;" ::: "memory");
            const uint32_t st = sbase + (uint32_t)s * SB;
            const bool ok = mbar_wait_bounded(st, (phases >> s) & 1u, wait_ns);
            phases ^= 1u << s;
            if (!__all_sync(kAll, ok)) return false;
            __syncwarp();
        }
        unsigned char *const stp = stages + (size_t)s * SB;
        const unsigned single = __ballot_sync(kAll, mine && (b.w.y & kSingleBit));
        unsigned tr = __ballot_sync(kAll, mine) & ~single;
        const unsigned m16 = (((b.w.y & 0xFFu) * (unsigned)__popc(b.w.w)) + 15u) & ~15u;
        while (tr) {
            const int i = __ffs(tr) - 1;
            tr &= tr - 1u;
            const unsigned y = __shfl_sync(kAll, b.w.y, i);
            const unsigned mi = __shfl_sync(kAll, b.w.w, i);
            const int pi = __shfl_sync(kAll, prec, i);
            const unsigned mt = __shfl_sync(kAll, m16, i);
            if (lane >= R) continue;
            const unsigned char *tb = stp + ((y >> 8) & 0xFFFu) * 16u;
            const unsigned wi = y & 0xFFu;
            if (pi == EVOCG_FP64) tile_rows<EVOCG_FP64, C, DOT>(tb, mt, wi, mi, lane, ltm, acc, ls, lc, cnt0);
            else if (pi == EVOCG_FP32) tile_rows<EVOCG_FP32, C, DOT>(tb, mt, wi, mi, lane, ltm, acc, ls, lc, cnt1);
            else tile_rows<EVOCG_BF16, C, DOT>(tb, mt, wi, mi, lane, ltm, acc, ls, lc, cnt2);
        }
        // single-entry tiles: the product on the copying lane, added by the row's lane
        unsigned sa = 0u, sb = 0u;
        if ((single >> lane) & 1u) {
            const unsigned char *sd = stp + kSingleSlots + (uint32_t)lane * 16u;
            if (prec == EVOCG_FP64) {
                const double pd = reinterpret_cast<const double *>(sd)[0] * reinterpret_cast<const double *>(sd)[1];
                sa = (unsigned)__double2loint(pd);
                sb = (unsigned)__double2hiint(pd);
                if (DOT) ++cnt0;
            } else {
                const unsigned wd = reinterpret_cast<const unsigned *>(sd)[0];
                const float a = prec == EVOCG_FP32 ? __uint_as_float(wd)
                                : __uint_as_float((b.w.x & 1u) ? (wd & 0xFFFF0000u) : (wd << 16));
                const float xv = reinterpret_cast<const float *>(sd)[2];
                const float pf = __fmul_rn(a, xv);
                sa = __float_as_uint(pf);
                sb = __float_as_uint(__fmaf_rn(a, xv, -pf));   // exact remainder
                if (DOT) { if (prec == EVOCG_FP32) ++cnt1; else ++cnt2; }
            }
        }
        const int srow = __ffs(b.w.w) - 1;
        unsigned sm = single;
        while (sm) {
            const int i = __ffs(sm) - 1;
            sm &= sm - 1u;
            const unsigned a = __shfl_sync(kAll, sa, i);
            const unsigned bb = __shfl_sync(kAll, sb, i);
            const int rr = __shfl_sync(kAll, srow, i);
            const int pi = __shfl_sync(kAll, prec, i);
            if (lane == rr) {
                if (pi == EVOCG_FP64) {
                    acc += __hiloint2double((int)bb, (int)a);
                } else {
                    acc_low(ls, lc, __uint_as_float(a));
                    lc = __fadd_rn(lc, __uint_as_float(bb));
                }
            }
        }
        // the stage is rewritten by a later batch's bulk copies (the async proxy)
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        return true;
    };

    auto load = [&](int64_t rec) -> Batch {
        Batch b;
        b.rec = rec;
        b.w = __ldcs(A.pdesc + rec + lane);
        b.prec = 0;
        if (!FORCE64 && !L.map_kind && lane > 0)
            b.prec = (int)__ldcs(A.recPrec + rec + lane);
        return b;
    };
    auto next_rec = [&](const Batch &b) -> int64_t {
        const unsigned nt = __shfl_sync(kAll, b.w.x, 0) & 0xFFu;
        const int64_t r = b.rec + 1 + nt;
        return r < rec_end ? r : -1;
    };

    int64_t rec0 = A.warpRec[wid];
    if (rec0 < rec_end) {
        Batch b0 = load(rec0);
        if (!FORCE64 && L.map_kind) b0.prec = batch_prec<FORCE64>(L, b0, lane);
        bool armed0 = issue(b0, 0);
        int64_t rec1 = next_rec(b0);
        Batch b1;
        b1.rec = -1;
        b1.w = make_uint4(0u, 0u, 0u, 0u);
        b1.prec = 0;
        if (rec1 >= 0) b1 = load(rec1);
        int s = 0;
        double acc = 0.0;
        float ls = 0.f, lc = 0.f;
        bool anylow = false;
        for (;;) {
            const bool have1 = b1.rec >= 0;
            bool armed1 = false;
            Batch b2;
            b2.rec = -1;
            b2.w = make_uint4(0u, 0u, 0u, 0u);
            b2.prec = 0;
            if (have1) {
                if (!FORCE64 && L.map_kind) b1.prec = batch_prec<FORCE64>(L, b1, lane);
                armed1 = issue(b1, s ^ 1);
                const int64_t rec2 = next_rec(b1);
                if (rec2 >= 0) b2 = load(rec2);
            }
            // compute batch 0 (its copies landed while batch 1's were issued)
            const unsigned h0 = __shfl_sync(kAll, b0.w.x, 0);
            if (!FORCE64) anylow |= __any_sync(kAll, lane >= 1 && lane <= (int)(h0 & 0xFFu) && b0.prec != EVOCG_FP64);
            if (!compute(b0, s, armed0, !armed1, acc, ls, lc)) {
                lost = true;
                break;
            }
            if (h0 & kLastBit) {   // the panel's rows are complete
                const int64_t row = (int64_t)__shfl_sync(kAll, b0.w.y, 0) * R + lane;
                if (lane < R && row < A.n) {
                    double yv = acc;
                    if (!FORCE64 && anylow) yv = (acc + f64_from_f32(ls)) + f64_from_f32(lc);
                    L.y[row] = yv;
                    if (DOT) dotp = fma(__ldg(L.x64 + row), yv, dotp);
                }
                acc = 0.0;
                ls = 0.f;
                lc = 0.f;
                anylow = false;
            }
            if (!have1) break;
            b0 = b1;
            armed0 = armed1;
            b1 = b2;
            s ^= 1;
        }
        if (lost) {   // report; let the other stage's copies land before the warp leaves
            if (lane == 0 && A.err) atomicExch(A.err, 1);
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            for (int t = 0; t < 2; ++t) {
                const uint32_t st = sbase + (uint32_t)t * SB;
                mbar_wait_bounded(st, (phases >> t) & 1u, kTestWaitNs);
            }
        }
    }
    if (DOT && L.census) {
        for (int o = 16; o; o >>= 1) {
            cnt0 += __shfl_xor_sync(kAll, cnt0, o);
            cnt1 += __shfl_xor_sync(kAll, cnt1, o);
            cnt2 += __shfl_xor_sync(kAll, cnt2, o);
        }
        if (lane == 0) {
            if (cnt0) atomicAdd(&L.st->census[0], (unsigned long long)cnt0);
            if (cnt1) atomicAdd(&L.st->census[1], (unsigned long long)cnt1);
            if (cnt2) atomicAdd(&L.st->census[2], (unsigned long long)cnt2);
        }
    }
    if (DOT) {   // this warp's p.q partial (lanes summed in a fixed tree)
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(kAll, dotp, o);
        if (lane == 0) L.pq[wid] = dotp;
    }
}

template <int R, int C, int SB, int MB, bool IL>
cudaError_t launch_v(const SpmvLaunch &L, cudaStream_t s)
{
    const int grid = L.A.panel_grid;
    const size_t sm = (size_t)2 * SB * (kPanelThreads / 32);
    if (L.force64) {
        if (L.dot) spmv_panel_kernel<R, C, true, true, SB, MB, IL><<<grid, kPanelThreads, sm, s>>>(L);
        else spmv_panel_kernel<R, C, true, false, SB, MB, IL><<<grid, kPanelThreads, sm, s>>>(L);
    } else {
        if (L.dot) spmv_panel_kernel<R, C, false, true, SB, MB, IL><<<grid, kPanelThreads, sm, s>>>(L);
        else spmv_panel_kernel<R, C, false, false, SB, MB, IL><<<grid, kPanelThreads, sm, s>>>(L);
    }
    return cudaGetLastError();
}

template <int R, int C, int SB, int MB, bool IL>
int grid_v(int sms)
{
    const int sm = 2 * SB * (kPanelThreads / 32);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, true, true, SB, MB, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, true, false, SB, MB, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, false, true, SB, MB, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, false, false, SB, MB, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_panel_kernel<R, C, false, true, SB, MB, IL>,
                                                      kPanelThreads, sm) != cudaSuccess || per < 1)
        per = 1;
    cudaGetLastError();
    return sms * per;
}

// Variants: (bytes of each of a warp's two stages, blocks per SM the registers are budgeted for,
// panels interleaved over the warps).
#define EVOCG_PANEL_VARIANTS(X)     \
    X(0, 4096, 6, false)            \
    X(1, 3072, 8, false)            \
    X(2, 2560, 8, false)            \
    X(3, 4608, 5, false)

template <int R, int C>
cudaError_t launch_RC(const SpmvLaunch &L, cudaStream_t s)
{
#define X(id, sb, mb, il) \
    if (L.A.panel_variant == id) return launch_v<R, C, sb, mb, il>(L, s);
    EVOCG_PANEL_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

template <int R, int C>
int grid_RC(int sms, int variant)
{
#define X(id, sb, mb, il) \
    if (variant == id) return grid_v<R, C, sb, mb, il>(sms);
    EVOCG_PANEL_VARIANTS(X)
#undef X
    return 0;
}

}  // namespace

cudaError_t launch_spmv_panel(const SpmvLaunch &L, cudaStream_t s)
{
    if (!L.A.pdesc || L.A.panel_grid <= 0) return cudaErrorInvalidValue;
    switch (L.A.T) {
    case 16: return launch_RC<16, 16>(L, s);
    case 32: return launch_RC<32, 32>(L, s);
    default: return cudaErrorInvalidValue;
    }
}

int panel_stage_bytes(int variant)
{
#define X(id, sb, mb, il) \
    if (variant == id) return sb;
    EVOCG_PANEL_VARIANTS(X)
#undef X
    return 0;
}

int panel_grid_for(int T, int sms, int variant)
{
    switch (T) {
    case 16: return grid_RC<16, 16>(sms, variant);
    case 32: return grid_RC<32, 32>(sms, variant);
    default: return 0;
    }
}

}  // namespace evocg
