// spmv_staged.cu -- the tile-wise mixed-precision SpMV (EvoCG, "Self-Evolving Precision
// Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 / Eq. 5) with every operand
// staged into shared memory by the Tensor Memory Accelerator, for sm_103a.
//
// Work mapping. Each warp owns a contiguous range of row blocks and walks their tiles in
// order, in batches fixed at build time (a static plan: staged_plan.cpp). Lane l owns local
// row l (rows l and l+32 for T = 64; lanes 16..31 idle in the arithmetic for T = 16) and
// keeps its row sums in registers for the whole row block: no cross-lane reduction, so an
// FP64 tile costs one FP64 fused multiply-add per entry and nothing more. Inside a tile the
// slots are slot-major over the nonempty rows, so at every k the lanes read consecutive
// slots; a lane finds its slot column with one popcount of the tile's row mask and runs
// exactly the tile's width w, skipping pads (local column T).
//
// Staging. A warp holds S stages of shared memory; every tile of a batch has a fixed slot
// in its stage, sized for FP64. For a batch, lane j issues two bulk asynchronous copies for
// tile j: the tile's slice of the value stream its precision selects (the 16-byte aligned
// cover of the slice: the same 32-byte sectors a plain load would fetch) and the x segment
// of the tile's column block in that precision; one lane copies the batch's local-column
// bytes, which are contiguous. Copies land on the stage's mbarrier with
// their byte count; the warp computes batch b while batches b+1 .. b+S-1 are in flight. So
// a warp keeps kilobytes of reads in flight for a few instructions per tile, instead of a
// dependent chain of global loads per tile. Matrix streams are read with an evict-first L2
// policy so that x, which every tile column re-reads, stays in L2.
//
// Tile descriptors are loaded two batches ahead and their precision resolved one batch
// ahead, so the issue step never waits on memory. A tile too large for a stage is computed
// from global memory directly. Every mbarrier wait is bounded: if it runs out, the kernel
// records the event in an error word the host reads, stops staging and returns.
//
// Arithmetic is that of the direct kernel: FP32 and BF16 products exact in FP32 pairs
// summed error-free, merged into the FP64 row sum once per row.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

namespace {

// Per tile size: consumer warps per block (plus one producer warp), stages per consumer,
// tiles per consumer batch (NC * NB <= 32: a producer round covers one batch of every
// consumer, one tile per lane), local-column bytes and value + x bytes per stage, and the
// resident blocks per SM the registers are capped for.
template <int NC_, int S_, int NB_, int CB_, int DB_, int MINB_>
struct StParams {
    static constexpr int NC = NC_, S = S_, NB = NB_, CB = CB_, DB = DB_, MINB = MINB_;
    static constexpr int NW = NC;        // plan warps per block (the consumers)
    static constexpr int THREADS = (NC + 1) * 32;
};
template <int T>
struct StCfg;
template <>
struct StCfg<16> : StParams<4, 3, 8, 512, 2560, 4> {};
// T = 32 (tuning constants, one macro each so a build can override them)
#ifndef EVOCG_ST32_NC
#define EVOCG_ST32_NC 2
#endif
#ifndef EVOCG_ST32_S
#define EVOCG_ST32_S 2
#endif
#ifndef EVOCG_ST32_NB
#define EVOCG_ST32_NB 16
#endif
#ifndef EVOCG_ST32_CB
#define EVOCG_ST32_CB 768
#endif
#ifndef EVOCG_ST32_DB
#define EVOCG_ST32_DB 4096
#endif
#ifndef EVOCG_ST32_MINB
#define EVOCG_ST32_MINB 8
#endif
template <>
struct StCfg<32> : StParams<EVOCG_ST32_NC, EVOCG_ST32_S, EVOCG_ST32_NB, EVOCG_ST32_CB, EVOCG_ST32_DB,
                            EVOCG_ST32_MINB> {};
template <>
struct StCfg<64> : StParams<4, 2, 8, 1024, 8192, 2> {};

// Stage layout (bytes from the stage base): header, per-tile info, local columns,
// values + x segments. Block layout: full and empty mbarriers of every consumer stage,
// then each consumer's S stages.
template <int T>
struct StLayout {
    using C = StCfg<T>;
    static constexpr int HDR = 0;                        // int64 tb, int32 nb, int32 direct
    static constexpr int INFO = 16;                      // NB x INFOB bytes
    static constexpr int INFOB = T > 32 ? 32 : 16;       // uint4 (+ the high row mask)
    static constexpr int COL = INFO + INFOB * C::NB;     // CB bytes
    static constexpr int DATA = COL + C::CB;             // DB bytes
    static constexpr int STAGE = (DATA + C::DB + 127) / 128 * 128;
    static constexpr int BARS = (2 * C::NC * C::S * 8 + 127) / 128 * 128;
    static constexpr int SMEM = BARS + C::NC * C::S * STAGE;
};

template <int T>
constexpr bool layout_ok()
{
    return StCfg<T>::S * StLayout<T>::STAGE <= 65536 && StCfg<T>::NC * StCfg<T>::NB <= 32 &&
           32 % StCfg<T>::NC == 0 && StCfg<T>::NB <= 32 / StCfg<T>::NC && StLayout<T>::SMEM <= 227 * 1024;
}
static_assert(layout_ok<16>() && layout_ok<32>() && layout_ok<64>(), "stage layout");

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWaitLimit = 1 << 24;   // try_wait polls before a stage wait is declared lost

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    for (int i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global -> shared bulk copy completing on an mbarrier. dst, src 16-byte aligned, bytes a
// positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

template <int T, bool FORCE64, bool DOT>
__global__ void __launch_bounds__(StCfg<T>::THREADS, StCfg<T>::MINB)
    spmv_staged_kernel(SpmvLaunch L)
{
    using C = StCfg<T>;
    using Y = StLayout<T>;
    constexpr int RPL = T > 32 ? 2 : 1;            // rows per lane (consumers)
    constexpr int G = 32 / C::NC;                   // producer lanes per consumer
    if ((DOT || L.gate) && L.st->done) return;      // a stopped solve: nothing to do
    extern __shared__ __align__(128) unsigned char sm[];
    const TilesView A = L.A;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const uint32_t sbase = smem_u32(sm);
    // full[c][s]: the stage's copies landed (producer arrival + bytes); empty[c][s]: the
    // consumer finished reading the stage
    auto full_bar = [&](int c, int st) { return sbase + 8u * (uint32_t)(c * C::S + st); };
    auto empty_bar = [&](int c, int st) { return sbase + 8u * (uint32_t)((C::NC + c) * C::S + st); };
    auto region = [&](int c) { return (uint32_t)Y::BARS + (uint32_t)(c * C::S * Y::STAGE); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * C::NC * C::S; ++i) mbar_init(sbase + 8u * i, 1u);
        fence_mbar_init();
    }
    __syncthreads();

    const int n = (int)A.n;
    double dotp = 0.0;
    unsigned cnt0 = 0, cnt1 = 0, cnt2 = 0;   // stored entries per precision (census)

    if (wib == C::NC) {
        // =============================== producer ===============================
        // Lane l serves consumer c = l / G, tile i = l % G of that consumer's current batch.
        const uint64_t pol = policy_evict_first();
        const int c = lane / G, i = lane % G;
        const int gw = blockIdx.x * C::NC + c;
        const int bBeg = A.warpBatch[gw], bEnd = A.warpBatch[gw + 1];
        int rounds = bEnd - bBeg;
#pragma unroll
        for (int o = 16; o; o >>= 1) rounds = max(rounds, __shfl_xor_sync(kFull, rounds, o));
        const uint32_t wreg = region(c);

        // Descriptors: raw for round r + 1 (loaded two rounds ahead) and resolved, with the
        // precision looked up, for round r (its precision load issued one round ahead); the
        // first tiles of rounds r + 2 and r + 3 (the batch pointers the raw loads index by)
        // are loaded one round before they are used. No load inside a round waits on
        // another load of that round.
        int64_t r_o0 = 0, r_tb = 0;
        int r_cb = 0, r_rb = 0, r_slot = 0, r_pt = 0, r_nb = 0, r_w = 0;
        uint64_t r_mask = 0;
        int64_t d_o0 = 0, d_tb = 0;
        int d_m = 0, d_cb = 0, d_rb = 0, d_slot = 0, d_nb = 0, d_prec = 0, d_w = 0;
        uint64_t d_mask = 0;
        auto batch_ptr = [&](int r) -> int64_t {   // first tile of round r (bEnd: past the end)
            const int bb = bBeg + r;
            return bb <= bEnd ? __ldg(A.batchTile + bb) : 0;
        };
        auto resolve = [&]() {   // d <- raw
            d_nb = r_nb; d_tb = r_tb; d_o0 = r_o0;
            d_m = r_w * __popcll(r_mask);   // slots of the tile
            d_cb = r_cb; d_rb = r_rb; d_slot = r_slot; d_w = r_w; d_mask = r_mask;
            if (FORCE64) d_prec = 0;
            else if (L.map_kind == EVOCG_MAP_PER_TILE) d_prec = r_pt;
            else d_prec = (i < r_nb) ? (int)__ldg(L.prec + r_cb) : 0;
        };
        auto load_raw = [&](int r, int64_t tb0, int64_t tb1) {   // tb0, tb1: rounds r, r + 1
            r_nb = 0;
            if (bBeg + r < bEnd) {
                r_tb = tb0;
                r_nb = (int)(tb1 - tb0);
                if (i < r_nb) {
                    const int64_t t = r_tb + i;
                    r_o0 = __ldg(A.tileNnzOff + t);
                    r_cb = __ldg(A.tileColIdx + t);
                    r_rb = __ldg(A.tileRowIdx + t);
                    r_slot = __ldg(A.tileSlot + t);
                    r_mask = __ldg(reinterpret_cast<const unsigned long long *>(A.rowMask) + t);
                    r_w = (int)__ldg(A.tileWidth + t);
                    r_pt = (!FORCE64 && L.map_kind == EVOCG_MAP_PER_TILE) ? (int)__ldg(L.prec + t) : 0;
                }
            }
        };
        int64_t tbA, tbB;   // first tiles of rounds r + 2 and r + 3 at the end of round r
        {
            const int64_t p0 = batch_ptr(0), p1 = batch_ptr(1), p2 = batch_ptr(2);
            tbA = p2;
            tbB = batch_ptr(3);
            load_raw(0, p0, p1);
            resolve();
            load_raw(1, p1, p2);
        }
        bool lost = false;
        for (int r = 0; r < rounds && !lost; ++r) {
            const int st = r % C::S;
            // this round's descriptors; the next round's resolve and the one after's raw
            // loads are issued at the end of the round
            const int nb = d_nb;
            const int64_t tb = d_tb, o0 = d_o0;
            const int m = d_m, cb = d_cb, rb = d_rb, slot = d_slot, prec = d_prec, tw = d_w;
            const uint64_t tmask = d_mask;
            const bool valid = i < nb;
            // wait until each consumer has released the stage this round refills
            bool timedout = false;
            if (r >= C::S && i == 0 && nb > 0)
                timedout = !mbar_wait_bounded(empty_bar(c, st), (uint32_t)(((r / C::S) - 1) & 1));
            if (__any_sync(kFull, timedout)) {   // a consumer stopped: issue nothing more
                if (lane == 0 && A.err) atomicExch(A.err, 1);
                lost = true;
                break;
            }
            fence_proxy_async();
            const uint32_t stg = wreg + (uint32_t)(st * Y::STAGE);     // consumer stage in sm
            const uint32_t srel = stg - wreg;                             // ... in its region
            const int slot0 = __shfl_sync(kFull, slot, 0, G);   // every lane takes part
            const bool direct = (nb == 1) && (slot0 == (int)kDirectSlot);
            const int vw = prec == 0 ? 8 : (prec == 1 ? 4 : 2);
            const int xw = prec == 0 ? 8 : 4;
            const int xb = T * xw;
            const int64_t vbyte0 = o0 * vw;
            const int64_t va0 = vbyte0 & ~(int64_t)15;
            const int vb = (int)(((vbyte0 + (int64_t)m * vw + 15) & ~(int64_t)15) - va0);
            const bool full_x = (cb + 1) * T <= n;
            const int64_t colFirst = __shfl_sync(kFull, o0, 0, G) & ~(int64_t)15;
            const int64_t lastEnd = __shfl_sync(kFull, o0 + m, nb > 0 ? nb - 1 : 0, G);
            const int colBytes = (int)(((lastEnd + 15) & ~(int64_t)15) - colFirst);
            int txl = (valid && !direct) ? vb + (full_x ? xb : 0) : 0;
#pragma unroll
            for (int o = G / 2; o; o >>= 1) txl += __shfl_xor_sync(kFull, txl, o, G);
            const uint32_t dOff = srel + Y::DATA + (uint32_t)slot;
            const uint32_t valS = dOff + (uint32_t)(vbyte0 - va0);
            const uint32_t xS = dOff + (uint32_t)(staged_slot_bytes(m, T) - 8 * T);
            const uint32_t colS = srel + Y::COL + (uint32_t)(o0 - colFirst);
            if (valid) {
                const uint32_t pw = ((uint32_t)prec << 16) | ((uint32_t)tw << 18);
                if (direct) {
                    *reinterpret_cast<int4 *>(sm + stg + Y::HDR) =
                        make_int4((int)(tb & 0xffffffff), (int)(tb >> 32), 1, 1);
                    *reinterpret_cast<uint4 *>(sm + stg + Y::INFO) =
                        make_uint4(0u, (uint32_t)rb, pw, (uint32_t)tmask);
                } else {
                    *reinterpret_cast<uint4 *>(sm + stg + Y::INFO + Y::INFOB * i) =
                        make_uint4(valS | (xS << 16), (uint32_t)rb, colS | pw, (uint32_t)tmask);
                    if (T > 32)
                        *reinterpret_cast<uint32_t *>(sm + stg + Y::INFO + Y::INFOB * i + 16) =
                            (uint32_t)(tmask >> 32);
                    if (!full_x) {  // the last column block of a matrix with T not dividing n
                        const int xb0 = cb * T;
                        if (prec == 0) {
                            double *dd = reinterpret_cast<double *>(sm + wreg + xS);
                            for (int k = 0; k < T; ++k) dd[k] = (xb0 + k < n) ? __ldg(L.x64 + xb0 + k) : 0.0;
                        } else {
                            const float *src = prec == 1 ? L.x32 : L.x16f;
                            float *dd = reinterpret_cast<float *>(sm + wreg + xS);
                            for (int k = 0; k < T; ++k) dd[k] = (xb0 + k < n) ? __ldg(src + xb0 + k) : 0.f;
                        }
                    }
                    if (i == 0)
                        *reinterpret_cast<int4 *>(sm + stg + Y::HDR) =
                            make_int4((int)(tb & 0xffffffff), (int)(tb >> 32), nb, 0);
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (i == 0 && nb > 0) {
                if (direct) mbar_arrive(full_bar(c, st));
                else mbar_arrive_expect_tx(full_bar(c, st), (uint32_t)(txl + colBytes));
            }
            __syncwarp();
            if (valid && !direct) {
                const unsigned char *vsrc =
                    prec == 0 ? reinterpret_cast<const unsigned char *>(A.v64)
                              : (prec == 1 ? reinterpret_cast<const unsigned char *>(A.v32)
                                           : reinterpret_cast<const unsigned char *>(A.v16));
                bulk_g2s_hint(sbase + wreg + dOff, vsrc + va0, (uint32_t)vb, full_bar(c, st), pol);
                if (full_x) {
                    const unsigned char *xsrc =
                        prec == 0 ? reinterpret_cast<const unsigned char *>(L.x64)
                                  : (prec == 1 ? reinterpret_cast<const unsigned char *>(L.x32)
                                               : reinterpret_cast<const unsigned char *>(L.x16f));
                    bulk_g2s(sbase + wreg + xS, xsrc + (size_t)cb * (size_t)xb, (uint32_t)xb, full_bar(c, st));
                }
                if (i == 0)
                    bulk_g2s_hint(sbase + stg + Y::COL, A.colIdx + colFirst, (uint32_t)colBytes, full_bar(c, st), pol);
            }
            resolve();
            load_raw(r + 2, tbA, tbB);
            tbA = tbB;
            tbB = batch_ptr(r + 4);
        }
    } else {
        // =============================== consumer ===============================
        const int gw = blockIdx.x * C::NC + wib;
        const bool rowlane = (T >= 32) || (lane < T);   // lanes that own a row
        const uint32_t wofs = region(wib);
        const int rbBeg = A.warpRb[gw], rbEnd = A.warpRb[gw + 1];
        const int nbat = A.warpBatch[gw + 1] - A.warpBatch[gw];

        double acc64[RPL];
        F32Pair accl[RPL];
        bool any64 = false, anylow = false;
        int cur_rb = rbBeg;
        auto start_rb = [&](int rb) {
#pragma unroll
            for (int q = 0; q < RPL; ++q) {
                acc64[q] = 0.0;
                accl[q].hi = 0.f;
                accl[q].lo = 0.f;
            }
            any64 = false;
            anylow = false;
        };
        auto finish_rb = [&](int rb) {
#pragma unroll
            for (int q = 0; q < RPL; ++q) {
                const int row = rb * T + lane + 32 * q;
                if (rowlane && row < n) {
                    double y = acc64[q];
                    if (anylow) {  // FP32 -> FP64 widening is exact
                        const double dd = (double)accl[q].hi + (double)accl[q].lo;
                        y = any64 ? y + dd : dd;
                    }
                    L.y[row] = y;
                    if (DOT) dotp = fma(__ldg(L.x64 + row), y, dotp);   // p.q of CG
                }
            }
        };
        auto zero_rows = [&](int z0, int z1) {   // row blocks [z0, z1) have no tiles
            for (int z = z0; z < z1; ++z)
#pragma unroll
                for (int q = 0; q < RPL; ++q) {
                    const int row = z * T + lane + 32 * q;
                    if (rowlane && row < n) L.y[row] = 0.0;
                }
        };
        auto goto_rb = [&](int rb) {
            if (rb == cur_rb) return;
            finish_rb(cur_rb);
            zero_rows(cur_rb + 1, rb);
            cur_rb = rb;
            start_rb(rb);
        };
        const uint32_t ltm = (1u << lane) - 1u;   // lanes below mine
        // one tile's products for my rows, operands in my shared-memory region (32-bit
        // offsets): my slot column j = popcount of the row mask below my row; w slots at
        // stride h = popcount of the mask; pads (column T) are skipped
        auto tile_staged = [&](const uint4 inf, uint32_t mhi) {
            const int prec = (int)((inf.z >> 16) & 3u);
            const int w = (int)((inf.z >> 18) & 127u);
            const uint32_t colo = wofs + (inf.z & 0xffffu), valo = wofs + (inf.x & 0xffffu);
            const uint32_t xo = wofs + (inf.x >> 16);
            const uint32_t mlo = inf.w;
            const uint32_t h = (uint32_t)(__popc(mlo) + (RPL == 2 ? __popc(mhi) : 0));
#pragma unroll
            for (int q = 0; q < RPL; ++q) {
                const uint32_t mq = q ? mhi : mlo;
                if (!((mq >> lane) & 1u)) continue;   // my row has no entry in this tile
                const uint32_t j = (uint32_t)((q ? __popc(mlo) : 0) + __popc(mq & ltm));
                if (prec == EVOCG_FP64) {
                    double a = acc64[q];
#pragma unroll 1
                    for (int k = 0; k < w; ++k) {
                        const uint32_t s = (uint32_t)k * h + j;
                        const uint32_t cc = sm[colo + s];
                        if (cc < (uint32_t)T) {
                            a = fma(*reinterpret_cast<const double *>(sm + valo + 8u * s),
                                    *reinterpret_cast<const double *>(sm + xo + 8u * cc), a);
                            if (L.census) ++cnt0;
                        }
                    }
                    acc64[q] = a;
                } else if (prec == EVOCG_FP32) {
#pragma unroll 1
                    for (int k = 0; k < w; ++k) {
                        const uint32_t s = (uint32_t)k * h + j;
                        const uint32_t cc = sm[colo + s];
                        if (cc < (uint32_t)T) {
                            accl[q].add_prod(*reinterpret_cast<const float *>(sm + valo + 4u * s),
                                             *reinterpret_cast<const float *>(sm + xo + 4u * cc));
                            if (L.census) ++cnt1;
                        }
                    }
                } else {
#pragma unroll 1
                    for (int k = 0; k < w; ++k) {  // BF16 x BF16 is exact in FP32
                        const uint32_t s = (uint32_t)k * h + j;
                        const uint32_t cc = sm[colo + s];
                        if (cc < (uint32_t)T) {
                            const uint16_t hb = *reinterpret_cast<const uint16_t *>(sm + valo + 2u * s);
                            accl[q].add(__fmul_rn(f32_from_bf16(hb),
                                                  *reinterpret_cast<const float *>(sm + xo + 4u * cc)));
                            if (L.census) ++cnt2;
                        }
                    }
                }
            }
            if (prec == EVOCG_FP64) any64 = true; else anylow = true;
        };
        // one tile's products straight from global memory (a tile larger than a stage)
        auto tile_direct = [&](int64_t t, int prec) {
            const int64_t off = __ldg(A.tileNnzOff + t);
            const int xb0 = __ldg(A.tileColIdx + t) * T;
            const uint64_t msk = __ldg(reinterpret_cast<const unsigned long long *>(A.rowMask) + t);
            const int w = (int)__ldg(A.tileWidth + t);
            const int64_t h = __popcll(msk);
#pragma unroll
            for (int q = 0; q < RPL; ++q) {
                const int r = lane + 32 * q;
                if (!rowlane || !((msk >> r) & 1ull)) continue;
                const int64_t j = __popcll(msk & ((1ull << r) - 1ull));
                for (int k = 0; k < w; ++k) {
                    const int64_t s = off + (int64_t)k * h + j;
                    const int cc = __ldg(A.colIdx + s);
                    if (cc >= T) continue;
                    const int jx = xb0 + cc;
                    if (prec == EVOCG_FP64) {
                        acc64[q] = fma(__ldg(A.v64 + s), __ldg(L.x64 + jx), acc64[q]);
                        if (L.census) ++cnt0;
                    } else if (prec == EVOCG_FP32) {
                        accl[q].add_prod(__ldg(A.v32 + s), __ldg(L.x32 + jx));
                        if (L.census) ++cnt1;
                    } else {
                        accl[q].add(__fmul_rn(f32_from_bf16(__ldg(A.v16 + s)), __ldg(L.x16f + jx)));
                        if (L.census) ++cnt2;
                    }
                }
            }
            if (prec == EVOCG_FP64) any64 = true; else anylow = true;
        };

        if (rbBeg < rbEnd) {
            start_rb(rbBeg);
            bool lost = false;
            for (int b = 0; b < nbat; ++b) {
                const int st = b % C::S;
                if (!mbar_wait_bounded(full_bar(wib, st), (uint32_t)((b / C::S) & 1))) {
                    lost = true;
                    if (lane == 0 && A.err) atomicExch(A.err, 1);
                    break;
                }
                const uint32_t stg = wofs + (uint32_t)(st * Y::STAGE);
                const int4 h = *reinterpret_cast<const int4 *>(sm + stg + Y::HDR);
                const uint32_t info = stg + Y::INFO;
                if (h.w) {  // one tile too large for a stage
                    const int64_t tb = (int64_t)(uint32_t)h.x | ((int64_t)h.y << 32);
                    const uint4 inf = *reinterpret_cast<const uint4 *>(sm + info);
                    goto_rb((int)inf.y);
                    tile_direct(tb, (int)((inf.z >> 16) & 3u));
                } else {
                    const int nb = h.z;
                    uint4 inf = *reinterpret_cast<const uint4 *>(sm + info);
                    uint32_t mhi = (T > 32) ? *reinterpret_cast<const uint32_t *>(sm + info + 16u) : 0u;
                    for (int jt = 0; jt < nb; ++jt) {
                        // the next tile's descriptor loads while this one computes
                        const uint32_t ia = info + (uint32_t)(Y::INFOB * (jt + 1 < nb ? jt + 1 : jt));
                        const uint4 infn = *reinterpret_cast<const uint4 *>(sm + ia);
                        const uint32_t mhin = (T > 32) ? *reinterpret_cast<const uint32_t *>(sm + ia + 16u) : 0u;
                        goto_rb((int)inf.y);
                        tile_staged(inf, mhi);
                        inf = infn;
                        mhi = mhin;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(wib, st));   // the stage may be refilled
            }
            if (!lost) {
                finish_rb(cur_rb);
                zero_rows(cur_rb + 1, rbEnd);
            }
        }
    }

    if (L.census && wib < C::NC) {   // stored entries per precision, pads not counted
        for (int o = 16; o; o >>= 1) {
            cnt0 += __shfl_xor_sync(kFull, cnt0, o);
            cnt1 += __shfl_xor_sync(kFull, cnt1, o);
            cnt2 += __shfl_xor_sync(kFull, cnt2, o);
        }
        if (lane == 0) {
            if (cnt0) atomicAdd(&L.st->census[0], (unsigned long long)cnt0);
            if (cnt1) atomicAdd(&L.st->census[1], (unsigned long long)cnt1);
            if (cnt2) atomicAdd(&L.st->census[2], (unsigned long long)cnt2);
        }
    }
    if (DOT && wib < C::NC) {   // this consumer warp's p.q partial (fixed shuffle tree)
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(kFull, dotp, o);
        if (lane == 0) L.pq[blockIdx.x * C::NC + wib] = dotp;
    }
}

template <int T>
cudaError_t staged_T(const SpmvLaunch &L, cudaStream_t s)
{
    constexpr int threads = StCfg<T>::THREADS;
    constexpr int smem = StLayout<T>::SMEM;
    if (L.force64) {
        if (L.dot) spmv_staged_kernel<T, true, true><<<L.grid, threads, smem, s>>>(L);
        else spmv_staged_kernel<T, true, false><<<L.grid, threads, smem, s>>>(L);
    } else {
        if (L.dot) spmv_staged_kernel<T, false, true><<<L.grid, threads, smem, s>>>(L);
        else spmv_staged_kernel<T, false, false><<<L.grid, threads, smem, s>>>(L);
    }
    return cudaGetLastError();
}

template <int T>
int staged_grid_T(int sms)
{
    constexpr int threads = StCfg<T>::THREADS;
    constexpr int smem = StLayout<T>::SMEM;
    const void *ks[4] = {(const void *)spmv_staged_kernel<T, true, true>,
                         (const void *)spmv_staged_kernel<T, true, false>,
                         (const void *)spmv_staged_kernel<T, false, true>,
                         (const void *)spmv_staged_kernel<T, false, false>};
    for (const void *k : ks)
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_staged_kernel<T, false, true>,
                                                      threads, smem) != cudaSuccess || per < 1) {
        cudaGetLastError();
        return 0;
    }
    const int g = sms * per;
    return g > kMaxBlocks ? kMaxBlocks : g;
}

template <int T>
void limits_T(StagedLimits *o)
{
    o->warps_per_block = StCfg<T>::NW;
    o->nb = StCfg<T>::NB;
    o->col_bytes = StCfg<T>::CB;
    o->data_bytes = StCfg<T>::DB;
}

}  // namespace

cudaError_t launch_spmv_staged(const SpmvLaunch &L, cudaStream_t s)
{
    switch (L.A.T) {
    case 16: return staged_T<16>(L, s);
    case 32: return staged_T<32>(L, s);
    case 64: return staged_T<64>(L, s);
    default: return cudaErrorInvalidValue;
    }
}

int staged_grid_for(int T, int sms)
{
    switch (T) {
    case 16: return staged_grid_T<16>(sms);
    case 32: return staged_grid_T<32>(sms);
    case 64: return staged_grid_T<64>(sms);
    default: return 0;
    }
}

int staged_warps_per_block(int T)
{
    switch (T) {
    case 16: return StCfg<16>::NC;
    case 32: return StCfg<32>::NC;
    case 64: return StCfg<64>::NC;
    default: return 0;
    }
}

bool staged_limits(int T, StagedLimits *out)
{
    switch (T) {
    case 16: limits_T<16>(out); return true;
    case 32: limits_T<32>(out); return true;
    case 64: limits_T<64>(out); return true;
    default: return false;
    }
}

}  // namespace evocg
