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
// Staging. Each warp owns one shared-memory stage. A panel's tiles are cut at run time into
// batches that fit it (the cut depends on the precisions, hence on the map): for a batch the
// lanes issue asynchronous global-to-shared copies (cp.async, 16 bytes per lane and
// instruction) of the 16-byte cover of the batch's local-column bytes, of every tile's value
// slice in the stream its precision selects, and of every tile's x segment in that
// precision; single-entry tiles (one row, width one: the panel-edge tiles of stencils, most
// of a stencil's tiles by count) copy just their value and x entry. The warp then waits for
// its own copies (cp.async.wait_group: a hardware wait on the issuing threads' copies, no
// polling) and computes the batch from shared memory. The next panel's descriptors and their
// precisions are loaded while the current panel is in flight. Registers no longer bound the
// bytes in flight, so an SM holds many warps with kilobytes in flight each. A tile too large
// for the stage on its own is computed from global memory level by level.
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
constexpr int kSingleBytes = 16;   // stage bytes of a single-entry tile: value word, x entry

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

// Asynchronous global -> shared copies; completion is awaited with cp_wait_all by the same
// threads. The 16-byte form bypasses L1 (streamed matrix data), the 4- and 8-byte forms
// allocate in L1 (x entries, which neighbouring panels read again).
__device__ __forceinline__ void cp16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
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

__device__ __forceinline__ unsigned lds_u8(uint32_t a)
{
    unsigned v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ unsigned lds_u16(uint32_t a)
{
    unsigned v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ unsigned lds_u32(uint32_t a)
{
    unsigned v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) { return __uint_as_float(lds_u32(a)); }
__device__ __forceinline__ double lds_f64(uint32_t a)
{
    double v;
    asm volatile("ld.shared.f64 %0, [%1];" : "=d"(v) : "r"(a));
    return v;
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

__device__ __forceinline__ int vsize(int pr) { return pr == EVOCG_FP64 ? 8 : pr == EVOCG_FP32 ? 4 : 2; }
__device__ __forceinline__ int xsize(int pr) { return pr == EVOCG_FP64 ? 8 : 4; }

// 16-byte chunks of the cover of slots [s0, s0 + m) in a stream of elements of sz bytes.
__device__ __forceinline__ int cover16(int64_t s0, int m, int sz)
{
    return (int)((((s0 + m) * sz + 15) & ~(int64_t)15) - ((s0 * sz) & ~(int64_t)15)) >> 4;
}

__device__ __forceinline__ int scan_incl(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kAll, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Record layout (panel_plan.cpp): header {tiles, panel, first slot lo, hi}; tile {slot offset
// from the panel's first slot, w | single-entry column << 8 | stored entries << 16, column
// block, row mask}. SB: stage bytes per warp; MB: blocks per SM the registers are sized for.
template <int R, int C, bool FORCE64, bool DOT, int SB, int MB>
__global__ void __launch_bounds__(kPanelThreads, MB) spmv_panel_kernel(SpmvLaunch L)
{
    static_assert(R == 16 || R == 32, "panel rows");
    static_assert(C == R, "this kernel reads tiles as wide as the panel is tall");
    // stage: single-entry slots, then local columns, then value covers and x segments
    constexpr int kColSt = 32 * kSingleBytes;
    constexpr int kData = SB - kColSt - 32;   // bytes for columns (+32 of alignment) and data
    static_assert(SB % 16 == 0 && kData >= 1024, "stage size");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    if ((DOT || L.gate) && L.st->done) return;
    const TilesView &A = L.A;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
    const uint32_t st0 = smem_addr(smem_raw + (size_t)wib * SB);
    const unsigned ltm = lanemask_lt();
    const int p_end = A.warpPanel[wid + 1];
    int p = A.warpPanel[wid];
    int64_t rec = A.warpRec[wid];
    double dotp = 0.0;
    unsigned cnt0 = 0, cnt1 = 0, cnt2 = 0;
    uint4 win = make_uint4(0u, 0u, 0u, 0u);
    int wprec = 0;
    if (p < p_end) {
        win = __ldcs(A.pdesc + rec + lane);
        const unsigned nt0 = __shfl_sync(kAll, win.x, 0);   // the header's tile count
        if (!FORCE64 && lane > 0 && lane <= (int)nt0)
            wprec = L.map_kind ? (int)__ldg(L.prec + (int)win.z) : (int)__ldcs(L.prec + (rec + lane - p - 1));
    }

    for (; p < p_end; ++p) {
        const unsigned nt = __shfl_sync(kAll, win.x, 0);
        const int64_t sbase = (int64_t)(((uint64_t)__shfl_sync(kAll, win.w, 0) << 32) |
                                        (uint64_t)__shfl_sync(kAll, win.z, 0));
        const int64_t nextrec = rec + 1 + nt;
        const bool more = p + 1 < p_end;
        uint4 nwin = make_uint4(0u, 0u, 0u, 0u);
        int nprec = 0;
        bool nprec_pending = false;   // a per-column-block map: resolved once nwin is in
        if (more) {
            nwin = __ldcs(A.pdesc + nextrec + lane);
            if (!FORCE64) {
                // tile index of lane's record in the next panel (its count is not known yet,
                // so the index is bounded by the tile count instead)
                const int64_t ti = nextrec + lane - (p + 1) - 1;
                if (L.map_kind) nprec_pending = true;
                else if (lane > 0 && ti < A.ntiles) nprec = (int)__ldcs(L.prec + ti);
            }
        }
        const int64_t row = (int64_t)p * R + lane;
        const bool rowok = lane < R && row < A.n;
        double xrow = 0.0;
        if (DOT && rowok) xrow = __ldg(L.x64 + row);

        double acc = 0.0;
        float ls = 0.f, lc = 0.f;
        bool anylow = false;
        for (int64_t r0 = rec; r0 <= rec + (int64_t)nt; r0 += 32) {
            const int64_t r = r0 + lane;
            const bool valid = r > rec && r <= rec + (int64_t)nt;
            uint4 d = win;
            int prec = wprec;
            if (r0 != rec) {   // tiles past the first 31 of the panel
                d = valid ? __ldcs(A.pdesc + r) : make_uint4(0u, 0u, 0u, 0u);
                prec = 0;
                if (!FORCE64 && valid)
                    prec = L.map_kind ? (int)__ldg(L.prec + (int)d.z) : (int)__ldcs(L.prec + (r - p - 1));
            }
            if (FORCE64 || !valid) prec = 0;
            const int w = (int)(d.y & 0xFFu);
            const unsigned mk = d.w;
            const int h = __popc(mk);
            const int m = w * h;                         // slots of the tile
            const int64_t s0 = sbase + (int64_t)d.x;     // its first slot
            const bool single = valid && w == 1 && h == 1;
            const bool regular = valid && !single;
            if (!FORCE64) anylow |= __any_sync(kAll, valid && prec != EVOCG_FP64);
            if (DOT && valid) {   // census: stored entries of the tile, by precision
                const unsigned e = d.y >> 16;
                if (prec == EVOCG_FP64) cnt0 += e; else if (prec == EVOCG_FP32) cnt1 += e; else cnt2 += e;
            }
            // stage bytes: value cover + x segment of a regular tile, and an upper bound of the
            // local-column bytes of every tile (its slots)
            const int dbytes = regular ? 16 * cover16(s0, m, vsize(prec)) + C * xsize(prec) : 0;
            const int need = valid ? dbytes + m : 0;
            unsigned left = __ballot_sync(kAll, valid);
            while (left) {
                // batch: the lowest tiles still left whose bytes fit the stage (a prefix)
                const bool in = (left >> lane) & 1u;
                const int incl = scan_incl(in ? need : 0, lane);
                unsigned take = __ballot_sync(kAll, in && incl <= kData);
                const bool big = take == 0u;   // the lowest tile left does not fit alone
                if (big) take = left & (0u - left);
                const bool mine = (take >> lane) & 1u;
                const unsigned treg = take & __ballot_sync(kAll, regular);
                const unsigned tsgl = take & __ballot_sync(kAll, single);
                // local columns of the batch: one cover of its contiguous slot range
                const int lo_l = __ffs(take) - 1, hi_l = 31 - __clz(take);
                const int64_t c_a = __shfl_sync(kAll, s0, lo_l) & ~(int64_t)15;
                const int64_t c_b = (__shfl_sync(kAll, s0 + m, hi_l) + 15) & ~(int64_t)15;
                const int ncol16 = (int)((c_b - c_a) >> 4);
                const uint32_t col_st = st0 + kColSt;
                // each regular tile's value cover and x segment, packed after the columns
                const int dincl = scan_incl(mine ? dbytes : 0, lane);
                const uint32_t vst = col_st + 16u * (uint32_t)ncol16 + (uint32_t)(dincl - (mine ? dbytes : 0));

                if (!big) {
                    // ---- issue the batch's copies
                    for (int q = lane; q < ncol16; q += 32) cp16(col_st + 16u * q, A.colIdx + c_a + 16 * q);
                    unsigned tr = treg;
                    while (tr) {
                        const int i = __ffs(tr) - 1;
                        tr &= tr - 1u;
                        const int pi = __shfl_sync(kAll, prec, i);
                        const int64_t si = __shfl_sync(kAll, s0, i);
                        const int mi = __shfl_sync(kAll, m, i);
                        const uint32_t vi = __shfl_sync(kAll, vst, i);
                        const int cbi = __shfl_sync(kAll, (int)d.z, i);
                        const int sz = vsize(pi);
                        const int64_t a = (si * sz) & ~(int64_t)15;
                        const int nv16 = cover16(si, mi, sz);
                        const unsigned char *vsrc =
                            pi == EVOCG_FP64 ? reinterpret_cast<const unsigned char *>(A.v64)
                            : pi == EVOCG_FP32 ? reinterpret_cast<const unsigned char *>(A.v32)
                                               : reinterpret_cast<const unsigned char *>(A.v16);
                        for (int q = lane; q < nv16; q += 32) cp16(vi + 16u * q, vsrc + a + 16 * q);
                        const uint32_t xst = vi + 16u * nv16;
                        const int64_t xj = (int64_t)cbi * C + lane;
                        if (lane < C && xj < A.n) {
                            if (pi == EVOCG_FP64) cp8(xst + 8u * lane, L.x64 + xj);
                            else cp4(xst + 4u * lane, (pi == EVOCG_FP32 ? L.x32 : L.x16f) + xj);
                        }
                    }
                    // single-entry tiles: the value word and the x entry into the lane's slot
                    if (mine && single) {
                        const uint32_t sd = st0 + (uint32_t)lane * kSingleBytes;
                        const int64_t xj = (int64_t)(int)d.z * C + (int64_t)((d.y >> 8) & 0xFFu);
                        if (prec == EVOCG_FP64) {
                            cp8(sd, A.v64 + s0);
                            cp8(sd + 8u, L.x64 + xj);
                        } else if (prec == EVOCG_FP32) {
                            cp4(sd, A.v32 + s0);
                            cp4(sd + 8u, L.x32 + xj);
                        } else {
                            cp4(sd, A.v16 + (s0 & ~(int64_t)1));   // the aligned pair holding it
                            cp4(sd + 8u, L.x16f + xj);
                        }
                    }
                }
                if (nprec_pending) {   // the next panel's precisions, while the copies fly
                    nprec_pending = false;
                    const unsigned nnt = __shfl_sync(kAll, nwin.x, 0);
                    if (lane > 0 && lane <= (int)nnt) nprec = (int)__ldg(L.prec + (int)nwin.z);
                }
                cp_wait_all();
                __syncwarp();

                // ---- compute the batch
                if (big) {   // one tile larger than the stage: level by level from global memory
                    const int pi = __shfl_sync(kAll, prec, lo_l);
                    const int64_t si = __shfl_sync(kAll, s0, lo_l);
                    const int wi = __shfl_sync(kAll, w, lo_l);
                    const unsigned mi = __shfl_sync(kAll, mk, lo_l);
                    const int cbi = __shfl_sync(kAll, (int)d.z, lo_l);
                    const int hi = __popc(mi);
                    const bool has = lane < R && ((mi >> lane) & 1u);
                    const int j = __popc(mi & ltm);
                    for (int k = 0; has && k < wi; ++k) {
                        const int64_t s = si + (int64_t)k * hi + j;
                        const int c = A.colIdx[s];
                        if (c >= C) continue;
                        const int64_t xj = (int64_t)cbi * C + c;
                        if (pi == EVOCG_FP64) {
                            acc = fma(__ldcs(A.v64 + s), __ldg(L.x64 + xj), acc);
                        } else if (pi == EVOCG_FP32) {
                            acc_prod(ls, lc, __ldcs(A.v32 + s), __ldg(L.x32 + xj));
                        } else {
                            const unsigned b = __ldcs(reinterpret_cast<const unsigned short *>(A.v16) + s);
                            acc_low(ls, lc, __fmul_rn(__uint_as_float(b << 16), __ldg(L.x16f + xj)));
                        }
                    }
                } else {
                    unsigned tr = treg;
                    while (tr) {
                        const int i = __ffs(tr) - 1;
                        tr &= tr - 1u;
                        const int pi = __shfl_sync(kAll, prec, i);
                        const int64_t si = __shfl_sync(kAll, s0, i);
                        const int wi = __shfl_sync(kAll, w, i);
                        const unsigned mi = __shfl_sync(kAll, mk, i);
                        const uint32_t vi = __shfl_sync(kAll, vst, i);
                        const int hi = __popc(mi);
                        if (!(lane < R && ((mi >> lane) & 1u))) continue;
                        const int j = __popc(mi & ltm);
                        const int sz = vsize(pi);
                        const uint32_t v0 = vi + (uint32_t)((si * sz) & 15) + (uint32_t)(sz * j);
                        const uint32_t xst = vi + 16u * cover16(si, hi * wi, sz);
                        const uint32_t c0 = col_st + (uint32_t)(si - c_a) + (uint32_t)j;
                        const uint32_t vstep = (uint32_t)(sz * hi);
                        if (pi == EVOCG_FP64) {
                            for (int k = 0; k < wi; ++k) {
                                const unsigned c = lds_u8(c0 + (uint32_t)(k * hi));
                                if (c < (unsigned)C) acc = fma(lds_f64(v0 + vstep * k), lds_f64(xst + 8u * c), acc);
                            }
                        } else if (pi == EVOCG_FP32) {
                            for (int k = 0; k < wi; ++k) {
                                const unsigned c = lds_u8(c0 + (uint32_t)(k * hi));
                                if (c < (unsigned)C) acc_prod(ls, lc, lds_f32(v0 + vstep * k), lds_f32(xst + 4u * c));
                            }
                        } else {
                            for (int k = 0; k < wi; ++k) {
                                const unsigned c = lds_u8(c0 + (uint32_t)(k * hi));
                                if (c < (unsigned)C)   // BF16 x BF16 is exact in FP32
                                    acc_low(ls, lc, __fmul_rn(__uint_as_float(lds_u16(v0 + vstep * k) << 16),
                                                              lds_f32(xst + 4u * c)));
                            }
                        }
                    }
                    // single-entry tiles: the product on the copying lane, added by the row's lane
                    unsigned sa = 0u, sb = 0u;
                    if (mine && single) {
                        const uint32_t sd = st0 + (uint32_t)lane * kSingleBytes;
                        if (prec == EVOCG_FP64) {
                            const double pd = lds_f64(sd) * lds_f64(sd + 8u);
                            sa = (unsigned)__double2loint(pd);
                            sb = (unsigned)__double2hiint(pd);
                        } else {
                            const unsigned wd = lds_u32(sd);
                            const float a = prec == EVOCG_FP32 ? __uint_as_float(wd)
                                            : __uint_as_float((s0 & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
                            const float xv = lds_f32(sd + 8u);
                            const float pf = __fmul_rn(a, xv);
                            sa = __float_as_uint(pf);
                            sb = __float_as_uint(__fmaf_rn(a, xv, -pf));   // exact remainder
                        }
                    }
                    const int srow = __ffs(mk) - 1;
                    unsigned sm = tsgl;
                    while (sm) {
                        const int i = __ffs(sm) - 1;
                        sm &= sm - 1u;
                        const unsigned a = __shfl_sync(kAll, sa, i);
                        const unsigned b = __shfl_sync(kAll, sb, i);
                        const int rr = __shfl_sync(kAll, srow, i);
                        const int pi = __shfl_sync(kAll, prec, i);
                        if (lane == rr) {
                            if (pi == EVOCG_FP64) {
                                acc += __hiloint2double((int)b, (int)a);
                            } else {
                                acc_low(ls, lc, __uint_as_float(a));
                                lc = __fadd_rn(lc, __uint_as_float(b));
                            }
                        }
                    }
                }
                __syncwarp();   // the stage is free for the next batch
                left &= ~take;
            }
        }
        if (nprec_pending) {
            const unsigned nnt = __shfl_sync(kAll, nwin.x, 0);
            if (lane > 0 && lane <= (int)nnt) nprec = (int)__ldg(L.prec + (int)nwin.z);
        }
        if (rowok) {
            double y = acc;
            if (!FORCE64 && anylow) y = (acc + f64_from_f32(ls)) + f64_from_f32(lc);
            L.y[row] = y;
            if (DOT) dotp = fma(xrow, y, dotp);
        }
        win = nwin;
        wprec = nprec;
        rec = nextrec;
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

template <int R, int C, int SB, int MB>
cudaError_t launch_v(const SpmvLaunch &L, cudaStream_t s)
{
    const int grid = L.A.panel_grid;
    const size_t sm = (size_t)SB * (kPanelThreads / 32);
    if (L.force64) {
        if (L.dot) spmv_panel_kernel<R, C, true, true, SB, MB><<<grid, kPanelThreads, sm, s>>>(L);
        else spmv_panel_kernel<R, C, true, false, SB, MB><<<grid, kPanelThreads, sm, s>>>(L);
    } else {
        if (L.dot) spmv_panel_kernel<R, C, false, true, SB, MB><<<grid, kPanelThreads, sm, s>>>(L);
        else spmv_panel_kernel<R, C, false, false, SB, MB><<<grid, kPanelThreads, sm, s>>>(L);
    }
    return cudaGetLastError();
}

template <int R, int C, int SB, int MB>
int grid_v(int sms)
{
    const int sm = SB * (kPanelThreads / 32);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, true, true, SB, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, true, false, SB, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, false, true, SB, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    cudaFuncSetAttribute(spmv_panel_kernel<R, C, false, false, SB, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_panel_kernel<R, C, false, true, SB, MB>,
                                                      kPanelThreads, sm) != cudaSuccess || per < 1)
        per = 1;
    cudaGetLastError();
    return sms * per;
}

// Variants: (stage bytes per warp, blocks per SM the registers are budgeted for).
template <int R, int C>
cudaError_t launch_RC(const SpmvLaunch &L, cudaStream_t s)
{
    switch (L.A.panel_variant) {
    case 1: return launch_v<R, C, 4096, 6>(L, s);
    case 2: return launch_v<R, C, 3072, 10>(L, s);
    case 3: return launch_v<R, C, 6144, 6>(L, s);
    default: return launch_v<R, C, 4096, 8>(L, s);
    }
}

template <int R, int C>
int grid_RC(int sms, int variant)
{
    switch (variant) {
    case 1: return grid_v<R, C, 4096, 6>(sms);
    case 2: return grid_v<R, C, 3072, 10>(sms);
    case 3: return grid_v<R, C, 6144, 6>(sms);
    default: return grid_v<R, C, 4096, 8>(sms);
    }
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

int panel_grid_for(int T, int sms, int variant)
{
    switch (T) {
    case 16: return grid_RC<16, 16>(sms, variant);
    case 32: return grid_RC<32, 32>(sms, variant);
    default: return 0;
    }
}

}  // namespace evocg
