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
// Staging. Each warp owns one shared-memory stage. A panel's tiles come in batches planned on
// the host (panel_plan.cpp: every tile sized for FP64, so the plan holds for any precision
// map), each tile with a fixed stage offset. For a batch the lanes issue asynchronous
// global-to-shared copies (cp.async): a tile's value slice in the stream its precision
// selects (16 bytes per lane and instruction; the builder aligns every tile with more than one
// slot to 8 slots and pads it to a multiple of 8, so slices are whole 16-byte chunks in every
// stream), its local-column bytes (8 per lane) and its x segment in that precision (one entry
// per lane); single-entry tiles (one row, width one: the panel-edge tiles of stencils, most of
// a stencil's tiles by count) copy just their value and x entry, one lane each. The warp then
// waits for its own copies (cp.async.wait_group: a hardware wait on the issuing threads'
// copies, no polling) and computes the batch from shared memory. The next panel's descriptors
// and their precisions are loaded while the current panel is in flight. A tile too large for
// the stage on its own is computed from global memory level by level.
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

// Record flags (panel_plan.cpp): single-entry tile, first tile of a batch, tile computed from
// global memory.
constexpr unsigned kSingleBit = 1u << 26, kBatchBit = 1u << 27, kDirectBit = 1u << 28;

// Record layout and batches: panel_plan.cpp. SB: stage bytes per warp (the plan's); MB: blocks
// per SM the registers are sized for; IL: panels interleaved over the warps.
template <int R, int C, bool FORCE64, bool DOT, int SB, int MB, bool IL>
__global__ void __launch_bounds__(kPanelThreads, MB) spmv_panel_kernel(SpmvLaunch L)
{
    static_assert(R == 16 || R == 32, "panel rows");
    static_assert(C == R, "this kernel reads tiles as wide as the panel is tall");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    if ((DOT || L.gate) && L.st->done) return;
    const TilesView &A = L.A;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
    const uint32_t st0 = smem_addr(smem_raw + (size_t)wib * SB);
    const unsigned ltm = lanemask_lt();
    // Panels of this warp: a contiguous range of the plan (IL = false), or every nwarps-th
    // panel from wid (IL = true: all warps sweep one window of the matrix together). Panel
    // q's header record is at q + tileRowPtr[q].
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t pstep = IL ? nwarps : 1;
    const int64_t p_end = IL ? A.nrb : A.warpPanel[wid + 1];
    int64_t p = IL ? wid : A.warpPanel[wid];
    int64_t rec = IL ? (p < p_end ? p + A.tileRowPtr[p] : 0) : A.warpRec[wid];
    int64_t tr_next = (IL && p + pstep < p_end) ? __ldg(A.tileRowPtr + p + pstep) : 0;
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

    for (; p < p_end; p += pstep) {
        const unsigned nt = __shfl_sync(kAll, win.x, 0);
        const int64_t sbase = (int64_t)(((uint64_t)__shfl_sync(kAll, win.w, 0) << 32) |
                                        (uint64_t)__shfl_sync(kAll, win.z, 0));
        const bool more = p + pstep < p_end;
        const int64_t nextrec = IL ? (more ? p + pstep + tr_next : 0) : rec + 1 + nt;
        if (IL) tr_next = (p + 2 * pstep < p_end) ? __ldg(A.tileRowPtr + p + 2 * pstep) : 0;
        uint4 nwin = make_uint4(0u, 0u, 0u, 0u);
        int nprec = 0;
        bool nprec_pending = false;   // a per-column-block map: resolved once nwin is in
        if (more) {
            nwin = __ldcs(A.pdesc + nextrec + lane);
            if (!FORCE64) {
                // tile index of lane's record in the next panel (its count is not known yet,
                // so the index is bounded by the tile count instead)
                const int64_t ti = nextrec + lane - (p + pstep) - 1;
                if (L.map_kind) nprec_pending = true;
                else if (lane > 0 && ti < A.ntiles) nprec = (int)__ldcs(L.prec + ti);
            }
        }
        // this panel's slots in every stream
        const unsigned char *ci = A.colIdx + sbase;
        const unsigned char *vb64 = reinterpret_cast<const unsigned char *>(A.v64 + sbase);
        const unsigned char *vb32 = reinterpret_cast<const unsigned char *>(A.v32 + sbase);
        const unsigned char *vb16 = reinterpret_cast<const unsigned char *>(A.v16 + sbase);

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
            if (!FORCE64) anylow |= __any_sync(kAll, valid && prec != EVOCG_FP64);
            const unsigned vmask = __ballot_sync(kAll, valid);
            const unsigned smask = __ballot_sync(kAll, valid && (d.y & kSingleBit));
            unsigned bmask = __ballot_sync(kAll, valid && (d.y & kBatchBit));
            while (bmask) {
                const int lo = __ffs(bmask) - 1;
                bmask &= bmask - 1u;
                const unsigned upto = bmask ? (1u << (__ffs(bmask) - 1)) - 1u : kAll;
                const unsigned take = vmask & upto & ~((1u << lo) - 1u);
                const unsigned treg = take & ~smask, tsgl = take & smask;
                const bool mine = (take >> lane) & 1u;
                const unsigned ylo = __shfl_sync(kAll, d.y, lo);
                if (ylo & kDirectBit) {   // a tile larger than the stage, from global memory
                    const int pi = __shfl_sync(kAll, prec, lo);
                    const unsigned so = __shfl_sync(kAll, d.x, lo);
                    const int cbi = __shfl_sync(kAll, (int)d.z, lo);
                    const unsigned mi = __shfl_sync(kAll, d.w, lo);
                    const int wi = (int)(ylo & 0xFFu), hi = __popc(mi);
                    const bool has = lane < R && ((mi >> lane) & 1u);
                    const unsigned s0 = so + (unsigned)__popc(mi & ltm);
                    for (int k = 0; has && k < wi; ++k) {
                        const unsigned s = s0 + (unsigned)(k * hi);
                        const unsigned c = ci[s];
                        if (c >= (unsigned)C) continue;
                        const int64_t xj = (int64_t)cbi * C + c;
                        if (pi == EVOCG_FP64) {
                            acc = fma(__ldcs(reinterpret_cast<const double *>(vb64) + s), __ldg(L.x64 + xj), acc);
                            if (DOT) ++cnt0;
                        } else if (pi == EVOCG_FP32) {
                            acc_prod(ls, lc, __ldcs(reinterpret_cast<const float *>(vb32) + s), __ldg(L.x32 + xj));
                            if (DOT) ++cnt1;
                        } else {
                            const unsigned b = __ldcs(reinterpret_cast<const unsigned short *>(vb16) + s);
                            acc_low(ls, lc, __fmul_rn(__uint_as_float(b << 16), __ldg(L.x16f + xj)));
                            if (DOT) ++cnt2;
                        }
                    }
                    continue;
                }
                // ---- issue the batch's copies
                unsigned tr = treg;
                while (tr) {
                    const int i = __ffs(tr) - 1;
                    tr &= tr - 1u;
                    const unsigned so = __shfl_sync(kAll, d.x, i);
                    const unsigned y = __shfl_sync(kAll, d.y, i);
                    const int cbi = __shfl_sync(kAll, (int)d.z, i);
                    const unsigned mi = __shfl_sync(kAll, d.w, i);
                    const int pi = __shfl_sync(kAll, prec, i);
                    const unsigned m8 = ((y & 0xFFu) * (unsigned)__popc(mi) + 7u) & ~7u;
                    const uint32_t st = st0 + ((y >> 8) & 0xFFFu) * 16u;
                    const unsigned sz = 8u >> pi;   // 8, 4, 2 bytes
                    const unsigned char *vs = (pi == EVOCG_FP64 ? vb64 : pi == EVOCG_FP32 ? vb32 : vb16) + so * sz;
                    const unsigned nv16 = (m8 * sz) >> 4;
                    for (unsigned q = lane; q < nv16; q += 32) cp16(st + 16u * q, vs + 16u * q);
                    const uint32_t cst = st + 8u * m8;
                    for (unsigned q = lane; q < (m8 >> 3); q += 32) cp8(cst + 8u * q, ci + so + 8u * q);
                    const uint32_t xst = cst + ((m8 + 15u) & ~15u);
                    const int64_t xj = (int64_t)cbi * C + lane;
                    if (lane < C && xj < A.n) {
                        if (pi == EVOCG_FP64) cp8(xst + 8u * lane, L.x64 + xj);
                        else cp4(xst + 4u * lane, (pi == EVOCG_FP32 ? L.x32 : L.x16f) + xj);
                    }
                }
                // single-entry tiles: their value and x entry into the lane's own 16-byte slot
                const bool sgl = mine && (d.y & kSingleBit);
                if (sgl) {
                    const uint32_t sd = st0 + (uint32_t)lane * 16u;
                    const int64_t xj = (int64_t)(int)d.z * C + (int64_t)((d.y >> 20) & 0x3Fu);
                    if (prec == EVOCG_FP64) {
                        cp8(sd, vb64 + 8u * d.x);
                        cp8(sd + 8u, L.x64 + xj);
                    } else if (prec == EVOCG_FP32) {
                        cp4(sd, vb32 + 4u * d.x);
                        cp4(sd + 8u, L.x32 + xj);
                    } else {
                        cp4(sd, vb16 + 2u * (d.x & ~1u));   // the aligned pair holding it
                        cp4(sd + 8u, L.x16f + xj);
                    }
                }
                if (nprec_pending) {   // the next panel's precisions, while the copies fly
                    nprec_pending = false;
                    const unsigned nnt = __shfl_sync(kAll, nwin.x, 0);
                    if (lane > 0 && lane <= (int)nnt) nprec = (int)__ldg(L.prec + (int)nwin.z);
                }
                cp_wait_all();
                __syncwarp();

                // ---- compute the batch from the stage
                tr = treg;
                while (tr) {
                    const int i = __ffs(tr) - 1;
                    tr &= tr - 1u;
                    const unsigned y = __shfl_sync(kAll, d.y, i);
                    const unsigned mi = __shfl_sync(kAll, d.w, i);
                    const int pi = __shfl_sync(kAll, prec, i);
                    if (lane >= R || !((mi >> lane) & 1u)) continue;
                    const unsigned wi = y & 0xFFu, hi = (unsigned)__popc(mi), j = (unsigned)__popc(mi & ltm);
                    const unsigned m8 = (wi * hi + 7u) & ~7u;
                    const uint32_t st = st0 + ((y >> 8) & 0xFFFu) * 16u;
                    const uint32_t cst = st + 8u * m8 + j;
                    const uint32_t xst = st + 8u * m8 + ((m8 + 15u) & ~15u);
                    if (pi == EVOCG_FP64) {
                        const uint32_t vst = st + 8u * j;
                        for (unsigned k = 0; k < wi; ++k) {
                            const unsigned c = lds_u8(cst + k * hi);
                            if (c < (unsigned)C) {
                                acc = fma(lds_f64(vst + 8u * k * hi), lds_f64(xst + 8u * c), acc);
                                if (DOT) ++cnt0;
                            }
                        }
                    } else if (pi == EVOCG_FP32) {
                        const uint32_t vst = st + 4u * j;
                        for (unsigned k = 0; k < wi; ++k) {
                            const unsigned c = lds_u8(cst + k * hi);
                            if (c < (unsigned)C) {
                                acc_prod(ls, lc, lds_f32(vst + 4u * k * hi), lds_f32(xst + 4u * c));
                                if (DOT) ++cnt1;
                            }
                        }
                    } else {
                        const uint32_t vst = st + 2u * j;
                        for (unsigned k = 0; k < wi; ++k) {
                            const unsigned c = lds_u8(cst + k * hi);
                            if (c < (unsigned)C) {   // BF16 x BF16 is exact in FP32
                                acc_low(ls, lc, __fmul_rn(__uint_as_float(lds_u16(vst + 2u * k * hi) << 16),
                                                          lds_f32(xst + 4u * c)));
                                if (DOT) ++cnt2;
                            }
                        }
                    }
                }
                // single-entry tiles: the product on the copying lane, added by the row's lane
                unsigned sa = 0u, sb = 0u;
                if (sgl) {
                    const uint32_t sd = st0 + (uint32_t)lane * 16u;
                    if (prec == EVOCG_FP64) {
                        const double pd = lds_f64(sd) * lds_f64(sd + 8u);
                        sa = (unsigned)__double2loint(pd);
                        sb = (unsigned)__double2hiint(pd);
                        if (DOT) ++cnt0;
                    } else {
                        const unsigned wd = lds_u32(sd);
                        const float a = prec == EVOCG_FP32 ? __uint_as_float(wd)
                                        : __uint_as_float((d.x & 1u) ? (wd & 0xFFFF0000u) : (wd << 16));
                        const float xv = lds_f32(sd + 8u);
                        const float pf = __fmul_rn(a, xv);
                        sa = __float_as_uint(pf);
                        sb = __float_as_uint(__fmaf_rn(a, xv, -pf));   // exact remainder
                        if (DOT) { if (prec == EVOCG_FP32) ++cnt1; else ++cnt2; }
                    }
                }
                const int srow = __ffs(d.w) - 1;
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
                __syncwarp();   // the stage is free for the next batch
            }
        }
        if (nprec_pending) {
            const unsigned nnt = __shfl_sync(kAll, nwin.x, 0);
            if (lane > 0 && lane <= (int)nnt) nprec = (int)__ldg(L.prec + (int)nwin.z);
        }
        const int64_t row = p * R + lane;
        if (lane < R && row < A.n) {
            double yv = acc;
            if (!FORCE64 && anylow) yv = (acc + f64_from_f32(ls)) + f64_from_f32(lc);
            L.y[row] = yv;
            if (DOT) dotp = fma(__ldg(L.x64 + row), yv, dotp);
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

template <int R, int C, int SB, int MB, bool IL>
cudaError_t launch_v(const SpmvLaunch &L, cudaStream_t s)
{
    const int grid = L.A.panel_grid;
    const size_t sm = (size_t)SB * (kPanelThreads / 32);
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
    const int sm = SB * (kPanelThreads / 32);
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

// Variants: (stage bytes per warp, blocks per SM the registers are budgeted for, panels
// interleaved over the warps).
#define EVOCG_PANEL_VARIANTS(X)     \
    X(0, 4096, 8, true)             \
    X(1, 4096, 8, false)            \
    X(2, 4096, 6, true)             \
    X(3, 6144, 6, true)

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
