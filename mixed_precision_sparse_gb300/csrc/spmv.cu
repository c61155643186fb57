// spmv.cu -- the direct tile-wise mixed-precision SpMV (EvoCG, "Self-Evolving Precision
// Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 / Eq. 5) for sm_103a, the kernel
// choice, the rounded x copies the SpMV reads, and the device rounding entry point. The
// row-block kernel (spmv_rowblock.cu, tiles of 32), the row-ELL kernel (spmv_rowell.cu, sparse
// tiles of 64) and the panel kernel (spmv_panel.cu, tiles of 16) run wherever their plans
// exist; this kernel runs the rest (tiles of 64 that hold several entries per row) and on
// request.
//
// Work mapping. A warp owns a row block (T rows) at a time and walks its tiles in
// ascending column block, so every row is summed in column order. Lane l owns local row
// l (T = 32), rows l and l+32 (T = 64), or, for T = 16, the two half-warps take
// alternate tiles of the row block and are merged at the end. Each lane keeps its rows'
// sums in registers for the whole row block: no cross-lane reduction at all. In a tile,
// a lane whose row is in the row mask reads its slots k*h + j (j = the mask's popcount
// below its row) for k < w and skips pads (local column T).
//
// Arithmetic. An FP64 tile costs exactly one FP64 fused multiply-add per entry, the
// floor for FP64 data. FP32 and BF16 tiles never touch the FP64 unit: their products
// are exact in an FP32 pair (BF16 x BF16 fits in FP32; FP32 x FP32 is split by one
// fused multiply-add), summed error-free (TwoSum) into an FP32 hi/lo pair, and merged
// into the FP64 row sum once per row: about 48 bits of the sum are kept, so a
// low-precision tile contributes its exactly rounded-operand products, as the paper's
// model asks, and the row sum stays an FP64 sum. GB300 issues FP64 at about 1/58 of
// the FP32 rate, so this split is what lets low-precision tiles run at memory speed.
//
// Operands. The x entries a low-precision tile reads are the FP32 / BF16 roundings of x
// scaled by the column factor 2^e_j, made once per SpMV (xcopies_kernel, or the CG
// p-update) with integer instructions.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

template <int T>
struct Geo {
    static constexpr int G = T < 32 ? T : 32;  // lanes per row group
    static constexpr int NG = 32 / G;          // row groups per warp
    static constexpr int RPL = T / G;          // rows per lane
};

template <int T, bool FORCE64, bool DOT>
__global__ void __launch_bounds__(kSpmvThreads, kSpmvMinBlocks) spmv_kernel(SpmvLaunch L)
{
    using Gm = Geo<T>;
    if ((DOT || L.gate) && L.st->done) return;  // a stopped solve: nothing to compute or count
    const TilesView A = L.A;
    const int lane = threadIdx.x & 31;
    const int grp = lane / Gm::G;
    const int gl = lane % Gm::G;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * wpb;
    const int64_t wid = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    double dotp = 0.0;
    unsigned cnt0 = 0, cnt1 = 0, cnt2 = 0;   // stored entries per precision (census)

    for (int64_t rb = wid; rb < A.nrb; rb += nwarps) {
        const int64_t t0 = A.tileRowPtr[rb], t1 = A.tileRowPtr[rb + 1];
        double acc64[Gm::RPL];
        F32Pair accl[Gm::RPL];
#pragma unroll
        for (int rr = 0; rr < Gm::RPL; ++rr) acc64[rr] = 0.0;
        bool any64 = false, anylow = false;
        for (int64_t t = t0 + grp; t < t1; t += Gm::NG) {
            const int64_t cb = A.tileColIdx[t];
            const int64_t off = A.tileNnzOff[t];
            const uint64_t msk = __ldg(reinterpret_cast<const unsigned long long *>(A.rowMask) + t);
            const int w = (int)__ldg(A.tileWidth + t);
            const int prec = FORCE64 ? 0 : (int)__ldg(L.prec + (L.map_kind ? cb : t));
            const int64_t h = __popcll(msk);
            const uint8_t *ci = A.colIdx + off;
            const int64_t xb = cb * T;
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int r = gl + rr * Gm::G;
                if (!((msk >> r) & 1ull)) continue;          // no entry of my row here
                const int64_t j = __popcll(msk & ((1ull << r) - 1ull));   // my slot column
                if (prec == EVOCG_FP64) {
                    const double *vv = A.v64 + off;
                    const double *xs = L.x64 + xb;
                    double a = acc64[rr];
                    for (int k = 0; k < w; ++k) {
                        const int64_t s = (int64_t)k * h + j;
                        const int c = __ldg(ci + s);
                        if (c < T) { a = fma(__ldg(vv + s), __ldg(xs + c), a); ++cnt0; }
                    }
                    acc64[rr] = a;
                } else if (prec == EVOCG_FP32) {
                    const float *vv = A.v32 + off;
                    const float *xs = L.x32 + xb;
                    for (int k = 0; k < w; ++k) {
                        const int64_t s = (int64_t)k * h + j;
                        const int c = __ldg(ci + s);
                        if (c < T) { accl[rr].add_prod(__ldg(vv + s), __ldg(xs + c)); ++cnt1; }
                    }
                } else {
                    const uint16_t *vv = A.v16 + off;
                    const float *xs = L.x16f + xb;
                    for (int k = 0; k < w; ++k) {  // BF16 x BF16 is exact in FP32
                        const int64_t s = (int64_t)k * h + j;
                        const int c = __ldg(ci + s);
                        if (c < T) {
                            accl[rr].add(__fmul_rn(f32_from_bf16(__ldg(vv + s)), __ldg(xs + c)));
                            ++cnt2;
                        }
                    }
                }
            }
            any64 |= (prec == EVOCG_FP64);
            anylow |= (prec != EVOCG_FP64);
        }
        if (Gm::NG == 2) {  // T = 16: fold the odd-tile half-warp into the even one
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                acc64[rr] += __shfl_down_sync(0xffffffffu, acc64[rr], 16);
                F32Pair o;
                o.hi = __shfl_down_sync(0xffffffffu, accl[rr].hi, 16);
                o.lo = __shfl_down_sync(0xffffffffu, accl[rr].lo, 16);
                accl[rr].merge(o);
            }
        }
        any64 = __any_sync(0xffffffffu, any64);
        anylow = __any_sync(0xffffffffu, anylow);
        if (grp == 0) {
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int64_t row = rb * T + gl + rr * Gm::G;
                if (row < A.n) {
                    double y = acc64[rr];
                    if (anylow) {
                        const double d = f64_from_f32(accl[rr].hi) + f64_from_f32(accl[rr].lo);
                        y = any64 ? y + d : d;
                    }
                    L.y[row] = y;
                    if (DOT) dotp = fma(__ldg(L.x64 + row), y, dotp);
                }
            }
        }
    }
    if (L.census) {
        for (int o = 16; o; o >>= 1) {
            cnt0 += __shfl_xor_sync(0xffffffffu, cnt0, o);
            cnt1 += __shfl_xor_sync(0xffffffffu, cnt1, o);
            cnt2 += __shfl_xor_sync(0xffffffffu, cnt2, o);
        }
        if (lane == 0) {
            if (cnt0) atomicAdd(&L.st->census[0], (unsigned long long)cnt0);
            if (cnt1) atomicAdd(&L.st->census[1], (unsigned long long)cnt1);
            if (cnt2) atomicAdd(&L.st->census[2], (unsigned long long)cnt2);
        }
    }
    if (DOT) {   // this warp's p.q partial (lanes summed in a fixed tree)
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(0xffffffffu, dotp, o);
        if (lane == 0) L.pq[wid] = dotp;
    }
}

// x copies for the low-precision tiles: x32_j = RN32(x_j) 2^e_j and x16f_j = RN16(x_j) 2^e_j,
// the BF16 value held in an FP32 container (4-byte copies stage it like x32).
__global__ void __launch_bounds__(kVecThreads)
    xcopies_kernel(int64_t n, const double *__restrict__ x, const int8_t *__restrict__ colExp,
                   float *__restrict__ x32, float *__restrict__ x16f)
{
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const double v = x[j];
        const float s = pow2f(colExp[j]);
        x32[j] = __fmul_rn(f32_from_f64_rn(v), s);
        x16f[j] = __fmul_rn(f32_from_bf16(bf16_from_f64_rn(v)), s);
    }
}

__global__ void __launch_bounds__(kVecThreads)
    round_kernel(int64_t n, const double *__restrict__ x, float *o32, uint16_t *o16)
{
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const double v = x[j];
        if (o32) o32[j] = f32_from_f64_rn(v);
        if (o16) o16[j] = bf16_from_f64_rn(v);
    }
}

template <int T>
static cudaError_t launch_T(const SpmvLaunch &L, cudaStream_t s)
{
    const int grid = L.grid;
    if (L.force64) {
        if (L.dot) spmv_kernel<T, true, true><<<grid, kSpmvThreads, 0, s>>>(L);
        else spmv_kernel<T, true, false><<<grid, kSpmvThreads, 0, s>>>(L);
    } else {
        if (L.dot) spmv_kernel<T, false, true><<<grid, kSpmvThreads, 0, s>>>(L);
        else spmv_kernel<T, false, false><<<grid, kSpmvThreads, 0, s>>>(L);
    }
    return cudaGetLastError();
}

int spmv_kind_for(const TilesView &A, int direct, int kind)
{
    if (direct) return SPMV_KIND_DIRECT;
    const int k = kind ? kind : A.spmv_kind;
    const bool rb = A.rbMeta && A.rb_grid > 0, el = A.elBase && A.el_grid > 0;
    const bool panel = A.pdesc && A.panel_grid > 0;
    if ((k == SPMV_KIND_ROWBLOCK || k == SPMV_KIND_AUTO) && rb) return SPMV_KIND_ROWBLOCK;
    if ((k == SPMV_KIND_ROWELL || k == SPMV_KIND_AUTO) && el) return SPMV_KIND_ROWELL;
    if ((k == SPMV_KIND_PANEL || k == SPMV_KIND_AUTO) && panel) return SPMV_KIND_PANEL;
    return SPMV_KIND_DIRECT;
}

static int chosen_kind(const SpmvLaunch &L) { return spmv_kind_for(L.A, L.direct, L.kind); }

int spmv_dot_partials(const SpmvLaunch &L)
{
    switch (chosen_kind(L)) {
    case SPMV_KIND_ROWBLOCK: return L.A.rb_grid;   // one per block
    case SPMV_KIND_ROWELL: return L.A.el_grid;     // one per block
    case SPMV_KIND_PANEL: return L.A.panel_grid * (kPanelThreads / 32);
    default: return L.grid * (kSpmvThreads / 32);
    }
}

cudaError_t launch_spmv(const SpmvLaunch &L, cudaStream_t s)
{
    switch (chosen_kind(L)) {
    case SPMV_KIND_ROWBLOCK: return launch_spmv_rowblock(L, s);
    case SPMV_KIND_ROWELL: return launch_spmv_rowell(L, s);
    case SPMV_KIND_PANEL: return launch_spmv_panel(L, s);
    default: return launch_spmv_direct(L, s);
    }
}

cudaError_t launch_spmv_direct(const SpmvLaunch &L, cudaStream_t s)
{
    switch (L.A.T) {
    case 16: return launch_T<16>(L, s);
    case 32: return launch_T<32>(L, s);
    case 64: return launch_T<64>(L, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int T>
static int grid_T(int sms)
{
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_kernel<T, false, true>, kSpmvThreads, 0) !=
            cudaSuccess || per < 1)
        per = 1;
    cudaGetLastError();
    const int g = sms * per;
    return g > kMaxBlocks ? kMaxBlocks : g;
}

int spmv_grid_for(int T, int sms)
{
    switch (T) {
    case 16: return grid_T<16>(sms);
    case 64: return grid_T<64>(sms);
    default: return grid_T<32>(sms);
    }
}

cudaError_t launch_xcopies(const TilesView &A, const double *x, float *x32, float *x16f,
                           int grid, cudaStream_t s)
{
    if (A.n == 0) return cudaSuccess;
    xcopies_kernel<<<grid, kVecThreads, 0, s>>>(A.n, x, A.colExp, x32, x16f);
    return cudaGetLastError();
}

cudaError_t launch_round(const double *x, int64_t n, float *o32, uint16_t *o16, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    int64_t g = (n + kVecThreads - 1) / kVecThreads;
    if (g > 4096) g = 4096;
    round_kernel<<<(int)g, kVecThreads, 0, s>>>(n, x, o32, o16);
    return cudaGetLastError();
}

}  // namespace evocg
