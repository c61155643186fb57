// spmv_rowell.cu -- the row-ELL tile-wise mixed-precision SpMV (EvoCG, "Self-Evolving Precision
// Control for Faster Conjugate Gradient", §3.3 EvoSpMV, Eq. 2 / Eq. 5) for matrices whose tiles
// of 64 hold about one entry per row (rowell_plan.cpp), on sm_103a.
//
// A warp owns a row block (64 rows: lane l has rows l and l + 32) and walks its ELL block two
// levels at a time for both rows: first the four slots' columns and precision codes (the
// per-slot copy of the tile map, or the column block's code of a per-column-block map), then
// their values in those formats and their x entries (FP64 x, or the scaled FP32 / BF16
// copies), then the products. Consecutive lanes read consecutive slots at every level, and
// every lane holds one of its rows' entries in every instruction (pads excepted), so each FP64
// fused multiply-add does a full warp of work. Arithmetic as in the tile kernels: one FP64 FMA
// per FP64 entry, FP32 and BF16 products exact in an FP32 pair summed error-free, joined to the
// FP64 row sum once per row.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kElU = 2;           // levels loaded together
constexpr int kElMinBlocks = 4;   // resident blocks of kElThreads per SM the registers are sized for

template <bool FORCE64, bool DOT>
__global__ void __launch_bounds__(kElThreads, kElMinBlocks) spmv_rowell_kernel(SpmvLaunch L)
{
    if ((DOT || L.gate) && L.st->done) return;  // a stopped solve: nothing to compute or count
    const TilesView &A = L.A;
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (kElThreads / 32);
    const int64_t wid = (int64_t)blockIdx.x * (kElThreads / 32) + (threadIdx.x >> 5);
    double dotp = 0.0;
    unsigned cnt[3] = {0u, 0u, 0u};
    for (int64_t rb = wid; rb < A.nrb; rb += nw) {
        const int64_t b0 = A.elBase[rb];
        const int W = (int)((A.elBase[rb + 1] - b0) >> 6);
        double acc[2] = {0.0, 0.0};
        F32Pair lp[2];
        for (int k0 = 0; k0 < W; k0 += kElU) {
            int col[2][kElU], pr[2][kElU];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < kElU; ++u) {
                    col[h][u] = -1;
                    pr[h][u] = EVOCG_FP64;
                    if (k0 + u < W) {
                        const int64_t s = b0 + (int64_t)(k0 + u) * 64 + h * 32 + lane;
                        col[h][u] = __ldcs(A.elCol + s);
                        if (!FORCE64 && !L.map_kind) pr[h][u] = (int)__ldcs(A.elPrec + s);
                    }
                }
            if (!FORCE64 && L.map_kind) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int u = 0; u < kElU; ++u)
                        if (col[h][u] >= 0) pr[h][u] = (int)__ldg(L.prec + (col[h][u] >> 6));
            }
            unsigned long long v[2][kElU], x[2][kElU];   // raw bits: FP64, or FP32 / BF16 low
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < kElU; ++u) {
                    v[h][u] = 0ull;
                    x[h][u] = 0ull;
                    const int c = col[h][u];
                    if (c < 0) continue;
                    const int64_t s = b0 + (int64_t)(k0 + u) * 64 + h * 32 + lane;
                    if (pr[h][u] == EVOCG_FP64) {
                        v[h][u] = (unsigned long long)__double_as_longlong(__ldcs(A.elV64 + s));
                        x[h][u] = (unsigned long long)__double_as_longlong(__ldg(L.x64 + c));
                    } else if (pr[h][u] == EVOCG_FP32) {
                        v[h][u] = __float_as_uint(__ldcs(A.elV32 + s));
                        x[h][u] = __float_as_uint(__ldg(L.x32 + c));
                    } else {
                        v[h][u] = __ldcs(A.elV16 + s);
                        x[h][u] = __float_as_uint(__ldg(L.x16f + c));
                    }
                }
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < kElU; ++u) {
                    if (col[h][u] < 0) continue;
                    if (pr[h][u] == EVOCG_FP64) {
                        acc[h] = fma(__longlong_as_double((long long)v[h][u]), __longlong_as_double((long long)x[h][u]),
                                     acc[h]);
                        ++cnt[0];
                    } else if (pr[h][u] == EVOCG_FP32) {
                        lp[h].add_prod(__uint_as_float((unsigned)v[h][u]), __uint_as_float((unsigned)x[h][u]));
                        ++cnt[1];
                    } else {   // BF16 x BF16: exact in FP32
                        lp[h].add(__fmul_rn(f32_from_bf16((uint16_t)v[h][u]), __uint_as_float((unsigned)x[h][u])));
                        ++cnt[2];
                    }
                }
        }
        const bool low = !FORCE64 && __any_sync(kAll, lp[0].hi != 0.f || lp[0].lo != 0.f ||
                                                         lp[1].hi != 0.f || lp[1].lo != 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = rb * 64 + h * 32 + lane;
            if (row < A.n) {
                double y = acc[h];
                if (low) y = acc[h] + (f64_from_f32(lp[h].hi) + f64_from_f32(lp[h].lo));
                L.y[row] = y;
                if (DOT) dotp = fma(__ldg(L.x64 + row), y, dotp);
            }
        }
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
        __shared__ double s_pq[kElThreads / 32];
        for (int o = 16; o; o >>= 1) dotp += __shfl_xor_sync(kAll, dotp, o);
        if (lane == 0) s_pq[threadIdx.x >> 5] = dotp;
        __syncthreads();
        if (threadIdx.x == 0) {
            double sum = 0.0;
            for (int i = 0; i < kElThreads / 32; ++i) sum += s_pq[i];
            L.pq[blockIdx.x] = sum;
        }
    }
}

// The per-slot copy of a per-tile precision map (pads: FP64, never read).
__global__ void __launch_bounds__(256) elprec_kernel(int64_t ns, const int32_t *__restrict__ tile,
                                                     const uint8_t *__restrict__ tilePrec, uint8_t *__restrict__ out)
{
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < ns; s += (int64_t)gridDim.x * blockDim.x) {
        const int32_t t = tile[s];
        out[s] = t >= 0 ? tilePrec[t] : (uint8_t)EVOCG_FP64;
    }
}

// Within every row of the row-ELL blocks, the slots put in (precision code, column) order, pads
// last: the kernel's lanes then meet one precision at most levels instead of branching over
// two or three (on the banded workload with the 40/40/20 map, 1.8 instead of 2.6 precisions per
// warp and level). The sum of a row is the same up to rounding order; with every tile in FP64
// the order is the plan's column order again. One thread per row; rows of more than
// kElSortMax slots keep their order. The permutation is applied in place by following its
// cycles, each slot moved once.
constexpr int kElSortMax = 64;

__global__ void __launch_bounds__(256) elsort_kernel(int64_t nrb, const int64_t *__restrict__ base,
                                                     int32_t *__restrict__ col, int32_t *__restrict__ tile,
                                                     double *__restrict__ v64, float *__restrict__ v32,
                                                     uint16_t *__restrict__ v16, uint8_t *__restrict__ prec)
{
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nrb * 64;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rb = q >> 6, b0 = base[rb] + (q & 63);
        const int w = (int)((base[rb + 1] - base[rb]) >> 6);
        if (w < 2 || w > kElSortMax) continue;
        uint64_t key[kElSortMax];
        uint8_t src[kElSortMax];   // src[i]: the slot that goes to position i
        for (int k = 0; k < w; ++k) {
            const int64_t s = b0 + (int64_t)k * 64;
            const int32_t c = col[s];
            key[k] = c < 0 ? ~0ull : ((uint64_t)prec[s] << 32) | (uint32_t)c;
            src[k] = (uint8_t)k;
        }
        for (int i = 1; i < w; ++i) {   // insertion sort of (key, slot); keys are distinct but pads
            const uint64_t kk = key[i];
            const uint8_t ss = src[i];
            int j = i - 1;
            while (j >= 0 && key[j] > kk) {
                key[j + 1] = key[j];
                src[j + 1] = src[j];
                --j;
            }
            key[j + 1] = kk;
            src[j + 1] = ss;
        }
        uint64_t done = 0;
        for (int st = 0; st < w; ++st) {
            if (((done >> st) & 1ull) || src[st] == st) continue;
            const int64_t s0 = b0 + (int64_t)st * 64;
            const int32_t tc = col[s0], tt = tile[s0];
            const double t64 = v64[s0];
            const float t32 = v32[s0];
            const uint16_t t16 = v16[s0];
            const uint8_t tp = prec[s0];
            int i = st;
            for (;;) {
                done |= 1ull << i;
                const int j = src[i];
                const int64_t di = b0 + (int64_t)i * 64;
                if (j == st) {
                    col[di] = tc; tile[di] = tt; v64[di] = t64; v32[di] = t32; v16[di] = t16; prec[di] = tp;
                    break;
                }
                const int64_t sj = b0 + (int64_t)j * 64;
                col[di] = col[sj]; tile[di] = tile[sj]; v64[di] = v64[sj]; v32[di] = v32[sj];
                v16[di] = v16[sj]; prec[di] = prec[sj];
                i = j;
            }
        }
    }
}

}  // namespace

int rowell_grid_for(int sms)
{
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_rowell_kernel<false, true>, kElThreads, 0) !=
            cudaSuccess || per < 1)
        per = 1;
    cudaGetLastError();
    const int g = sms * per;
    return g > kMaxBlocks ? kMaxBlocks : g;
}

cudaError_t launch_spmv_rowell(const SpmvLaunch &L, cudaStream_t s)
{
    const int g = L.A.el_grid;
    if (g <= 0 || !L.A.elBase) return cudaErrorInvalidValue;
    if (L.force64) {
        if (L.dot) spmv_rowell_kernel<true, true><<<g, kElThreads, 0, s>>>(L);
        else spmv_rowell_kernel<true, false><<<g, kElThreads, 0, s>>>(L);
    } else {
        if (L.dot) spmv_rowell_kernel<false, true><<<g, kElThreads, 0, s>>>(L);
        else spmv_rowell_kernel<false, false><<<g, kElThreads, 0, s>>>(L);
    }
    return cudaGetLastError();
}

cudaError_t launch_elprec(int64_t ns, const int32_t *tile, const uint8_t *tilePrec, uint8_t *out, cudaStream_t s)
{
    if (ns <= 0) return cudaSuccess;
    int64_t g = (ns + 255) / 256;
    if (g > 8192) g = 8192;
    elprec_kernel<<<(int)g, 256, 0, s>>>(ns, tile, tilePrec, out);
    return cudaGetLastError();
}

cudaError_t launch_elsort(int64_t nrb, const int64_t *base, int32_t *col, int32_t *tile, double *v64,
                          float *v32, uint16_t *v16, uint8_t *prec, cudaStream_t s)
{
    if (nrb <= 0) return cudaSuccess;
    int64_t g = (nrb * 64 + 255) / 256;
    if (g > 8192) g = 8192;
    elsort_kernel<<<(int)g, 256, 0, s>>>(nrb, base, col, tile, v64, v32, v16, prec);
    return cudaGetLastError();
}

}  // namespace evocg
