// spmv.cu -- launchers of the tile-wise mixed-precision SpMV (the kernel body lives in
// spmv_kernel.cuh), the rounded x copies it reads, and the device rounding entry point.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"
#include "spmv_kernel.cuh"

namespace evocg {

// Last block of a grid: true in every thread of the block whose ticket comes last.
__device__ __forceinline__ bool last_block(DevState *st, int slot)
{
    __shared__ bool amLast;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&st->tickets[slot], 1u);
        amLast = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (amLast) __threadfence();
    return amLast;
}

// Deterministic block sum of one double per thread (fixed shuffle tree, fixed order);
// the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double v)
{
    __shared__ double ws[32];
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) ws[w] = v;
    __syncthreads();
    double s = 0.0;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += ws[i];
    return s;
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src)
{
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)v, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)((uint64_t)v >> 32), src);
    return (int64_t)(((uint64_t)hi << 32) | lo);
}

template <int T, bool FORCE64, bool DOT>
__global__ void __launch_bounds__(kSpmvThreads) spmv_kernel(SpmvLaunch L)
{
    using Gm = Geo<T>;
    if (DOT && L.st->done) return;  // a stopped solve: nothing to compute or count
    const TilesView A = L.A;
    const unsigned lane = lane_id();
    const int gl = (int)(lane % Gm::G);
    const int64_t wpb = blockDim.x >> 5;
    const int64_t W = (int64_t)gridDim.x * wpb;
    const int64_t w = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t rbA = w * A.nrb / W, rbB = (w + 1) * A.nrb / W;
    double dotp = 0.0;
    unsigned long long cnt0 = 0, cnt1 = 0, cnt2 = 0;
    double acc[Gm::RPL];
    F32Pair pr[Gm::RPL];
#pragma unroll
    for (int rr = 0; rr < Gm::RPL; ++rr) acc[rr] = 0.0;
    bool any64 = false, anylow = false;
    int64_t rb_cur = rbA;

    // write the rows of rb_cur, zero rows of the empty row blocks before new_rb, move on
    auto flush_to = [&](int64_t new_rb) {
#pragma unroll
        for (int rr = 0; rr < Gm::RPL; ++rr) {
            const int64_t row = rb_cur * T + gl + rr * Gm::G;
            if ((int)lane < Gm::G && row < A.n) {
                double y = acc[rr];
                if (anylow) {
                    const double d = f64_from_f32(pr[rr].hi) + f64_from_f32(pr[rr].lo);
                    y = any64 ? y + d : d;
                }
                L.y[row] = y;
                if (DOT) dotp = fma(__ldg(L.x64 + row), y, dotp);
            }
            acc[rr] = 0.0;
            pr[rr] = F32Pair();
        }
        for (int64_t rb = rb_cur + 1; rb < new_rb; ++rb)
#pragma unroll
            for (int rr = 0; rr < Gm::RPL; ++rr) {
                const int64_t row = rb * T + gl + rr * Gm::G;
                if ((int)lane < Gm::G && row < A.n) L.y[row] = 0.0;
            }
        any64 = false;
        anylow = false;
        rb_cur = new_rb;
    };

    if (rbA < rbB) {
        int64_t t = A.tileRowPtr[rbA];
        const int64_t tEnd = A.tileRowPtr[rbB];
        while (t < tEnd) {
            const int64_t rb0 = rb_cur;
            // ends of the row blocks rb0 .. rb0+31 (capped at this warp's range)
            const int64_t wend = __ldg(A.tileRowPtr + min(rb0 + 1 + (int64_t)lane, rbB));
            const int64_t wlast = shfl64(wend, 31);
            if (wlast <= t) {  // those 32 row blocks have no tiles left
                flush_to(min(rb0 + 32, rbB));
                continue;
            }
            const int64_t cend = min(min(t + 32, tEnd), wlast);
            const int nt = (int)(cend - t);
            // row ends of the first two tiles, while the descriptors load
            RowEnds<T> R0, R1;
            load_rowends<T>(A, t, 0, nt, R0);
            load_rowends<T>(A, t, 1, nt, R1);
            // descriptors of the chunk: lane u holds tile t+u
            const int64_t tt = t + lane;
            int cbv = 0, pv = 0;
            int64_t ov = 0;
            if ((int)lane < nt) {
                cbv = __ldcs(A.tileColIdx + tt);
                ov = __ldcs(A.tileNnzOff + tt);
                pv = FORCE64 ? 0 : (int)__ldg(L.prec + (L.map_kind ? (int64_t)cbv : tt));
                if (L.census) {
                    const unsigned long long c = (unsigned long long)(__ldcs(A.tileNnzOff + tt + 1) - ov);
                    if (pv == 0) cnt0 += c; else if (pv == 1) cnt1 += c; else cnt2 += c;
                }
            }
            int drb = 0;  // row block of tile tt, counted from rb0: window ends <= tt
#pragma unroll
            for (int step = 16; step; step >>= 1)
                if (shfl64(wend, drb + step - 1) <= tt) drb += step;
            const int64_t offbase = shfl64(ov, 0);
            const uint32_t dw0 = (uint32_t)cbv | ((uint32_t)pv << 28);
            const uint32_t dw1 = (uint32_t)(ov - offbase) | ((uint32_t)drb << 24);

            TileStage<T> S0, S1;
            load_stage<T>(A, L, dw0, dw1, offbase, 0, nt, R0, S0);
            for (int u = 0; u < nt; ++u) {
                load_stage<T>(A, L, dw0, dw1, offbase, u + 1, nt, R1, S1);
                load_rowends<T>(A, t, u + 2, nt, R1);
                const int64_t rbu = rb0 + S0.drb;
                if (rbu != rb_cur) flush_to(rbu);
                any64 |= (S0.prec == EVOCG_FP64);
                anylow |= (S0.prec != EVOCG_FP64);
                compute_stage<T>(A, L, S0, acc, pr);
                S0 = S1;
            }
            t = cend;
        }
        flush_to(rbB);
    }
    if (L.census) {
        for (int o = 16; o; o >>= 1) {
            cnt0 += __shfl_xor_sync(0xffffffffu, cnt0, o);
            cnt1 += __shfl_xor_sync(0xffffffffu, cnt1, o);
            cnt2 += __shfl_xor_sync(0xffffffffu, cnt2, o);
        }
        if (lane == 0) {
            if (cnt0) atomicAdd(&L.st->census[0], cnt0);
            if (cnt1) atomicAdd(&L.st->census[1], cnt1);
            if (cnt2) atomicAdd(&L.st->census[2], cnt2);
        }
    }
    if (DOT) {
        DevState *st = L.st;
        const double s = block_sum(dotp);
        if (threadIdx.x == 0) L.partials[blockIdx.x] = s;
        if (last_block(st, TK_SPMV)) {
            double v = 0.0;
            for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) v += __ldcg(L.partials + i);
            const double sigma = block_sum(v);
            if (threadIdx.x == 0) {
                st->tickets[TK_SPMV] = 0;
                if (!st->done) {
                    if (!(sigma > 0.0) || !isfinite(sigma)) {
                        st->status = EVOCG_EBREAKDOWN;
                        st->done = 1;
                    } else {
                        st->sigma = sigma;
                        st->alpha = st->rho / sigma;
                    }
                }
            }
        }
    }
}

// x copies for the low-precision tiles: x32_j = RN32(x_j) 2^e_j, x16_j = RN16(x_j) 2^e_j.
__global__ void __launch_bounds__(kVecThreads)
    xcopies_kernel(int64_t n, const double *__restrict__ x, const int8_t *__restrict__ colExp,
                   float *__restrict__ x32, uint16_t *__restrict__ x16)
{
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const double v = x[j];
        const float s = pow2f(colExp[j]);
        x32[j] = __fmul_rn(f32_from_f64_rn(v), s);
        x16[j] = (uint16_t)(__float_as_uint(__fmul_rn(f32_from_bf16(bf16_from_f64_rn(v)), s)) >> 16);
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

cudaError_t launch_spmv(const SpmvLaunch &L, cudaStream_t s)
{
    switch (L.A.T) {
    case 16: return launch_T<16>(L, s);
    case 32: return launch_T<32>(L, s);
    case 64: return launch_T<64>(L, s);
    default: return cudaErrorInvalidValue;
    }
}

int spmv_grid_for(int T, int sms)
{
    int per = 0;
    cudaError_t e;
    switch (T) {
    case 16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_kernel<16, false, true>, kSpmvThreads, 0); break;
    case 64: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_kernel<64, false, true>, kSpmvThreads, 0); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, spmv_kernel<32, false, true>, kSpmvThreads, 0); break;
    }
    if (e != cudaSuccess || per < 1) per = 2;
    int g = sms * per;
    return g > kMaxBlocks ? kMaxBlocks : g;
}

cudaError_t launch_xcopies(const TilesView &A, const double *x, float *x32, uint16_t *x16,
                           int grid, cudaStream_t s)
{
    if (A.n == 0) return cudaSuccess;
    xcopies_kernel<<<grid, kVecThreads, 0, s>>>(A.n, x, A.colExp, x32, x16);
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
