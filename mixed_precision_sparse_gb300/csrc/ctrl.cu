// ctrl.cu -- in-loop precision controllers (EvoCG, "Self-Evolving Precision Control for
// Faster Conjugate Gradient", §3.2.2 Eq. 8-10 state and action, §3.2.3 policy network,
// §3.4 device-side inference, §4.7 residual-threshold rule) for sm_103a.
//
// The policy runs one warp per column block (segment of C = T entries of p). The FP64
// segment is normalised without FP64 instructions: its largest magnitude fixes a power
// of two that brings the entries into [-2, 2] by an exponent shift, the shifted entries
// are rounded to FP32 on the integer pipe, and the norm, phi and the three layers run
// in FP32 on the CUDA cores with weights staged in shared memory (transposed, so lanes
// read consecutive banks). The decision is the argmax of the logits, ties to the lower
// code (the higher precision).
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

namespace {

constexpr int kMlpThreads = 256;
constexpr int kMlpWarps = kMlpThreads / 32;

// v * 2^-e for an FP64 bit pattern, by exponent arithmetic; results below the FP64
// normal range are flushed to zero (they are < 2^-1022 relative to the segment maximum).
__device__ __forceinline__ uint64_t scale_bits(uint64_t u, int e)
{
    const int ef = (int)((u >> 52) & 0x7FF);
    if (ef == 0) return u & 0x8000000000000000ull;
    const int nf = ef - e;
    if (nf <= 0) return u & 0x8000000000000000ull;
    if (nf >= 2047) return (u & 0x8000000000000000ull) | 0x7FF0000000000000ull;
    return (u & 0x800FFFFFFFFFFFFFull) | ((uint64_t)nf << 52);
}

template <int T>
__global__ void __launch_bounds__(kMlpThreads)
    mlp_kernel(int64_t n, const double *__restrict__ p, const float *__restrict__ W, int H1,
               int H2, double delta, uint8_t *__restrict__ cbPrec, float *__restrict__ logits,
               DevState *gate)
{
    if (gate) {
        if (gate->done || (gate->k % gate->kstar) != 0) return;
        if (blockIdx.x == 0 && threadIdx.x == 0) gate->ctrl_calls += 1;
    }
    __shared__ float W1t[T * kMlpHiddenMax];              // [c][o]
    __shared__ float W2t[kMlpHiddenMax * kMlpHiddenMax];  // [c][o]
    __shared__ float W3s[3 * kMlpHiddenMax];
    __shared__ float b1s[kMlpHiddenMax], b2s[kMlpHiddenMax], b3s[4];
    __shared__ float phis[kMlpWarps][T];
    __shared__ float h1s[kMlpWarps][kMlpHiddenMax];
    // packed layout: W1 (H1 x T), b1, W2 (H2 x H1), b2, W3 (3 x H2), b3
    const float *gW1 = W, *gb1 = gW1 + H1 * T, *gW2 = gb1 + H1, *gb2 = gW2 + H2 * H1;
    const float *gW3 = gb2 + H2, *gb3 = gW3 + 3 * H2;
    for (int i = threadIdx.x; i < H1 * T; i += blockDim.x) {
        const int o = i / T, c = i % T;
        W1t[c * kMlpHiddenMax + o] = gW1[i];
    }
    for (int i = threadIdx.x; i < H2 * H1; i += blockDim.x) {
        const int o = i / H1, c = i % H1;
        W2t[c * kMlpHiddenMax + o] = gW2[i];
    }
    for (int i = threadIdx.x; i < 3 * H2; i += blockDim.x) W3s[i] = gW3[i];
    for (int i = threadIdx.x; i < H1; i += blockDim.x) b1s[i] = gb1[i];
    for (int i = threadIdx.x; i < H2; i += blockDim.x) b2s[i] = gb2[i];
    if (threadIdx.x < 3) b3s[threadIdx.x] = gb3[threadIdx.x];
    __syncthreads();

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t ncb = (n + T - 1) / T;
    const uint64_t dbits = (uint64_t)__double_as_longlong(delta);
    constexpr int PL = (T + 31) / 32;  // entries per lane
    for (int64_t seg = (int64_t)blockIdx.x * kMlpWarps + w; seg < ncb;
         seg += (int64_t)gridDim.x * kMlpWarps) {
        // ---- phi = p_i / max(||p_i||, delta) (Eq. 8), without FP64 arithmetic
        uint64_t u[PL];
        uint64_t m = 0;
#pragma unroll
        for (int h = 0; h < PL; ++h) {
            const int c = lane + 32 * h;
            const int64_t j = seg * T + c;
            u[h] = (c < T && j < n) ? (uint64_t)__double_as_longlong(p[j]) : 0ull;
            const uint64_t a = u[h] & 0x7FFFFFFFFFFFFFFFull;
            m = a > m ? a : m;
        }
        for (int o = 16; o; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, m, o);
            m = other > m ? other : m;
        }
        const int mef = (int)(m >> 52);
        const int e = (mef == 0) ? 0 : mef - 1023;   // floor(log2 max |p|); zero segment -> 0
        float ps[PL];
        float ss = 0.f;
#pragma unroll
        for (int h = 0; h < PL; ++h) {
            ps[h] = (mef == 0) ? 0.f : __uint_as_float(rne_bits_from_f64<23>(scale_bits(u[h], e)));
            ss = __fmaf_rn(ps[h], ps[h], ss);
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float nrm = sqrtf(ss);                        // ||p_i|| * 2^-e
        const float dsc = __uint_as_float(rne_bits_from_f64<23>(scale_bits(dbits, e)));
        const float den = (nrm > dsc) ? nrm : dsc;          // max(||p_i||, delta) * 2^-e
#pragma unroll
        for (int h = 0; h < PL; ++h) {
            const int c = lane + 32 * h;
            if (c < T) phis[w][c] = (den > 0.f) ? __fdiv_rn(ps[h], den) : 0.f;
        }
        __syncwarp();
        // ---- layer 1: lane takes outputs lane and lane + 32
        float a0 = 0.f, a1 = 0.f;
        if (lane < H1) a0 = b1s[lane];
        if (lane + 32 < H1) a1 = b1s[lane + 32];
#pragma unroll 8
        for (int c = 0; c < T; ++c) {
            const float f = phis[w][c];
            a0 = __fmaf_rn(W1t[c * kMlpHiddenMax + lane], f, a0);
            a1 = __fmaf_rn(W1t[c * kMlpHiddenMax + lane + 32], f, a1);
        }
        if (lane < H1) h1s[w][lane] = a0 > 0.f ? a0 : 0.f;
        if (lane + 32 < H1) h1s[w][lane + 32] = a1 > 0.f ? a1 : 0.f;
        __syncwarp();
        // ---- layer 2
        float c0 = 0.f, c1 = 0.f;
        if (lane < H2) c0 = b2s[lane];
        if (lane + 32 < H2) c1 = b2s[lane + 32];
        for (int c = 0; c < H1; ++c) {
            const float f = h1s[w][c];
            c0 = __fmaf_rn(W2t[c * kMlpHiddenMax + lane], f, c0);
            c1 = __fmaf_rn(W2t[c * kMlpHiddenMax + lane + 32], f, c1);
        }
        const float g0 = (lane < H2 && c0 > 0.f) ? c0 : 0.f;
        const float g1 = (lane + 32 < H2 && c1 > 0.f) ? c1 : 0.f;
        // ---- head: three dot products over H2, reduced across the warp
        float z[3];
#pragma unroll
        for (int o = 0; o < 3; ++o) {
            float t = 0.f;
            if (lane < H2) t = __fmul_rn(W3s[o * H2 + lane], g0);
            if (lane + 32 < H2) t = __fmaf_rn(W3s[o * H2 + lane + 32], g1, t);
            for (int s = 16; s; s >>= 1) t += __shfl_xor_sync(0xffffffffu, t, s);
            z[o] = t + b3s[o];
        }
        if (lane == 0) {
            int best = 0;
            if (z[1] > z[best]) best = 1;
            if (z[2] > z[best]) best = 2;
            cbPrec[seg] = (uint8_t)best;
            if (logits) {
                logits[3 * seg] = z[0];
                logits[3 * seg + 1] = z[1];
                logits[3 * seg + 2] = z[2];
            }
        }
        __syncwarp();
    }
}

// Threshold rule on a given p (one thread per segment), for one-off decisions.
__global__ void threshold_kernel(int64_t n, int T, const double *__restrict__ p, uint64_t lo_bits,
                                 uint64_t hi_bits, uint8_t *__restrict__ cbPrec)
{
    const int64_t ncb = (n + T - 1) / T;
    for (int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; seg < ncb;
         seg += (int64_t)gridDim.x * blockDim.x) {
        uint64_t m = 0;
        for (int c = 0; c < T; ++c) {
            const int64_t j = seg * T + c;
            if (j >= n) break;
            const uint64_t a = (uint64_t)__double_as_longlong(p[j]) & 0x7FFFFFFFFFFFFFFFull;
            m = a > m ? a : m;
        }
        cbPrec[seg] = (m < lo_bits) ? EVOCG_BF16 : (m < hi_bits) ? EVOCG_FP32 : EVOCG_FP64;
    }
}

__global__ void broadcast_kernel(int64_t ntiles, const int32_t *__restrict__ tileColIdx,
                                 const uint8_t *__restrict__ cbPrec, uint8_t *__restrict__ tilePrec)
{
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < ntiles;
         t += (int64_t)gridDim.x * blockDim.x)
        tilePrec[t] = cbPrec[tileColIdx[t]];
}

int grid_for(int64_t items, int per_block, int cap)
{
    int64_t g = (items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    return (int)(g > cap ? cap : g);
}

}  // namespace

cudaError_t launch_ctrl_mlp(const TilesView &A, const double *p, const float *W, int H1, int H2,
                            double delta, uint8_t *cbPrec, float *logits, const DevState *gate,
                            cudaStream_t s)
{
    const int64_t ncb = A.nrb;
    if (ncb == 0) return cudaSuccess;
    const int grid = grid_for(ncb, kMlpWarps, 4096);
    DevState *g = const_cast<DevState *>(gate);
    switch (A.T) {
    case 16: mlp_kernel<16><<<grid, kMlpThreads, 0, s>>>(A.n, p, W, H1, H2, delta, cbPrec, logits, g); break;
    case 32: mlp_kernel<32><<<grid, kMlpThreads, 0, s>>>(A.n, p, W, H1, H2, delta, cbPrec, logits, g); break;
    case 64: mlp_kernel<64><<<grid, kMlpThreads, 0, s>>>(A.n, p, W, H1, H2, delta, cbPrec, logits, g); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_ctrl_threshold(const TilesView &A, const double *p, double eps_lo,
                                  double eps_hi, uint8_t *cbPrec, cudaStream_t s)
{
    if (A.nrb == 0) return cudaSuccess;
    threshold_kernel<<<grid_for(A.nrb, 256, 4096), 256, 0, s>>>(
        A.n, A.T, p, (uint64_t)__builtin_bit_cast(long long, eps_lo),
        (uint64_t)__builtin_bit_cast(long long, eps_hi), cbPrec);
    return cudaGetLastError();
}

cudaError_t launch_broadcast_map(const TilesView &A, const uint8_t *cbPrec, uint8_t *tilePrec,
                                 cudaStream_t s)
{
    if (A.ntiles == 0) return cudaSuccess;
    broadcast_kernel<<<grid_for(A.ntiles, 256, 8192), 256, 0, s>>>(A.ntiles, A.tileColIdx, cbPrec, tilePrec);
    return cudaGetLastError();
}

}  // namespace evocg
