// ctrl.cu -- in-loop precision controllers (EvoCG, "Self-Evolving Precision Control for
// Faster Conjugate Gradient", §3.2.2 Eq. 8-10 state and action, §3.2.3 policy network,
// §3.4 device-side inference, §4.7 residual-threshold rule) for sm_103a.
//
// The policy runs one warp per column block (segment of C = T entries of p), on a grid of
// the blocks that fit on the SMs at once: every block stages the weights (25 KB for T = 32)
// in shared memory once and its warps then walk the segments in a grid stride. The FP64
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

// Weights as the kernel stages them (upload_mlp writes this layout): W1 transposed [c][o]
// (T x 64), W2 transposed [c][o] (64 x 64), W3 row-major (3 x H2, stride H2, in 3 x 64
// words), b1 (64), b2 (64), b3 (4); zero where a width is below 64.
template <int T>
__host__ __device__ constexpr int mlp_words() { return T * kMlpHiddenMax + kMlpHiddenMax * kMlpHiddenMax + 3 * kMlpHiddenMax + 2 * kMlpHiddenMax + 4; }

// Segments a warp evaluates together: every weight read from shared memory serves S of them.
template <int T>
__host__ __device__ constexpr int mlp_segs() { return T <= 32 ? 4 : 2; }

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
    constexpr int S = mlp_segs<T>();
    constexpr int kW = mlp_words<T>();
    static_assert(kW % 4 == 0, "the staged weights are copied as float4");
    __shared__ __align__(16) float wsm[kW];
    __shared__ float phis[kMlpWarps][S][T];
    __shared__ float h1s[kMlpWarps][S][kMlpHiddenMax];
    const float *W1t = wsm, *W2t = W1t + T * kMlpHiddenMax, *W3s = W2t + kMlpHiddenMax * kMlpHiddenMax;
    const float *b1s = W3s + 3 * kMlpHiddenMax, *b2s = b1s + kMlpHiddenMax, *b3s = b2s + kMlpHiddenMax;
    for (int i = threadIdx.x; i < kW / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(wsm)[i] = __ldg(reinterpret_cast<const float4 *>(W) + i);
    __syncthreads();

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t ncb = (n + T - 1) / T;
    const int64_t npass = (ncb + S - 1) / S;
    const uint64_t dbits = (uint64_t)__double_as_longlong(delta);
    constexpr int PL = (T + 31) / 32;  // entries per lane
    for (int64_t pass = (int64_t)blockIdx.x * kMlpWarps + w; pass < npass;
         pass += (int64_t)gridDim.x * kMlpWarps) {
        const int64_t seg0 = pass * S;
        // ---- phi = p_i / max(||p_i||, delta) (Eq. 8) for the S segments, without FP64
        // arithmetic; all their loads first
        uint64_t u[S][PL];
#pragma unroll
        for (int sg = 0; sg < S; ++sg)
#pragma unroll
            for (int h = 0; h < PL; ++h) {
                const int c = lane + 32 * h;
                const int64_t j = (seg0 + sg) * T + c;
                u[sg][h] = (c < T && seg0 + sg < ncb && j < n) ? (uint64_t)__double_as_longlong(p[j]) : 0ull;
            }
#pragma unroll
        for (int sg = 0; sg < S; ++sg) {
            uint64_t m = 0;
#pragma unroll
            for (int h = 0; h < PL; ++h) {
                const uint64_t a = ((uint64_t)abs_hi((uint32_t)(u[sg][h] >> 32)) << 32) | (uint32_t)u[sg][h];
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
                ps[h] = (mef == 0) ? 0.f : __uint_as_float(rne_bits_dev<23>(scale_bits(u[sg][h], e)));
                ss = __fmaf_rn(ps[h], ps[h], ss);
            }
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float nrm = sqrtf(ss);                        // ||p_i|| * 2^-e
            const float dsc = __uint_as_float(rne_bits_dev<23>(scale_bits(dbits, e)));
            const float den = (nrm > dsc) ? nrm : dsc;          // max(||p_i||, delta) * 2^-e
#pragma unroll
            for (int h = 0; h < PL; ++h) {
                const int c = lane + 32 * h;
                if (c < T) phis[w][sg][c] = (den > 0.f) ? __fdiv_rn(ps[h], den) : 0.f;
            }
        }
        __syncwarp();
        // ---- layer 1: lane takes outputs lane and lane + 32 of every segment
        float a0[S], a1[S];
#pragma unroll
        for (int sg = 0; sg < S; ++sg) {
            a0[sg] = lane < H1 ? b1s[lane] : 0.f;
            a1[sg] = lane + 32 < H1 ? b1s[lane + 32] : 0.f;
        }
#pragma unroll 4
        for (int c = 0; c < T; ++c) {
            const float wa = W1t[c * kMlpHiddenMax + lane], wb = W1t[c * kMlpHiddenMax + lane + 32];
#pragma unroll
            for (int sg = 0; sg < S; ++sg) {
                const float f = phis[w][sg][c];
                a0[sg] = __fmaf_rn(wa, f, a0[sg]);
                a1[sg] = __fmaf_rn(wb, f, a1[sg]);
            }
        }
#pragma unroll
        for (int sg = 0; sg < S; ++sg) {
            if (lane < H1) h1s[w][sg][lane] = a0[sg] > 0.f ? a0[sg] : 0.f;
            if (lane + 32 < H1) h1s[w][sg][lane + 32] = a1[sg] > 0.f ? a1[sg] : 0.f;
        }
        __syncwarp();
        // ---- layer 2
        float c0[S], c1[S];
#pragma unroll
        for (int sg = 0; sg < S; ++sg) {
            c0[sg] = lane < H2 ? b2s[lane] : 0.f;
            c1[sg] = lane + 32 < H2 ? b2s[lane + 32] : 0.f;
        }
#pragma unroll 4
        for (int c = 0; c < H1; ++c) {
            const float wa = W2t[c * kMlpHiddenMax + lane], wb = W2t[c * kMlpHiddenMax + lane + 32];
#pragma unroll
            for (int sg = 0; sg < S; ++sg) {
                const float f = h1s[w][sg][c];
                c0[sg] = __fmaf_rn(wa, f, c0[sg]);
                c1[sg] = __fmaf_rn(wb, f, c1[sg]);
            }
        }
        // ---- head: three dot products over H2, reduced across the warp, per segment
#pragma unroll
        for (int sg = 0; sg < S; ++sg) {
            const int64_t seg = seg0 + sg;
            const float g0 = (lane < H2 && c0[sg] > 0.f) ? c0[sg] : 0.f;
            const float g1 = (lane + 32 < H2 && c1[sg] > 0.f) ? c1[sg] : 0.f;
            float z[3];
#pragma unroll
            for (int o = 0; o < 3; ++o) {
                float t = 0.f;
                if (lane < H2) t = __fmul_rn(W3s[o * H2 + lane], g0);
                if (lane + 32 < H2) t = __fmaf_rn(W3s[o * H2 + lane + 32], g1, t);
                for (int sh = 16; sh; sh >>= 1) t += __shfl_xor_sync(0xffffffffu, t, sh);
                z[o] = t + b3s[o];
            }
            if (lane == 0 && seg < ncb) {
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

int64_t mlp_staged_words(int T)
{
    switch (T) {
    case 16: return mlp_words<16>();
    case 32: return mlp_words<32>();
    case 64: return mlp_words<64>();
    default: return 0;
    }
}

void mlp_stage_weights(const float *packed, int T, int H1, int H2, float *out)
{
    const int64_t words = mlp_staged_words(T);
    for (int64_t i = 0; i < words; ++i) out[i] = 0.f;
    const float *W1 = packed, *b1 = W1 + (int64_t)H1 * T, *W2 = b1 + H1, *b2 = W2 + (int64_t)H2 * H1;
    const float *W3 = b2 + H2, *b3 = W3 + 3 * H2;
    float *W1t = out, *W2t = W1t + (int64_t)T * kMlpHiddenMax, *W3s = W2t + kMlpHiddenMax * kMlpHiddenMax;
    float *b1s = W3s + 3 * kMlpHiddenMax, *b2s = b1s + kMlpHiddenMax, *b3s = b2s + kMlpHiddenMax;
    for (int o = 0; o < H1; ++o)
        for (int c = 0; c < T; ++c) W1t[c * kMlpHiddenMax + o] = W1[(int64_t)o * T + c];
    for (int o = 0; o < H2; ++o)
        for (int c = 0; c < H1; ++c) W2t[c * kMlpHiddenMax + o] = W2[(int64_t)o * H1 + c];
    for (int i = 0; i < 3 * H2; ++i) W3s[i] = W3[i];
    for (int o = 0; o < H1; ++o) b1s[o] = b1[o];
    for (int o = 0; o < H2; ++o) b2s[o] = b2[o];
    for (int k = 0; k < 3; ++k) b3s[k] = b3[k];
}

int mlp_grid_for(int T, int sms)
{
    int per = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (T) {
    case 16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, mlp_kernel<16>, kMlpThreads, 0); break;
    case 32: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, mlp_kernel<32>, kMlpThreads, 0); break;
    case 64: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, mlp_kernel<64>, kMlpThreads, 0); break;
    default: break;
    }
    if (e != cudaSuccess || per < 1) per = 1;
    cudaGetLastError();
    return sms * per;
}

cudaError_t launch_ctrl_mlp(const TilesView &A, const double *p, const float *W, int H1, int H2,
                            double delta, uint8_t *cbPrec, float *logits, const DevState *gate,
                            cudaStream_t s)
{
    const int64_t ncb = A.nrb;
    if (ncb == 0) return cudaSuccess;
    // one pass of resident blocks (each stages the weights once), at most one warp per segment
    const int grid = grid_for(ncb, kMlpWarps, A.mlp_grid > 0 ? A.mlp_grid : 4096);
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
