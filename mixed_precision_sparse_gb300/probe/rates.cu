// rates.cu -- arithmetic-rate probe for the GPU the kernels run on (not part of the solver).
//
// Measures, with every SM full of independent chains, how many of one operation an SM
// completes per clock: FP64 FMA, FP32 FMA, the hardware FP64 -> FP32 and FP32 -> FP64
// conversions, and the integer-pipe FP64 -> FP32 rounding of fpconv.cuh. These are the
// figures behind the SpMV's and the CG kernels' choices (one FP64 FMA per FP64 entry, FP32
// pairs for low-precision entries, conversions on the integer pipe).
//
// Each thread runs kChains independent chains for `iters` steps, every SM holding the same
// number of resident blocks; operations per second from CUDA events around the second of two
// launches, and per clock per SM at the device's maximum SM clock (a lower bound on the
// per-clock rate when the clock ran lower).
#include <cuda_runtime.h>

#include <cstdint>

#include "fpconv.cuh"

namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

enum Kind { FMA64 = 0, FMA32 = 1, CVT64TO32 = 2, CVT32TO64 = 3, INTRND64TO32 = 4, NKIND = 5 };

template <int K>
__global__ void __launch_bounds__(kThreads) rate_kernel(int iters, double m, double c, double *sink)
{
    double d[kChains];
    float f[kChains];
    long long u[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        d[i] = 1.0 + 1e-3 * (threadIdx.x + i);
        f[i] = (float)d[i];
        u[i] = __double_as_longlong(d[i]) + i;
    }
    const float mf = (float)m, cf = (float)c;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            if (K == FMA64) {
                d[i] = fma(d[i], m, c);
            } else if (K == FMA32) {
                f[i] = fmaf(f[i], mf, cf);
            } else if (K == CVT64TO32) {   // one conversion, one 64-bit integer add, one FP32 add
                u[i] += 1;
                f[i] += __double2float_rn(__longlong_as_double(u[i]));
            } else if (K == CVT32TO64) {   // one conversion, one integer add, one FP64 compare-free move
                u[i] += (long long)__double_as_longlong((double)__int_as_float((int)u[i] | 0x3f800000));
            } else {                       // fpconv.cuh's integer rounding, one 64-bit add, one FP32 add
                u[i] += 1;
                f[i] += evocg::f32_from_f64_rn(__longlong_as_double(u[i]));
            }
        }
    }
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += d[i] + (double)f[i] + (double)(u[i] & 1);
    sink[(int64_t)blockIdx.x * kThreads + threadIdx.x] = s;
}

template <int K>
cudaError_t launch(int grid, int iters, double *sink, cudaStream_t s)
{
    rate_kernel<K><<<grid, kThreads, 0, s>>>(iters, 1.0 - 1e-12, 1e-12, sink);
    return cudaGetLastError();
}

cudaError_t launch_kind(int kind, int grid, int iters, double *sink, cudaStream_t s)
{
    switch (kind) {
    case FMA64: return launch<FMA64>(grid, iters, sink, s);
    case FMA32: return launch<FMA32>(grid, iters, sink, s);
    case CVT64TO32: return launch<CVT64TO32>(grid, iters, sink, s);
    case CVT32TO64: return launch<CVT32TO64>(grid, iters, sink, s);
    case INTRND64TO32: return launch<INTRND64TO32>(grid, iters, sink, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Runs probe `kind` (0 FP64 FMA, 1 FP32 FMA, 2 FP64->FP32 cvt, 3 FP32->FP64 cvt, 4 integer
// rounding FP64->FP32) on the current device with `blocks_per_sm` resident blocks of 256
// threads per SM and `iters` steps of 8 chains per thread. Outputs: operations per second
// (CUDA events; the second of two launches), operations per clock per SM at the maximum SM
// clock, and the launch's milliseconds. Returns 0, or a CUDA error code (nothing is left
// allocated).
extern "C" int evocg_rate_probe(int kind, int blocks_per_sm, int iters, double *ops_per_s,
                                double *ops_per_clk_sm, double *ms)
{
    if (kind < 0 || kind >= NKIND || blocks_per_sm < 1 || blocks_per_sm > 8 || iters < 1) return (int)cudaErrorInvalidValue;
    int dev = 0, sms = 0, khz = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
    if (e != cudaSuccess) return (int)e;
    const int grid = sms * blocks_per_sm;
    double *sink = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    e = cudaMalloc(&sink, sizeof(double) * (size_t)grid * kThreads);
    if (e == cudaSuccess) e = cudaEventCreate(&a);
    if (e == cudaSuccess) e = cudaEventCreate(&b);
    float t = 0.f;
    if (e == cudaSuccess) e = launch_kind(kind, grid, iters, sink, 0);   // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(a, 0);
    if (e == cudaSuccess) e = launch_kind(kind, grid, iters, sink, 0);
    if (e == cudaSuccess) e = cudaEventRecord(b, 0);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, a, b);
    if (e == cudaSuccess) {
        const double ops = (double)grid * kThreads * kChains * (double)iters;
        *ms = t;
        *ops_per_s = ops / (t * 1e-3);
        *ops_per_clk_sm = *ops_per_s / ((double)sms * (double)khz * 1e3);
    }
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
    cudaFree(sink);
    return (int)e;
}
