// cg.cu -- fused CG / Jacobi-PCG vector kernels (EvoCG, "Self-Evolving Precision Control
// for Faster Conjugate Gradient": the solver lines of Algorithm 1, §2.1 Fig. 1, §3.4
// fused step, §4.6 Jacobi-PCG) for sm_103a.
//
// One iteration is three kernels in a CUDA graph: the SpMV (with one p.q partial per block),
// cg_update (alpha from those partials; r, z and the two dot products;
// its last block forms beta, the history entry and the stop flag, and drives the graph's
// while node), and cg_pupdate (x += alpha p, then p, the rounded copies of p that the next SpMV reads, and
// the threshold controller's decisions). Reductions are per-thread FP64 partials in a
// fixed order, a fixed shuffle tree per block, and a last-block sum over the blocks in
// index order: bit-reproducible from run to run. FP64 instructions are only the method's
// own (one per axpy or dot term); conversions and comparisons run on the integer pipe.
#include <cuda_runtime.h>

#include "evocg_internal.h"
#include "fpconv.cuh"

namespace evocg {

__device__ __forceinline__ bool last_block_cg(DevState *st, int slot)
{
    __shared__ bool amLast;
    __syncthreads();
    if (threadIdx.x == 0) {   // thread 0 wrote the block's partial: publish it, take a ticket
        __threadfence();
        const unsigned t = atomicAdd(&st->tickets[slot], 1u);
        amLast = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (amLast) __threadfence();
    return amLast;
}

__device__ __forceinline__ double block_sum_cg(double v)
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

// Two block sums (blockDim.x == kVecThreads) with the same result bits as block_sum_cg but
// far fewer FP64 warp instructions (each costs a sub-partition's FP64 unit 64 cycles however
// few lanes it adds): the values go to shared memory, and warp 0 (for a) and warp 1 (for b)
// replay every warp's shuffle tree there, level by level (level o: 8o sums, a warp's
// position j < o plus position j + o), then add the eight warp totals in warp order.
// The results are valid in every thread.
__device__ __forceinline__ void tree_sum2(double a, double b, double &sa, double &sb)
{
    __shared__ double buf[2][kVecThreads];
    __shared__ double res[2];
    static_assert(kVecThreads == 256, "the tree below replays eight warps");
    __syncthreads();   // earlier readers of res are done
    buf[0][threadIdx.x] = a;
    buf[1][threadIdx.x] = b;
    __syncthreads();
    const int wr = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (wr < 2) {
        double *v = buf[wr];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            for (int i = l; i < 8 * o; i += 32) {
                const int k = 32 * (i / o) + (i % o);
                v[k] = v[k] + v[k + o];
            }
            __syncwarp();
        }
        if (l == 0) {
            double t = 0.0;
            for (int w = 0; w < kVecThreads / 32; ++w) t += v[32 * w];
            res[wr] = t;
        }
    }
    __syncthreads();
    sa = res[0];
    sb = res[1];
}

// Sum of gridDim.x partials in a fixed order; valid in thread 0 of the calling block.
__device__ __forceinline__ double sum_partials(const double *part)
{
    double v = 0.0;
    for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) v += __ldcg(part + i);
    return block_sum_cg(v);
}

__device__ __forceinline__ uint64_t abs_bits(double v)
{
    const uint64_t u = (uint64_t)__double_as_longlong(v);
    return ((uint64_t)abs_hi((uint32_t)(u >> 32)) << 32) | (uint32_t)u;
}

// Threshold rule of EvoCG §4.7 on segments of T entries held by T/2 consecutive lanes
// (two entries per lane): m = max |p| over the segment, compared through the bit
// patterns of non-negative doubles (which order like the values; a NaN compares above
// every threshold and keeps FP64). Every lane of the warp must call it.
template <int T>
__device__ __forceinline__ void threshold_segments(uint64_t m, int64_t pair, int64_t ncb,
                                                   uint64_t lo_bits, uint64_t hi_bits,
                                                   uint8_t *cbPrec)
{
    constexpr int W = T / 2;
#pragma unroll
    for (int o = W / 2; o; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, m, o);
        m = other > m ? other : m;
    }
    if ((threadIdx.x & (W - 1)) == 0) {
        const int64_t seg = (2 * pair) / T;
        if (seg < ncb) cbPrec[seg] = (m < lo_bits) ? EVOCG_BF16 : (m < hi_bits) ? EVOCG_FP32 : EVOCG_FP64;
    }
}

// Rounded copies of p for the next SpMV's low-precision tiles (x32, x16f) and its
// threshold features; entries past n are zero.
__device__ __forceinline__ void write_copies(const CgLaunch &L, int64_t j, double v)
{
    const float s = pow2f(L.A.colExp[j]);
    L.x32[j] = __fmul_rn(f32_from_f64_rn(v), s);
    L.x16f[j] = __fmul_rn(f32_from_bf16(bf16_from_f64_rn(v)), s);
}

// The same for the pair j, j + 1 (j even): one 2-byte exponent load, 8-byte stores.
__device__ __forceinline__ void write_copies2(const CgLaunch &L, int64_t j, double v0, double v1)
{
    const char2 e = *reinterpret_cast<const char2 *>(L.A.colExp + j);
    const float s0 = pow2f(e.x), s1 = pow2f(e.y);
    *reinterpret_cast<float2 *>(L.x32 + j) =
        make_float2(__fmul_rn(f32_from_f64_rn(v0), s0), __fmul_rn(f32_from_f64_rn(v1), s1));
    *reinterpret_cast<float2 *>(L.x16f + j) =
        make_float2(__fmul_rn(f32_from_bf16(bf16_from_f64_rn(v0)), s0),
                    __fmul_rn(f32_from_bf16(bf16_from_f64_rn(v1)), s1));
}

// The relative threshold option: both cut points times ||b||_inf (= ||r_0||_inf with x0 = 0),
// before the first decision. Block maxima of |b| through the bit patterns (non-negative
// doubles order like their patterns), the last block scales.
__global__ void __launch_bounds__(kVecThreads) threshold_scale_kernel(CgLaunch L)
{
    DevState *st = L.st;
    uint64_t m = 0;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < L.n; j += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t a = abs_bits(L.b[j]);
        m = a > m ? a : m;
    }
    for (int o = 16; o; o >>= 1) {
        const uint64_t t = __shfl_xor_sync(0xffffffffu, m, o);
        m = t > m ? t : m;
    }
    __shared__ uint64_t wm[kVecThreads / 32];
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < kVecThreads / 32; ++i) m = wm[i] > m ? wm[i] : m;
        L.partials[blockIdx.x] = __longlong_as_double((long long)m);
    }
    if (last_block_cg(st, TK_SCALE) && threadIdx.x == 0) {
        uint64_t g = 0;
        for (int i = 0; i < (int)gridDim.x; ++i) {
            const uint64_t v = (uint64_t)__double_as_longlong(__ldcg(L.partials + i));
            g = v > g ? v : g;
        }
        const double binf = __longlong_as_double((long long)g);
        st->tickets[TK_SCALE] = 0;
        st->eps_hi *= binf;
        st->eps_lo = 0.1 * st->eps_hi;   // 0.1 eps' with eps' = eps ||b||_inf, as the host forms 0.1 eps
    }
}

cudaError_t launch_threshold_scale(const CgLaunch &L, cudaStream_t s)
{
    threshold_scale_kernel<<<L.vec_grid, kVecThreads, 0, s>>>(L);
    return cudaGetLastError();
}

// Start (restart = 0) or FP64-finish restart (restart = 1, after q = A x in FP64):
//   r = b (x = 0) or r = b - q; z = D^-1 r; p = z; rho = r.z; ||r||^2.
template <int T>
__global__ void __launch_bounds__(kVecThreads) cg_init_kernel(CgLaunch L, int restart)
{
    DevState *st = L.st;
    const int64_t n = L.n, npairs = (n + 1) / 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const bool thr = (L.ctrl == EVOCG_CTRL_THRESHOLD) && !restart;
    const uint64_t lo_bits = (uint64_t)__double_as_longlong(st->eps_lo);
    const uint64_t hi_bits = (uint64_t)__double_as_longlong(st->eps_hi);
    const int64_t ncb = (n + T - 1) / T;
    double rz = 0.0, rr = 0.0;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < npairs;
         base += stride) {
        const int64_t pair = base + lane;
        uint64_t m = 0;
        if (pair < npairs) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t j = 2 * pair + h;
                if (j >= n) break;
                double r = L.b[j];
                if (restart) r = r - L.q[j];
                else L.x[j] = 0.0;
                L.r[j] = r;
                double z = r;
                if (L.jacobi) { z = L.dinv[j] * r; L.z[j] = z; }
                L.p[j] = z;
                write_copies(L, j, z);
                rz = fma(r, z, rz);
                rr = fma(r, r, rr);
                const uint64_t ab = abs_bits(z);
                m = ab > m ? ab : m;
            }
        }
        if (thr) threshold_segments<T>(m, pair, ncb, lo_bits, hi_bits, L.cbPrec);
    }
    const double s_rz = block_sum_cg(rz);
    const double s_rr = block_sum_cg(rr);
    if (threadIdx.x == 0) {
        L.partials[blockIdx.x] = s_rz;
        L.partials[kMaxBlocks + blockIdx.x] = s_rr;
    }
    if (last_block_cg(st, TK_INIT)) {
        const double RZ = sum_partials(L.partials);
        const double RR = sum_partials(L.partials + kMaxBlocks);
        if (threadIdx.x == 0) {
            st->tickets[TK_INIT] = 0;
            st->rho = L.jacobi ? RZ : RR;
            st->rr = RR;
            st->xstep = 0;
            if (!restart) {
                st->nr0 = sqrt(RR);
                st->k = 0;
                L.hist[0] = 1.0;
                st->status = EVOCG_OK;
                st->converged = 0;
                if (thr) st->ctrl_calls += 1;
            }
            st->done = 0;
            if (RR == 0.0) {             // b = 0 (or an exact restart residual of zero)
                st->done = 1;
                st->converged = 1;
                st->status = EVOCG_OK;
            } else if (st->k >= st->maxit) {
                st->done = 1;
                st->status = EVOCG_ENOTCONV;
            }
            if (L.use_cond) cudaGraphSetConditional(L.cond, st->done ? 0u : 1u);
        }
    }
}

// sigma = p.q from the SpMV's partials (one per warp or per block, summed in order, identically
// in every block), alpha = rho / sigma; then r -= alpha q; z = D^-1 r; r.z and ||r||^2 (x +=
// alpha p is left to the p-update, which reads p anyway). The last block appends the history
// entry, tests convergence and forms beta. A sigma that is not finite and positive stops the
// solve with EVOCG_EBREAKDOWN.
__global__ void __launch_bounds__(kVecThreads, kUpdMinBlocks) cg_update_kernel(CgLaunch L, int npq)
{
    DevState *st = L.st;
    const int64_t n = L.n, nfull = n / 2;   // whole pairs; an odd last entry separately
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool jac = L.jacobi != 0;
    // Every thread takes two pairs per pass (pair and pair + stride) and holds the next
    // pass's q, r, dinv in registers while it does this pass's arithmetic, so that the loads
    // stay in flight under the FP64 instructions (4 per entry with Jacobi, which on this part
    // take about as long as streaming the entries). The first pass's loads go out before
    // sigma is known: they do not depend on it.
    double2 q[2], r[2], d[2];
    auto ld2 = [](const double *a, int64_t j) { return *reinterpret_cast<const double2 *>(a + j); };
    auto load = [&](int64_t pr) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t ph = pr + h * stride;
            q[h] = r[h] = d[h] = make_double2(0.0, 0.0);
            if (ph < nfull) {
                q[h] = ld2(L.q, 2 * ph);
                r[h] = ld2(L.r, 2 * ph);
                if (jac) d[h] = ld2(L.dinv, 2 * ph);
            }
        }
    };
    int64_t pair = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    load(pair);
    if (st->done) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            st->xstep = 0;
            if (L.use_cond) cudaGraphSetConditional(L.cond, 0u);
        }
        return;
    }
    __shared__ double s_alpha;
    {
        double v = 0.0;
        for (int i = threadIdx.x; i < npq; i += blockDim.x) v += __ldcg(L.pq + i);
        double sigma, unused;
        tree_sum2(v, 0.0, sigma, unused);
        if (threadIdx.x == 0) {
            const bool ok = (sigma > 0.0) && isfinite(sigma);
            s_alpha = ok ? st->rho / sigma : 0.0;
            if (blockIdx.x == 0) {
                st->sigma = sigma;
                st->xstep = ok ? 1 : 0;
                if (ok) {
                    st->alpha = s_alpha;
                } else {
                    st->status = EVOCG_EBREAKDOWN;
                    st->done = 1;
                    if (L.use_cond) cudaGraphSetConditional(L.cond, 0u);
                }
            }
            if (!ok) s_alpha = __longlong_as_double(0x7FF8000000000000ll);   // NaN marks the stop
        }
        __syncthreads();
    }
    const double alpha = s_alpha;
    if (isnan(alpha)) return;   // every block saw the same sigma
    // two sets of dot-product partials, so that the FP64 pipe does not wait on one chain
    double rzs[2] = {0.0, 0.0}, rrs[2] = {0.0, 0.0};
    for (; pair < nfull; pair += 2 * stride) {
        double2 cq[2], cr[2], cd[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) { cq[h] = q[h]; cr[h] = r[h]; cd[h] = d[h]; }
        load(pair + 2 * stride);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t ph = pair + h * stride;
            if (ph >= nfull) break;
            double2 rv = cr[h];
            rv.x = fma(-alpha, cq[h].x, rv.x);
            rv.y = fma(-alpha, cq[h].y, rv.y);
            *reinterpret_cast<double2 *>(L.r + 2 * ph) = rv;
            rrs[h] = fma(rv.x, rv.x, rrs[h]);
            rrs[h] = fma(rv.y, rv.y, rrs[h]);
            if (jac) {
                double2 z;
                z.x = cd[h].x * rv.x;
                z.y = cd[h].y * rv.y;
                *reinterpret_cast<double2 *>(L.z + 2 * ph) = z;
                rzs[h] = fma(rv.x, z.x, rzs[h]);
                rzs[h] = fma(rv.y, z.y, rzs[h]);
            }
        }
    }
    if ((n & 1) && blockIdx.x == 0 && threadIdx.x == 0) {   // odd last entry
        const int64_t j = n - 1;
        const double rv = fma(-alpha, L.q[j], L.r[j]);
        L.r[j] = rv;
        rrs[1] = fma(rv, rv, rrs[1]);
        if (jac) {
            const double z = L.dinv[j] * rv;
            L.z[j] = z;
            rzs[1] = fma(rv, z, rzs[1]);
        }
    }
    double s_rz, s_rr;
    tree_sum2(rzs[0] + rzs[1], rrs[0] + rrs[1], s_rz, s_rr);
    if (threadIdx.x == 0) {
        L.partials[blockIdx.x] = s_rz;
        L.partials[kMaxBlocks + blockIdx.x] = s_rr;
    }
    if (last_block_cg(st, TK_UPDATE)) {
        double a = 0.0, b = 0.0;   // as sum_partials, both at once
        for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) {
            a += __ldcg(L.partials + i);
            b += __ldcg(L.partials + kMaxBlocks + i);
        }
        double RZ, RR;
        tree_sum2(a, b, RZ, RR);
        if (threadIdx.x == 0) {
            st->tickets[TK_UPDATE] = 0;
            const int k = st->k + 1;
            st->k = k;
            st->rr = RR;
            const double h = sqrt(RR) / st->nr0;
            L.hist[k] = h;
            if (h <= st->rtol) {
                st->done = 1;
                st->converged = 1;
                st->status = EVOCG_OK;
            } else if (k >= st->maxit) {
                st->done = 1;
                st->status = EVOCG_ENOTCONV;
            } else {
                const double rho_new = L.jacobi ? RZ : RR;
                st->beta = rho_new / st->rho;
                st->rho = rho_new;
            }
            if (L.use_cond) cudaGraphSetConditional(L.cond, st->done ? 0u : 1u);
        }
    }
}

// x += alpha p with the p of this iteration (when the update formed a valid alpha), then
// p = z + beta p, its rounded copies and the threshold rule when it is due; after the last
// iteration only the x step.
template <int T>
__global__ void __launch_bounds__(kVecThreads, kUpdMinBlocks) cg_pupdate_kernel(CgLaunch L)
{
    DevState *st = L.st;
    const int64_t n = L.n, npairs = (n + 1) / 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    const double *zsrc = L.jacobi ? L.z : L.r;
    // One pair per lane and pass; the next pass's p, x, z are loaded before this pass's
    // arithmetic, and the first pass's before the solve state is read (none depends on it).
    double2 p, x, z;
    auto load = [&](int64_t base) {
        const int64_t j = 2 * (base + lane);
        p = x = z = make_double2(0.0, 0.0);
        if (j + 1 < n) {
            p = *reinterpret_cast<const double2 *>(L.p + j);
            x = *reinterpret_cast<const double2 *>(L.x + j);
            z = *reinterpret_cast<const double2 *>(zsrc + j);
        }
    };
    int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
    load(base);
    const bool xs = st->xstep != 0, pdue = !st->done;
    if (!xs && !pdue) return;
    const double alpha = st->alpha, beta = st->beta;
    const bool thr = pdue && (L.ctrl == EVOCG_CTRL_THRESHOLD) && (st->k % st->kstar == 0);
    const uint64_t lo_bits = (uint64_t)__double_as_longlong(st->eps_lo);
    const uint64_t hi_bits = (uint64_t)__double_as_longlong(st->eps_hi);
    const int64_t ncb = (n + T - 1) / T;
    for (; base < npairs; base += stride) {
        double2 cp = p, cx = x;
        const double2 cz = z;
        load(base + stride);
        const int64_t pair = base + lane;
        uint64_t m = 0;
        if (pair < npairs) {
            const int64_t j = 2 * pair;
            if (j + 1 < n) {
                if (xs) {
                    cx.x = fma(alpha, cp.x, cx.x);
                    cx.y = fma(alpha, cp.y, cx.y);
                    *reinterpret_cast<double2 *>(L.x + j) = cx;
                }
                if (pdue) {
                    cp.x = fma(beta, cp.x, cz.x);
                    cp.y = fma(beta, cp.y, cz.y);
                    *reinterpret_cast<double2 *>(L.p + j) = cp;
                    write_copies2(L, j, cp.x, cp.y);
                    if (thr) {
                        const uint64_t a0 = abs_bits(cp.x), a1 = abs_bits(cp.y);
                        m = a0 > a1 ? a0 : a1;
                    }
                }
            } else {   // odd last entry
                double pv = L.p[j];
                if (xs) L.x[j] = fma(alpha, pv, L.x[j]);
                if (pdue) {
                    pv = fma(beta, pv, zsrc[j]);
                    L.p[j] = pv;
                    write_copies(L, j, pv);
                    m = abs_bits(pv);
                }
            }
        }
        if (thr) threshold_segments<T>(m, pair, ncb, lo_bits, hi_bits, L.cbPrec);
    }
    if (thr && blockIdx.x == 0 && threadIdx.x == 0) st->ctrl_calls += 1;
}

// FP64 true residual ||b - q||^2 and ||b||^2 with q = A x from an all-FP64 SpMV.
__global__ void __launch_bounds__(kVecThreads) true_residual_kernel(CgLaunch L)
{
    DevState *st = L.st;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    double num = 0.0, den = 0.0;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < L.n; j += stride) {
        const double b = L.b[j];
        const double d = b - L.q[j];
        num = fma(d, d, num);
        den = fma(b, b, den);
    }
    const double s_n = block_sum_cg(num);
    const double s_d = block_sum_cg(den);
    if (threadIdx.x == 0) {
        L.partials[blockIdx.x] = s_n;
        L.partials[kMaxBlocks + blockIdx.x] = s_d;
    }
    if (last_block_cg(st, TK_TRUE)) {
        const double N = sum_partials(L.partials);
        const double D = sum_partials(L.partials + kMaxBlocks);
        if (threadIdx.x == 0) {
            st->tickets[TK_TRUE] = 0;
            st->tr_num = N;
            st->tr_den = D;
        }
    }
}

template <int T>
static cudaError_t init_T(const CgLaunch &L, int restart, cudaStream_t s)
{
    cg_init_kernel<T><<<L.vec_grid, kVecThreads, 0, s>>>(L, restart);
    return cudaGetLastError();
}

cudaError_t launch_cg_init(const CgLaunch &L, int restart, cudaStream_t s)
{
    switch (L.T) {
    case 16: return init_T<16>(L, restart, s);
    case 32: return init_T<32>(L, restart, s);
    case 64: return init_T<64>(L, restart, s);
    default: return cudaErrorInvalidValue;
    }
}

// Row k of the decision log = the column-block map the SpMV of iteration k reads (k = the
// iterations done so far); nothing once the solve has stopped or past the log's rows.
__global__ void __launch_bounds__(kVecThreads)
    log_map_kernel(const uint8_t *__restrict__ cbPrec, uint8_t *__restrict__ log, int64_t ncb,
                   int64_t rows, const DevState *st)
{
    if (st->done) return;
    const int64_t k = st->k;
    if (k < 0 || k >= rows) return;
    uint8_t *row = log + k * ncb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ncb;
         i += (int64_t)gridDim.x * blockDim.x)
        row[i] = cbPrec[i];
}

// One loop body: [MLP controller] -> [decision log] -> SpMV (+ p.q, alpha) -> update -> p-update.
cudaError_t launch_cg_body(const CgLaunch &L, int force64, cudaStream_t s)
{
    cudaError_t e;
    if (!force64 && L.ctrl == EVOCG_CTRL_MLP) {
        e = launch_ctrl_mlp(L.A, L.p, L.mlpW, L.H1, L.H2, L.delta, L.cbPrec, nullptr, L.st, s);
        if (e != cudaSuccess) return e;
    }
    if (!force64 && L.ctrl != EVOCG_CTRL_STATIC && L.map_log) {
        const int64_t ncb = L.A.nrb;
        int64_t g = (ncb + kVecThreads - 1) / kVecThreads;
        if (g > 1024) g = 1024;
        log_map_kernel<<<(int)g, kVecThreads, 0, s>>>(L.cbPrec, L.map_log, ncb, L.map_log_rows, L.st);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    SpmvLaunch S{};
    S.A = L.A;
    S.x64 = L.p;
    S.x32 = L.x32;
    S.x16f = L.x16f;
    S.y = L.q;
    S.prec = (L.ctrl == EVOCG_CTRL_STATIC) ? L.prec : L.cbPrec;
    S.map_kind = (L.ctrl == EVOCG_CTRL_STATIC) ? L.map_kind : EVOCG_MAP_PER_COLBLOCK;
    S.force64 = force64;
    S.dot = 1;             // p.q partials (per warp or per block), summed by the update kernel
    S.pq = L.pq;
    S.gate = 1;
    S.partials = L.partials;
    S.st = L.st;
    S.census = 1;
    S.grid = L.spmv_grid;
    const int npq = spmv_dot_partials(S);
    if (npq > kMaxPq) return cudaErrorInvalidConfiguration;
    e = launch_spmv(S, s);
    if (e != cudaSuccess) return e;
    cg_update_kernel<<<L.upd_grid, kVecThreads, 0, s>>>(L, npq);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (L.T) {
    case 16: cg_pupdate_kernel<16><<<L.upd_grid, kVecThreads, 0, s>>>(L); break;
    case 32: cg_pupdate_kernel<32><<<L.upd_grid, kVecThreads, 0, s>>>(L); break;
    default: cg_pupdate_kernel<64><<<L.upd_grid, kVecThreads, 0, s>>>(L); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_true_residual(const CgLaunch &L, cudaStream_t s)
{
    SpmvLaunch S{};
    S.A = L.A;
    S.x64 = L.x;
    S.y = L.q;
    S.force64 = 1;
    S.dot = 0;
    S.st = L.st;
    S.census = 0;
    S.grid = L.spmv_grid;
    cudaError_t e = launch_spmv(S, s);
    if (e != cudaSuccess) return e;
    true_residual_kernel<<<L.vec_grid, kVecThreads, 0, s>>>(L);
    return cudaGetLastError();
}

}  // namespace evocg
