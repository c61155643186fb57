// spmv_noalloc.cu -- an SpMV entry point that never allocates memory.
//
// evocg_spmv keeps the FP32 and BF16 roundings of x in buffers the library allocates with
// cudaMalloc. Some programs cannot let a library do that at call time: cudaMalloc may
// synchronise the whole device, it is not allowed while a stream is being captured into
// a graph, and services that own all device memory through their own pool (or that run
// under a fixed memory budget) forbid allocations they did not plan. For those callers
// this file holds the scratch in a fixed array that is part of the loaded module: it is
// reserved once, when the library is loaded on a device, and never grows.
#include <cuda.h>   // CUcontext; the driver call is reached through the runtime's entry point table
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "evocg_internal.h"

namespace {

// Largest x length the allocation-free SpMV accepts.
constexpr int64_t kNoAllocMaxN = 1 << 20;

// Scratch for the rounded copies of x: kNoAllocMaxN FP32 roundings followed by
// kNoAllocMaxN BF16 roundings (held in FP32 containers). 8 MiB; every GPU that loads this
// library holds it until the process exits. Host code must not take this name as a
// device address: it only names the symbol for cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[2 * kNoAllocMaxN];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// The scratch's device address, looked up once per device and context: the module (and with
// it the array) is loaded again in a new context, for instance after cudaDeviceReset, so an
// address is only reused while the context it was looked up in is still the current one.
struct ScratchAddr {
    CUcontext ctx;
    float *ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

int current_context(CUcontext *out)
{
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) {
            cudaGetLastError();
            return evocg::fail(EVOCG_ECUDA, "cuCtxGetCurrent is not available from the CUDA runtime");
        }
        fn = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    *out = nullptr;
    if (fn(out) != CUDA_SUCCESS) return evocg::fail(EVOCG_ECUDA, "cuCtxGetCurrent failed");
    return EVOCG_OK;
}

// Device address of the scratch in the current device's current context, looked up with
// cudaGetSymbolAddress on the first call in that context.
int scratch_for_current_device(float **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return evocg::cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return evocg::fail(EVOCG_EDEVICE, "device index out of range");
    e = cudaSetDevice(dev);   // binds the device's primary context to this thread
    if (e != cudaSuccess) return evocg::cuda_fail(e, "cudaSetDevice");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    CUcontext ctx = nullptr;
    int rc = current_context(&ctx);
    if (rc) return rc;
    if (!g_scratch[dev].ptr || g_scratch[dev].ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return evocg::cuda_fail(e, "cudaGetSymbolAddress (allocation-free SpMV scratch)");
        g_scratch[dev].ptr = static_cast<float *>(p);
        g_scratch[dev].ctx = ctx;
    }
    *out = g_scratch[dev].ptr;
    return EVOCG_OK;
}

}  // namespace

extern "C" int evocg_spmv_noalloc(evocg_tiles_t A, const double *x, double *y, void *stream)
{
    evocg::set_error("");
    if (!A || (A->n > 0 && (!x || !y))) return evocg::fail(EVOCG_EINVAL, "NULL argument");
    if (A->n > kNoAllocMaxN)
        return evocg::fail(EVOCG_EINVAL, "evocg_spmv_noalloc: n = " + std::to_string(A->n) +
                                             " exceeds the fixed scratch of " +
                                             std::to_string(kNoAllocMaxN) + " entries");
    if (A->n == 0) return EVOCG_OK;
    for (const void *p : {static_cast<const void *>(x), static_cast<const void *>(y)}) {
        cudaPointerAttributes at;
        cudaError_t e = cudaPointerGetAttributes(&at, p);
        if (e != cudaSuccess || (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)) {
            cudaGetLastError();
            return evocg::fail(EVOCG_EINVAL, "evocg_spmv_noalloc needs device pointers for x and y");
        }
    }
    float *scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    float *x32 = scratch, *x16f = scratch + kNoAllocMaxN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every entry of the copies below n is rewritten here, so nothing needs clearing
    cudaError_t e = evocg::launch_xcopies(A->view(), x, x32, x16f, A->vec_grid, s);
    if (e != cudaSuccess) return evocg::cuda_fail(e, "launch x copies (allocation-free)");
    evocg::SpmvLaunch S{};
    S.A = A->view();
    S.x64 = x;
    S.x32 = x32;
    S.x16f = x16f;
    S.y = y;
    S.prec = (A->map_kind == EVOCG_MAP_PER_TILE) ? A->tilePrec : A->cbPrec;
    S.map_kind = A->map_kind;
    S.force64 = 0;
    S.dot = 0;
    S.st = nullptr;
    S.census = 0;
    S.grid = A->spmv_grid;
    // only kernels without device waits: a lost wait could not be reported by this call
    S.direct = evocg::spmv_kind_for(A->view(), 0, 0) == evocg::SPMV_KIND_PANEL ? 1 : 0;
    e = evocg::launch_spmv(S, s);
    if (e != cudaSuccess) return evocg::cuda_fail(e, "launch spmv (allocation-free)");
    return EVOCG_OK;
}
