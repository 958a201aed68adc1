// fw_noalloc.cu -- fw_delta_forward_noalloc: the forward for callers that
// cannot allocate device memory when they call it.
//
// The bf16 forward needs a workspace (the per-chunk operand images the prep
// kernel hands to the scan kernel).  fw_delta_forward takes it from the
// caller; this entry point instead uses a fixed array in the library's own
// device memory, FW_NOALLOC_SCRATCH_BYTES long, and then runs exactly the same
// checks and kernels as fw_delta_forward.  It never calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The array is a file-scope __device__ variable: in host code its name is
// only a stand-in, so its device address is looked up with
// cudaGetSymbolAddress with the device current.  The address belongs to the
// context that loaded the library's device code, so it is cached per
// (device, context) pair: a new context on the device (after
// cudaDeviceReset, or a context the caller made current through the driver
// API) is looked up afresh instead of reusing an address from a context that
// no longer exists.
#include "fastweight.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

static __device__ __align__(256) unsigned char g_fw_noalloc_scratch[FW_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];
CUcontext g_scratch_ctx[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The driver's cuCtxGetCurrent, reached through the runtime (the library
// does not link the driver library itself).
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// Device address of the scratch array in the current context.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get)
        return cudaErrorDeviceUninitialized;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        // (with no context current yet, the lookup itself sets up the
        // device's primary context, which is then the one recorded)
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fw_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx))
            return cudaErrorDeviceUninitialized;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" FW_API int fw_delta_forward_noalloc(const void *q, const void *k, const void *v,
                                               const void *beta, const float *W0, float *W_final,
                                               void *y, int B, int H, int L, int d_key, int nu,
                                               int d_v, int chunk, int io_dtype, float eps,
                                               void *stream) {
    // Same shape rules as fw_delta_forward; a shape it rejects reports 0 here
    // and is rejected again, with its own code, by the call below.
    const size_t need = fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, io_dtype);
    if (need > FW_NOALLOC_SCRATCH_BYTES)
        return FW_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need > 0 && (int64_t)B * H > 0 && L > 0 && scratch_address(&scratch) != cudaSuccess)
        return FW_ERR_CUDA;
    return fw_delta_forward(q, k, v, beta, W0, W_final, y, scratch, need, B, H, L, d_key, nu, d_v,
                            chunk, io_dtype, eps, stream);
}
