// fw_api.cu -- the C ABI (include/fastweight.h): argument checks on the host,
// then dispatch to the sm_103a kernels.  Nothing is enqueued unless every
// check passes; the library never allocates device memory.
#include "fastweight.h"
#include "fw_common.cuh"
#include "fw_forward_tc.h"
#include "fw_stack.h"

#include <climits>
#include <cmath>
#include <mutex>

namespace fw {
cudaError_t launch_rowscan(const void *q, const void *k, const void *v, const void *beta,
                           const float *W0, float *Wout, void *y, int BH, int L, int d_key, int nu,
                           int d_v, int bf16, float eps, cudaStream_t st);
} // namespace fw

// Device-side status word (bit fw::kStatusTimeout: a bounded wait gave up).
static __device__ unsigned g_fw_device_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

struct DeviceInfo {
    int num_sms;
    unsigned *status;
};

// Per-device facts, looked up once per device with that device current.
cudaError_t device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fw_device_status);
        if (e != cudaSuccess)
            return e;
        g_num_sms[dev] = sms;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    out->num_sms = g_num_sms[dev];
    out->status = g_status_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(int d) { return d == FW_DTYPE_F32 || d == FW_DTYPE_BF16; }
// Longest sequence: chunk counts are formed as (L + chunk - 1) / chunk in int.
constexpr int kMaxL = INT_MAX - 64;

bool dkey_supported(int d_key) {
    return d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128;
}
bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.f; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FW_OK : FW_ERR_CUDA; }

} // namespace

namespace fw {
// Address of the current device's status word (for the self-test entry points).
cudaError_t status_word(unsigned **out) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e == cudaSuccess)
        *out = di.status;
    return e;
}
} // namespace fw

extern "C" {

FW_API const char *fw_status_string(int status) {
    switch (status) {
    case FW_OK: return "FW_OK";
    case FW_ERR_INVALID_ARG: return "FW_ERR_INVALID_ARG: invalid argument";
    case FW_ERR_UNSUPPORTED: return "FW_ERR_UNSUPPORTED: shape or dtype outside the compiled set";
    case FW_ERR_CUDA: return "FW_ERR_CUDA: a CUDA call failed";
    case FW_ERR_TIMEOUT: return "FW_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "unknown fw_status";
    }
}

FW_API int fw_dpfp(const void *x, void *phi, int64_t rows, int d_key, int nu, int in_dtype,
                   int out_dtype, float eps, void *stream) {
    if (rows < 0 || d_key <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 || !dtype_ok(in_dtype) ||
        !dtype_ok(out_dtype) || !eps_ok(eps))
        return FW_ERR_INVALID_ARG;
    if (!dkey_supported(d_key))
        return FW_ERR_UNSUPPORTED;
    if (rows == 0)
        return FW_OK; // empty: the pointers are not used and may be NULL
    if (!x || !phi || !aligned16(x) || !aligned16(phi))
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return FW_ERR_CUDA;
    e = fw::launch_dpfp(x, phi, rows, d_key, nu, in_dtype == FW_DTYPE_BF16, out_dtype == FW_DTYPE_BF16,
                        eps, di.num_sms, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

namespace {

// Shape checks shared by the forward and its workspace query.
// Returns FW_OK, FW_ERR_INVALID_ARG or FW_ERR_UNSUPPORTED.
int check_forward_shape(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int io_dtype) {
    if (B < 0 || H < 0 || L < 0 || d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 ||
        !dtype_ok(io_dtype) || !(chunk == 16 || chunk == 32 || chunk == 64))
        return FW_ERR_INVALID_ARG;
    if (L > kMaxL)
        return FW_ERR_UNSUPPORTED;
    if (!dkey_supported(d_key))
        return FW_ERR_UNSUPPORTED;
    const int d_dot = 2 * d_key * nu;
    if (io_dtype == FW_DTYPE_F32)
        return d_dot <= 1024 ? FW_OK : FW_ERR_UNSUPPORTED;
    return fw::tc_forward_supported(d_key, nu, d_v, chunk) ? FW_OK : FW_ERR_UNSUPPORTED;
}

} // namespace

FW_API size_t fw_delta_forward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v,
                                              int chunk, int io_dtype) {
    if (check_forward_shape(B, H, L, d_key, nu, d_v, chunk, io_dtype) != FW_OK)
        return 0;
    if (io_dtype == FW_DTYPE_F32)
        return 0;
    return fw::tc_forward_workspace_bytes(B, H, L, d_key, nu, d_v, chunk);
}

FW_API int fw_delta_forward_kernel_count(int B, int H, int L, int d_key, int nu, int d_v, int chunk,
                                         int io_dtype) {
    if (check_forward_shape(B, H, L, d_key, nu, d_v, chunk, io_dtype) != FW_OK)
        return -1;
    if ((int64_t)B * H == 0 || L == 0)
        return 0;
    if (io_dtype == FW_DTYPE_F32)
        return 1;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return -1;
    return fw::tc_forward_kernel_count(B, H, L, d_key, nu, d_v, chunk, di.num_sms);
}

FW_API int fw_delta_forward(const void *q, const void *k, const void *v, const void *beta,
                            const float *W0, float *W_final, void *y, void *workspace,
                            size_t workspace_bytes, int B, int H, int L, int d_key, int nu,
                            int d_v, int chunk, int io_dtype, float eps, void *stream) {
    if (!eps_ok(eps))
        return FW_ERR_INVALID_ARG;
    const int rc = check_forward_shape(B, H, L, d_key, nu, d_v, chunk, io_dtype);
    if (rc != FW_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t BH = (int64_t)B * H;
    if (BH == 0)
        return FW_OK; // empty: no pointer is used and any may be NULL
    if ((W0 && !aligned16(W0)) || (W_final && !aligned16(W_final)))
        return FW_ERR_INVALID_ARG;
    if (L > 0) {
        if (!q || !k || !v || !beta || !y)
            return FW_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) || !aligned16(y) ||
            (workspace && !aligned16(workspace)))
            return FW_ERR_INVALID_ARG;
        const size_t need = fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, io_dtype);
        if (need > 0 && (!workspace || workspace_bytes < need))
            return FW_ERR_INVALID_ARG;
    }
    if (BH > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    const int d_dot = 2 * d_key * nu;
    if (L == 0) {
        // no token: the final state is the initial one
        if (!W_final)
            return FW_OK;
        const size_t bytes = sizeof(float) * (size_t)BH * d_v * d_dot;
        if (W0 == W_final)
            return FW_OK;
        cudaError_t e = W0 ? cudaMemcpyAsync(W_final, W0, bytes, cudaMemcpyDeviceToDevice, st)
                           : cudaMemsetAsync(W_final, 0, bytes, st);
        return cuda_status(e);
    }
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return FW_ERR_CUDA;
    if (io_dtype == FW_DTYPE_F32) {
        e = fw::launch_rowscan(q, k, v, beta, W0, W_final, y, (int)BH, L, d_key, nu, d_v, 0, eps, st);
        return cuda_status(e);
    }
    e = fw::tc_forward_launch(q, k, v, beta, W0, W_final, y, workspace, B, H, L, d_key, nu, d_v,
                              chunk, eps, di.num_sms, di.status, st);
    return cuda_status(e);
}

namespace {

// The projected q, k, v, beta inside the workspace, each 256-byte aligned,
// then the forward's own workspace.
struct ProjLayout {
    size_t q, k, v, beta, fwd, bytes;
};
ProjLayout proj_layout(int B, int L, int H, int d_key, int d_v, size_t fwd_bytes) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t tok = (size_t)B * H * L;
    ProjLayout p;
    p.q = 0;
    p.k = up(p.q + tok * d_key * 2);
    p.v = up(p.k + tok * d_key * 2);
    p.beta = up(p.v + tok * d_v * 2);
    p.fwd = up(p.beta + tok * 2);
    p.bytes = p.fwd + fwd_bytes;
    return p;
}

} // namespace

FW_API size_t fw_delta_forward_projected_workspace_size(int B, int L, int d_model, int H, int d_key, int nu,
                                                        int d_v, int chunk) {
    if (d_model <= 0 || d_model % 64 || H <= 0 || check_forward_shape(B, H, L, d_key, nu, d_v, chunk,
                                                                      FW_DTYPE_BF16) != FW_OK)
        return 0;
    return proj_layout(B, L, H, d_key, d_v, fw::tc_forward_workspace_bytes(B, H, L, d_key, nu, d_v, chunk))
        .bytes;
}

FW_API int fw_delta_forward_projected(const void *x, const void *W_all, int ldw, const float *W0, float *W_final,
                                      void *y, void *workspace, size_t workspace_bytes, int B, int L, int d_model,
                                      int H, int d_key, int nu, int d_v, int chunk, float eps, void *stream) {
    if (!eps_ok(eps) || d_model <= 0 || d_model % 64 || H <= 0)
        return FW_ERR_INVALID_ARG;
    const int rc = check_forward_shape(B, H, L, d_key, nu, d_v, chunk, FW_DTYPE_BF16);
    if (rc != FW_OK)
        return rc;
    const int64_t N = (int64_t)H * (2 * d_key + d_v + 1);
    if (ldw % 8 || ldw < (N + 7) / 8 * 8)
        return FW_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t BH = (int64_t)B * H;
    if (BH == 0)
        return FW_OK;
    if ((W0 && !aligned16(W0)) || (W_final && !aligned16(W_final)))
        return FW_ERR_INVALID_ARG;
    if (BH > (int64_t)1 << 30 || (int64_t)B * L > (int64_t)1 << 30 || N > 65535 * 128)
        return FW_ERR_UNSUPPORTED;
    const int d_dot = 2 * d_key * nu;
    if (L == 0) {
        if (!W_final || W0 == W_final)
            return FW_OK;
        const size_t bytes = sizeof(float) * (size_t)BH * d_v * d_dot;
        return cuda_status(W0 ? cudaMemcpyAsync(W_final, W0, bytes, cudaMemcpyDeviceToDevice, st)
                              : cudaMemsetAsync(W_final, 0, bytes, st));
    }
    if (!x || !W_all || !y || !aligned16(x) || !aligned16(W_all) || !aligned16(y))
        return FW_ERR_INVALID_ARG;
    const ProjLayout pl =
        proj_layout(B, L, H, d_key, d_v, fw::tc_forward_workspace_bytes(B, H, L, d_key, nu, d_v, chunk));
    if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes)
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return FW_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // Where the forward runs as its two kernels, the projections are folded
    // into the first (q, k, v and beta never reach global memory): two
    // launches from x.  Otherwise the projection GEMM, then the forward.
    if (fw::tc_prepare_x_supported(d_key, d_v) &&
        fw::tc_forward_kernel_count(B, H, L, d_key, nu, d_v, chunk, di.num_sms) == 2) {
        e = fw::tc_prepare_x_launch(x, W_all, ldw, ws + pl.fwd, B, H, L, d_model, d_key, nu, d_v, chunk, eps,
                                    di.num_sms, di.status, st);
        if (e != cudaSuccess)
            return cuda_status(e);
        return cuda_status(fw::tc_scan_launch(ws + pl.fwd, W0, W_final, y, B, H, L, d_key, nu, d_v, chunk,
                                              di.num_sms, di.status, st));
    }
    e = fw::launch_project(x, W_all, ldw, ws + pl.q, ws + pl.k, ws + pl.v, ws + pl.beta, B, L, H, d_key, d_v, d_model,
                           false, di.status, st);
    if (e != cudaSuccess)
        return cuda_status(e);
    e = fw::tc_forward_launch(ws + pl.q, ws + pl.k, ws + pl.v, ws + pl.beta, W0, W_final, y, ws + pl.fwd, B, H, L,
                              d_key, nu, d_v, chunk, eps, di.num_sms, di.status, st);
    return cuda_status(e);
}

namespace {

int check_backward_shape(int B, int H, int L, int d_key, int nu, int d_v, int io_dtype) {
    if (B < 0 || H < 0 || L < 0 || d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 ||
        !dtype_ok(io_dtype))
        return FW_ERR_INVALID_ARG;
    if (L > kMaxL)
        return FW_ERR_UNSUPPORTED;
    if (!dkey_supported(d_key) || 2 * d_key * nu > 1024 || fw::backward_smem_bytes(d_key, nu, d_v) > (size_t)227 * 1024)
        return FW_ERR_UNSUPPORTED;
    return FW_OK;
}

} // namespace

FW_API size_t fw_delta_backward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v, int io_dtype) {
    if (check_backward_shape(B, H, L, d_key, nu, d_v, io_dtype) != FW_OK)
        return 0;
    const int64_t BH = (int64_t)B * H;
    if (BH > (int64_t)1 << 30) // fw_delta_backward rejects it too
        return 0;
    return fw::backward_workspace_bytes((int)BH, L, d_key, nu, d_v);
}

FW_API int fw_delta_backward(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                             const void *dy, const float *dW_final, void *dq, void *dk, void *dv, void *dbeta,
                             float *dW0, void *workspace, size_t workspace_bytes, int B, int H, int L, int d_key,
                             int nu, int d_v, int io_dtype, float eps, void *stream) {
    if (!eps_ok(eps))
        return FW_ERR_INVALID_ARG;
    const int rc = check_backward_shape(B, H, L, d_key, nu, d_v, io_dtype);
    if (rc != FW_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t BH = (int64_t)B * H;
    if (BH == 0)
        return FW_OK;
    if ((W0 && !aligned16(W0)) || (dW_final && !aligned16(dW_final)) || (dW0 && !aligned16(dW0)))
        return FW_ERR_INVALID_ARG;
    if (BH > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    const int d_dot = 2 * d_key * nu;
    if (L == 0) { // no token: dL/dW0 = dL/dW_final
        if (!dW0 || dW0 == dW_final)
            return FW_OK;
        const size_t bytes = sizeof(float) * (size_t)BH * d_v * d_dot;
        return cuda_status(dW_final ? cudaMemcpyAsync(dW0, dW_final, bytes, cudaMemcpyDeviceToDevice, st)
                                    : cudaMemsetAsync(dW0, 0, bytes, st));
    }
    const void *in[] = {q, k, v, beta, dy, dq, dk, dv, dbeta};
    for (const void *p : in)
        if (!p || !aligned16(p))
            return FW_ERR_INVALID_ARG;
    const size_t need = fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, io_dtype);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return FW_ERR_CUDA;
    return cuda_status(fw::launch_backward(q, k, v, beta, W0, dy, dW_final, dq, dk, dv, dbeta, dW0,
                                           static_cast<float *>(workspace), (int)BH, L, d_key, nu, d_v,
                                           io_dtype == FW_DTYPE_BF16, eps, di.num_sms, st));
}

namespace {

int check_linear_shape(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int normalize, int io_dtype) {
    if (B < 0 || H < 0 || L < 0 || d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 ||
        !dtype_ok(io_dtype) || !(chunk == 16 || chunk == 32 || chunk == 64) || (normalize != 0 && normalize != 1))
        return FW_ERR_INVALID_ARG;
    if (L > kMaxL)
        return FW_ERR_UNSUPPORTED;
    if (!dkey_supported(d_key) || io_dtype != FW_DTYPE_BF16)
        return FW_ERR_UNSUPPORTED;
    return fw::tc_linear_supported(d_key, nu, d_v, chunk, normalize) ? FW_OK : FW_ERR_UNSUPPORTED;
}

} // namespace

FW_API size_t fw_linear_forward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v, int chunk,
                                               int normalize, int io_dtype) {
    if (check_linear_shape(B, H, L, d_key, nu, d_v, chunk, normalize, io_dtype) != FW_OK)
        return 0;
    return fw::tc_linear_workspace_bytes(B, H, L, d_key, nu, d_v, chunk, normalize);
}

FW_API int fw_linear_forward(const void *q, const void *k, const void *v, const float *W0, const float *z0,
                             float *W_final, float *z_final, void *y, void *workspace, size_t workspace_bytes,
                             int B, int H, int L, int d_key, int nu, int d_v, int chunk, int normalize,
                             int io_dtype, float eps, void *stream) {
    if (!eps_ok(eps))
        return FW_ERR_INVALID_ARG;
    const int rc = check_linear_shape(B, H, L, d_key, nu, d_v, chunk, normalize, io_dtype);
    if (rc != FW_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t BH = (int64_t)B * H;
    if (BH == 0)
        return FW_OK; // empty: no pointer is used and any may be NULL
    if ((W0 && !aligned16(W0)) || (W_final && !aligned16(W_final)) || (z0 && !aligned16(z0)) ||
        (z_final && !aligned16(z_final)))
        return FW_ERR_INVALID_ARG;
    if (L > 0) {
        if (!q || !k || !v || !y || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y))
            return FW_ERR_INVALID_ARG;
        const size_t need = fw_linear_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, normalize, io_dtype);
        if (!workspace || !aligned16(workspace) || workspace_bytes < need)
            return FW_ERR_INVALID_ARG;
    }
    if (BH > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    const int d_dot = 2 * d_key * nu;
    if (L == 0) {
        // no token: the final state is the initial one
        cudaError_t e = cudaSuccess;
        if (W_final && W_final != W0) {
            const size_t bytes = sizeof(float) * (size_t)BH * d_v * d_dot;
            e = W0 ? cudaMemcpyAsync(W_final, W0, bytes, cudaMemcpyDeviceToDevice, st)
                   : cudaMemsetAsync(W_final, 0, bytes, st);
        }
        if (e == cudaSuccess && normalize && z_final && z_final != z0) {
            const size_t bytes = sizeof(float) * (size_t)BH * d_dot;
            e = z0 ? cudaMemcpyAsync(z_final, z0, bytes, cudaMemcpyDeviceToDevice, st)
                   : cudaMemsetAsync(z_final, 0, bytes, st);
        }
        return cuda_status(e);
    }
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return FW_ERR_CUDA;
    e = fw::tc_linear_launch(q, k, v, W0, normalize ? z0 : nullptr, W_final, normalize ? z_final : nullptr, y,
                             workspace, B, H, L, d_key, nu, d_v, chunk, normalize, eps, di.num_sms, di.status, st);
    return cuda_status(e);
}

namespace {

// Checks shared by the two phases of the bf16 forward.  Returns FW_OK with
// *empty set when nothing has to be enqueued.
int check_phase(int B, int H, int L, int d_key, int nu, int d_v, int chunk, const void *workspace,
                size_t workspace_bytes, bool *empty) {
    const int rc = check_forward_shape(B, H, L, d_key, nu, d_v, chunk, FW_DTYPE_BF16);
    if (rc != FW_OK)
        return rc;
    *empty = (int64_t)B * H == 0 || L == 0;
    if (*empty)
        return FW_OK;
    if ((int64_t)B * H > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    const size_t need = fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, FW_DTYPE_BF16);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return FW_ERR_INVALID_ARG;
    return FW_OK;
}

} // namespace

FW_API int fw_delta_forward_prepare(const void *q, const void *k, const void *v, const void *beta,
                                    void *workspace, size_t workspace_bytes, int B, int H, int L,
                                    int d_key, int nu, int d_v, int chunk, float eps, void *stream) {
    if (!eps_ok(eps))
        return FW_ERR_INVALID_ARG;
    bool empty = false;
    const int rc = check_phase(B, H, L, d_key, nu, d_v, chunk, workspace, workspace_bytes, &empty);
    if (rc != FW_OK || empty)
        return rc;
    if (!q || !k || !v || !beta || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta))
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return FW_ERR_CUDA;
    return cuda_status(fw::tc_prepare_launch(q, k, v, beta, workspace, B, H, L, d_key, nu, d_v, chunk, eps,
                                             di.num_sms, di.status, static_cast<cudaStream_t>(stream)));
}

FW_API int fw_delta_forward_scan(const void *workspace, size_t workspace_bytes, const float *W0,
                                 float *W_final, void *y, int B, int H, int L, int d_key, int nu, int d_v,
                                 int chunk, void *stream) {
    bool empty = false;
    const int rc = check_phase(B, H, L, d_key, nu, d_v, chunk, workspace, workspace_bytes, &empty);
    if (rc != FW_OK)
        return rc;
    if ((W0 && !aligned16(W0)) || (W_final && !aligned16(W_final)))
        return FW_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (empty) {
        // no token: the final state is the initial one
        if ((int64_t)B * H == 0 || !W_final || W0 == W_final)
            return FW_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * d_v * (2 * d_key * nu);
        return cuda_status(W0 ? cudaMemcpyAsync(W_final, W0, bytes, cudaMemcpyDeviceToDevice, st)
                              : cudaMemsetAsync(W_final, 0, bytes, st));
    }
    if (!y || !aligned16(y))
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return FW_ERR_CUDA;
    return cuda_status(fw::tc_scan_launch(workspace, W0, W_final, y, B, H, L, d_key, nu, d_v, chunk,
                                          di.num_sms, di.status, st));
}

FW_API int fw_delta_decode_step(const void *q, const void *k, const void *v, const void *beta,
                                float *W, void *y, int B, int H, int d_key, int nu, int d_v,
                                int io_dtype, float eps, void *stream) {
    if (!eps_ok(eps) || B < 0 || H < 0 || d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 ||
        !dtype_ok(io_dtype))
        return FW_ERR_INVALID_ARG;
    if (!dkey_supported(d_key) || 2 * d_key * nu > 1024)
        return FW_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0)
        return FW_OK; // empty: no pointer is used and any may be NULL
    if (!q || !k || !v || !beta || !W || !y)
        return FW_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) || !aligned16(W) ||
        !aligned16(y))
        return FW_ERR_INVALID_ARG;
    if (BH > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return FW_ERR_CUDA;
    e = fw::launch_decode(q, k, v, beta, W, y, (int)BH, d_key, nu, d_v, io_dtype == FW_DTYPE_BF16,
                          eps, di.num_sms, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

namespace {

int check_stack_shape(int n_layers, int B, int H, int d_key, int nu, int d_v, int d_model, int d_ff) {
    if (n_layers < 0 || B < 0 || H <= 0 || d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * (int64_t)d_key - 1 ||
        d_model <= 0 || d_ff <= 0)
        return FW_ERR_INVALID_ARG;
    if (!dkey_supported(d_key) || 2 * d_key * nu > 1024 || d_model % 128 || d_model > 1024 || ((int64_t)H * d_v) % 64 ||
        d_ff % 64 || (int64_t)H * (2 * d_key + d_v + 1) > 65535 * 128 || d_ff > 65535 * 128 ||
        (int64_t)B * H > (int64_t)1 << 30)
        return FW_ERR_UNSUPPORTED;
    return FW_OK;
}

} // namespace

FW_API size_t fw_decode_stack_workspace_size(int B, int H, int d_key, int d_v, int d_model, int d_ff) {
    if (check_stack_shape(0, B, H, d_key, 1, d_v, d_model, d_ff) != FW_OK)
        return 0;
    return fw::stack_layout(B, H, d_key, d_v, d_model, d_ff).bytes;
}

FW_API int fw_decode_stack_step(const fw_stack_layer *layers, int n_layers, const float *x, const float *ln_gamma,
                                const float *ln_beta, float *out, void *workspace, size_t workspace_bytes, int B,
                                int H, int d_key, int nu, int d_v, int d_model, int d_ff, int ldw_in, float eps,
                                float ln_eps, void *stream) {
    if (!eps_ok(eps) || !eps_ok(ln_eps))
        return FW_ERR_INVALID_ARG;
    const int rc = check_stack_shape(n_layers, B, H, d_key, nu, d_v, d_model, d_ff);
    if (rc != FW_OK)
        return rc;
    const int64_t N = (int64_t)H * (2 * d_key + d_v + 1);
    if (n_layers > 0 && (ldw_in % 8 || ldw_in < (N + 7) / 8 * 8))
        return FW_ERR_INVALID_ARG;
    if (B == 0)
        return FW_OK; // no sequence: nothing is read or written
    if (!x || !out || !aligned16(x) || !aligned16(out) || (ln_gamma && !aligned16(ln_gamma)) ||
        (ln_beta && !aligned16(ln_beta)))
        return FW_ERR_INVALID_ARG;
    if (n_layers > 0 && !layers)
        return FW_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const fw_stack_layer &ly = layers[l];
        if (!ly.W_in || !ly.W_o || !ly.W_1 || !ly.W_2 || !ly.W)
            return FW_ERR_INVALID_ARG;
        const void *ptrs[] = {ly.W_in, ly.W_o, ly.b_o, ly.ln_gamma, ly.ln_beta, ly.W_1, ly.b_1, ly.W_2, ly.b_2, ly.W};
        for (const void *p : ptrs)
            if (p && !aligned16(p))
                return FW_ERR_INVALID_ARG;
    }
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < fw::stack_layout(B, H, d_key, d_v, d_model, d_ff).bytes)
        return FW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return FW_ERR_CUDA;
    return cuda_status(fw::stack_step_launch(layers, n_layers, x, ln_gamma, ln_beta, out, workspace, B, H, d_key, nu,
                                             d_v, d_model, d_ff, ldw_in, eps, ln_eps, di.num_sms, di.status,
                                             static_cast<cudaStream_t>(stream)));
}

FW_API int fw_device_status(void *stream) {
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return FW_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FW_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, di.status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FW_ERR_CUDA;
    if (word != 0 && cudaMemset(di.status, 0, sizeof(word)) != cudaSuccess)
        return FW_ERR_CUDA;
    return (word & fw::kStatusTimeout) ? FW_ERR_TIMEOUT : FW_OK;
}

} // extern "C"
