// fw_stack.cu -- one token through a stack of fast-weight Transformer layers,
// each layer's fast weights persisting across tokens (the token-wise model).
//
// Method (Fast Weights Transformer guide: the token_wise variant keeps one
// weight list entry per layer and passes each token through all layers in
// turn, then applies the final LayerNorm; a layer adds the fast-weight
// attention's output to its input, normalises the sum, and adds the
// feed-forward block's output; the attention module projects q, k, v and
// beta (bias-free, beta through the sigmoid), steps its fast weights with
// the delta rule on DPFP features, and maps the heads' concatenated output
// back to the model width with a linear layer; the feed-forward block is
// linear, ReLU, linear):
//   per layer l, for every sequence b of the batch (x_b: the residual stream)
//     q, k, v, beta = proj_l(x_b);  y_b = decode step of W_l with them
//     x_b <- x_b + y_b W_o,l + b_o,l
//     x_b <- x_b + relu(LN_l(x_b) W_1,l + b_1,l) W_2,l + b_2,l
//   out_b = LN_final(x_b)
// Dropout is the identity (inference).
//
// Every step is a kernel of this library: the projections and the three
// dense layers run on the tcgen05 GEMM of fw_project.cu, the state update
// on the decode kernel, the norms on the row kernel below; consecutive
// kernels are chained by programmatic dependent launch, so one token of an
// L-layer stack is 6 L + 2 operations (a split GEMM adds its reduction
// kernel) that a caller can capture as one graph.
// The residual stream is fp32; the activations the tensor cores read (a bf16
// copy of x written beside it, y, LN output, the hidden layer) are bf16.
#include "fw_forward_tc.h"
#include "fw_common.cuh"
#include "fw_stack.h"

#include <algorithm>

namespace fw {

namespace {

constexpr int kLnRows = 8; // rows per 256-thread CTA, one warp each

FW_DEV void ln_store4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
FW_DEV void ln_store4(__nv_bfloat16 *p, float a, float b, float c, float d) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

// One warp per row; lane l holds columns 128 c + 4 l .. + 3 for c < D / 128.
// Mean first, then the mean squared deviation (two passes over registers).
template <class TO>
__global__ void __launch_bounds__(32 * kLnRows)
    layernorm_kernel(const float *__restrict__ x, const float *__restrict__ gamma, const float *__restrict__ beta,
                     TO *__restrict__ out, int M, int D, float eps) {
    griddep_launch_dependents();
    griddep_wait(); // x is the preceding kernel's output
    x = after_wait(x);
    gamma = after_wait(gamma);
    beta = after_wait(beta);
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x * kLnRows + (threadIdx.x >> 5);
    if (m >= M)
        return;
    const int nc = D / 128;
    const float *row = x + (size_t)m * D;
    float4 r[8];
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        if (c < nc) {
            r[c] = __ldcg(reinterpret_cast<const float4 *>(row + 128 * c) + lane);
            s += (r[c].x + r[c].y) + (r[c].z + r[c].w);
        }
    const float mean = warp_sum(s) / (float)D;
    float q = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        if (c < nc) {
            const float a = r[c].x - mean, b = r[c].y - mean, cc = r[c].z - mean, d = r[c].w - mean;
            q += (a * a + b * b) + (cc * cc + d * d);
        }
    const float inv = rsqrtf(warp_sum(q) / (float)D + eps);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        if (c < nc) {
            const int col = 128 * c + 4 * lane;
            float4 g = make_float4(1.f, 1.f, 1.f, 1.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (gamma)
                g = __ldcg(reinterpret_cast<const float4 *>(gamma + col));
            if (beta)
                b = __ldcg(reinterpret_cast<const float4 *>(beta + col));
            ln_store4(out + (size_t)m * D + col, (r[c].x - mean) * inv * g.x + b.x, (r[c].y - mean) * inv * g.y + b.y,
                      (r[c].z - mean) * inv * g.z + b.z, (r[c].w - mean) * inv * g.w + b.w);
        }
}

// The layer stack's input rounded to bf16: the first projection's A.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ y,
                                                      int64_t n8) {
    griddep_launch_dependents();
    griddep_wait(); // x may be the preceding kernel's output
    x = after_wait(x);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        float v[8];
        load8(x + 8 * i, v);
        store8(y + 8 * i, v);
    }
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

} // namespace

cudaError_t launch_layernorm(const float *x, const float *gamma, const float *beta, void *out, bool out_bf16, int M,
                             int D, float eps, cudaStream_t st) {
    const dim3 grid((unsigned)((M + kLnRows - 1) / kLnRows));
    if (out_bf16)
        return launch_pdl(layernorm_kernel<__nv_bfloat16>, grid, dim3(32 * kLnRows), 0, st, x, gamma, beta,
                          static_cast<__nv_bfloat16 *>(out), M, D, eps);
    return launch_pdl(layernorm_kernel<float>, grid, dim3(32 * kLnRows), 0, st, x, gamma, beta,
                      static_cast<float *>(out), M, D, eps);
}

StackLayout stack_layout(int B, int H, int d_key, int d_v, int d_model, int d_ff) {
    const size_t bh = (size_t)B * H;
    StackLayout p;
    p.q = 0;
    p.k = up256(p.q + bh * d_key * 2);
    p.v = up256(p.k + bh * d_key * 2);
    p.beta = up256(p.v + bh * d_v * 2);
    p.y = up256(p.beta + bh * 2);
    p.z = up256(p.y + bh * d_v * 2);
    p.h = up256(p.z + (size_t)B * d_model * 2);
    p.x = up256(p.h + (size_t)B * d_ff * 2);
    p.x16 = up256(p.x + (size_t)B * d_model * 4);
    p.stats = up256(p.x16 + (size_t)B * d_model * 2);
    p.bytes = up256(p.stats + (size_t)B * (d_model / 128 + 1) * 8);
    return p;
}

cudaError_t stack_step_launch(const fw_stack_layer *layers, int n_layers, const float *x, const float *ln_gamma,
                              const float *ln_beta, float *out, void *workspace, int B, int H, int d_key, int nu,
                              int d_v, int d_model, int d_ff, int ldw_in, float eps, float ln_eps, int num_sms,
                              unsigned *status, cudaStream_t st) {
    const StackLayout pl = stack_layout(B, H, d_key, d_v, d_model, d_ff);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *xr = reinterpret_cast<float *>(ws + pl.x);
    void *x16 = ws + pl.x16;
    // each layer's norm folded into its first feed-forward map: the output
    // map leaves the statistics of x's rows, and the feed-forward GEMM forms
    // its A = LN(x) itself (else a LayerNorm kernel between the two)
    const bool ln_fused = d_model % 128 == 0 && dense_ln_supported(B, d_ff, d_model);
    float2 *stats = reinterpret_cast<float2 *>(ws + pl.stats);
    cudaError_t e = cudaSuccess;
    if (n_layers > 0) {
        const int64_t n8 = (int64_t)B * d_model / 8;
        e = launch_pdl(to_bf16_kernel, dim3((unsigned)std::min<int64_t>((n8 + 255) / 256, 4 * num_sms)), dim3(256),
                           0, st, x, static_cast<__nv_bfloat16 *>(x16), n8);
    }
    for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
        const fw_stack_layer &ly = layers[l];
        const float *xin = l == 0 ? x : xr;
        e = launch_project(x16, ly.W_in, ldw_in, ws + pl.q, ws + pl.k, ws + pl.v, ws + pl.beta, B, 1, H, d_key, d_v,
                           d_model, true, status, st);
        if (e == cudaSuccess)
            e = launch_decode(ws + pl.q, ws + pl.k, ws + pl.v, ws + pl.beta, ly.W, ws + pl.y, B * H, d_key, nu, d_v,
                              1, eps, num_sms, st);
        if (e == cudaSuccess) // x <- x + y W_o + b_o
            e = launch_dense(ws + pl.y, ly.W_o, H * d_v, B, d_model, ly.b_o, xin, xr, false, nullptr, true,
                             ln_fused ? stats : nullptr, nullptr, status, st);
        if (e == cudaSuccess && !ln_fused)
            e = launch_layernorm(xr, ly.ln_gamma, ly.ln_beta, ws + pl.z, true, B, d_model, ln_eps, st);
        if (e == cudaSuccess) { // hidden = relu(LN(x) W_1 + b_1)
            const DenseLn ln = {xr, stats, ly.ln_gamma, ly.ln_beta, ln_eps, d_model / 128};
            e = launch_dense(ws + pl.z, ly.W_1, d_model, B, d_ff, ly.b_1, nullptr, ws + pl.h, true, nullptr, true,
                             nullptr, ln_fused ? &ln : nullptr, status, st);
        }
        if (e == cudaSuccess) // x <- x + hidden W_2 + b_2, and its bf16 copy for the next projection
            e = launch_dense(ws + pl.h, ly.W_2, d_ff, B, d_model, ly.b_2, xr, xr, false, x16, true, nullptr, nullptr,
                             status, st);
    }
    if (e == cudaSuccess)
        e = launch_layernorm(n_layers ? xr : x, ln_gamma, ln_beta, out, false, B, d_model, ln_eps, st);
    return e;
}

} // namespace fw
