// fw_stack.h -- host interface of the token-wise layer stack (fw_stack.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "fastweight.h"

namespace fw {

// Byte offsets of the per-token scratch inside the caller's workspace, each
// 256-byte aligned: q, k [B, H, d_key], v, y [B, H, d_v], beta [B, H] (bf16),
// the norm's output z [B, d_model] and the hidden layer h [B, d_ff] (bf16),
// the residual stream x [B, d_model] (fp32) and its bf16 copy x16, and the
// per-row statistics of x for the norm folded into the feed-forward map
// ([B][d_model / 128] float2).
struct StackLayout {
    size_t q, k, v, beta, y, z, h, x, x16, stats, bytes;
};
StackLayout stack_layout(int B, int H, int d_key, int d_v, int d_model, int d_ff);

// Enqueue one token through every layer (arguments validated by the caller).
cudaError_t stack_step_launch(const fw_stack_layer *layers, int n_layers, const float *x, const float *ln_gamma,
                              const float *ln_beta, float *out, void *workspace, int B, int H, int d_key, int nu,
                              int d_v, int d_model, int d_ff, int ldw_in, float eps, float ln_eps, int num_sms,
                              unsigned *status, cudaStream_t st);

} // namespace fw
