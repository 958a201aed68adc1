// fw_forward_tc.h -- host interface of the bf16 chunked forward (tcgen05).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fw {

cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *beta, float *W,
                          void *y, int BH, int d_key, int nu, int d_v, int bf16, float eps,
                          int num_sms, cudaStream_t st);

// True if the bf16 tensor-core forward is compiled for this shape.
bool tc_forward_supported(int d_key, int nu, int d_v, int chunk);

// Device workspace bytes the bf16 forward needs for this shape.
size_t tc_forward_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk);

// The two phases of the bf16 forward (arguments validated by the caller):
// per-chunk preparation into the workspace, then the serial state scan.
cudaError_t tc_prepare_launch(const void *q, const void *k, const void *v, const void *beta, void *workspace,
                              int B, int H, int L, int d_key, int nu, int d_v, int chunk, float eps, int num_sms,
                              unsigned *status, cudaStream_t st);
cudaError_t tc_scan_launch(const void *workspace, const float *W0, float *W_final, void *y, int B, int H, int L,
                           int d_key, int nu, int d_v, int chunk, int num_sms, unsigned *status, cudaStream_t st);

// Kernels tc_forward_launch enqueues for this shape: 1 (one cooperative
// launch, the flags zeroed by a memset before it), 2 (prep, then scan), or
// -1 on a CUDA error.
int tc_forward_kernel_count(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int num_sms);

// Enqueue the bf16 forward: both phases (arguments validated by the caller),
// as one launch or as the two kernels.
cudaError_t tc_forward_launch(const void *q, const void *k, const void *v, const void *beta,
                              const float *W0, float *W_final, void *y, void *workspace, int B,
                              int H, int L, int d_key, int nu, int d_v, int chunk, float eps,
                              int num_sms, unsigned *status, cudaStream_t st);

// The prep with the projection prologue folded in: q, k, v and beta of each
// chunk computed from x [B*L, d_model] and W_all [d_model, ldw] (the layout
// launch_project reads) inside the prep kernel, then the records written as
// tc_prepare_launch writes them.  d_key <= 64, d_v <= 64, d_model % 64 == 0;
// x and W_all 16-byte aligned (arguments validated by the caller).
bool tc_prepare_x_supported(int d_key, int d_v);
cudaError_t tc_prepare_x_launch(const void *x, const void *W_all, int ldw, void *workspace, int B, int H, int L,
                                int d_model, int d_key, int nu, int d_v, int chunk, float eps, int num_sms,
                                unsigned *status, cudaStream_t st);

// A 2-D TMA map of a row-major bf16 matrix [rows, cols] (row stride ld
// elements) in boxes of box_rows x 64 columns, 128-byte swizzle.
cudaError_t make_bf16_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows);

// The sum rule (linear attention), bf16 I/O: W_i = W_{i-1} + v_i phi(k_i)^T,
// y_i = W_i phi(q_i), divided by z_i . phi(q_i) (z_i = sum of phi(k)) when
// normalize != 0.  Arguments validated by the caller.
bool tc_linear_supported(int d_key, int nu, int d_v, int chunk, int normalize);
size_t tc_linear_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int normalize);
cudaError_t tc_linear_launch(const void *q, const void *k, const void *v, const float *W0, const float *z0,
                             float *W_final, float *z_final, void *y, void *workspace, int B, int H, int L,
                             int d_key, int nu, int d_v, int chunk, int normalize, float eps, int num_sms,
                             unsigned *status, cudaStream_t st);

// The backward of the delta rule (fp32 arithmetic, fp32 or bf16 I/O).  Where
// backward_chunked_supported() holds, the chunk-parallel form
// (fw_backward_chunk.cu); otherwise one CTA per (b,h) and block of 16 rows of
// W, token by token, with those rows of W and of its gradient in shared
// memory.  Arguments validated by the caller.
size_t backward_smem_bytes(int d_key, int nu, int d_v);
size_t backward_workspace_bytes(int BH, int L, int d_key, int nu, int d_v);
cudaError_t launch_backward(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                            const void *gy, const float *gWL, void *gq, void *gk, void *gv, void *gbeta,
                            float *gW0, float *scratch, int BH, int L, int d_key, int nu, int d_v, int bf16,
                            float eps, int num_sms, cudaStream_t st);
// The chunk-parallel backward (chunks of 64 tokens): d_dot <= 512, d_v <= 128.
// It reads phi(k), phi(q) (fp32, made by launch_dpfp), writes gv and gW0,
// and leaves per token [g_phi(q) | g_phi(k) | gbeta | pad] (2 d_dot + 4
// floats) in part for the DPFP-backward kernel; buf holds
// backward_chunked_buffer_floats() floats of intermediate chunk data.
bool backward_chunked_supported(int d_key, int nu, int d_v, int L);
size_t backward_chunked_buffer_floats(int BH, int L, int d_key, int nu, int d_v);
cudaError_t launch_backward_chunked(const float *phk, const float *phq, const void *v, const void *beta,
                                    const float *W0, const void *gy, const float *gWL, void *gv, float *gW0,
                                    float *part, float *buf, int BH, int L, int d_dot, int d_v, int bf16,
                                    cudaStream_t st);
// K1, the standalone DPFP map: phi [rows, 2 d_key nu] of x [rows, d_key]
// (bf16 or fp32 each way; arguments validated by the caller).
cudaError_t launch_dpfp(const void *x, void *phi, int64_t rows, int d_key, int nu, int in_bf16, int out_bf16,
                        float eps, int num_sms, cudaStream_t st);

// The dense layers run on one tcgen05 GEMM fed by TMA (fw_project.cu).  When
// the output tiles alone would leave most SMs idle, K is split into up to 8
// slices, each tile's slices one thread-block cluster whose CTAs add their
// fp32 partial tiles in slice order through distributed shared memory.
int gemm_slices(int M, int N, int K);
size_t project_smem_bytes();

// The projection prologue: q, k, v, beta (bf16, [B,H,L,*]) = x [B*L, d_model]
// (bf16) times W_all = [W_q | W_k | W_v | W_beta] ([d_model, ldw], the first
// N = H (2 d_key + d_v + 1) columns used; beta through the sigmoid).
// d_model % 64 == 0, ldw % 8 == 0, ldw >= N rounded up to 8; x and W_all
// 16-byte aligned.  w_early: the kernel may read the weights before the
// preceding kernel on the stream has completed (only where that kernel is
// one of this library's, which never write a weight).
cudaError_t launch_project(const void *x, const void *Wall, int ldw, void *q, void *k, void *v, void *beta, int B,
                           int L, int H, int d_key, int d_v, int d_model, bool w_early, unsigned *status,
                           cudaStream_t st);

// A dense layer's A operand as the LayerNorm of fp32 rows x [M, K]
// (biased variance over K; gamma, beta fp32 [K] or null for 1 and 0),
// rounded to bf16, from the per-row statistics of x that the dense layer
// which wrote x left in `stats`: (mean, sum of squared deviations) of each
// 128-column part, [M][parts], parts = K / 128.
struct DenseLn {
    const float *x;
    const float2 *stats;
    const float *gamma, *beta;
    float eps;
    int parts;
};
// Whether launch_dense can take its A as a DenseLn for these sizes: K a
// multiple of 128, and at most two K steps of 64 per K slice (x's fp32 tiles
// are staged in the two ring stages those steps leave free).
bool dense_ln_supported(int M, int N, int K);

// A dense layer: P = A W + bias with A [M, K] bf16 and W [K, N] bf16
// (row-major), then out = resid + P (fp32; resid may be NULL or equal to
// out; out_bf16_copy, when not NULL, receives the same values in bf16) or,
// with relu, out = bf16(max(P, 0)).  K % 64 == 0, N % 8 == 0; bias (fp32
// [N]) may be NULL.  w_early as for launch_project.  stats (fp32 output
// only, N % 128 == 0; or null): the output rows' statistics for a DenseLn
// of a later layer.  ln (or null): A is that LayerNorm instead, computed in
// the kernel (A then only sizes the unused tensor map).
cudaError_t launch_dense(const void *A, const void *W, int K, int M, int N, const float *bias, const float *resid,
                         void *out, bool relu, void *out_bf16_copy, bool w_early, float2 *stats, const DenseLn *ln,
                         unsigned *status, cudaStream_t st);

// Row-wise layer normalisation (biased variance): out[m] = (x[m] - mean) /
// sqrt(var + eps) * gamma + beta over D columns; x fp32 [M, D]; out bf16
// (out_bf16) or fp32.  D % 128 == 0, D <= 1024.
cudaError_t launch_layernorm(const float *x, const float *gamma, const float *beta, void *out, bool out_bf16, int M,
                             int D, float eps, cudaStream_t st);

} // namespace fw
