/*
 * fastweight.h -- C ABI of the GB300 (sm_103a) delta-rule fast-weight layer
 * core with the DPFP feature map.
 *
 * The method is the one the Fast Weights Transformer guide (xdnf.cn/news/308600,
 * a walk-through of "Linear Transformers Are Secretly Fast Weight Memory
 * Systems", arXiv:2102.11174) describes:
 *
 *   phi(k)   = DPFP(k): x = ReLU([k, -k]) (length 2*d_key); for i = 1..nu the
 *              block i of phi is x * roll(x, i), where roll follows
 *              torch.roll(shifts=i) (position j holds x[(j - i) mod 2*d_key]);
 *              phi is then divided by (sum(phi) + eps).  d_dot = 2*d_key*nu.
 *              [section "DPFP: projection formula and hyper-parameters", the
 *              normalisation formula and the DPFP source shown with it]
 *   vbar_t   = W_{t-1} phi(k_t)
 *   W_t      = W_{t-1} + beta_t (v_t - vbar_t) outer phi(k_t)
 *   y_t      = W_t phi(q_t)         (the read uses the updated W)
 *              [section "FastWeightsAttention: the new update rule" and its
 *              forward-pass loop; W starts from zero per (batch, head) unless
 *              an initial state is given]
 *
 * There is no normaliser z and no 1/sqrt(d) scale: phi is already normalised
 * (same section).
 *
 * Conventions shared by every call
 *   - All tensor arguments are CALLER-OWNED DEVICE pointers to contiguous,
 *     row-major memory (the last dimension is fastest).  The library never
 *     allocates or frees device memory and keeps no pointer after a call
 *     returns.
 *   - Activations use the [B, H, L, d] layout (batch, head, token, feature).
 *     The fast-weight state W is fp32 [B, H, d_v, d_dot], the layout of the
 *     guide's forward pass (weights of shape [batch, heads, d_value, d_key]).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns; results are
 *     ready once the stream has reached that point.
 *   - Every argument is checked on the host BEFORE anything is enqueued: a
 *     call that returns an error has launched nothing and touched no memory.
 *   - Pointers must be 16-byte aligned (FW_ERR_INVALID_ARG otherwise).
 *     When an operation is empty (rows == 0, B*H == 0, or L == 0 for the
 *     activations of fw_delta_forward) the pointers of the empty tensors are
 *     not used and may be NULL.
 *   - No call has a CPU fallback: shapes outside the compiled tile set give
 *     FW_ERR_UNSUPPORTED.
 *   - Return values are fw_status codes; fw_status_string() names them.
 */
#ifndef FASTWEIGHT_H
#define FASTWEIGHT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FW_API __attribute__((visibility("default")))
#else
#define FW_API
#endif

typedef enum fw_status {
    FW_OK = 0,
    FW_ERR_INVALID_ARG = 1, /* null or misaligned pointer, non-positive size, nu out of range */
    FW_ERR_UNSUPPORTED = 2, /* valid arguments outside the compiled shapes / dtypes */
    FW_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
    FW_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see fw_device_status) */
} fw_status;

typedef enum fw_dtype {
    FW_DTYPE_F32 = 0, /* IEEE binary32 */
    FW_DTYPE_BF16 = 1 /* bfloat16 */
} fw_dtype;

/* Name of a status code (static string, never NULL). */
FW_API const char *fw_status_string(int status);

/*
 * fw_dpfp -- the DPFP feature map with its sum-normalisation, one fused pass.
 * [Fast Weights Transformer guide, section "DPFP: projection formula and
 * hyper-parameters" and the normalisation formula with its source]
 *
 *   x    : [rows, d_key] in in_dtype          (read)
 *   phi  : [rows, 2*d_key*nu] in out_dtype    (written)
 *   rows : >= 0 (0 enqueues nothing);  d_key in {8, 16, 32, 64, 128};
 *   nu   : 1 .. 2*d_key-1;  eps >= 0 (the guide's default is 1e-6).
 *   A row whose phi sums to zero gives phi = 0 (0 / (0 + eps)).
 * Errors: FW_ERR_INVALID_ARG for null/misaligned pointers, rows < 0,
 * d_key <= 0, nu out of range, eps < 0 or an unknown dtype;
 * FW_ERR_UNSUPPORTED for other d_key; FW_ERR_CUDA if the launch fails.
 */
FW_API int fw_dpfp(const void *x, void *phi, int64_t rows, int d_key, int nu, int in_dtype,
                   int out_dtype, float eps, void *stream);

/*
 * Bytes of device workspace fw_delta_forward needs for this shape (0 when it
 * needs none; also 0 for arguments it would reject).  The caller allocates it.
 */
FW_API size_t fw_delta_forward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v,
                                              int chunk, int io_dtype);

/*
 * fw_delta_forward -- the delta-rule recurrence over a whole sequence, for
 * every (batch, head) pair, with the DPFP map of q and k fused in.
 * [Fast Weights Transformer guide, section "FastWeightsAttention: the new
 * update rule" and its forward-pass loop; the chunked evaluation with the
 * memory passed from chunk to chunk follows the lucidrains
 * fast-weight-attention write-up, section 4.2, which gives the interface
 * (tokens in, output and next memory out) but no algorithm.]
 *
 *   q, k     : [B, H, L, d_key]  io_dtype             (read)
 *   v        : [B, H, L, d_v]    io_dtype             (read)
 *   beta     : [B, H, L]         io_dtype, in [0, 1]  (read)
 *   W0       : [B, H, d_v, d_dot] fp32 initial state, or NULL for zeros
 *   W_final  : [B, H, d_v, d_dot] fp32 final state, or NULL to skip it;
 *              W_final == W0 (in place) is allowed
 *   y        : [B, H, L, d_v]    io_dtype             (written)
 *   workspace: device scratch of at least fw_delta_forward_workspace_size()
 *              bytes (may be NULL when that size is 0); its contents on entry
 *              do not matter and are garbage on return
 *   chunk    : tokens per chunk of the chunked evaluation, in {16, 32, 64};
 *              L need not be a multiple of it (the last chunk is partial).
 *              The result does not depend on it beyond rounding.
 *   io_dtype : FW_DTYPE_F32 -- fp32 arithmetic on CUDA cores, token by token
 *              (chunk is validated but only tiles the work);
 *              FW_DTYPE_BF16 -- bf16 operands on the tcgen05 tensor cores
 *              with fp32 accumulation and an fp32 state.
 *   eps      : DPFP normaliser (1e-6 in the guide).
 * Other pointers must not alias each other.
 * Errors: FW_ERR_INVALID_ARG (null required pointer, misaligned pointer,
 * non-positive size, nu out of range, workspace too small);
 * FW_ERR_UNSUPPORTED (shapes outside the compiled set: d_key in {8, 16, 32,
 * 64, 128}; for bf16 also d_v in {16, 32, 64, 128} and the state must fit
 * the tensor memory); FW_ERR_CUDA (launch failure).  A device-side bounded
 * wait that gives up is reported by fw_device_status().
 */
FW_API int fw_delta_forward(const void *q, const void *k, const void *v, const void *beta,
                            const float *W0, float *W_final, void *y, void *workspace,
                            size_t workspace_bytes, int B, int H, int L, int d_key, int nu,
                            int d_v, int chunk, int io_dtype, float eps, void *stream);

/*
 * How many of this library's kernels fw_delta_forward enqueues for this shape
 * on the current device.  (An engineering query: the pages have no
 * counterpart.)  With bf16 I/O the forward has two phases -- preparing every
 * chunk, then walking the chunks in order -- run either as two kernels (2) or
 * as one cooperative launch in which the walk overlaps the rest of the
 * preparation (1; a memset of the workspace's ready flags precedes it).  The
 * one launch is taken where the preparation needs more than one wave of CTAs
 * and the walking CTAs leave SMs free; both give the same bits.  fp32 I/O: 1.
 * 0 when nothing is launched (B*H == 0 or L == 0); -1 for arguments
 * fw_delta_forward would reject, or a CUDA error.
 */
FW_API int fw_delta_forward_kernel_count(int B, int H, int L, int d_key, int nu, int d_v, int chunk,
                                         int io_dtype);

/*
 * Bytes of device workspace fw_delta_forward_projected needs (0 for
 * arguments it would reject).  The caller allocates it.
 */
FW_API size_t fw_delta_forward_projected_workspace_size(int B, int L, int d_model, int H, int d_key,
                                                        int nu, int d_v, int chunk);

/*
 * fw_delta_forward_projected -- the layer core from the token activations:
 * the bias-free projections of the attention module (q, k, v of every head
 * and one beta per head through the sigmoid) on the tensor cores, then
 * fw_delta_forward on their bf16 results.  [Fast Weights Transformer guide,
 * the attention module's projections and the sigmoid on beta, then the
 * sections cited for fw_delta_forward.]
 *
 *   x        : [B, L, d_model] bf16 token activations            (read)
 *   W_all    : [d_model, ldw]  bf16, the four weight matrices side by side:
 *              columns [0, H d_key) W_q, then H d_key of W_k, H d_v of W_v
 *              and H of W_beta (head h owns columns h d .. (h + 1) d - 1 of
 *              its block); ldw % 8 == 0 and ldw >= H (2 d_key + d_v + 1)
 *              rounded up to 8 (the padding columns are read, not used)
 *   W0, W_final, y, chunk, eps : as for fw_delta_forward (y [B, H, L, d_v])
 *   workspace: device scratch of fw_delta_forward_projected_workspace_size()
 *              bytes: room for the projected q, k, v, beta, then the
 *              forward's workspace
 * q, k, v and beta are rounded to bf16 once (fp32 accumulation).
 * Errors as for fw_delta_forward; FW_ERR_INVALID_ARG also for d_model not a
 * multiple of 64 or a bad ldw.
 * Kernels: where fw_delta_forward_kernel_count() of the shape is 2 and
 * d_key, d_v <= 64, the projections run inside the forward's first kernel
 * (each chunk's prep computes its own rows of q, k, v and beta from x with
 * TMA-fed tensor-core MMAs; they never reach global memory), then the walk
 * over the chunks: two launches from x.  Otherwise the projections' GEMM
 * (when B L is small, K is split across the CTAs of a thread-block cluster,
 * which add their partial tiles in the same kernel) writes q, k, v, beta to
 * the workspace and fw_delta_forward follows.
 * Launches are chained by programmatic dependent launch.
 */
FW_API int fw_delta_forward_projected(const void *x, const void *W_all, int ldw, const float *W0,
                                      float *W_final, void *y, void *workspace, size_t workspace_bytes,
                                      int B, int L, int d_model, int H, int d_key, int nu, int d_v,
                                      int chunk, float eps, void *stream);

/*
 * Bytes of device workspace fw_delta_backward needs for this shape (0 for
 * arguments it would reject).  The caller allocates it.
 */
FW_API size_t fw_delta_backward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v,
                                               int io_dtype);

/*
 * fw_delta_backward -- gradients of the delta-rule forward (fw_delta_forward,
 * any chunk: the result does not depend on it) with respect to q, k, v, beta
 * and the initial state, given the gradients of y and of the final state.
 * [The chain rule applied in reverse token order to the recurrence of the
 * Fast Weights Transformer guide, section "FastWeightsAttention: the new
 * update rule", and through its DPFP map; the pages print no backward, the
 * guide trains through the loop with autograd.]
 *
 *   q, k, v, beta : as for fw_delta_forward                 (read)
 *   W0       : [B, H, d_v, d_dot] fp32 initial state, or NULL for zeros
 *   dy       : [B, H, L, d_v]     io_dtype, dL/dy           (read)
 *   dW_final : [B, H, d_v, d_dot] fp32 dL/dW_final, or NULL for zeros
 *   dq, dk   : [B, H, L, d_key]   io_dtype                  (written)
 *   dv       : [B, H, L, d_v]     io_dtype                  (written)
 *   dbeta    : [B, H, L]          io_dtype                  (written)
 *   dW0      : [B, H, d_v, d_dot] fp32 dL/dW0, or NULL to skip it
 *   workspace: device scratch of fw_delta_backward_workspace_size() bytes
 * fp32 arithmetic on CUDA cores for both I/O dtypes, after the DPFP map of
 * every k and q (fp32, into the workspace).  For d_dot <= 512 and d_v <= 128
 * the chunk-parallel form: the transpose of the forward's chunk algebra
 * (chunks of 64 tokens), as a per-chunk preparation kernel, a scan of the
 * chunk-start states, a reverse scan of their gradients (both split over
 * blocks of 16 rows of the state) and a per-chunk gradient kernel.  Other
 * shapes (d_dot <= 1024) walk the tokens one at a time: one CTA per
 * (batch, head) and block of 16 rows of the state, with those rows of the
 * state and of its gradient in shared memory.  Either way a last kernel
 * takes the DPFP backward of q and k.
 * The result does not depend on the run (fixed summation orders).
 * Errors as for fw_delta_forward.
 */
FW_API int fw_delta_backward(const void *q, const void *k, const void *v, const void *beta,
                             const float *W0, const void *dy, const float *dW_final, void *dq,
                             void *dk, void *dv, void *dbeta, float *dW0, void *workspace,
                             size_t workspace_bytes, int B, int H, int L, int d_key, int nu,
                             int d_v, int io_dtype, float eps, void *stream);

/*
 * Bytes of device workspace fw_linear_forward needs for this shape (0 for
 * arguments it would reject).  The caller allocates it.
 */
FW_API size_t fw_linear_forward_workspace_size(int B, int H, int L, int d_key, int nu, int d_v,
                                               int chunk, int normalize, int io_dtype);

/*
 * fw_linear_forward -- the sum rule that the delta rule replaces: linear
 * self-attention with the DPFP kernel, written as a fast-weight recurrence.
 * [Fast Weights Transformer guide, section on the fast form of linear
 * self-attention: W_i = W_{i-1} + v_i outer phi(k_i), z_i = z_{i-1} +
 * phi(k_i), y_i = W_i phi(q_i) / (z_i . phi(q_i)).]  The guide gives no
 * guard for a zero denominator; here y_i = 0 where z_i . phi(q_i) == 0
 * (every phi is non-negative, so the numerator is 0 there as well).
 *
 *   q, k     : [B, H, L, d_key]   bf16              (read)
 *   v        : [B, H, L, d_v]     bf16              (read)
 *   W0       : [B, H, d_v, d_dot] fp32 initial state, or NULL for zeros
 *   z0       : [B, H, d_dot]      fp32 initial normaliser, or NULL for zeros
 *   W_final  : [B, H, d_v, d_dot] fp32 final state, or NULL to skip it
 *   z_final  : [B, H, d_dot]      fp32 final normaliser, or NULL to skip it
 *              (W_final == W0 and z_final == z0 in place are allowed)
 *   y        : [B, H, L, d_v]     bf16              (written)
 *   workspace: device scratch of at least fw_linear_forward_workspace_size()
 *              bytes; contents on entry do not matter, garbage on return
 *   chunk    : in {16, 32, 64}, as for fw_delta_forward
 *   normalize: 1 divides by z . phi(q); 0 returns W phi(q) (z0 and z_final
 *              are then not used)
 *   io_dtype : FW_DTYPE_BF16 (the tensor-core path; FW_DTYPE_F32 returns
 *              FW_ERR_UNSUPPORTED)
 *   eps      : DPFP normaliser (1e-6 in the guide)
 * Errors as for fw_delta_forward; with normalize the state must also fit the
 * tensor memory with 16 more channels (padded d_dot + d_v + 16 <= 512).
 */
FW_API int fw_linear_forward(const void *q, const void *k, const void *v, const float *W0,
                             const float *z0, float *W_final, float *z_final, void *y,
                             void *workspace, size_t workspace_bytes, int B, int H, int L,
                             int d_key, int nu, int d_v, int chunk, int normalize, int io_dtype,
                             float eps, void *stream);

/*
 * fw_delta_forward_prepare / fw_delta_forward_scan -- the two phases of the
 * bf16 fw_delta_forward, callable on their own (bf16 I/O only).  Enqueuing
 * prepare then scan on one stream computes exactly what fw_delta_forward
 * computes for the same arguments.
 *   prepare: every chunk of every (batch, head) in parallel -- DPFP of the
 *            chunk's q and k, the chunk's Gram matrix and the triangular
 *            solve of the chunked form, and the products that do not involve
 *            the state -- written to `workspace`.  Reads q, k, v, beta.
 *   scan:    the chunks of each (batch, head) in order -- the state passes
 *            from chunk to chunk, y and the final state are written.  Reads
 *            the workspace written by prepare (and W0), not q, k, v, beta.
 * [the chunked evaluation of the update rule of the Fast Weights Transformer
 * guide; the split into a parallel and a serial phase is this library's]
 * Arguments and errors as fw_delta_forward (io_dtype is bf16).  The
 * workspace must stay untouched between the two calls.
 */
FW_API int fw_delta_forward_prepare(const void *q, const void *k, const void *v, const void *beta,
                                    void *workspace, size_t workspace_bytes, int B, int H, int L,
                                    int d_key, int nu, int d_v, int chunk, float eps, void *stream);
FW_API int fw_delta_forward_scan(const void *workspace, size_t workspace_bytes, const float *W0,
                                 float *W_final, void *y, int B, int H, int L, int d_key, int nu, int d_v,
                                 int chunk, void *stream);

/* Size of the library's own scratch array used by fw_delta_forward_noalloc. */
#define FW_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * fw_delta_forward_noalloc -- fw_delta_forward for callers that must not
 * allocate device memory at call time.  The pages have no counterpart: this
 * is an interface variant, not part of the method.
 *
 * Who needs it: a host program whose memory pool owns the GPU's memory and
 * forbids further cudaMalloc, or a serving loop that cannot afford the
 * implicit device synchronisation cudaMalloc / cudaFree may cause.  Such a
 * caller cannot hand fw_delta_forward a workspace it would first have to
 * allocate.
 *
 * What it does: the bf16 path's workspace is taken from a fixed array inside
 * the library, FW_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU where the
 * library's device code is loaded, held until the process exits.  Then the
 * same checks and kernels as fw_delta_forward run, with the same arguments
 * minus the workspace pair.  No cudaMalloc, cudaFree or other allocating call
 * is made.
 *   - Shapes whose workspace (fw_delta_forward_workspace_size) exceeds
 *     FW_NOALLOC_SCRATCH_BYTES return FW_ERR_UNSUPPORTED before anything is
 *     enqueued.  fp32 I/O needs no workspace and is never limited.
 *   - The array's device address is looked up (cudaGetSymbolAddress) the
 *     first time this function runs in a context on a device, with that
 *     device current, and kept for that context; a new context on the device
 *     (after cudaDeviceReset, for instance) is looked up afresh.
 *   - Every call on a device shares the one array, and its contents from the
 *     previous call are left in place (nothing needs them to be zero).  Calls
 *     that may run at the same time on the GPU (different streams without an
 *     ordering between them) race on it and give undefined results: order
 *     them, e.g. by issuing them on one stream.
 */
FW_API int fw_delta_forward_noalloc(const void *q, const void *k, const void *v, const void *beta,
                                    const float *W0, float *W_final, void *y, int B, int H, int L,
                                    int d_key, int nu, int d_v, int chunk, int io_dtype, float eps,
                                    void *stream);

/*
 * fw_delta_decode_step -- one new token per (batch, head) against a
 * persistent fast-weight state, updated in place.  Every element of W is read
 * once and written once.
 * [Fast Weights Transformer guide, section "token_wise variant" (one token at
 * a time, the weights kept from step to step) and section "inference and
 * sampling"; the arithmetic is the update rule above for one token]
 *
 *   q, k : [B, H, d_key] io_dtype;  v, y : [B, H, d_v] io_dtype;
 *   beta : [B, H] io_dtype;  W : [B, H, d_v, d_dot] fp32, read and written.
 * Errors: as fw_delta_forward (d_key in {8, 16, 32, 64, 128}, d_dot <= 1024).
 */
FW_API int fw_delta_decode_step(const void *q, const void *k, const void *v, const void *beta,
                                float *W, void *y, int B, int H, int d_key, int nu, int d_v,
                                int io_dtype, float eps, void *stream);

/*
 * One layer of the token-wise stack (fw_decode_stack_step): the weights of
 * its fast-weight attention module and feed-forward block, and its fast
 * weights.  All pointers are device pointers; bf16 matrices are row-major
 * [in, out] (P = x W); every bias may be NULL (zero) and each norm's gamma /
 * beta may be NULL (one / zero).
 */
typedef struct fw_stack_layer {
    const void *W_in;      /* bf16 [d_model, ldw_in]: [W_q | W_k | W_v | W_beta], the
                              layout of fw_delta_forward_projected's W_all            */
    const void *W_o;       /* bf16 [H d_v, d_model]: the module's output map          */
    const float *b_o;      /* fp32 [d_model]                                          */
    const float *ln_gamma; /* fp32 [d_model]: the norm before the feed-forward block  */
    const float *ln_beta;  /* fp32 [d_model]                                          */
    const void *W_1;       /* bf16 [d_model, d_ff]                                    */
    const float *b_1;      /* fp32 [d_ff]                                             */
    const void *W_2;       /* bf16 [d_ff, d_model]                                    */
    const float *b_2;      /* fp32 [d_model]                                          */
    float *W;              /* fp32 [B, H, d_v, d_dot]: this layer's fast weights,
                              read and written (persist from token to token)          */
} fw_stack_layer;

/*
 * Bytes of device workspace fw_decode_stack_step needs (0 for a shape it
 * would reject).  The caller allocates it.
 */
FW_API size_t fw_decode_stack_workspace_size(int B, int H, int d_key, int d_v, int d_model, int d_ff);

/*
 * fw_decode_stack_step -- one new token of B sequences through n_layers
 * fast-weight Transformer layers, each layer's fast weights kept from token
 * to token, then the final LayerNorm.
 * [Fast Weights Transformer guide, section "token_wise variant" (one weight
 * entry per layer; each token passes through every layer in turn, then the
 * final norm), section "layer and model assembly" (attention output added to
 * the input, LayerNorm, feed-forward block of linear, ReLU, linear added
 * again; no norm before the attention), section "module structure" (q, k, v
 * and beta projections without bias, beta through the sigmoid, the output
 * linear layer with bias); dropout is the identity at inference]
 *
 *   layers   : HOST array of n_layers fw_stack_layer (read during the call only)
 *   x        : [B, d_model] fp32, the token's input to layer 0       (read)
 *   ln_gamma, ln_beta : fp32 [d_model], the final norm (NULL: one / zero)
 *   out      : [B, d_model] fp32, the final norm's output          (written)
 *   workspace: device scratch of fw_decode_stack_workspace_size() bytes
 *   ldw_in   : row stride of every layer's W_in, as for
 *              fw_delta_forward_projected (ldw % 8 == 0, >= N rounded up to 8)
 *   eps      : DPFP eps;  ln_eps: the norms' eps (1e-5 in PyTorch)
 * Per layer: q, k, v, beta = x W_in (beta through the sigmoid, all rounded to
 * bf16), y = fw_delta_decode_step on the layer's W, x += y W_o + b_o,
 * x += relu(LN(x) W_1 + b_1) W_2 + b_2.  The residual stream x is fp32;
 * what the tensor cores read (x, y, LN(x), the hidden layer) is rounded to
 * bf16 and every product accumulates in fp32.  Six operations per layer
 * plus a cast and the final norm.  A dense layer whose K is split across
 * CTAs adds the slices inside its kernel, and where the first feed-forward
 * map's K slices are at most two steps of 64 (as at the 256-sequence,
 * d_model 512 shape), that GEMM forms LN(x) itself from statistics the
 * output map leaves: 5 n_layers + 2 kernels there, else 6 n_layers + 2; all
 * on `stream`, chained by programmatic dependent launch (capturable in one
 * CUDA graph).
 * Errors: FW_ERR_INVALID_ARG for bad sizes, NULL or unaligned pointers, a
 * small workspace; FW_ERR_UNSUPPORTED for d_key outside {8, 16, 32, 64, 128},
 * d_dot > 1024, d_model not a multiple of 128 or above 1024, H d_v or d_ff
 * not a multiple of 64.
 */
FW_API int fw_decode_stack_step(const fw_stack_layer *layers, int n_layers, const float *x,
                                const float *ln_gamma, const float *ln_beta, float *out,
                                void *workspace, size_t workspace_bytes, int B, int H, int d_key,
                                int nu, int d_v, int d_model, int d_ff, int ldw_in, float eps,
                                float ln_eps, void *stream);

/*
 * fw_device_status -- waits for `stream`, then reports and clears the
 * device-side status word of the current device: FW_ERR_TIMEOUT if any
 * kernel of this library gave up a bounded wait (its outputs are then
 * undefined) since the last call, FW_OK otherwise, FW_ERR_CUDA if the
 * synchronisation itself failed.  Not an error path of the math: with valid
 * inputs the waits always complete.
 */
FW_API int fw_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTWEIGHT_H */
