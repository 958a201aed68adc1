// fw_project.cu -- the projection prologue of the fast-weight layer: q, k, v
// and beta of every head from the token activations x, on tcgen05 tensor
// cores.
//
// Method (Fast Weights Transformer guide, the attention module's
// projections: bias-free linear maps of the model width to the heads' query,
// key and value widths, and one scalar per head for beta followed by the
// sigmoid): with the four weight matrices side by side as one
// W_all = [W_q | W_k | W_v | W_beta] of d_model rows and
// N = H (2 d_key + d_v + 1) columns, P = x W_all, then
//   q[b, h, t, :] = P[b L + t, h d_key : (h + 1) d_key], k and v likewise,
//   beta[b, h, t] = sigmoid(P[b L + t, 2 H d_key + H d_v + h]),
// each rounded once to bf16 (fp32 accumulation).
//
// The same kernel serves the other dense layers of the token-wise layer
// stack (the attention module's output map, the two linear maps of the
// feed-forward block): P = A W plus a bias, then either added to a residual
// stream (fp32) or passed through ReLU (bf16 out).  A may be fp32 (the
// residual stream, rounded to bf16 as it is staged) or bf16.
//
// Mapping: one CTA of 128 threads per 128 x 128 tile of P; K walked in steps
// of 64 with two shared-memory stages, so the loads of the next step overlap
// the MMAs of the current one.  A = x rows (K-major, 128-byte swizzle), B =
// W_all rows (MN-major, 64-column blocks); the fp32 accumulator lives in
// TMEM; each thread owns one output row and routes every 8 columns to their
// head in q, k, v (16-byte stores) or beta (sigmoid).
#include "fw_forward_tc.h"
#include "fw_tc.cuh"

namespace fw {

namespace {

using namespace tc;

constexpr int kProjThreads = 128;
constexpr int kProjStage = 32768; // A 16 KB + B 16 KB per stage

enum { kEpiHeads = 0, kEpiBiasResid = 1, kEpiBiasRelu = 2 };

// Where the epilogue puts P: the heads' q, k, v, beta ([B, H, L, *] bf16),
// or one row-major [M, ldo] output (fp32 plus a residual, or bf16 after ReLU).
struct GemmOut {
    __nv_bfloat16 *q, *k, *v, *beta;
    int L, H, d_key, d_v;
    const float *bias, *resid;
    float *out_f32;
    __nv_bfloat16 *out_bf16;
    int ldo;
};

FW_DEV uint32_t ptile_b_chunk(int kr, int n8) { // MN-major B: rows k, 64-column blocks of 8 KB
    return (uint32_t)(n8 >> 6) * 8192u + (uint32_t)kr * 128u + ((uint32_t)(((n8 & 63) >> 3) ^ (kr & 7)) << 4);
}

// 8 columns n .. n + 7 of row m of P routed to their head in q, k, v, or
// to beta through the sigmoid (one head per column).
FW_DEV void heads_out(const GemmOut &o, const float *acc, int m, int n, int N) {
    const int H = o.H, d_key = o.d_key, d_v = o.d_v, L = o.L;
    const int b_ = m / L, t = m - b_ * L;
    const int Nq = H * d_key, Nv = H * d_v;
    __nv_bfloat16 *q = o.q, *k = o.k, *v = o.v, *beta = o.beta;
    if (n < 2 * Nq + Nv) {          // q, k or v: all 8 in one head
        __nv_bfloat16 *dst;
        if (n < Nq)
            dst = q + (((size_t)b_ * H + n / d_key) * L + t) * d_key + n % d_key;
        else if (n < 2 * Nq)
            dst = k + (((size_t)b_ * H + (n - Nq) / d_key) * L + t) * d_key + (n - Nq) % d_key;
        else
            dst = v + (((size_t)b_ * H + (n - 2 * Nq) / d_v) * L + t) * d_v + (n - 2 * Nq) % d_v;
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            t8[e] = acc[e];
        store8(dst, t8);
    } else {                        // beta: one head per column
        for (int e = 0; e < 8 && n + e < N; ++e) {
            const int h = n + e - 2 * Nq - Nv;
            beta[((size_t)b_ * H + h) * L + t] = __float2bfloat16_rn(1.0f / (1.0f + expf(-acc[e])));
        }
    }
}

// 8 columns n .. n + 7 of row m of P plus the bias, then added to the
// residual row (fp32 out; the residual may be the output itself) or passed
// through ReLU (bf16 out).
template <int EPI>
FW_DEV void bias_out(const GemmOut &o, const float *acc, int m, int n) {
    float t8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        t8[e] = acc[e] + (o.bias ? __ldcg(o.bias + n + e) : 0.f);
    const size_t off = (size_t)m * o.ldo + n;
    if (EPI == kEpiBiasResid) {
        if (o.resid) {
            float r[8];
            load8(o.resid + off, r);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                t8[e] += r[e];
        }
        store8(o.out_f32 + off, t8);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            t8[e] = fmaxf(t8[e], 0.f);
        store8(o.out_bf16 + off, t8);
    }
}

// One thread's row of the A tile for one K step (64 columns), held in
// registers between its load and its store into shared memory.
template <class TA> struct ARow;
template <> struct ARow<__nv_bfloat16> {
    uint4 r[8];
    FW_DEV void load(const __nv_bfloat16 *p, bool in) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            r[c] = in ? __ldcg(reinterpret_cast<const uint4 *>(p) + c) : make_uint4(0, 0, 0, 0);
    }
    FW_DEV uint4 chunk(int c) const { return r[c]; }
};
template <> struct ARow<float> {
    float4 r[16];
    FW_DEV void load(const float *p, bool in) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            r[c] = in ? __ldcg(reinterpret_cast<const float4 *>(p) + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    FW_DEV uint4 chunk(int c) const { // 8 columns, rounded to bf16
        const float4 a = r[2 * c], b = r[2 * c + 1];
        return make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
};

template <class TA, int EPI>
__global__ void __launch_bounds__(kProjThreads)
    project_kernel(const TA *__restrict__ x, const __nv_bfloat16 *__restrict__ Wall, int ldw, int K, int M, int N,
                   GemmOut o, unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = (uint64_t *)(smem + 2 * kProjStage); // [2] MMAs of a stage done
    uint32_t *slot = (uint32_t *)(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128;
    const int nkb = K / 64;

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 128);
        tmem_relinquish();
    }
    griddep_launch_dependents();
    griddep_wait(); // x and W_all may be the preceding kernel's output
    x = after_wait(x);
    Wall = after_wait(Wall);
    o.bias = after_wait(o.bias);
    o.resid = after_wait(o.resid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;

    // the next stage's tiles go through registers: A row tid (8 chunks), B
    // rows (tid + 128 i) / 16 (chunks (tid + 128 i) % 16)
    ARow<TA> ra;
    uint4 rb[8];
    auto load = [&](int kb) {
        const int k0 = 64 * kb;
        const int m = m0 + tid;
        ra.load(x + (size_t)(m < M ? m : 0) * K + k0, m < M);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + kProjThreads * i, kr = idx >> 4, n = n0 + 8 * (idx & 15);
            rb[i] = n < N ? __ldcg(reinterpret_cast<const uint4 *>(Wall + (size_t)(k0 + kr) * ldw + n))
                          : make_uint4(0, 0, 0, 0);
        }
    };
    auto store = [&](int s) {
        uint8_t *a = smem + s * kProjStage, *b = a + 16384;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(a + kmajor_chunk(tid, 8 * c, 128)) = ra.chunk(c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + kProjThreads * i;
            *reinterpret_cast<uint4 *>(b + ptile_b_chunk(idx >> 4, 8 * (idx & 15))) = rb[i];
        }
    };

    bool ok = true;
    load(0);
    for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb & 1;
        if (kb >= 2) // the MMAs that read this stage two steps ago are done
            ok = mbar_wait(bar + s, (uint32_t)(((kb - 2) >> 1) & 1), status);
        if (__syncthreads_or(!ok))
            break;
        store(s);
        if (kb + 1 < nkb)
            load(kb + 1); // in flight while this step's MMAs run
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a = smem_u32(smem + s * kProjStage), b = a + 16384;
            const uint32_t idesc = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int st = 0; st < 4; ++st)
                mma_bf16(tm, desc_sw128(a + kmajor_step(st, 128), 16, 1024),
                         desc_sw128(b + (uint32_t)st * 2048u, 8192, 1024), idesc, (kb > 0 || st > 0) ? 1u : 0u);
            mma_commit(bar + s);
        }
    }
    if (ok) { // the last step's commit covers every MMA
        const int s = (nkb - 1) & 1;
        ok = mbar_wait(bar + s, (uint32_t)(((nkb - 1) >> 1) & 1), status);
    }
    tc_fence_after();
    if (!__syncthreads_or(!ok)) {
        const int m = m0 + tid;
        const uint32_t lane_base = tmem_lane_base(warp);
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float acc[16];
            tmem_ld16(tm + lane_base + (uint32_t)c0, acc);
            tmem_ld_wait();
            if (m >= M)
                continue;
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8) {
                const int n = n0 + c0 + h8; // 8 columns n .. n + 7 of P
                if (n >= N)
                    break;
                if (EPI == kEpiHeads)
                    heads_out(o, acc + h8, m, n, N);
                else
                    bias_out<EPI>(o, acc + h8, m, n);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, 128);
}

} // namespace

size_t project_smem_bytes() { return 2 * (size_t)kProjStage + 64 + 1024; }

template <class TA, int EPI>
cudaError_t launch_gemm_t(const void *A, const void *W, int ldw, int K, int M, int N, const GemmOut &o,
                          unsigned *status, cudaStream_t st) {
    const size_t smem = project_smem_bytes();
    auto kern = project_kernel<TA, EPI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)((M + 127) / 128), (unsigned)((N + 127) / 128));
    return launch_pdl(kern, grid, dim3(kProjThreads), smem, st, static_cast<const TA *>(A),
                      static_cast<const __nv_bfloat16 *>(W), ldw, K, M, N, o, status);
}

cudaError_t launch_project(const void *x, const void *Wall, int ldw, void *q, void *k, void *v, void *beta, int B,
                           int L, int H, int d_key, int d_v, int d_model, unsigned *status, cudaStream_t st,
                           bool x_f32) {
    GemmOut o = {};
    o.q = static_cast<__nv_bfloat16 *>(q);
    o.k = static_cast<__nv_bfloat16 *>(k);
    o.v = static_cast<__nv_bfloat16 *>(v);
    o.beta = static_cast<__nv_bfloat16 *>(beta);
    o.L = L;
    o.H = H;
    o.d_key = d_key;
    o.d_v = d_v;
    const int M = B * L, N = H * (2 * d_key + d_v + 1);
    return x_f32 ? launch_gemm_t<float, kEpiHeads>(x, Wall, ldw, d_model, M, N, o, status, st)
                 : launch_gemm_t<__nv_bfloat16, kEpiHeads>(x, Wall, ldw, d_model, M, N, o, status, st);
}

cudaError_t launch_dense(const void *A, const void *W, int K, int M, int N, const float *bias, const float *resid,
                         void *out, bool relu, unsigned *status, cudaStream_t st) {
    GemmOut o = {};
    o.bias = bias;
    o.resid = resid;
    o.ldo = N;
    if (relu) {
        o.out_bf16 = static_cast<__nv_bfloat16 *>(out);
        return launch_gemm_t<__nv_bfloat16, kEpiBiasRelu>(A, W, N, K, M, N, o, status, st);
    }
    o.out_f32 = static_cast<float *>(out);
    return launch_gemm_t<__nv_bfloat16, kEpiBiasResid>(A, W, N, K, M, N, o, status, st);
}

} // namespace fw
