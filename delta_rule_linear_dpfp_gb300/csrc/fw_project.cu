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

FW_DEV uint32_t ptile_b_chunk(int kr, int n8) { // MN-major B: rows k, 64-column blocks of 8 KB
    return (uint32_t)(n8 >> 6) * 8192u + (uint32_t)kr * 128u + ((uint32_t)(((n8 & 63) >> 3) ^ (kr & 7)) << 4);
}

__global__ void __launch_bounds__(kProjThreads)
    project_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ Wall, int ldw,
                   __nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ k, __nv_bfloat16 *__restrict__ v,
                   __nv_bfloat16 *__restrict__ beta, int M, int L, int H, int d_key, int d_v, int d_model, int N,
                   unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = (uint64_t *)(smem + 2 * kProjStage); // [2] MMAs of a stage done
    uint32_t *slot = (uint32_t *)(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128;
    const int nkb = d_model / 64;

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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;

    // the next stage's tiles go through registers: A row tid (8 chunks), B
    // rows (tid + 128 i) / 16 (chunks (tid + 128 i) % 16)
    uint4 ra[8], rb[8];
    auto load = [&](int kb) {
        const int k0 = 64 * kb;
        const int m = m0 + tid;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            ra[c] = m < M ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)m * d_model + k0) + c)
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + kProjThreads * i, kr = idx >> 4, n = n0 + 8 * (idx & 15);
            rb[i] = n < N ? __ldg(reinterpret_cast<const uint4 *>(Wall + (size_t)(k0 + kr) * ldw + n))
                          : make_uint4(0, 0, 0, 0);
        }
    };
    auto store = [&](int s) {
        uint8_t *a = smem + s * kProjStage, *b = a + 16384;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(a + kmajor_chunk(tid, 8 * c, 128)) = ra[c];
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
        const int b_ = m / L, t = m - b_ * L;
        const int Nq = H * d_key, Nv = H * d_v;
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
                        t8[e] = acc[h8 + e];
                    store8(dst, t8);
                } else {                        // beta: one head per column
                    for (int e = 0; e < 8 && n + e < N; ++e) {
                        const int h = n + e - 2 * Nq - Nv;
                        beta[((size_t)b_ * H + h) * L + t] = __float2bfloat16_rn(1.0f / (1.0f + expf(-acc[h8 + e])));
                    }
                }
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

cudaError_t launch_project(const void *x, const void *Wall, int ldw, void *q, void *k, void *v, void *beta, int B,
                           int L, int H, int d_key, int d_v, int d_model, unsigned *status, cudaStream_t st) {
    const int M = B * L, N = H * (2 * d_key + d_v + 1);
    const size_t smem = project_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)((M + 127) / 128), (unsigned)((N + 127) / 128));
    return launch_pdl(project_kernel, grid, dim3(kProjThreads), smem, st, static_cast<const __nv_bfloat16 *>(x),
                      static_cast<const __nv_bfloat16 *>(Wall), ldw, static_cast<__nv_bfloat16 *>(q),
                      static_cast<__nv_bfloat16 *>(k), static_cast<__nv_bfloat16 *>(v),
                      static_cast<__nv_bfloat16 *>(beta), M, L, H, d_key, d_v, d_model, N, status);
}

} // namespace fw
