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
// stream (fp32) or passed through ReLU (bf16 out).  A and W are bf16.
//
// Mapping: one CTA of 128 threads per 128 x 128 tile of P and per slice of
// K (split-K when the tiles alone would leave most SMs idle).  K is walked
// in steps of 64 through a ring of four shared-memory stages filled by TMA
// tensor copies (A: a 128-row x 64-column box of x, K-major; B: two 64 x 64
// boxes of W_all, MN-major; both with the 128-byte swizzle the MMA
// descriptors name), so up to four steps of loads are in flight while the
// tensor core works.  One thread issues the copies, another the MMAs
// (tcgen05, fp32 accumulator in TMEM); the ring's full / empty mbarriers
// order them.  The epilogue reads TMEM, one output row per thread: with one
// slice it finishes the tile at once; with several, every CTA stores its
// fp32 partial tile and a second kernel adds the partials in slice order
// (the same sum on every run) and finishes them.  Finishing routes every 8 columns to their head
// in q, k, v (16-byte stores) or beta (sigmoid), or adds the bias and then
// the residual (fp32, optionally also a bf16 copy) or applies ReLU (bf16).
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "fw_forward_tc.h"
#include "fw_tc.cuh"

namespace fw {

namespace {

using namespace tc;

constexpr int kProjThreads = 128;
constexpr int kStages = 4;
constexpr int kStageBytes = 32768; // A 16 KB + B 16 KB
// K is split when the output tiles alone would occupy fewer than half the
// SMs, into slices that bring the grid to about kTargetCtas CTAs: measured
// on the layer stack's GEMMs (M = 256), splitting every one of them, with
// its extra reduction kernel, beat splitting only the long (K = 2048) one
// by 13% per token (471 vs 540 us).
constexpr int kTargetCtas = 148;

enum { kEpiHeads = 0, kEpiBiasResid = 1, kEpiBiasRelu = 2 };

// Where the epilogue puts P: the heads' q, k, v, beta ([B, H, L, *] bf16),
// or one row-major [M, ldo] output (fp32 plus a residual, with an optional
// bf16 copy, or bf16 after ReLU).
struct GemmOut {
    __nv_bfloat16 *q, *k, *v, *beta;
    int L, H, d_key, d_v;
    const float *bias, *resid;
    float *out_f32;
    __nv_bfloat16 *out_bf16;
    int ldo;
};

// 8 columns n .. n + 7 of row m of P routed to their head in q, k, v, or
// to beta through the sigmoid (one head per column).
FW_DEV void heads_out(const GemmOut &o, const float *acc, int m, int n, int N) {
    const int H = o.H, d_key = o.d_key, d_v = o.d_v, L = o.L;
    const int b_ = m / L, t = m - b_ * L;
    const int Nq = H * d_key, Nv = H * d_v;
    if (n < 2 * Nq + Nv) {          // q, k or v: all 8 in one head
        __nv_bfloat16 *dst;
        if (n < Nq)
            dst = o.q + (((size_t)b_ * H + n / d_key) * L + t) * d_key + n % d_key;
        else if (n < 2 * Nq)
            dst = o.k + (((size_t)b_ * H + (n - Nq) / d_key) * L + t) * d_key + (n - Nq) % d_key;
        else
            dst = o.v + (((size_t)b_ * H + (n - 2 * Nq) / d_v) * L + t) * d_v + (n - 2 * Nq) % d_v;
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            t8[e] = acc[e];
        store8(dst, t8);
    } else {                        // beta: one head per column
        for (int e = 0; e < 8 && n + e < N; ++e) {
            const int h = n + e - 2 * Nq - Nv;
            o.beta[((size_t)b_ * H + h) * L + t] = __float2bfloat16_rn(1.0f / (1.0f + expf(-acc[e])));
        }
    }
}

// 8 columns n .. n + 7 of row m of P plus the bias, then added to the
// residual row (fp32 out, and its bf16 copy when asked; the residual may be
// the output itself) or passed through ReLU (bf16 out).
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
        if (o.out_bf16)
            store8(o.out_bf16 + off, t8);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            t8[e] = fmaxf(t8[e], 0.f);
        store8(o.out_bf16 + off, t8);
    }
}

template <int EPI>
FW_DEV void finish16(const GemmOut &o, const float *acc, int m, int n, int N) {
#pragma unroll
    for (int h8 = 0; h8 < 16; h8 += 8) {
        if (n + h8 >= N)
            break;
        if (EPI == kEpiHeads)
            heads_out(o, acc + h8, m, n + h8, N);
        else
            bias_out<EPI>(o, acc + h8, m, n + h8);
    }
}

// grid (M tiles, N tiles, K slices); K slice z covers K steps
// [z * per, min(nk, (z + 1) * per)) of 64.  part: [slices][M tiles * 128][N
// tiles * 128] fp32 partial tiles (used with slices > 1 only).
template <int EPI>
__global__ void __launch_bounds__(kProjThreads)
    gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, int K, int M, int N,
                int per, GemmOut o, float *part, unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = (uint64_t *)(smem + kStages * kStageBytes); // [kStages] a stage's copies landed
    uint64_t *empty = full + kStages;                            // [kStages] a stage's MMAs are done
    uint64_t *done = empty + kStages;                            // every MMA is done
    uint32_t *slot = (uint32_t *)(done + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128, z = blockIdx.z, slices = gridDim.z;
    const int nk = K / 64, kb0 = z * per, nkl = min(nk, kb0 + per) - kb0;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(done, 1);
        fence_barrier_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ta)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tb)) : "memory");
    }
    if (warp == 0) {
        tmem_alloc(slot, 128);
        tmem_relinquish();
    }
    griddep_launch_dependents();
    griddep_wait(); // A and W may be the preceding kernel's output
    o.bias = after_wait(o.bias);
    o.resid = after_wait(o.resid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {          // producer: the TMA copies of each K step
        int issued = 0;
        for (int i = 0; i < nkl; ++i) {
            const int s = i % kStages;
            if (i >= kStages && !mbar_wait(empty + s, (uint32_t)((i / kStages - 1) & 1), status)) {
                ok = false;
                break;
            }
            uint8_t *a = smem + s * kStageBytes, *b = a + 16384;
            const int k0 = 64 * (kb0 + i);
            mbar_arrive_expect_tx(full + s, kStageBytes);
            tma_load_2d(a, &ta, k0, m0, full + s);
            tma_load_2d(b, &tb, n0, k0, full + s);
            tma_load_2d(b + 8192, &tb, n0 + 64, k0, full + s);
            issued = i + 1;
        }
        // before the CTA can leave, every copy issued has landed (bounded)
        for (int i = max(0, issued - kStages); i < issued; ++i)
            mbar_wait(full + i % kStages, (uint32_t)((i / kStages) & 1), status);
    } else if (warp == 1 && lane == 0) {   // the MMAs of each K step
        const uint32_t idesc = idesc_bf16(128, 128, 0, 1);
        for (int i = 0; i < nkl; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(full + s, (uint32_t)((i / kStages) & 1), status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_u32(smem + s * kStageBytes), b = a + 16384;
#pragma unroll
            for (int st = 0; st < 4; ++st)
                mma_bf16(tm, desc_sw128(a + kmajor_step(st, 128), 16, 1024),
                         desc_sw128(b + (uint32_t)st * 2048u, 8192, 1024), idesc, (i > 0 || st > 0) ? 1u : 0u);
            mma_commit(empty + s);
        }
        mma_commit(done);
    }
    __syncwarp();
    ok = mbar_wait(done, 0, status) && ok;
    tc_fence_after();
    if (__syncthreads_or(!ok)) {
        tc_fence_before();
        __syncthreads();
        if (warp == 0)
            tmem_dealloc(tm, 128);
        return;
    }
    const int m = m0 + tid;
    const uint32_t lane_base = tmem_lane_base(warp);
    if (slices == 1) {
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float acc[16];
            tmem_ld16(tm + lane_base + (uint32_t)c0, acc);
            tmem_ld_wait();
            if (m < M && n0 + c0 < N)
                finish16<EPI>(o, acc, m, n0 + c0, N);
        }
    } else { // this slice's fp32 partial tile; splitk_reduce_kernel adds the slices
        const size_t ldp = (size_t)gridDim.y * 128, rows = (size_t)gridDim.x * 128;
        float *mine = part + ((size_t)z * rows + m) * ldp + n0;
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float acc[16];
            tmem_ld16(tm + lane_base + (uint32_t)c0, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                __stcg(reinterpret_cast<float4 *>(mine + c0 + j), make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, 128);
}

// The slices of a split-K GEMM added in slice order (so the sum does not
// depend on which CTA finished first), then finished like a one-slice tile.
// One thread per 8 columns of a row; the loads of up to 8 slices are issued
// before any is added.  part: [slices][Mp][ldp] fp32.
template <int EPI>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *part, int slices, int Mp, int ldp, int M, int N,
                                                            GemmOut o) {
    griddep_launch_dependents();
    griddep_wait(); // the partial tiles are the preceding kernel's
    part = after_wait(part);
    o.bias = after_wait(o.bias);
    o.resid = after_wait(o.resid);
    const int g8 = (N + 7) / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)M * g8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / g8), n = 8 * (int)(i % g8);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[e] = 0.f;
        for (int z0 = 0; z0 < slices; z0 += 8) {
            float4 f[8][2];
#pragma unroll
            for (int zz = 0; zz < 8; ++zz)
                if (z0 + zz < slices) {
                    const float4 *src = reinterpret_cast<const float4 *>(part + ((size_t)(z0 + zz) * Mp + m) * ldp + n);
                    f[zz][0] = __ldcg(src);
                    f[zz][1] = __ldcg(src + 1);
                }
#pragma unroll
            for (int zz = 0; zz < 8; ++zz)
                if (z0 + zz < slices) {
                    acc[0] += f[zz][0].x;
                    acc[1] += f[zz][0].y;
                    acc[2] += f[zz][0].z;
                    acc[3] += f[zz][0].w;
                    acc[4] += f[zz][1].x;
                    acc[5] += f[zz][1].y;
                    acc[6] += f[zz][1].z;
                    acc[7] += f[zz][1].w;
                }
        }
        if (EPI == kEpiHeads)
            heads_out(o, acc, m, n, N);
        else
            bias_out<EPI>(o, acc, m, n);
    }
}

// ------------------------------------------------------------ tensor maps
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// A row-major bf16 matrix [rows, cols] with row stride ld (elements) seen as
// boxes of box_rows x 64 columns with the 128-byte swizzle; out-of-range
// elements read as zero.
cudaError_t make_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows) {
    EncodeTiled fn = encoder();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

} // namespace

cudaError_t make_bf16_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows) {
    return make_map(map, base, rows, cols, ld, box_rows);
}

int gemm_slices(int M, int N, int K) {
    const int tiles = ((M + 127) / 128) * ((N + 127) / 128), nk = K / 64;
    if (tiles >= kTargetCtas / 2 || nk <= 1)
        return 1;
    const int want = std::min(nk, (kTargetCtas + tiles - 1) / tiles);
    const int per = (nk + want - 1) / want;
    return (nk + per - 1) / per;
}

size_t gemm_scratch_bytes(int M, int N, int K) {
    const int sl = gemm_slices(M, N, K);
    if (sl == 1)
        return 0;
    const size_t tm = (M + 127) / 128, tn = (N + 127) / 128;
    return (size_t)sl * tm * 128 * tn * 128 * 4;
}

size_t project_smem_bytes() { return (size_t)kStages * kStageBytes + (2 * kStages + 1) * 8 + 16 + 1024; }

template <int EPI>
cudaError_t launch_gemm_t(const void *A, const void *W, int ldw, int K, int M, int N, const GemmOut &o, void *scratch,
                          unsigned *status, cudaStream_t st) {
    CUtensorMap ta, tb;
    cudaError_t e = make_map(&ta, A, M, K, K, 128);
    if (e == cudaSuccess)
        e = make_map(&tb, W, K, N, ldw, 64);
    if (e != cudaSuccess)
        return e;
    const size_t smem = project_smem_bytes();
    auto kern = gemm_kernel<EPI>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int sl = gemm_slices(M, N, K), nk = K / 64, per = (nk + sl - 1) / sl;
    const int tm = (M + 127) / 128, tn = (N + 127) / 128;
    if (sl > 1 && !scratch)
        return cudaErrorInvalidValue;
    float *part = static_cast<float *>(scratch);
    const dim3 grid((unsigned)tm, (unsigned)tn, (unsigned)sl);
    e = launch_pdl(kern, grid, dim3(kProjThreads), smem, st, ta, tb, K, M, N, per, o, part, status);
    if (e != cudaSuccess || sl == 1)
        return e;
    const int64_t work = (int64_t)M * ((N + 7) / 8);
    return launch_pdl(splitk_reduce_kernel<EPI>, dim3((unsigned)std::min<int64_t>((work + 255) / 256, 1184)),
                      dim3(256), 0, st, (const float *)part, sl, tm * 128, tn * 128, M, N, o);
}

cudaError_t launch_project(const void *x, const void *Wall, int ldw, void *q, void *k, void *v, void *beta, int B,
                           int L, int H, int d_key, int d_v, int d_model, void *scratch, unsigned *status,
                           cudaStream_t st) {
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
    return launch_gemm_t<kEpiHeads>(x, Wall, ldw, d_model, M, N, o, scratch, status, st);
}

cudaError_t launch_dense(const void *A, const void *W, int K, int M, int N, const float *bias, const float *resid,
                         void *out, bool relu, void *out_bf16_copy, void *scratch, unsigned *status,
                         cudaStream_t st) {
    GemmOut o = {};
    o.bias = bias;
    o.resid = resid;
    o.ldo = N;
    if (relu) {
        o.out_bf16 = static_cast<__nv_bfloat16 *>(out);
        return launch_gemm_t<kEpiBiasRelu>(A, W, N, K, M, N, o, scratch, status, st);
    }
    o.out_f32 = static_cast<float *>(out);
    o.out_bf16 = static_cast<__nv_bfloat16 *>(out_bf16_copy);
    return launch_gemm_t<kEpiBiasResid>(A, W, N, K, M, N, o, scratch, status, st);
}

} // namespace fw
