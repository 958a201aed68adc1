// fw_selftest.cu -- one-CTA tcgen05 GEMM (D = A B^T, M = 128) through the same
// primitives and 128-byte-swizzled operand layouts as the bf16 forward, so a
// GPU test can pin them against a plain matrix product.
#include "fastweight_selftest.h"
#include "fw_tc.cuh"

namespace fw {
cudaError_t status_word(unsigned **out);
}

namespace {

using namespace fw::tc;

// Element (m, k) of an operand with M/N index m and contraction index k.
//   K-major:  the tile's rows are m (R = rows of the operand), columns k.
//   MN-major: the tile's rows are k (R = K), columns m.
__device__ uint32_t operand_off(int m, int k, int rows, int K, int mn) {
    return mn ? kmajor_off(k, m, K) : kmajor_off(m, k, rows);
}

__device__ uint64_t operand_desc(uint32_t base, int s, int rows, int K, int mn, int swap) {
    if (!mn)
        return desc_sw128(base + kmajor_step(s, rows), 16, 1024);
    const uint32_t lbo = (uint32_t)K * 128u, sbo = 1024u; // 64-column blocks, 8-row groups
    return swap ? desc_sw128(base + (uint32_t)s * 2048u, sbo, lbo)
                : desc_sw128(base + (uint32_t)s * 2048u, lbo, sbo);
}

constexpr int kRegionA = 64 * 1024;  // A tile region (the tile itself is <= 32 KB)
constexpr int kRegionB = 96 * 1024;  // B tile region (the tile itself is <= 64 KB)

__global__ void __launch_bounds__(128) umma_selftest_kernel(const float *A, const float *B, float *D, int N,
                                                            int K, int a_mn, int b_mn, int swap,
                                                            unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u); // stays a shared pointer
    uint8_t *ta = smem;
    uint8_t *tb = smem + kRegionA;
    uint64_t *bar = (uint64_t *)(smem + kRegionA + kRegionB);
    uint32_t *slot = (uint32_t *)(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t ncols = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));

    // zero both regions so any read outside the staged tile sees finite data
    for (int i = tid; i < (kRegionA + kRegionB) / 16; i += 128)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, ncols);
        tmem_relinquish();
    }
    __syncthreads();
    for (int i = tid; i < 128 * K; i += 128) {
        const int m = i / K, k = i % K;
        *reinterpret_cast<__nv_bfloat16 *>(ta + operand_off(m, k, 128, K, a_mn)) = __float2bfloat16_rn(A[i]);
    }
    for (int i = tid; i < N * K; i += 128) {
        const int n = i / K, k = i % K;
        *reinterpret_cast<__nv_bfloat16 *>(tb + operand_off(n, k, N, K, b_mn)) = __float2bfloat16_rn(B[i]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *slot;
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, N, a_mn, b_mn);
        for (int s = 0; s < K / 16; ++s)
            mma_bf16(taddr, operand_desc(smem_u32(ta), s, 128, K, a_mn, swap),
                     operand_desc(smem_u32(tb), s, N, K, b_mn, swap), idesc, s > 0);
        mma_commit(bar);
    }
    const bool ok = mbar_wait(bar, 0, status);
    tc_fence_after();
    if (ok) {
        const int row = 32 * warp + lane;
        for (int c0 = 0; c0 < N; c0 += 16) {
            float r[16];
            tmem_ld16(taddr + tmem_lane_base(warp) + (uint32_t)c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                D[row * N + c0 + j] = r[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(taddr, ncols);
}

} // namespace

extern "C" FW_API int fw_selftest_umma(const float *A, const float *B, float *D, int N, int K, int a_mn,
                                       int b_mn, int swap_mn, void *stream) {
    if (!A || !B || !D || ((uintptr_t)A & 15) || ((uintptr_t)B & 15) || ((uintptr_t)D & 15))
        return FW_ERR_INVALID_ARG;
    if (!(N == 16 || N == 32 || N == 64 || N == 128 || N == 256) ||
        !(K == 16 || K == 32 || K == 64 || K == 128) || (a_mn | b_mn | swap_mn) & ~1)
        return FW_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (fw::status_word(&status) != cudaSuccess)
        return FW_ERR_CUDA;
    const size_t smem = kRegionA + kRegionB + 64 + 1024;
    if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return FW_ERR_CUDA;
    umma_selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(A, B, D, N, K, a_mn, b_mn,
                                                                              swap_mn, status);
    return cudaGetLastError() == cudaSuccess ? FW_OK : FW_ERR_CUDA;
}

namespace {

// One CTA waits on an mbarrier that nothing arrives at: the bounded wait
// gives up after limit_ns, records the timeout and the kernel returns.
__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        (void)mbar_wait_ns(&bar, 0, status, limit_ns);
    __syncthreads();
}

// A ready flag that nothing ever sets.
__device__ unsigned g_selftest_flag;

__global__ void flag_timeout_kernel(uint64_t limit_ns, unsigned *status) {
    if (threadIdx.x == 0)
        (void)flag_wait_ns(&g_selftest_flag, status, limit_ns);
    __syncthreads();
}

} // namespace

extern "C" FW_API int fw_selftest_flag_timeout(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 100000)
        return FW_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (fw::status_word(&status) != cudaSuccess)
        return FW_ERR_CUDA;
    flag_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000u, status);
    return cudaGetLastError() == cudaSuccess ? FW_OK : FW_ERR_CUDA;
}

extern "C" FW_API int fw_selftest_wait_timeout(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 100000)
        return FW_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (fw::status_word(&status) != cudaSuccess)
        return FW_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000u, status);
    return cudaGetLastError() == cudaSuccess ? FW_OK : FW_ERR_CUDA;
}
