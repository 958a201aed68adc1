// fw_forward_tc.cu -- the bf16 chunked delta-rule forward on tcgen05 tensor
// cores (fp32 accumulation, fp32 state).
//
// Method: the recurrence of the Fast Weights Transformer guide (section
// "FastWeightsAttention: the new update rule"), evaluated chunk by chunk with
// the memory passed between chunks (the chunked interface of the lucidrains
// fast-weight-attention write-up, section 4.2).  The pages give no chunk
// algorithm; this one follows from the recurrence.  Per chunk of C tokens
// with state S (d_v x d_dot) at its start, K = phi(k), Q = phi(q) (C x d_dot),
// V (C x d_v), beta (C):
//   A   = strict_lower(diag(beta) K K^T),  T = (I + A)^-1 diag(beta)
//   U   = T (V - K S^T)                     (the C write vectors u_t)
//   Y   = Q S^T + tril_incl(Q K^T) U        (reads use the updated W)
//   S  <- S + U^T K
// This is the WY / "UT transform" form of a product of Householder-like
// factors (Bischof and Van Loan 1987; Joffrain et al. 2006; applied to the
// delta rule by Yang et al. 2024), written here from the algebra above.
//
// Two kernels:
//  * chunk_prep_kernel, one CTA per (chunk, batch*head), all in parallel:
//    DPFP of the chunk's k and q rows straight into a 128 x Dp bf16 operand
//    tile [K; Q] (rows 0..63 keys, 64..127 queries; shuffle-based roll as in
//    the standalone DPFP kernel), one tcgen05 MMA chain [K; Q] K^T for the
//    Gram matrix and Q K^T, the unit-lower inverse (I + A)^-1 by 16 x 16 block
//    forward substitution in fp32, T and P T on CUDA cores.  It writes the
//    [K; Q] tile and the [T; P T] tile to the workspace as byte images of
//    the swizzled shared-memory operands.
//  * chunk_scan_kernel, one CTA per (block of DVB value channels,
//    batch*head): rows of W evolve independently, so the state is split by
//    value channel.  The CTA walks the chunks in order: bulk-copies the two
//    images into shared memory, then
//      MMA1  D1 = [K; Q] S^T           (rows 0..63: K S^T, 64..127: Q S^T)
//      X    = V - K S^T  -> bf16 operand tile
//      MMA2  D2 = [T; P T] X           (rows 0..63: U, 64..127: P U)
//      Y    = Q S^T + P U -> y;  U -> bf16 operand tile
//      MMA3  S^T += K^T U              (fp32, resident in tensor memory)
//      S^T  -> bf16 operand tile for the next chunk's MMA1
//    The next chunk's images are copied in as soon as MMA3 has consumed the
//    current ones.
//
// Partial chunks are padded to 64 token rows with zero phi rows and
// beta = 0, which makes the padded rows of T, P and U exactly zero.
#include "fw_dpfp.cuh"
#include "fw_forward_tc.h"
#include "fw_tc.cuh"

namespace fw {
namespace {

using namespace tc;

constexpr int kTile = 64;    // token rows of a chunk tile (chunk <= 64, padded)
constexpr int kThreads = 128;
constexpr int LDS = 65;      // fp32 row stride of the 64 x 64 work matrices
constexpr int kTpBytes = 128 * 128; // [T; P T]: 128 rows x 64 bf16

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ inline int padded_ddot(int d_dot) { return round_up(d_dot, 128); }
__host__ __device__ inline size_t image_bytes(int Dp) { return (size_t)256 * Dp + kTpBytes; }

FW_DEV uint8_t *align1024(uint8_t *p) { return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023); }

FW_DEV uint4 pack8(const float *v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    return u;
}

// ---------------------------------------------------------------------------
// (I + A)^-1 for a strictly lower 64 x 64 A, by 16 x 16 blocks:
//   diagonal blocks by forward substitution (one column per thread), then
//   block row I: N_IJ = -N_II * sum_{K=J}^{I-1} A_IK N_KJ   (J < I).
// A, N: [64][LDS]; R: [16][LDS] scratch.  All 128 threads; ends synchronised.
FW_DEV void unit_lower_inverse(const float *A, float *N, float *R, int tid) {
    for (int i = tid; i < 64 * LDS; i += kThreads)
        N[i] = 0.f;
    __syncthreads();
    if (tid < 64) {
        const int o = 16 * (tid >> 4), j = tid & 15;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < i; ++s)
                acc = fmaf(-A[(o + i) * LDS + o + s], col[s], acc);
            col[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            N[(o + i) * LDS + o + j] = col[i];
    }
    __syncthreads();
    for (int I = 1; I < 4; ++I) {
        for (int idx = tid; idx < 256 * I; idx += kThreads) {
            const int J = idx >> 8, ii = (idx >> 4) & 15, jj = idx & 15;
            float acc = 0.f;
            for (int K = J; K < I; ++K) {
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    acc = fmaf(A[(16 * I + ii) * LDS + 16 * K + s], N[(16 * K + s) * LDS + 16 * J + jj], acc);
            }
            R[ii * LDS + 16 * J + jj] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < 256 * I; idx += kThreads) {
            const int J = idx >> 8, ii = (idx >> 4) & 15, jj = idx & 15;
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < 16; ++s)
                acc = fmaf(N[(16 * I + ii) * LDS + 16 * I + s], R[s * LDS + 16 * J + jj], acc);
            N[(16 * I + ii) * LDS + 16 * J + jj] = -acc;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
template <int DK>
__global__ void __launch_bounds__(kThreads)
    chunk_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ beta, uint8_t *__restrict__ ws, int L, int C,
                      int nch, int nu, int Dp, float eps, unsigned *status) {
    constexpr int G = DK / 4, RPW = 32 / G, N2 = 2 * DK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *kq = smem;                          // [K; Q] tile, 128 x Dp bf16 K-major SW128
    float *Am = (float *)(smem + 256 * Dp);      // A, later P T
    float *Nm = Am + 64 * LDS;                   // (I + A)^-1, later T
    float *Pm = Nm + 64 * LDS;                   // tril_incl(Q K^T)
    float *Rm = Pm + 64 * LDS;                   // block-solve scratch [16][LDS]
    float *bs = Rm + 16 * LDS;                   // beta of the chunk (0 on padded rows)
    uint64_t *bar = (uint64_t *)(bs + 64);
    uint32_t *slot = (uint32_t *)(bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * C, Lc = min(C, L - t0);
    const int d_dot = N2 * nu;
    uint8_t *img = ws + ((size_t)bh * nch + c) * image_bytes(Dp);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 64);
        tmem_relinquish();
    }
    if (tid < 64)
        bs[tid] = tid < Lc ? __bfloat162float(beta[bh * L + t0 + tid]) : 0.f;

    // DPFP rows: r < 64 are keys, r >= 64 queries of token r & 63
    {
        const int g = lane % G, base_lane = lane - g;
        for (int r0 = 0; r0 < 128; r0 += 4 * RPW) {
            const int r = r0 + warp * RPW + lane / G;
            const int t = r & 63;
            const bool valid = t < Lc;
            const __nv_bfloat16 *src = (r < 64 ? k : q) + ((size_t)bh * L + t0 + (valid ? t : 0)) * DK;
            float x[8];
            dpfp_load_x<G>(src, g, valid, x);
            const float denom = dpfp_row_sum<G>(x, g, base_lane, nu) + eps;
            for (int i = 1; i <= nu; ++i) {
                float p[8];
                dpfp_block_dispatch<G>(x, p, g, base_lane, i);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    p[e] = __fdiv_rn(p[e], denom);
                const uint4 u = pack8(p);
                const uint32_t off = kmajor_chunk(r, (i - 1) * N2 + 8 * g, 128);
                *reinterpret_cast<uint4 *>(kq + off) = u;
                *reinterpret_cast<uint4 *>(img + off) = u;
            }
        }
        const int padc = (Dp - d_dot) / 8; // zero columns d_dot .. Dp-1
        for (int idx = tid; idx < 128 * padc; idx += kThreads) {
            const int r = idx / padc, m = d_dot + 8 * (idx % padc);
            const uint32_t off = kmajor_chunk(r, m, 128);
            *reinterpret_cast<uint4 *>(kq + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(img + off) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;

    // Gram: D[128 x 64] = [K; Q] K^T  (B = the first 64 rows of the same tile)
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
        const uint32_t base = smem_u32(kq);
        for (int s = 0; s < Dp / 16; ++s) {
            const uint64_t d = desc_sw128(base + kmajor_step(s, 128), 16, 1024);
            mma_bf16(tm, d, d, idesc, s > 0);
        }
        mma_commit(bar);
    }
    const bool ok = mbar_wait(bar, 0, status);
    tc_fence_after();
    const bool abort = __syncthreads_or(!ok);
    if (!abort) {
        float gr[16];
        for (int cb = 0; cb < 64; cb += 16) {
            tmem_ld16(tm + tmem_lane_base(warp) + (uint32_t)cb, gr);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s = cb + j;
                if (tid < 64)
                    Am[tid * LDS + s] = s < tid ? bs[tid] * gr[j] : 0.f;
                else
                    Pm[(tid - 64) * LDS + s] = s <= tid - 64 ? gr[j] : 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, 64);
    if (abort)
        return;

    unit_lower_inverse(Am, Nm, Rm, tid);
    for (int idx = tid; idx < 64 * 64; idx += kThreads) // T = (I + A)^-1 diag(beta)
        Nm[(idx >> 6) * LDS + (idx & 63)] *= bs[idx & 63];
    __syncthreads();
    {   // P T (both lower triangular) into Am
        const int i = tid & 63, j0 = (tid >> 6) * 32;
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            acc[j] = 0.f;
        for (int kk = j0; kk < 64; ++kk) {
            const float p = Pm[i * LDS + kk];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                acc[j] = fmaf(p, Nm[kk * LDS + j0 + j], acc[j]);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 32; ++j)
            Am[i * LDS + j0 + j] = acc[j];
    }
    __syncthreads();
    {   // [T; P T] image, bf16 K-major SW128 (one 64-column block)
        const float *src = tid < 64 ? Nm + tid * LDS : Am + (tid - 64) * LDS;
        uint8_t *tp = img + 256 * Dp;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v8[e] = src[8 * cc + e];
            *reinterpret_cast<uint4 *>(tp + kmajor_chunk(tid, 8 * cc, 128)) = pack8(v8);
        }
    }
}

// ---------------------------------------------------------------------------
// Row `row` of an MN-major SW128 operand tile whose rows are the contraction
// index and whose columns are value channels (64-column blocks `blk` bytes
// apart): write n values v[0..n) as bf16.
template <int DVB>
FW_DEV void write_vrow(uint8_t *tile, int row, const float *v, uint32_t blk) {
#pragma unroll
    for (int j0 = 0; j0 < DVB; j0 += 8) {
        const uint32_t off = (uint32_t)(j0 >> 6) * blk + (uint32_t)row * 128u +
                             ((uint32_t)(((j0 & 63) >> 3) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(tile + off) = pack8(v + j0);
    }
}

template <int DVB>
FW_DEV void tmem_ld_row(uint32_t taddr, float *r) {
#pragma unroll
    for (int j0 = 0; j0 < DVB; j0 += 16)
        tmem_ld16(taddr + (uint32_t)j0, r + j0);
}

template <int DVB>
__global__ void __launch_bounds__(kThreads)
    chunk_scan_kernel(const __nv_bfloat16 *__restrict__ v, const float *W0, float *Wf,
                      __nv_bfloat16 *__restrict__ y, const uint8_t *__restrict__ ws, int L, int C,
                      int nch, int d_v, int d_dot, int Dp, unsigned *status) {
    constexpr int VB = (DVB + 63) / 64;         // 64-column blocks of the value tiles
    constexpr int DS = DVB < 32 ? 32 : DVB;     // TMEM columns per accumulator region
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t kq_bytes = 256u * (uint32_t)Dp;
    const uint32_t img_bytes = kq_bytes + kTpBytes;
    uint8_t *kq = smem;                                  // [K; Q]  128 x Dp
    uint8_t *tp = kq + kq_bytes;                         // [T; P T] 128 x 64
    uint8_t *st = tp + kTpBytes;                         // S: rows d, columns v (MN-major)
    uint8_t *xt = st + (size_t)VB * Dp * 128;            // X: rows t, columns v
    uint8_t *ut = xt + VB * 8192;                        // U: rows t, columns v
    uint64_t *bar_load = (uint64_t *)(ut + VB * 8192);
    uint64_t *bar_mma = bar_load + 1;
    uint32_t *slot = (uint32_t *)(bar_mma + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int v0 = blockIdx.x * DVB;
    const int64_t bh = blockIdx.y;
    const int MB = Dp / 128;
    const int need = (2 + MB) * DS;
    const uint32_t ncols = need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
    const uint8_t *img0 = ws + (size_t)bh * nch * img_bytes;
    const bool has_w0 = W0 != nullptr;
    const uint32_t lb = tmem_lane_base(warp);

    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;
    const uint32_t tD1 = tm, tD2 = tm + DS, tS = tm + 2 * DS;
    const uint32_t kq_s = smem_u32(kq), tp_s = smem_u32(tp), st_s = smem_u32(st), xt_s = smem_u32(xt),
                   ut_s = smem_u32(ut);

    if (tid == 0) { // chunk 0's operand images
        mbar_arrive_expect_tx(bar_load, img_bytes);
        bulk_g2s(kq, img0, kq_bytes, bar_load);
        bulk_g2s(tp, img0 + kq_bytes, kTpBytes, bar_load);
    }
    // initial state: S^T in TMEM (fp32) and S as the bf16 operand of MMA1
    for (int mb = 0; mb < MB; ++mb) {
        const int d = 128 * mb + tid;
        float w[DVB];
#pragma unroll
        for (int j = 0; j < DVB; ++j)
            w[j] = (has_w0 && d < d_dot) ? W0[((size_t)bh * d_v + v0 + j) * d_dot + d] : 0.f;
        if (has_w0) {
#pragma unroll
            for (int j0 = 0; j0 < DVB; j0 += 16)
                tmem_st16(tS + (uint32_t)(mb * DS + j0) + lb, w + j0);
        }
        write_vrow<DVB>(st, d, w, (uint32_t)Dp * 128u);
    }
    if (has_w0)
        tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    uint32_t mma_phase = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * C, Lc = min(C, L - t0);
        float vrow[DVB];
        if (tid < 64) { // value rows of this chunk (zero on padded rows)
            if (tid < Lc) {
                const __nv_bfloat16 *src = v + ((size_t)bh * L + t0 + tid) * d_v + v0;
#pragma unroll
                for (int j0 = 0; j0 < DVB; j0 += 8) {
                    float tmp[8];
                    load8(src + j0, tmp);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        vrow[j0 + e] = tmp[e];
                }
            } else {
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    vrow[j] = 0.f;
            }
        }
        bool ok = mbar_wait(bar_load, (uint32_t)(c & 1), status);
        if (__syncthreads_or(!ok))
            break;

        // MMA1: D1 = [K; Q] S^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, DVB, 0, 1);
            for (int s = 0; s < Dp / 16; ++s)
                mma_bf16(tD1, desc_sw128(kq_s + kmajor_step(s, 128), 16, 1024),
                         desc_sw128(st_s + (uint32_t)s * 2048u, (uint32_t)Dp * 128u, 1024), idesc, s > 0);
            mma_commit(bar_mma);
        }
        ok = mbar_wait(bar_mma, mma_phase, status);
        mma_phase ^= 1;
        if (__syncthreads_or(!ok))
            break;
        tc_fence_after();
        float qs[DVB]; // warps 2-3: Q S^T of token tid - 64
        {
            float d1[DVB];
            tmem_ld_row<DVB>(tD1 + lb, d1);
            tmem_ld_wait();
            if (tid < 64) {
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    d1[j] = vrow[j] - d1[j]; // X = V - K S^T
                write_vrow<DVB>(xt, tid, d1, 8192u);
            } else {
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    qs[j] = d1[j];
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // MMA2: D2 = [T; P T] X
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, DVB, 0, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tD2, desc_sw128(tp_s + (uint32_t)s * 32u, 16, 1024),
                         desc_sw128(xt_s + (uint32_t)s * 2048u, 8192, 1024), idesc, s > 0);
            mma_commit(bar_mma);
        }
        ok = mbar_wait(bar_mma, mma_phase, status);
        mma_phase ^= 1;
        if (__syncthreads_or(!ok))
            break;
        tc_fence_after();
        {
            float d2[DVB];
            tmem_ld_row<DVB>(tD2 + lb, d2);
            tmem_ld_wait();
            if (tid < 64) {
                write_vrow<DVB>(ut, tid, d2, 8192u); // U
            } else if (tid - 64 < Lc) {             // y = Q S^T + P U
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    d2[j] += qs[j];
                __nv_bfloat16 *dst = y + ((size_t)bh * L + t0 + (tid - 64)) * d_v + v0;
#pragma unroll
                for (int j0 = 0; j0 < DVB; j0 += 8)
                    *reinterpret_cast<uint4 *>(dst + j0) = pack8(d2 + j0);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // MMA3: S^T += K^T U  (K^T: the key rows of the [K; Q] tile read MN-major)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, DVB, 1, 1);
            for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tS + (uint32_t)(mb * DS),
                             desc_sw128(kq_s + (uint32_t)(2 * mb) * 16384u + (uint32_t)s * 2048u, 16384, 1024),
                             desc_sw128(ut_s + (uint32_t)s * 2048u, 8192, 1024), idesc,
                             (s > 0 || c > 0 || has_w0) ? 1u : 0u);
            mma_commit(bar_mma);
        }
        ok = mbar_wait(bar_mma, mma_phase, status);
        mma_phase ^= 1;
        if (__syncthreads_or(!ok))
            break;
        tc_fence_after();
        if (tid == 0 && c + 1 < nch) { // the tiles are consumed: fetch the next chunk's
            const uint8_t *img = img0 + (size_t)(c + 1) * img_bytes;
            mbar_arrive_expect_tx(bar_load, img_bytes);
            bulk_g2s(kq, img, kq_bytes, bar_load);
            bulk_g2s(tp, img + kq_bytes, kTpBytes, bar_load);
        }
        for (int mb = 0; mb < MB; ++mb) {
            const int d = 128 * mb + tid;
            float sv[DVB];
            tmem_ld_row<DVB>(tS + (uint32_t)(mb * DS) + lb, sv);
            tmem_ld_wait();
            if (c + 1 < nch) {
                write_vrow<DVB>(st, d, sv, (uint32_t)Dp * 128u);
            } else if (Wf && d < d_dot) {
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    Wf[((size_t)bh * d_v + v0 + j) * d_dot + d] = sv[j];
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, ncols);
}

// ---------------------------------------------------------------- host side
size_t prep_smem(int Dp) { return (size_t)256 * Dp + (3 * 64 + 16) * LDS * 4 + 64 * 4 + 16 + 1024; }

size_t scan_smem(int Dp, int dvb) {
    const int VB = (dvb + 63) / 64;
    return (size_t)256 * Dp + kTpBytes + (size_t)VB * Dp * 128 + 2 * (size_t)VB * 8192 + 32 + 1024;
}

int tmem_cols(int Dp, int dvb) { return (2 + Dp / 128) * (dvb < 32 ? 32 : dvb); }

constexpr size_t kMaxSmem = 227 * 1024;

bool fits(int Dp, int dvb) {
    return scan_smem(Dp, dvb) <= kMaxSmem && prep_smem(Dp) <= kMaxSmem && tmem_cols(Dp, dvb) <= 512;
}

// Channels per scan CTA: 16 spreads the serial chunk walk over the most CTAs;
// 32 only when 16 would exceed two CTAs per SM.
int choose_dvb(int BH, int d_v, int Dp, int num_sms) {
    int dvb = 16;
    while (dvb < d_v && dvb < 32 && (int64_t)BH * (d_v / dvb) > 2 * (int64_t)num_sms && fits(Dp, 2 * dvb))
        dvb *= 2;
    return dvb;
}

template <int DK>
cudaError_t launch_prep(const void *q, const void *k, const void *beta, uint8_t *ws, int BH, int L, int C,
                        int nch, int nu, int Dp, float eps, unsigned *status, cudaStream_t st) {
    const size_t smem = prep_smem(Dp);
    auto kern = chunk_prep_kernel<DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<dim3((unsigned)nch, (unsigned)BH), kThreads, smem, st>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(beta), ws, L, C, nch, nu, Dp, eps, status);
    return cudaGetLastError();
}

template <int DVB>
cudaError_t launch_scan(const void *v, const float *W0, float *Wf, void *y, const uint8_t *ws, int BH, int L,
                        int C, int nch, int d_v, int d_dot, int Dp, unsigned *status, cudaStream_t st) {
    const size_t smem = scan_smem(Dp, DVB);
    auto kern = chunk_scan_kernel<DVB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<dim3((unsigned)(d_v / DVB), (unsigned)BH), kThreads, smem, st>>>(
        static_cast<const __nv_bfloat16 *>(v), W0, Wf, static_cast<__nv_bfloat16 *>(y), ws, L, C, nch, d_v,
        d_dot, Dp, status);
    return cudaGetLastError();
}

} // namespace

bool tc_forward_supported(int d_key, int nu, int d_v, int chunk) {
    if (!(d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128))
        return false;
    if (!(d_v == 16 || d_v == 32 || d_v == 64 || d_v == 128))
        return false;
    if (chunk < 1 || chunk > kTile)
        return false;
    const int Dp = padded_ddot(2 * d_key * nu);
    return fits(Dp, 16);
}

size_t tc_forward_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk) {
    (void)d_v;
    const int nch = (L + chunk - 1) / chunk;
    return (size_t)B * H * nch * image_bytes(padded_ddot(2 * d_key * nu));
}

cudaError_t tc_forward_launch(const void *q, const void *k, const void *v, const void *beta,
                              const float *W0, float *W_final, void *y, void *workspace, int B,
                              int H, int L, int d_key, int nu, int d_v, int chunk, float eps,
                              int num_sms, unsigned *status, cudaStream_t st) {
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const int Dp = padded_ddot(d_dot);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    switch (d_key) {
    case 8: e = launch_prep<8>(q, k, beta, ws, BH, L, chunk, nch, nu, Dp, eps, status, st); break;
    case 16: e = launch_prep<16>(q, k, beta, ws, BH, L, chunk, nch, nu, Dp, eps, status, st); break;
    case 32: e = launch_prep<32>(q, k, beta, ws, BH, L, chunk, nch, nu, Dp, eps, status, st); break;
    case 64: e = launch_prep<64>(q, k, beta, ws, BH, L, chunk, nch, nu, Dp, eps, status, st); break;
    case 128: e = launch_prep<128>(q, k, beta, ws, BH, L, chunk, nch, nu, Dp, eps, status, st); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess)
        return e;
    const int dvb = choose_dvb(BH, d_v, Dp, num_sms);
    switch (dvb) {
    case 16: return launch_scan<16>(v, W0, W_final, y, ws, BH, L, chunk, nch, d_v, d_dot, Dp, status, st);
    case 32: return launch_scan<32>(v, W0, W_final, y, ws, BH, L, chunk, nch, d_v, d_dot, Dp, status, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace fw
