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
//   A  = strict_lower(diag(beta) K K^T),   T = (I + A)^-1 diag(beta)
//   U  = T (V - K S^T)                     (the C write vectors u_t)
//   Y  = Q S^T + P U,  P = tril_incl(Q K^T) (reads use the updated W)
//   S <- S + U^T K
// This is the WY / "UT transform" form of a product of Householder-like
// factors (Bischof and Van Loan 1987; Joffrain et al. 2006; applied to the
// delta rule by Yang et al. 2024), written here from the algebra above.
// Everything that does not involve S is moved out of the serial chain:
//   W' = T K,  U' = T V,  Q' = Q - P W',  Y' = P U'
//   =>  U = U' - W' S^T,   Y = Y' + Q' S^T,   S <- S + U^T K,
// so one MMA, [W'; Q'] S^T, gives what both U and Y need.
//
// Two kernels:
//  * chunk_prep_kernel, one CTA of 256 threads per (chunk, batch*head), all
//    chunks in parallel: DPFP of the chunk's k and q rows straight into a
//    128 x Dp bf16 operand tile [K; Q] (the shuffle-based roll of the
//    standalone DPFP kernel); tcgen05 MMA [K; Q] K^T for the Gram matrix and
//    Q K^T; (I + A)^-1 by 16 x 16 block forward substitution in fp32 on CUDA
//    cores; tcgen05 MMA [I; P] T = [T; P T]; tcgen05 MMA [T; P T] [K | V] =
//    [W', P W' | U', Y'].  It writes one record per chunk to the workspace:
//    the [W'; Q'] and K tiles as byte images of the swizzled shared-memory
//    operands the scan uses, and U', Y' in fp32.
//  * chunk_scan_kernel, one CTA of 128 threads per (block of DVB value
//    channels, batch*head): rows of W evolve independently, so the state is
//    split by value channel.  Per chunk, in order:
//      MMA1  D1 = [W'; Q'] S^T     -> U = U' - D1[0:64] (bf16 tile),
//                                     y = Y' + D1[64:128] (stored)
//      MMA3  S^T += K^T U           (fp32 state resident in tensor memory)
//      S^T -> bf16 operand tile for the next MMA1
//    The [W'; Q'] image of chunk c+1 is bulk-copied in as soon as MMA1 has
//    read chunk c's; K images are double-buffered, two chunks ahead.
//    The serial walk is bound by how fast MMAs issue: one thread issues a
//    tcgen05.mma about every 80 SM cycles whatever N (up to 128), while two
//    or more warps issuing at once reach about 44 cycles each in aggregate.
//    So MMA1 is issued by two threads (warps 0 and 1), each over half of the
//    contraction into its own accumulator (the read-out adds the two), and
//    MMA3 by one thread per 128-row block of S^T (warp mb).  Every
//    accumulator is written by one thread only, so no two threads' MMAs
//    ever need ordering against each other.
//
// Partial chunks are padded to 64 token rows with zero phi rows and
// beta = 0, which makes the padded rows of T, P, W', Q', U' and Y' zero.
#include "fw_dpfp.cuh"
#include "fw_forward_tc.h"
#include "fw_tc.cuh"

namespace fw {
namespace {

using namespace tc;

constexpr int kTile = 64;          // token rows of a chunk tile (chunk <= 64, padded)
constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 128;
constexpr int LDS = 68;            // fp32 row stride of the 64 x 64 work matrices (16-byte rows)
constexpr int kMaxDp = 384;        // padded d_dot the scan's shared memory holds

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ inline int padded_ddot(int d_dot) { return round_up(d_dot, 128); }

// One chunk's record in the workspace (byte offsets; all 1024-aligned).
struct Record {
    size_t a, k, up, yp, bytes;
};
__host__ __device__ inline Record record_layout(int Dp, int d_v) {
    Record r;
    r.a = 0;                                // [W'; Q']: 128 x Dp bf16, K-major SW128
    r.k = (size_t)256 * Dp;                 // K: 64 x Dp bf16, K-major SW128 (64-row blocks)
    r.up = r.k + (size_t)128 * Dp;          // U': 64 x d_v fp32, [d_v/4][64 rows][4 channels]
    r.yp = r.up + (size_t)256 * d_v;        // Y': 64 x d_v fp32, same layout
    r.bytes = r.yp + (size_t)256 * d_v;
    return r;
}

// First 1024-byte boundary at or after the dynamic shared-memory base.  The
// result is the base plus an offset, never a pointer rebuilt from an integer,
// so the compiler still knows it addresses shared memory and emits shared
// (not generic) loads and stores through it.
FW_DEV uint8_t *align1024(uint8_t *p) { return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u); }

FW_DEV uint4 pack8(const float *v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    return u;
}

FW_DEV void unpack8(uint4 u, float *v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

FW_DEV uint32_t tmem_cols_pow2(int need) {
    return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// ---------------------------------------------------------------------------
// Element offset helpers of the T operand tile (rows k, columns n; MN-major,
// 128-byte rows, 16-byte chunks swizzled by k & 7).
FW_DEV uint32_t ttile_chunk(int kk, int n) { return (uint32_t)kk * 128u + ((uint32_t)((n >> 3) ^ (kk & 7)) << 4); }

// (I + A)^-1 for a strictly lower 64 x 64 A, by 16 x 16 blocks:
//   diagonal blocks by forward substitution (one column per thread), then
//   block row I: N_IJ = -N_II * sum_{K=J}^{I-1} A_IK N_KJ   (J < I).
// A, N: [64][LDS]; R: [16][LDS] scratch; all 16-byte aligned.  Only the
// blocks on and below the diagonal of N are written (the ones above are
// zero and never read here).  As each block of N is final it also goes out,
// times beta of its column, in bf16 to the T operand tile tt (T = N diag(beta));
// the blocks above the diagonal are written as zeros.  NT threads (>= 256);
// ends synchronised.
template <int NT>
FW_DEV void unit_lower_inverse(const float *A, float *N, float *R, const float *bs, uint8_t *tt, int tid) {
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
        const float bj = bs[o + j];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            N[(o + i) * LDS + o + j] = col[i];
            *reinterpret_cast<__nv_bfloat16 *>(tt + ttile_chunk(o + i, o + j) + 2 * (j & 7)) =
                __float2bfloat16_rn(col[i] * bj);
        }
    } else if (tid < 64 + 192) { // zero chunks of the 6 blocks above the diagonal
        const int idx = tid - 64, blk = idx >> 5;
        const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const int kk = 16 * I + ((idx & 31) >> 1), n0 = 16 * J + 8 * (idx & 1);
        *reinterpret_cast<uint4 *>(tt + ttile_chunk(kk, n0)) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // off-diagonal blocks; each thread computes 4 adjacent outputs of a row
    // from 16-byte loads, so every A (or N) element it loads feeds 4 FMAs
    for (int I = 1; I < 4; ++I) {
        for (int idx = tid; idx < 64 * I; idx += NT) {
            const int J = idx >> 6, ii = (idx >> 2) & 15, j0 = 16 * J + 4 * (idx & 3);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int K = J; K < I; ++K) {
                const float *ar = A + (16 * I + ii) * LDS + 16 * K;
#pragma unroll
                for (int s4 = 0; s4 < 16; s4 += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(ar + s4);
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 n = *reinterpret_cast<const float4 *>(N + (16 * K + s4 + e) * LDS + j0);
                        acc.x = fmaf(av[e], n.x, acc.x);
                        acc.y = fmaf(av[e], n.y, acc.y);
                        acc.z = fmaf(av[e], n.z, acc.z);
                        acc.w = fmaf(av[e], n.w, acc.w);
                    }
                }
            }
            *reinterpret_cast<float4 *>(R + ii * LDS + j0) = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < 64 * I; idx += NT) {
            const int ii = (idx >> 2) & 15, j0 = 16 * (idx >> 6) + 4 * (idx & 3);
            const float *nr = N + (16 * I + ii) * LDS + 16 * I;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int s4 = 0; s4 < 16; s4 += 4) {
                const float4 nn = *reinterpret_cast<const float4 *>(nr + s4);
                const float nv[4] = {nn.x, nn.y, nn.z, nn.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 r = *reinterpret_cast<const float4 *>(R + (s4 + e) * LDS + j0);
                    acc.x = fmaf(nv[e], r.x, acc.x);
                    acc.y = fmaf(nv[e], r.y, acc.y);
                    acc.z = fmaf(nv[e], r.z, acc.z);
                    acc.w = fmaf(nv[e], r.w, acc.w);
                }
            }
            const int kk = 16 * I + ii;
            *reinterpret_cast<float4 *>(N + kk * LDS + j0) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
            uint2 t4;
            t4.x = pack_bf16x2(-acc.x * bs[j0], -acc.y * bs[j0 + 1]);
            t4.y = pack_bf16x2(-acc.z * bs[j0 + 2], -acc.w * bs[j0 + 3]);
            *reinterpret_cast<uint2 *>(tt + ttile_chunk(kk, j0) + 2 * (j0 & 7)) = t4;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// DPFP of one row of the [K; Q] tile by two threads (d_key <= 64).  Row x =
// ReLU([k, -k]) has n = 2 DK entries; the thread with hs = 0 owns
// x[0 .. DK-1] = ReLU(k), the one with hs = 1 owns x[DK .. n-1] = ReLU(-k)
// (the same DK raw values, opposite sign).  Block i of phi needs
// x[j] * x[(j - i) mod n] (torch.roll(shifts=i), DPFP source of the Fast
// Weights Transformer guide), so besides its own half the thread builds the
// NUMAX entries that precede it around the row: going back h places from
// the start of a half crosses ceil(h / DK) half boundaries (each one flips
// the sign) and lands on raw index (-h) mod DK.  Every index is static and
// every product a register operation; the two halves of a row add their
// sums with one shuffle (partner lane ^ 8).
template <int DK, int NUMAX>
FW_DEV void dpfp_half_row(const uint4 (&raw)[DK / 8], int hs, int r, int nu, float eps, uint8_t *kq) {
    constexpr int N2 = 2 * DK;
    const float sg = hs ? -1.f : 1.f;
    float kf[DK];
#pragma unroll
    for (int c8 = 0; c8 < DK / 8; ++c8)
        unpack8(raw[c8], kf + 8 * c8);
    float xs[NUMAX + DK]; // xs[NUMAX + t] = x[hs DK + t],  xs[NUMAX - h] = x[(hs DK - h) mod n]
#pragma unroll
    for (int h = 1; h <= NUMAX; ++h) {
        const int m = (DK - h % DK) % DK;               // raw index (static)
        const bool flip = ((h + DK - 1) / DK) & 1;      // odd number of half boundaries crossed
        xs[NUMAX - h] = fmaxf((flip ? -sg : sg) * kf[m], 0.f);
    }
#pragma unroll
    for (int t = 0; t < DK; ++t)
        xs[NUMAX + t] = fmaxf(sg * kf[t], 0.f);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 1; i <= NUMAX; ++i) {
        if (i <= nu) {
#pragma unroll
            for (int t = 0; t < DK; ++t)
                acc[t & 3] = fmaf(xs[NUMAX + t], xs[NUMAX + t - i], acc[t & 3]);
        }
    }
    float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 8);
    const float inv = 1.0f / (sum + eps);
#pragma unroll
    for (int i = 1; i <= NUMAX; ++i) {
        if (i <= nu) {
#pragma unroll
            for (int c8 = 0; c8 < DK / 8; ++c8) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    p[e] = (xs[NUMAX + 8 * c8 + e] * xs[NUMAX + 8 * c8 + e - i]) * inv;
                *reinterpret_cast<uint4 *>(kq + kmajor_chunk(r, (i - 1) * N2 + hs * DK + 8 * c8, 128)) = pack8(p);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// SUM = false: the delta rule.  SUM = true: the sum rule (linear attention):
// W' = 0, Q' = Q, U' = V', Y' = P V' with V' = V (d_vr channels) followed,
// when d_v > d_vr, by a 16-channel block whose first channel is 1 on every
// token (its running sum is z, its output the denominator z . phi(q)).  The
// scan is the same for both rules.
template <int DK, bool SUM>
__global__ void __launch_bounds__(kPrepThreads, 2)
    chunk_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ beta,
                      uint8_t *__restrict__ ws, int L, int C, int nch, int nu, int Dp, int d_v, int d_vr,
                      float eps, unsigned *status) {
    constexpr int G = DK / 4, RPW = 32 / G, N2 = 2 * DK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *kq = smem;                                  // [K; Q]: 128 x Dp, K-major
    uint8_t *ip = kq + 256 * Dp;                         // [I; P]: 128 x 64, K-major A
    uint8_t *tp = ip;                                    // [T; P T] replaces [I; P] once read
    uint8_t *tt = ip + 16384;                            // T: rows k, columns n (MN-major B)
    float *Am = (float *)(tt + 8192);                    // A = strict_lower(beta K K^T)
    float *Nm = Am + 64 * LDS;                           // (I + A)^-1
    float *Rm = Nm + 64 * LDS;                           // block-solve scratch [16][LDS]
    float *bs = Rm + 16 * LDS;                           // beta (0 on padded rows)
    uint8_t *vt = (uint8_t *)Am;                         // V (MN-major B), once A and N are done
    // MMA completion: the Gram matrix (2 issuers), [I; P] T (2 issuers; the
    // sum rule's [I; P] V' by 1), the final product (one issuer per accumulator)
    uint64_t *bar_g = (uint64_t *)(bs + 64);
    uint64_t *bar_i = bar_g + 1;
    uint64_t *bar_f = bar_g + 2;
    uint32_t *slot = (uint32_t *)(bar_g + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sp = warp & 3, half = warp >> 2;           // TMEM sub-partition, column half
    const int row = 32 * sp + lane;                      // accumulator row of this thread
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * C, Lc = min(C, L - t0);
    const int d_dot = N2 * nu;
    const Record rc = record_layout(Dp, d_v);
    uint8_t *rec = ws + ((size_t)bh * nch + c) * rc.bytes;
    const uint32_t ncols = tmem_cols_pow2(max(64, Dp + d_v));

    // This chunk's q, k and v rows are pulled into L2 while the preceding
    // kernel finishes (a prefetch is safe before the wait: see l2_prefetch).
    if (tid == 0) {
        const size_t tok = (size_t)bh * L + t0;
        l2_prefetch(k + tok * DK, (uint32_t)(Lc * DK * 2));
        l2_prefetch(q + tok * DK, (uint32_t)(Lc * DK * 2));
        if ((d_vr * 2) % 16 == 0)
            l2_prefetch(v + tok * d_vr, (uint32_t)(Lc * d_vr * 2));
    }
    griddep_wait(); // the inputs may be, and the workspace may still be read by, the preceding kernel
    q = after_wait(q);
    k = after_wait(k);
    v = after_wait(v);
    beta = after_wait(beta);
    // Only now may the scan start its prologue (on free SMs): it reads the
    // caller's W0 before its own wait, which is safe once everything enqueued
    // before this kernel has completed, as it has here.
    griddep_launch_dependents();
    // Global loads first, all in flight before any is used: the key and query
    // rows for the DPFP, the chunk's V rows (kept in registers until their
    // tile's space is free) and beta (stored to shared memory after the DPFP).
    constexpr bool kHalfRows = DK <= 64;
    constexpr int kRaw = kHalfRows ? DK / 8 : 128 / (8 * RPW);
    uint4 raw[kRaw];
    // kHalfRows: thread = (row r, half hs of x); lanes l and l ^ 8 share a row
    const int hs = (lane >> 3) & 1;
    const int hr = 16 * warp + ((lane & 7) | ((lane >> 4) << 3));
    if constexpr (kHalfRows) {
        const int t = hr & 63;
        const __nv_bfloat16 *src = (hr < 64 ? k : q) + ((size_t)bh * L + t0 + t) * DK;
#pragma unroll
        for (int c8 = 0; c8 < kRaw; ++c8)
            raw[c8] = t < Lc ? __ldcg(reinterpret_cast<const uint4 *>(src) + c8) : make_uint4(0, 0, 0, 0);
    } else {
        const int g = lane % G;
#pragma unroll
        for (int ps = 0; ps < kRaw; ++ps) {
            const int r = ps * 8 * RPW + warp * RPW + lane / G;
            const int t = r & 63;
            raw[ps] = make_uint4(0, 0, 0, 0);
            if (t < Lc)
                raw[ps] = __ldcg(reinterpret_cast<const uint4 *>((r < 64 ? k : q) + ((size_t)bh * L + t0 + t) * DK +
                                                               8 * (g % (G / 2))));
        }
    }
    constexpr int kVChunks = 4; // 64 * 128 / 8 / kPrepThreads
    uint4 vpre[kVChunks];
    const int vcpr = d_vr / 8;
#pragma unroll
    for (int i = 0; i < kVChunks; ++i) {
        const int idx = tid + i * kPrepThreads, t = idx / vcpr, j = 8 * (idx % vcpr);
        vpre[i] = make_uint4(0, 0, 0, 0);
        if (idx < 64 * vcpr && t < Lc)
            vpre[i] = __ldcg(reinterpret_cast<const uint4 *>(v + ((size_t)bh * L + t0 + t) * d_vr + j));
    }
    float beta_t = 0.f;
    if (!SUM && tid < Lc && tid < 64)
        beta_t = __bfloat162float(beta[bh * L + t0 + tid]);

    if (tid == 0) {
        mbar_init(bar_g, 2);
        mbar_init(bar_i, SUM ? 1 : 2);
        mbar_init(bar_f, (uint32_t)(Dp / 128 + 1));
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, ncols);
        tmem_relinquish();
    }
    // DPFP rows: r < 64 are keys, r >= 64 queries of token r & 63.
    if constexpr (kHalfRows) {
        dpfp_half_row<DK, kMaxDp / (2 * DK)>(raw, hs, hr, nu, eps, kq);
    } else {
        const int g = lane % G, base_lane = lane - g;
#pragma unroll
        for (int ps = 0; ps < kRaw; ++ps) {
            const int r = ps * 8 * RPW + warp * RPW + lane / G;
            float x[8];
            {
                float kv[8];
                unpack8(raw[ps], kv);
                const bool neg = g >= G / 2;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = fmaxf(neg ? -kv[e] : kv[e], 0.f);
            }
            dpfp_row_emit<G, 3>(x, g, base_lane, nu, eps, [&](int i, float (&p)[8]) {
                *reinterpret_cast<uint4 *>(kq + kmajor_chunk(r, (i - 1) * N2 + 8 * g, 128)) = pack8(p);
            });
        }
    }
    {
        const int padc = (Dp - d_dot) / 8; // zero columns d_dot .. Dp-1
        for (int idx = tid; idx < 128 * padc; idx += kPrepThreads) {
            const int r = idx / padc, m = d_dot + 8 * (idx % padc);
            *reinterpret_cast<uint4 *>(kq + kmajor_chunk(r, m, 128)) = make_uint4(0, 0, 0, 0);
        }
    }
    if (tid < 64)
        bs[tid] = beta_t; // 0 on padded rows
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;
    const uint32_t lb = tmem_lane_base(warp);
    // MMAs are issued by lane 0 of several warps at once (one thread issues a
    // tcgen05.mma about every 80 SM cycles; several warps together reach
    // about 44 each), every accumulator by one thread only
    const bool lead = lane == 0;

    // MMA: [K; Q] K^T  (B = the first 64 rows of the same tile), warp 0 over
    // the first half of the contraction into columns 0..63, warp 1 over the
    // second into 64..127.  The key rows of the tile are final here and go
    // out as the record's K image (bulk copies of the 64-row halves of each
    // 64-column block) while the rest of the chunk is worked out.
    if (tid == 0) {
        for (int kb = 0; kb < Dp / 64; ++kb)
            bulk_s2g(rec + rc.k + (size_t)kb * 8192, kq + (size_t)kb * 16384, 8192);
        bulk_commit();
    }
    if (lead && warp < 2) {
        const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
        const uint32_t base = smem_u32(kq);
        const int s0 = warp * (Dp / 32);
        for (int s = s0; s < s0 + Dp / 32; ++s) {
            const uint64_t d = desc_sw128(base + kmajor_step(s, 128), 16, 1024);
            mma_bf16(tm + (uint32_t)(64 * warp), d, d, idesc, s > s0);
        }
        mma_commit(bar_g);
    }
    bool ok = mbar_wait(bar_g, 0, status);
    tc_fence_after();
    if (__syncthreads_or(!ok))
        goto teardown;
    {   // A (keys) and P (queries); [I; P] operand tile
        float gr[32], g2[32];
        tmem_ld16(tm + lb + (uint32_t)(32 * half), gr);
        tmem_ld16(tm + lb + (uint32_t)(32 * half + 16), gr + 16);
        tmem_ld16(tm + lb + (uint32_t)(64 + 32 * half), g2);
        tmem_ld16(tm + lb + (uint32_t)(64 + 32 * half + 16), g2 + 16);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
            gr[j] += g2[j];
        if (SUM && row < 64) { // the I row only (no triangular solve)
#pragma unroll
            for (int j = 0; j < 32; ++j)
                gr[j] = 32 * half + j == row ? 1.f : 0.f;
        } else if (row < 64) { // A row (16-byte stores; rows are 16-byte aligned) and the I row
            const float br = bs[row];
#pragma unroll
            for (int j4 = 0; j4 < 32; j4 += 4) {
                float a4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 32 * half + j4 + e;
                    a4[e] = s < row ? br * gr[j4 + e] : 0.f;
                    gr[j4 + e] = s == row ? 1.f : 0.f;
                }
                *reinterpret_cast<float4 *>(Am + row * LDS + 32 * half + j4) = make_float4(a4[0], a4[1], a4[2], a4[3]);
            }
        } else {        // P row: Q K^T on and below the diagonal
#pragma unroll
            for (int j = 0; j < 32; ++j)
                gr[j] = 32 * half + j <= row - 64 ? gr[j] : 0.f;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            *reinterpret_cast<uint4 *>(ip + kmajor_chunk(row, 32 * half + 8 * cc, 128)) = pack8(gr + 8 * cc);
    }
    tc_fence_before();
    __syncthreads();

    if constexpr (SUM) {
        // V' (values, then the ones block when normalising) into the A / N space
        // as the MN-major B operand, then [I; P] V' = [V'; P V'] = [U'; Y'].
#pragma unroll
        for (int i = 0; i < kVChunks; ++i) {
            const int idx = tid + i * kPrepThreads, t = idx / vcpr, j = 8 * (idx % vcpr);
            if (idx < 64 * vcpr)
                *reinterpret_cast<uint4 *>(vt + (uint32_t)(j >> 6) * 8192u + (uint32_t)t * 128u +
                                           ((uint32_t)(((j & 63) >> 3) ^ (t & 7)) << 4)) = vpre[i];
        }
        if (d_v > d_vr && tid < 128) { // channel d_vr = 1 on the chunk's tokens, the rest of the block 0
            const int t = tid >> 1, j = d_vr + 8 * (tid & 1);
            const uint4 one = make_uint4((tid & 1) == 0 && t < Lc ? 0x3f80u : 0u, 0, 0, 0); // bf16 1.0 in the low half
            *reinterpret_cast<uint4 *>(vt + (uint32_t)(j >> 6) * 8192u + (uint32_t)t * 128u +
                                       ((uint32_t)(((j & 63) >> 3) ^ (t & 7)) << 4)) = one;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a = smem_u32(ip), bv = smem_u32(vt);
            const uint32_t idv = idesc_bf16(128, d_v, 0, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tm + (uint32_t)Dp, desc_sw128(a + (uint32_t)s * 32u, 16, 1024),
                         desc_sw128(bv + (uint32_t)s * 2048u, 8192, 1024), idv, s > 0);
            mma_commit(bar_i);
            bulk_wait_read(); // the K image has been read out of the key rows
        }
        ok = mbar_wait(bar_i, 0, status);
        tc_fence_after();
        if (__syncthreads_or(!ok))
            goto teardown;
        // Record out: [W'; Q'] = [0; Q] (the key rows of the tile zeroed)
        const int cpr = Dp / 8;
        for (int idx = tid; idx < 64 * cpr; idx += kPrepThreads)
            *reinterpret_cast<uint4 *>(kq + kmajor_chunk(idx / cpr, 8 * (idx % cpr), 128)) = make_uint4(0, 0, 0, 0);
    } else {
        // (I + A)^-1, and T = (I + A)^-1 diag(beta) as the MN-major operand tile
        // (rows k, columns n); ends synchronised, so A and N's space is free for V
        unit_lower_inverse<kPrepThreads>(Am, Nm, Rm, bs, tt, tid);
    #pragma unroll
        for (int i = 0; i < kVChunks; ++i) {
            const int idx = tid + i * kPrepThreads, t = idx / vcpr, j = 8 * (idx % vcpr);
            if (idx < 64 * vcpr)
                *reinterpret_cast<uint4 *>(vt + (uint32_t)(j >> 6) * 8192u + (uint32_t)t * 128u +
                                           ((uint32_t)(((j & 63) >> 3) ^ (t & 7)) << 4)) = vpre[i];
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // MMA: [I; P] T = [T; P T], contraction halves by warps 0 and 1 into
        // columns 0..63 and 64..127
        if (lead && warp < 2) {
            const uint32_t idesc = idesc_bf16(128, 64, 0, 1);
            const uint32_t a = smem_u32(ip), b = smem_u32(tt);
    #pragma unroll
            for (int s = 2 * warp; s < 2 * warp + 2; ++s)
                mma_bf16(tm + (uint32_t)(64 * warp), desc_sw128(a + (uint32_t)s * 32u, 16, 1024),
                         desc_sw128(b + (uint32_t)s * 2048u, 8192, 1024), idesc, s > 2 * warp);
            mma_commit(bar_i);
        }
        ok = mbar_wait(bar_i, 0, status);
        tc_fence_after();
        if (__syncthreads_or(!ok))
            goto teardown;
        {
            float tr[32], t2[32];
            tmem_ld16(tm + lb + (uint32_t)(32 * half), tr);
            tmem_ld16(tm + lb + (uint32_t)(32 * half + 16), tr + 16);
            tmem_ld16(tm + lb + (uint32_t)(64 + 32 * half), t2);
            tmem_ld16(tm + lb + (uint32_t)(64 + 32 * half + 16), t2 + 16);
            tmem_ld_wait();
    #pragma unroll
            for (int j = 0; j < 32; ++j)
                tr[j] += t2[j];
    #pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4 *>(tp + kmajor_chunk(row, 32 * half + 8 * cc, 128)) = pack8(tr + 8 * cc);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // MMA: [T; P T] [K | V] = [W', P W' | U', P U']  (columns 0..Dp-1 |
        // Dp..Dp+d_v-1): warp j issues the 128 columns of block j, warp Dp/128
        // the V columns
        if (lead && warp <= Dp / 128) {
            const uint32_t a = smem_u32(tp), bk = smem_u32(kq), bv = smem_u32(vt);
            const uint32_t idk = idesc_bf16(128, 128, 0, 1), idv = idesc_bf16(128, d_v, 0, 1);
            const int j = warp;
            if (j < Dp / 128) {
    #pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + (uint32_t)(128 * j), desc_sw128(a + (uint32_t)s * 32u, 16, 1024),
                             desc_sw128(bk + (uint32_t)(2 * j) * 16384u + (uint32_t)s * 2048u, 16384, 1024), idk,
                             s > 0);
            } else {
    #pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + (uint32_t)Dp, desc_sw128(a + (uint32_t)s * 32u, 16, 1024),
                             desc_sw128(bv + (uint32_t)s * 2048u, 8192, 1024), idv, s > 0);
            }
            mma_commit(bar_f);
        }
        if (tid == 0)
            bulk_wait_read(); // the K image has been read out of the key rows
        ok = mbar_wait(bar_f, 0, status);
        tc_fence_after();
        if (__syncthreads_or(!ok))
            goto teardown;
        // Record out.  W' replaces the key rows and Q' = Q - P W' the query rows
        // of the [K; Q] tile in place (the K image's bulk read of the key rows
        // finished before the barrier above); the tile goes out as one bulk copy.
        for (int c0 = 32 * half; c0 < Dp; c0 += 64) { // 32 columns per pass (Dp % 64 == 0)
            float w[32];
            tmem_ld16(tm + lb + (uint32_t)c0, w);
            tmem_ld16(tm + lb + (uint32_t)(c0 + 16), w + 16);
            tmem_ld_wait();
    #pragma unroll
            for (int h2 = 0; h2 < 4; ++h2) {
                uint4 *dst = reinterpret_cast<uint4 *>(kq + kmajor_chunk(row, c0 + 8 * h2, 128));
                if (row >= 64) {
                    float qv[8];
                    unpack8(*dst, qv);
    #pragma unroll
                    for (int e = 0; e < 8; ++e)
                        w[8 * h2 + e] = qv[e] - w[8 * h2 + e];
                }
                *dst = pack8(w + 8 * h2);
            }
        }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(rec + rc.a, kq, 256u * (uint32_t)Dp);
        bulk_commit();
    }
    // U' (rows < 64) and Y' (rows >= 64) go straight from registers to the
    // record in fp32 as [d_v/4][64][4], so a warp's 16-byte stores are one
    // contiguous run
    {
        float *uy = reinterpret_cast<float *>(rec + (row < 64 ? rc.up : rc.yp)) + 4 * (row & 63);
        for (int c0 = 16 * half; c0 < d_v; c0 += 32) {
            float w[16];
            tmem_ld16(tm + lb + (uint32_t)(Dp + c0), w);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(uy + 256 * ((c0 + e) >> 2)) = make_float4(w[e], w[e + 1], w[e + 2], w[e + 3]);
        }
    }
teardown:
    if (tid == 0)
        bulk_wait_all(); // the bulk copies are done before the CTA retires
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, ncols);
}

// ---------------------------------------------------------------------------
// 16-byte chunk holding columns j0 .. j0+7 of row `row` of an MN-major SW128
// operand tile whose rows are the contraction index and whose columns are
// value channels (64-column blocks `blk` bytes apart).
FW_DEV uint32_t vtile_chunk(int row, int j0, uint32_t blk) {
    return (uint32_t)(j0 >> 6) * blk + (uint32_t)row * 128u + ((uint32_t)(((j0 & 63) >> 3) ^ (row & 7)) << 4);
}

// One CTA walks the chunks of one (batch, head) for DVB value channels.
// Everything per thread is done 16 value channels at a time.  NA = number
// of [W'; Q'] buffers (2: the image of chunk c + 2 is fetched as soon as
// MMA1 has read chunk c's; 1: chunk c + 1's, into the same buffer).  NKB = number
// of K buffers (2: K images two chunks ahead; 1: the next K image is
// fetched as soon as MMA3 has read the current one).
// ZN = true (the normalised sum rule): the CTA's block is 16 value channels
// followed by the record's 16-channel normaliser block (channel d_vr holds
// the running z, its output the denominator z . phi(q)); DVB = 32, and y is
// written as the ratio of the value columns to that denominator (0 where it
// is 0).  d_v = the record's channel count, d_vr = the value channels of y,
// W0 and W_final; z0 / zf: the normaliser state in and out ([B,H,d_dot]).
template <int DVB, int NKB, int NA, bool ZN>
__global__ void __launch_bounds__(kScanThreads)
    chunk_scan_kernel(const float *W0, float *Wf, const float *z0, float *zf, __nv_bfloat16 *__restrict__ y,
                      const uint8_t *__restrict__ ws, int L, int C, int nch, int d_v, int d_vr, int d_dot, int Dp,
                      unsigned *status) {
    static_assert(!ZN || DVB == 32, "the normalised form takes 16 value + 16 normaliser channels");
    constexpr int DS = DVB < 32 ? 32 : DVB;          // TMEM columns per accumulator region
    constexpr int VB = (DVB + 63) / 64;              // 64-column blocks of the value tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Record rc = record_layout(Dp, d_v);
    const uint32_t a_bytes = 256u * (uint32_t)Dp, k_bytes = 128u * (uint32_t)Dp;
    const uint32_t sblk = 128u * (uint32_t)Dp;       // bytes of one 64-column block of the S tile
    uint8_t *at0 = smem;                              // [W'; Q']  128 x Dp (NA buffers)
    uint8_t *at1 = NA == 2 ? at0 + a_bytes : at0;
    uint8_t *kt0 = at0 + NA * a_bytes;                // K image(s)
    uint8_t *kt1 = NKB == 2 ? kt0 + k_bytes : kt0;
    uint8_t *st = kt0 + NKB * k_bytes;                // S: rows d, columns v (MN-major)
    uint8_t *ut = st + VB * sblk;                     // U: rows t, columns v (MN-major)
    uint64_t *bar_a = (uint64_t *)(ut + VB * 8192);  // [2]
    uint64_t *bar_k = bar_a + 2;                      // [2]
    uint64_t *bar_m1 = bar_a + 4;                     // MMA1 done (both issuers)
    uint64_t *bar_m3 = bar_a + 5;                     // MMA3 done (every block's issuer)
    uint32_t *slot = (uint32_t *)(bar_a + 6);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int v0 = blockIdx.x * (ZN ? 16 : DVB);
    const int64_t bh = blockIdx.y;
    // record channel of the CTA's column j (column groups of 4 stay contiguous)
    auto chan = [&](int j) { return (ZN && j >= 16) ? d_vr + (j - 16) : v0 + j; };
    const int MB = Dp / 128;
    const uint32_t ncols = tmem_cols_pow2((2 + MB) * DS);
    const uint8_t *rec0 = ws + (size_t)bh * nch * rc.bytes;
    const bool has_w0 = W0 != nullptr || (ZN && z0 != nullptr);
    const uint32_t lb = tmem_lane_base(warp);

    if (tid == 0) {
        mbar_init(bar_a, 1);
        mbar_init(bar_a + 1, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_k + 1, 1);
        mbar_init(bar_m1, 2);
        mbar_init(bar_m3, (uint32_t)MB);
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
    // D1 as two partial sums (contraction halves), then the MB blocks of S^T
    const uint32_t tD1 = tm, tD1b = tm + DS, tS = tm + 2 * DS;
    const bool lead = (tid & 31) == 0;
    const uint32_t st_s = smem_u32(st), ut_s = smem_u32(ut);
    const uint32_t kt0_s = smem_u32(kt0), kt1_s = smem_u32(kt1);

    // initial state: S^T in TMEM (fp32) and S as the bf16 operand of MMA1.
    // W0 is the caller's and never written by the prep kernel, which lets
    // this kernel start only after its own wait (so everything enqueued
    // before the prep has completed): it runs before the wait for the prep.
    for (int mb = 0; mb < MB; ++mb) {
        const int d = 128 * mb + tid;
#pragma unroll
        for (int j0 = 0; j0 < DVB; j0 += 16) {
            float w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int jj = j0 + j;
                if (ZN && jj >= 16)
                    w[j] = (jj == 16 && z0 && d < d_dot) ? z0[(size_t)bh * d_dot + d] : 0.f;
                else
                    w[j] = (W0 && d < d_dot) ? W0[((size_t)bh * d_vr + v0 + jj) * d_dot + d] : 0.f;
            }
            if (has_w0)
                tmem_st16(tS + (uint32_t)(mb * DS + j0) + lb, w);
            *reinterpret_cast<uint4 *>(st + vtile_chunk(d, j0, sblk)) = pack8(w);
            *reinterpret_cast<uint4 *>(st + vtile_chunk(d, j0 + 8, sblk)) = pack8(w + 8);
        }
    }
    if (has_w0)
        tmem_st_wait();
    // the workspace records are the prep kernel's: wait for it to complete
    // (and let the next kernel on the stream start its set-up meanwhile)
    griddep_launch_dependents();
    griddep_wait();
    rec0 = after_wait(rec0);
    // On an early exit (a wait that gave up) thread 0 waits, bounded, for the
    // bulk loads still in flight, so that none lands after the CTA has left.
    // Which are in flight follows from the chunk and the step that failed
    // (0: its [W'; Q'] image, 1: MMA1, 2: its K image, 3: MMA3): the image of
    // chunk j sits in buffer j % NA (j % NKB), in that buffer's phase j / NA.
    auto drain = [&](int c, int step) {
        if (tid != 0)
            return;
        const int a_hi = min(nch - 1, step >= 2 ? c + NA : c + NA - 1);
        for (int j = step >= 1 ? c + 1 : c; j <= a_hi; ++j)
            mbar_wait(bar_a + (NA == 2 ? (j & 1) : 0), (uint32_t)((NA == 2 ? j >> 1 : j) & 1), status);
        const int k_hi = min(nch - 1, c + NKB - 1);
        for (int j = step >= 3 ? c + 1 : c; j <= k_hi; ++j)
            mbar_wait(bar_k + (NKB == 2 ? (j & 1) : 0), (uint32_t)((NKB == 2 ? j >> 1 : j) & 1), status);
    };
    if (tid == 0) { // chunk 0's [W'; Q'] and the first K image(s)
        mbar_arrive_expect_tx(bar_a, a_bytes);
        bulk_g2s(at0, rec0 + rc.a, a_bytes, bar_a);
        if (NA == 2 && nch > 1) {
            mbar_arrive_expect_tx(bar_a + 1, a_bytes);
            bulk_g2s(at1, rec0 + rc.bytes + rc.a, a_bytes, bar_a + 1);
        }
        mbar_arrive_expect_tx(bar_k, k_bytes);
        bulk_g2s(kt0, rec0 + rc.k, k_bytes, bar_k);
        if (NKB == 2 && nch > 1) {
            mbar_arrive_expect_tx(bar_k + 1, k_bytes);
            bulk_g2s(kt1, rec0 + rc.bytes + rc.k, k_bytes, bar_k + 1);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // U' (rows 0..63, threads 0..63) or Y' (threads 64..127) of a chunk,
    // [d_v/4][64][4] in the record: each 16-byte load of a warp is one
    // 512-byte run.  Chunk c + 1's are loaded as soon as chunk c's are used.
    float pre[DVB];
    auto load_pre = [&](int cc) {
        const float *src = (const float *)(rec0 + (size_t)cc * rc.bytes + (tid < 64 ? rc.up : rc.yp)) + 4 * (tid & 63);
#pragma unroll
        for (int j = 0; j < DVB; j += 4) {
            const float4 f = __ldcg(reinterpret_cast<const float4 *>(src + 64 * chan(j)));
            pre[j] = f.x;
            pre[j + 1] = f.y;
            pre[j + 2] = f.z;
            pre[j + 3] = f.w;
        }
    };
    load_pre(0);
    uint32_t m1_phase = 0, m3_phase = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * C, Lc = min(C, L - t0), kb = NKB == 2 ? (c & 1) : 0, ab = NA == 2 ? (c & 1) : 0;
        const uint32_t a_parity = NA == 2 ? (uint32_t)((c >> 1) & 1) : (uint32_t)(c & 1);
        const uint32_t k_parity = NKB == 2 ? (uint32_t)((c >> 1) & 1) : (uint32_t)(c & 1);
        const uint8_t *rec = rec0 + (size_t)c * rc.bytes;
        // U' (rows 0..63, threads 0..63) or Y' (threads 64..127) of this chunk
        bool ok = mbar_wait(bar_a + ab, a_parity, status);
        if (__syncthreads_or(!ok)) {
            drain(c, 0);
            break;
        }

        // MMA1: D1 = [W'; Q'] S^T, warp 0 over the first half of the
        // contraction into tD1, warp 1 over the second into tD1b
        if (lead && warp < 2) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, DVB, 0, 1);
            const int s0 = warp * (Dp / 32);
            for (int s = s0; s < s0 + Dp / 32; ++s)
                mma_bf16(warp ? tD1b : tD1, desc_sw128(smem_u32(ab ? at1 : at0) + kmajor_step(s, 128), 16, 1024),
                         desc_sw128(st_s + (uint32_t)s * 2048u, sblk, 1024), idesc, s > s0);
            mma_commit(bar_m1);
        }
        ok = mbar_wait(bar_m1, m1_phase, status);
        m1_phase ^= 1;
        if (__syncthreads_or(!ok)) {
            drain(c, 1);
            break;
        }
        tc_fence_after();
        if (tid == 0 && c + NA < nch) { // this [W'; Q'] buffer is consumed: fetch a later chunk's
            mbar_arrive_expect_tx(bar_a + ab, a_bytes);
            bulk_g2s(ab ? at1 : at0, rec + (size_t)NA * rc.bytes + rc.a, a_bytes, bar_a + ab);
        }
        {
            float d1[DVB], d1b[DVB];
#pragma unroll
            for (int j0 = 0; j0 < DVB; j0 += 16) { // every load in flight, then one wait
                tmem_ld16(tD1 + lb + (uint32_t)j0, d1 + j0);
                tmem_ld16(tD1b + lb + (uint32_t)j0, d1b + j0);
            }
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < DVB; ++j)
                d1[j] += d1b[j];
            if (tid < 64) {                           // U = U' - W' S^T
#pragma unroll
                for (int j0 = 0; j0 < DVB; j0 += 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        d1[j0 + j] = pre[j0 + j] - d1[j0 + j];
                    *reinterpret_cast<uint4 *>(ut + vtile_chunk(tid, j0, 8192u)) = pack8(d1 + j0);
                    *reinterpret_cast<uint4 *>(ut + vtile_chunk(tid, j0 + 8, 8192u)) = pack8(d1 + j0 + 8);
                }
            } else if (tid - 64 < Lc) {               // y = Y' + Q' S^T
#pragma unroll
                for (int j = 0; j < DVB; ++j)
                    d1[j] += pre[j];
                if constexpr (ZN) {                   // the ratio to the normaliser column
                    const float den = d1[16];
                    const float inv = den != 0.f ? 1.0f / den : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        d1[j] *= inv;
                }
                __nv_bfloat16 *dst = y + ((size_t)bh * L + t0 + (tid - 64)) * d_vr + v0;
#pragma unroll
                for (int j0 = 0; j0 < (ZN ? 16 : DVB); j0 += 8)
                    *reinterpret_cast<uint4 *>(dst + j0) = pack8(d1 + j0);
            }
        }
        if (c + 1 < nch)
            load_pre(c + 1);
        fence_async_smem();
        tc_fence_before();
        ok = mbar_wait(bar_k + kb, k_parity, status);
        if (__syncthreads_or(!ok)) {
            drain(c, 2);
            break;
        }

        // MMA3: S^T += K^T U   (K^T: the K image read MN-major); block mb of
        // S^T by warp mb
        if (lead && warp < MB) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, DVB, 1, 1);
            const uint32_t kbase = kb ? kt1_s : kt0_s;
            const int mb = warp;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS + (uint32_t)(mb * DS),
                         desc_sw128(kbase + (uint32_t)(2 * mb) * 8192u + (uint32_t)s * 2048u, 8192, 1024),
                         desc_sw128(ut_s + (uint32_t)s * 2048u, 8192, 1024), idesc,
                         (s > 0 || c > 0 || has_w0) ? 1u : 0u);
            mma_commit(bar_m3);
        }
        ok = mbar_wait(bar_m3, m3_phase, status);
        m3_phase ^= 1;
        if (__syncthreads_or(!ok)) {
            drain(c, 3);
            break;
        }
        tc_fence_after();
        if (tid == 0 && c + NKB < nch) { // this K buffer is consumed: fetch a later chunk's
            mbar_arrive_expect_tx(bar_k + kb, k_bytes);
            bulk_g2s(kb ? kt1 : kt0, rec + (size_t)NKB * rc.bytes + rc.k, k_bytes, bar_k + kb);
        }
        for (int mb = 0; mb < MB; ++mb) {
            const int d = 128 * mb + tid;
            float sv[DVB];
#pragma unroll
            for (int j0 = 0; j0 < DVB; j0 += 16) // every load in flight, then one wait
                tmem_ld16(tS + (uint32_t)(mb * DS + j0) + lb, sv + j0);
            tmem_ld_wait();
#pragma unroll
            for (int j0 = 0; j0 < DVB; j0 += 16) {
                if (c + 1 < nch) {
                    *reinterpret_cast<uint4 *>(st + vtile_chunk(d, j0, sblk)) = pack8(sv + j0);
                    *reinterpret_cast<uint4 *>(st + vtile_chunk(d, j0 + 8, sblk)) = pack8(sv + j0 + 8);
                } else if (d < d_dot) {
                    if (ZN && j0 >= 16) {             // the normaliser state: column 16
                        if (j0 == 16 && zf && blockIdx.x == 0)
                            zf[(size_t)bh * d_dot + d] = sv[16];
                    } else if (Wf) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            Wf[((size_t)bh * d_vr + v0 + j0 + j) * d_dot + d] = sv[j0 + j];
                    }
                }
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
size_t prep_smem(int Dp, int d_v) {
    const int VB = (d_v + 63) / 64;
    (void)VB; // the V tile (<= 16 KB) reuses the fp32 work space (37 KB)
    return (size_t)256 * Dp + 16384 + 8192 + (2 * 64 + 16) * LDS * 4 + 64 * 4 + 32 + 1024;
}

size_t scan_smem(int Dp, int dvb, int nkb, int na) {
    const int VB = (dvb + 63) / 64;
    return (size_t)na * 256 * Dp + (size_t)nkb * 128 * Dp + (size_t)VB * 128 * Dp + (size_t)VB * 8192 + 64 + 1024;
}

constexpr size_t kMaxSmem = 227 * 1024;

bool fits(int Dp, int d_v, int dvb) {
    return Dp <= kMaxDp && Dp + d_v <= 512 && scan_smem(Dp, dvb, 1, 1) <= kMaxSmem && prep_smem(Dp, d_v) <= kMaxSmem;
}

// Value channels per scan CTA: 16 (32 with the normaliser block).  The walk
// over the chunks is serial, so the per-chunk latency decides: a tcgen05.mma
// of M = 128 costs about the same for any N up to 128, but the per-thread
// work between the MMAs (TMEM loads, the U and S tiles, y) grows with the
// channel count.  Measured on the b4h8 L512 and nu = 3 L2048 workloads, 16
// channels per CTA beat 32 and 64 (scan 14.4 / 18.5 / 24.5 us and
// 80 / 96 / 141 us).
constexpr int kDVB = 16;

// Two K buffers when they fit in shared memory, else one; then two [W'; Q']
// buffers when those fit as well.
int choose_nkb(int Dp, int dvb) { return scan_smem(Dp, dvb, 2, 1) <= kMaxSmem ? 2 : 1; }
int choose_na(int Dp, int dvb) { return scan_smem(Dp, dvb, choose_nkb(Dp, dvb), 2) <= kMaxSmem ? 2 : 1; }

template <int DK, bool SUM>
cudaError_t launch_prep(const void *q, const void *k, const void *v, const void *beta, uint8_t *ws, int BH,
                        int L, int C, int nch, int nu, int Dp, int d_v, int d_vr, float eps, unsigned *status,
                        cudaStream_t st) {
    const size_t smem = prep_smem(Dp, d_v);
    auto kern = chunk_prep_kernel<DK, SUM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3((unsigned)nch, (unsigned)BH), dim3(kPrepThreads), smem, st,
                      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                      static_cast<const __nv_bfloat16 *>(v), static_cast<const __nv_bfloat16 *>(beta), ws, L, C,
                      nch, nu, Dp, d_v, d_vr, eps, status);
}

template <int DVB, int NKB, int NA, bool ZN>
cudaError_t launch_scan(const float *W0, float *Wf, const float *z0, float *zf, void *y, const uint8_t *ws, int BH,
                        int L, int C, int nch, int d_v, int d_vr, int d_dot, int Dp, unsigned *status,
                        cudaStream_t st) {
    const size_t smem = scan_smem(Dp, DVB, NKB, NA);
    auto kern = chunk_scan_kernel<DVB, NKB, NA, ZN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    // programmatic dependent launch: the scan's CTAs may be scheduled while
    // the preceding kernel (the prep) finishes; they wait in griddep_wait
    // before reading its output
    const dim3 grid((unsigned)(ZN ? d_vr / 16 : d_v / DVB), (unsigned)BH);
    return launch_pdl(kern, grid, dim3(kScanThreads), smem, st, W0, Wf, z0, zf, static_cast<__nv_bfloat16 *>(y), ws,
                      L, C, nch, d_v, d_vr, d_dot, Dp, status);
}

template <int DVB, bool ZN>
cudaError_t launch_scan_bufs(const float *W0, float *Wf, const float *z0, float *zf, void *y, const uint8_t *ws,
                             int BH, int L, int C, int nch, int d_v, int d_vr, int d_dot, int Dp, unsigned *status,
                             cudaStream_t st) {
    if (choose_nkb(Dp, DVB) == 2) {
        if (choose_na(Dp, DVB) == 2)
            return launch_scan<DVB, 2, 2, ZN>(W0, Wf, z0, zf, y, ws, BH, L, C, nch, d_v, d_vr, d_dot, Dp, status, st);
        return launch_scan<DVB, 2, 1, ZN>(W0, Wf, z0, zf, y, ws, BH, L, C, nch, d_v, d_vr, d_dot, Dp, status, st);
    }
    return launch_scan<DVB, 1, 1, ZN>(W0, Wf, z0, zf, y, ws, BH, L, C, nch, d_v, d_vr, d_dot, Dp, status, st);
}

} // namespace

bool tc_forward_supported(int d_key, int nu, int d_v, int chunk) {
    if (!(d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128))
        return false;
    if (!(d_v == 16 || d_v == 32 || d_v == 64 || d_v == 128))
        return false;
    if (chunk < 1 || chunk > kTile)
        return false;
    return fits(padded_ddot(2 * d_key * nu), d_v, kDVB);
}

size_t tc_forward_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk) {
    const int nch = (L + chunk - 1) / chunk;
    return (size_t)B * H * nch * record_layout(padded_ddot(2 * d_key * nu), d_v).bytes;
}

namespace {

template <bool SUM>
cudaError_t prep_dispatch(const void *q, const void *k, const void *v, const void *beta, void *workspace, int B,
                          int H, int L, int d_key, int nu, int d_v, int d_vr, int chunk, float eps, unsigned *status,
                          cudaStream_t st) {
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int Dp = padded_ddot(2 * d_key * nu);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    switch (d_key) {
    case 8: return launch_prep<8, SUM>(q, k, v, beta, ws, BH, L, chunk, nch, nu, Dp, d_v, d_vr, eps, status, st);
    case 16: return launch_prep<16, SUM>(q, k, v, beta, ws, BH, L, chunk, nch, nu, Dp, d_v, d_vr, eps, status, st);
    case 32: return launch_prep<32, SUM>(q, k, v, beta, ws, BH, L, chunk, nch, nu, Dp, d_v, d_vr, eps, status, st);
    case 64: return launch_prep<64, SUM>(q, k, v, beta, ws, BH, L, chunk, nch, nu, Dp, d_v, d_vr, eps, status, st);
    case 128: return launch_prep<128, SUM>(q, k, v, beta, ws, BH, L, chunk, nch, nu, Dp, d_v, d_vr, eps, status, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

cudaError_t tc_prepare_launch(const void *q, const void *k, const void *v, const void *beta, void *workspace,
                              int B, int H, int L, int d_key, int nu, int d_v, int chunk, float eps,
                              unsigned *status, cudaStream_t st) {
    return prep_dispatch<false>(q, k, v, beta, workspace, B, H, L, d_key, nu, d_v, d_v, chunk, eps, status, st);
}

cudaError_t tc_scan_launch(const void *workspace, const float *W0, float *W_final, void *y, int B, int H, int L,
                           int d_key, int nu, int d_v, int chunk, int num_sms, unsigned *status, cudaStream_t st) {
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const int Dp = padded_ddot(d_dot);
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    (void)num_sms;
    return launch_scan_bufs<kDVB, false>(W0, W_final, nullptr, nullptr, y, ws, BH, L, chunk, nch, d_v, d_v, d_dot, Dp,
                                         status, st);
}

cudaError_t tc_forward_launch(const void *q, const void *k, const void *v, const void *beta,
                              const float *W0, float *W_final, void *y, void *workspace, int B,
                              int H, int L, int d_key, int nu, int d_v, int chunk, float eps,
                              int num_sms, unsigned *status, cudaStream_t st) {
    const cudaError_t e = tc_prepare_launch(q, k, v, beta, workspace, B, H, L, d_key, nu, d_v, chunk, eps, status, st);
    if (e != cudaSuccess)
        return e;
    return tc_scan_launch(workspace, W0, W_final, y, B, H, L, d_key, nu, d_v, chunk, num_sms, status, st);
}

// ------------------------------------------------ the sum rule (linear attention)
bool tc_linear_supported(int d_key, int nu, int d_v, int chunk, int normalize) {
    if (!(d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128))
        return false;
    if (!(d_v == 16 || d_v == 32 || d_v == 64 || d_v == 128))
        return false;
    if (chunk < 1 || chunk > kTile)
        return false;
    return fits(padded_ddot(2 * d_key * nu), d_v + (normalize ? 16 : 0), normalize ? 32 : kDVB);
}

size_t tc_linear_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int normalize) {
    const int nch = (L + chunk - 1) / chunk;
    return (size_t)B * H * nch * record_layout(padded_ddot(2 * d_key * nu), d_v + (normalize ? 16 : 0)).bytes;
}

// The same two kernels as the delta rule: the prep in its sum-rule form
// (records with W' = 0, Q' = Q, U' = V', Y' = P V'), then the scan, which
// with W' = 0 reduces to y = Y' + Q S^T, S += K^T V'.  With the normaliser,
// V' carries a ones column whose state is z and whose output is the
// denominator, and each scan CTA takes that block beside its 16 channels.
cudaError_t tc_linear_launch(const void *q, const void *k, const void *v, const float *W0, const float *z0,
                             float *W_final, float *z_final, void *y, void *workspace, int B, int H, int L,
                             int d_key, int nu, int d_v, int chunk, int normalize, float eps, int num_sms,
                             unsigned *status, cudaStream_t st) {
    (void)num_sms;
    const int dv2 = d_v + (normalize ? 16 : 0);
    cudaError_t e = prep_dispatch<true>(q, k, v, nullptr, workspace, B, H, L, d_key, nu, dv2, d_v, chunk, eps,
                                        status, st);
    if (e != cudaSuccess)
        return e;
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const int Dp = padded_ddot(d_dot);
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    if (normalize)
        return launch_scan_bufs<32, true>(W0, W_final, z0, z_final, y, ws, BH, L, chunk, nch, dv2, d_v, d_dot, Dp,
                                          status, st);
    return launch_scan_bufs<kDVB, false>(W0, W_final, nullptr, nullptr, y, ws, BH, L, chunk, nch, d_v, d_v, d_dot,
                                         Dp, status, st);
}

} // namespace fw
