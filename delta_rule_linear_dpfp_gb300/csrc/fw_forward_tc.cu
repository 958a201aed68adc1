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
#include <algorithm>

#include "fw_dpfp.cuh"
#include "fw_forward_tc.h"
#include "fw_tc.cuh"

namespace fw {
namespace {

using namespace tc;

constexpr int kTile = 64;          // token rows of a chunk tile (chunk <= 64, padded)
constexpr int kPrepThreads = 256;
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

__host__ __device__ inline uint32_t tmem_cols_pow2(int need) {
    return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// ---------------------------------------------------------------------------
// Element offset helpers of the T operand tile (rows k, columns n; MN-major,
// 128-byte rows, 16-byte chunks swizzled by k & 7).
FW_DEV uint32_t ttile_chunk(int kk, int n) { return (uint32_t)kk * 128u + ((uint32_t)((n >> 3) ^ (kk & 7)) << 4); }

// (I + A)^-1 for a strictly lower 64 x 64 A: the four 16 x 16 diagonal
// blocks by forward substitution (one column per thread), then the blocks
// below the diagonal by doubling (16 -> 32 -> 64, below).
// A, N: [64][LDS]; R: [16][LDS] scratch (used as [32][32]); all 16-byte
// aligned.  Only the blocks on and below the diagonal of N are written (the
// ones above are zero and never read here).  As each block of N is final it
// also goes out, times beta of its column, in bf16 to the T operand tile tt
// (T = N diag(beta)); the blocks above the diagonal are written as zeros.
// NT threads (>= 256); ends synchronised.
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
    // The blocks below the diagonal by doubling the block size: with
    // P = (I + A_11)^-1 and Q = (I + A_22)^-1 known for the two diagonal
    // blocks of a 2 x 2 partition, (I + A)^-1 = [P 0; -Q A_21 P  Q].  Level 1
    // takes the two 32 x 32 diagonal blocks at once (16 x 16 halves), level 2
    // the whole 64 x 64; each level is two products, R = A_21 P, then
    // -Q R.  Each thread computes 4 adjacent outputs of a row from 16-byte
    // loads, so every A (or N) element it loads feeds 4 FMAs.  R is used as
    // [32][32].  Only blocks on and below the diagonal of N are read.
    auto t_out = [&](int kk, int j0, float4 v) { // N row kk, columns j0..j0+3 -> N and the T tile
        *reinterpret_cast<float4 *>(N + kk * LDS + j0) = v;
        uint2 t4;
        t4.x = pack_bf16x2(v.x * bs[j0], v.y * bs[j0 + 1]);
        t4.y = pack_bf16x2(v.z * bs[j0 + 2], v.w * bs[j0 + 3]);
        *reinterpret_cast<uint2 *>(tt + ttile_chunk(kk, j0) + 2 * (j0 & 7)) = t4;
    };
    // level 1: blocks b = 0, 1 of 32 rows; R_b = A_{2b+1,2b} N_{2b,2b} (16 x 16)
    const int b1 = tid >> 6, i1 = (tid >> 2) & 15, j1 = 4 * (tid & 3);
    if (tid < 128) {
        const int c0 = 32 * b1, r0 = c0 + 16;
        const float *ar = A + (r0 + i1) * LDS + c0;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s4 = 0; s4 < 16; s4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(ar + s4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 n = *reinterpret_cast<const float4 *>(N + (c0 + s4 + e) * LDS + c0 + j1);
                acc.x = fmaf(av[e], n.x, acc.x);
                acc.y = fmaf(av[e], n.y, acc.y);
                acc.z = fmaf(av[e], n.z, acc.z);
                acc.w = fmaf(av[e], n.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(R + (16 * b1 + i1) * 32 + j1) = acc;
    }
    __syncthreads();
    // N_{2b+1,2b} = -N_{2b+1,2b+1} R_b
    if (tid < 128) {
        const int c0 = 32 * b1, r0 = c0 + 16;
        const float *nr = N + (r0 + i1) * LDS + r0;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s4 = 0; s4 < 16; s4 += 4) {
            const float4 nn = *reinterpret_cast<const float4 *>(nr + s4);
            const float nv[4] = {nn.x, nn.y, nn.z, nn.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 r = *reinterpret_cast<const float4 *>(R + (16 * b1 + s4 + e) * 32 + j1);
                acc.x = fmaf(nv[e], r.x, acc.x);
                acc.y = fmaf(nv[e], r.y, acc.y);
                acc.z = fmaf(nv[e], r.z, acc.z);
                acc.w = fmaf(nv[e], r.w, acc.w);
            }
        }
        t_out(r0 + i1, c0 + j1, make_float4(-acc.x, -acc.y, -acc.z, -acc.w));
    }
    __syncthreads();
    // level 2: R = A[32:64, 0:32] P with P = N[0:32, 0:32] (its block (0, 1)
    // is above the diagonal: columns 16..31 sum over rows 16..31 only)
    const int i2 = tid >> 3, j2 = 4 * (tid & 7);
    if (tid < 256) {
        const float *ar = A + (32 + i2) * LDS;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k4 = j2 >= 16 ? 16 : 0; k4 < 32; k4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(ar + k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 n = *reinterpret_cast<const float4 *>(N + (k4 + e) * LDS + j2);
                acc.x = fmaf(av[e], n.x, acc.x);
                acc.y = fmaf(av[e], n.y, acc.y);
                acc.z = fmaf(av[e], n.z, acc.z);
                acc.w = fmaf(av[e], n.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(R + i2 * 32 + j2) = acc;
    }
    __syncthreads();
    // N[32:64, 0:32] = -Q R with Q = N[32:64, 32:64] (rows 0..15 of Q sum
    // over its columns 0..15 only)
    if (tid < 256) {
        const float *nr = N + (32 + i2) * LDS + 32;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k4 = 0; k4 < (i2 < 16 ? 16 : 32); k4 += 4) {
            const float4 nn = *reinterpret_cast<const float4 *>(nr + k4);
            const float nv[4] = {nn.x, nn.y, nn.z, nn.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 r = *reinterpret_cast<const float4 *>(R + (k4 + e) * 32 + j2);
                acc.x = fmaf(nv[e], r.x, acc.x);
                acc.y = fmaf(nv[e], r.y, acc.y);
                acc.z = fmaf(nv[e], r.z, acc.z);
                acc.w = fmaf(nv[e], r.w, acc.w);
            }
        }
        t_out(32 + i2, j2, make_float4(-acc.x, -acc.y, -acc.z, -acc.w));
    }
    __syncthreads();
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
// Shared-memory layout of the prep (one chunk at a time).
struct PrepSmem {
    uint8_t *kq;     // [K; Q]: 128 x Dp, K-major
    uint8_t *ip;     // [I; P]: 128 x 64, K-major A; [T; P T] replaces it once read
    uint8_t *tt;     // T: rows k, columns n (MN-major B)
    float *Am;       // A = strict_lower(beta K K^T)
    float *Nm;       // (I + A)^-1
    float *Rm;       // block-solve scratch [16][LDS]
    float *bs;       // beta (0 on padded rows)
    uint8_t *vt;     // V (MN-major B), once A and N are done
    // MMA completion: the Gram matrix (2 issuers), [I; P] T (2 issuers; the
    // sum rule's [I; P] V' by 1), the final product (one issuer per accumulator)
    uint64_t *bar_g, *bar_i, *bar_f;
    uint32_t *slot;  // TMEM base address
};

// The barriers and the TMEM slot take the first kPrepHead bytes (the
// projection prologue of chunk_prep_x_kernel keeps its own barriers there
// too, and streams its operands through the space after them).
constexpr int kPrepHead = 1024;
FW_DEV PrepSmem prep_layout(uint8_t *smem, int Dp) {
    PrepSmem m;
    m.bar_g = (uint64_t *)smem;
    m.bar_i = m.bar_g + 1;
    m.bar_f = m.bar_g + 2;
    m.slot = (uint32_t *)(m.bar_g + 3);
    m.kq = smem + kPrepHead;
    m.ip = m.kq + 256 * Dp;
    m.tt = m.ip + 16384;
    m.Am = (float *)(m.tt + 8192);
    m.Nm = m.Am + 64 * LDS;
    m.Rm = m.Nm + 64 * LDS;
    m.bs = m.Rm + 16 * LDS;
    m.vt = (uint8_t *)m.Am;
    return m;
}

struct PrepArgs {
    const __nv_bfloat16 *q, *k, *v, *beta;
    uint8_t *ws;
    int L, C, nch, nu, Dp, d_v, d_vr;
    float eps;
    unsigned *status;
};

__host__ __device__ inline uint32_t prep_tmem_cols(int Dp, int d_v) { return tmem_cols_pow2(Dp + d_v > 64 ? Dp + d_v : 64); }

// The chunk's inputs in registers: the key and query rows for the DPFP, the
// V rows (kept until their tile's space is free) and beta (stored to shared
// memory after the DPFP).
template <int DK> struct PrepRegs {
    static constexpr int G = DK / 4, RPW = 32 / G;
    static constexpr bool kHalfRows = DK <= 64;
    static constexpr int kRaw = kHalfRows ? DK / 8 : 128 / (8 * RPW);
    static constexpr int kVChunks = 4; // 64 * 128 / 8 / kPrepThreads
    uint4 raw[kRaw];
    uint4 vpre[kVChunks];
    __nv_bfloat16 beta_raw; // converted only where it is stored, so its load's latency is not waited for early
};

// Global loads of chunk c of (b,h), all in flight before any is used.
template <int DK, bool SUM>
FW_DEV void prep_load(const PrepArgs &g, int c, int64_t bh, int tid, PrepRegs<DK> &r) {
    using R = PrepRegs<DK>;
    const int warp = tid >> 5, lane = tid & 31;
    const int t0 = c * g.C, Lc = min(g.C, g.L - t0);
    if constexpr (R::kHalfRows) { // thread = (row r, half hs of x); lanes l and l ^ 8 share a row
        const int hr = 16 * warp + ((lane & 7) | ((lane >> 4) << 3));
        const int t = hr & 63;
        const __nv_bfloat16 *src = (hr < 64 ? g.k : g.q) + ((size_t)bh * g.L + t0 + t) * DK;
#pragma unroll
        for (int c8 = 0; c8 < R::kRaw; ++c8)
            r.raw[c8] = t < Lc ? __ldcg(reinterpret_cast<const uint4 *>(src) + c8) : make_uint4(0, 0, 0, 0);
    } else {
        const int gg = lane % R::G;
#pragma unroll
        for (int ps = 0; ps < R::kRaw; ++ps) {
            const int rr = ps * 8 * R::RPW + warp * R::RPW + lane / R::G;
            const int t = rr & 63;
            r.raw[ps] = make_uint4(0, 0, 0, 0);
            if (t < Lc)
                r.raw[ps] = __ldcg(reinterpret_cast<const uint4 *>((rr < 64 ? g.k : g.q) + ((size_t)bh * g.L + t0 + t) * DK +
                                                                  8 * (gg % (R::G / 2))));
        }
    }
    const int vcpr = g.d_vr / 8;
#pragma unroll
    for (int i = 0; i < R::kVChunks; ++i) {
        const int idx = tid + i * kPrepThreads, t = idx / vcpr, j = 8 * (idx % vcpr);
        r.vpre[i] = make_uint4(0, 0, 0, 0);
        if (idx < 64 * vcpr && t < Lc)
            r.vpre[i] = __ldcg(reinterpret_cast<const uint4 *>(g.v + ((size_t)bh * g.L + t0 + t) * g.d_vr + j));
    }
    r.beta_raw = __float2bfloat16_rn(0.f);
    if (!SUM && tid < Lc && tid < 64)
        r.beta_raw = g.beta[bh * g.L + t0 + tid];
}

// Barriers and tensor memory of a prep CTA (once per CTA; published by the
// first barrier inside prep_compute).
template <bool SUM>
FW_DEV void prep_init(const PrepSmem &m, int Dp, int d_v, int tid) {
    if (tid == 0) {
        mbar_init(m.bar_g, 2);
        mbar_init(m.bar_i, SUM ? 1 : 2);
        mbar_init(m.bar_f, (uint32_t)(Dp / 128 + 1));
        fence_barrier_init();
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(m.slot, prep_tmem_cols(Dp, d_v));
        tmem_relinquish();
    }
}

// Chunk c of (b,h), from the DPFP to the record: [W'; Q'] and K images, U'
// and Y'.  `parity` is the phase of this chunk on the CTA's three MMA
// barriers (each completes once per chunk).  Ends with every bulk copy done
// reading shared memory (and, with wait_writes, fully complete: before a
// ready flag is set) and a CTA barrier; false if a wait gave up.
template <int DK, bool SUM>
FW_DEV bool prep_compute(const PrepArgs &g, const PrepSmem &m, const PrepRegs<DK> &regs, int c, int64_t bh,
                         uint32_t parity, int tid, bool wait_writes) {
    using R = PrepRegs<DK>;
    constexpr int G = R::G, RPW = R::RPW, N2 = 2 * DK;
    constexpr bool kHalfRows = R::kHalfRows;
    constexpr int kRaw = R::kRaw, kVChunks = R::kVChunks;
    uint8_t *kq = m.kq, *ip = m.ip, *tp = m.ip, *tt = m.tt, *vt = m.vt;
    float *Am = m.Am, *Nm = m.Nm, *Rm = m.Rm, *bs = m.bs;
    uint64_t *bar_g = m.bar_g, *bar_i = m.bar_i, *bar_f = m.bar_f;
    const auto &raw = regs.raw;
    const auto &vpre = regs.vpre;

    const int nu = g.nu, Dp = g.Dp, d_v = g.d_v, d_vr = g.d_vr;
    const float eps = g.eps;
    unsigned *status = g.status;
    const int warp = tid >> 5, lane = tid & 31;
    const int sp = warp & 3, half = warp >> 2;           // TMEM sub-partition, column half
    const int row = 32 * sp + lane;                      // accumulator row of this thread
    const int t0 = c * g.C, Lc = min(g.C, g.L - t0);
    const int d_dot = N2 * nu;
    const Record rc = record_layout(Dp, d_v);
    uint8_t *rec = g.ws + ((size_t)bh * g.nch + c) * rc.bytes;
    const int hs = (lane >> 3) & 1;
    const int hr = 16 * warp + ((lane & 7) | ((lane >> 4) << 3));
    const int vcpr = d_vr / 8;
    (void)G; (void)RPW; (void)kRaw; (void)t0;
    bool ok = true;
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
        bs[tid] = __bfloat162float(regs.beta_raw); // 0 on padded rows
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *m.slot;
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
    ok = mbar_wait(bar_g, parity, status);
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
        ok = mbar_wait(bar_i, parity, status);
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
        ok = mbar_wait(bar_i, parity, status);
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
        ok = mbar_wait(bar_f, parity, status);
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
    // U' (rows < 64) and Y' (rows >= 64) in fp32 as the record's
    // [d_v/4][64][4] blocks, U' then Y' (contiguous in the record): where they
    // fit, staged in the fp32 work space (free once the last MMA has read V)
    // and sent as one bulk copy; else stored from registers (16-byte stores,
    // one contiguous run per warp)
    {
        const uint32_t uy_bytes = 512u * (uint32_t)d_v;
        const bool staged = uy_bytes <= (uint32_t)((2 * 64 + 16) * LDS + 64) * 4u;
        float *uy = staged ? Am + (row < 64 ? 0 : 64 * d_v) + 4 * (row & 63)
                           : reinterpret_cast<float *>(rec + (row < 64 ? rc.up : rc.yp)) + 4 * (row & 63);
        for (int c0 = 16 * half; c0 < d_v; c0 += 32) {
            float w[16];
            tmem_ld16(tm + lb + (uint32_t)(Dp + c0), w);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(uy + 256 * ((c0 + e) >> 2)) = make_float4(w[e], w[e + 1], w[e + 2], w[e + 3]);
        }
        if (staged) {
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                bulk_s2g(rec + rc.up, Am, uy_bytes);
                bulk_commit();
            }
        }
    }
teardown:
    if (tid == 0) {
        if (wait_writes)
            bulk_wait_all();  // every bulk copy of the chunk is complete
        else
            bulk_wait_read(); // the copies are done with shared memory (the writes land before the kernel ends)
    }
    tc_fence_before();
    return !__syncthreads_or(!ok);
}

// Pull chunk c of (b,h)'s q, k and v rows into L2 (a prefetch: no data
// reaches the thread, and L2 is the point of coherence).
template <int DK>
FW_DEV void prep_prefetch(const PrepArgs &g, int c, int64_t bh) {
    const int t0 = c * g.C, Lc = min(g.C, g.L - t0);
    const size_t tok = (size_t)bh * g.L + t0;
    l2_prefetch(g.k + tok * DK, (uint32_t)(Lc * DK * 2));
    l2_prefetch(g.q + tok * DK, (uint32_t)(Lc * DK * 2));
    if ((g.d_vr * 2) % 16 == 0)
        l2_prefetch(g.v + tok * g.d_vr, (uint32_t)(Lc * g.d_vr * 2));
}

// A persistent prep CTA: chunks job0, job0 + stride, ... in chunk-major
// order (job = c * BH + bh), each prepared as one chunk_prep_kernel CTA
// prepares it, the next chunk's rows pulled into L2 while the current one is
// worked out.  flags (or null): chunk c of (b,h)'s ready flag, set once its
// record is complete.  False if a wait gave up.
template <int DK, bool SUM>
FW_DEV bool prep_jobs(const PrepArgs &g, const PrepSmem &m, int BH, int job0, int stride, unsigned *flags,
                      int tid) {
    const int jobs = BH * g.nch;
    prep_init<SUM>(m, g.Dp, g.d_v, tid);
    uint32_t parity = 0;
    bool ok = true;
    for (int job = job0; job < jobs; job += stride, parity ^= 1u) {
        const int c = job / BH;
        const int64_t bh = job % BH;
        if (tid == 0 && job + stride < jobs)
            prep_prefetch<DK>(g, (job + stride) / BH, (job + stride) % BH);
        PrepRegs<DK> r;
        prep_load<DK, SUM>(g, c, bh, tid, r);
        if (!prep_compute<DK, SUM>(g, m, r, c, bh, parity, tid, flags != nullptr)) {
            ok = false;
            break;
        }
        if (flags && tid == 0)
            flag_set(flags + (size_t)bh * g.nch + c);
    }
    if ((tid >> 5) == 0)
        tmem_dealloc(*m.slot, prep_tmem_cols(g.Dp, g.d_v));
    return ok;
}

// The prep as a persistent grid (where the chunks need more than one wave of
// chunk_prep_kernel CTAs): CTA i prepares chunks i, i + gridDim.x, ...
template <int DK, bool SUM>
__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_persistent_kernel(PrepArgs g, int BH) {
    extern __shared__ uint8_t smem_raw[];
    const PrepSmem m = prep_layout(align1024(smem_raw), g.Dp);
    const int tid = threadIdx.x;
    if (tid == 0 && (int)blockIdx.x < BH * g.nch) // the first chunk's rows while the preceding kernel finishes
        prep_prefetch<DK>(g, (int)blockIdx.x / BH, (int)blockIdx.x % BH);
    griddep_wait(); // the inputs may be, and the workspace may still be read by, the preceding kernel
    PrepArgs a = g;
    a.q = after_wait(a.q);
    a.k = after_wait(a.k);
    a.v = after_wait(a.v);
    a.beta = after_wait(a.beta);
    griddep_launch_dependents();
    prep_jobs<DK, SUM>(a, m, BH, (int)blockIdx.x, (int)gridDim.x, nullptr, tid);
}

template <int DK, bool SUM>
__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_kernel(PrepArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const PrepSmem m = prep_layout(align1024(smem_raw), g.Dp);
    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * g.C, Lc = min(g.C, g.L - t0);
    // This chunk's q, k and v rows are pulled into L2 while the preceding
    // kernel finishes (a prefetch is safe before the wait: see l2_prefetch).
    if (tid == 0) {
        const size_t tok = (size_t)bh * g.L + t0;
        l2_prefetch(g.k + tok * DK, (uint32_t)(Lc * DK * 2));
        l2_prefetch(g.q + tok * DK, (uint32_t)(Lc * DK * 2));
        if ((g.d_vr * 2) % 16 == 0)
            l2_prefetch(g.v + tok * g.d_vr, (uint32_t)(Lc * g.d_vr * 2));
    }
    griddep_wait(); // the inputs may be, and the workspace may still be read by, the preceding kernel
    PrepArgs a = g;
    a.q = after_wait(a.q);
    a.k = after_wait(a.k);
    a.v = after_wait(a.v);
    a.beta = after_wait(a.beta);
    // Only now may the scan start its prologue (on free SMs): it reads the
    // caller's W0 before its own wait, which is safe once everything enqueued
    // before this kernel has completed, as it has here.
    griddep_launch_dependents();
    PrepRegs<DK> r;
    prep_load<DK, SUM>(a, c, bh, tid, r);
    prep_init<SUM>(m, a.Dp, a.d_v, tid);
    prep_compute<DK, SUM>(a, m, r, c, bh, 0, tid, false);
    if ((tid >> 5) == 0)
        tmem_dealloc(*m.slot, prep_tmem_cols(a.Dp, a.d_v));
}

// ---------------------------------------------------------------------------
// The projection prologue folded into the prep (the attention module's
// bias-free projections of the Fast Weights Transformer guide, section
// "module structure": q, k, v = x W, beta = sigmoid(x w_beta)) for one chunk
// of one head:
//   P = x[the chunk's rows] [W_q | W_k | W_v | W_beta](head h's columns)
// K (d_model) is walked in steps of 64 through a ring of NS stages of TMA copies
// placed after the prep's barrier block (the prep's own tiles are not in use
// yet): the chunk's 64 rows of x (K-major) and three 64 x 64 boxes of W_all
// (MN-major), head h's q, k and v columns.  Warp 1 issues q | k and warp 2
// v (N = 128 and 64, one accumulator each); the MMAs take M = 128 rows of x,
// the 64 past the box being the stage's next bytes, whose products land in
// accumulator lanes nobody reads.  Warps 4 and 5 meanwhile form beta's
// pre-activation x w_beta on CUDA cores from the same x rows (one thread per
// row, w_beta's column staged once).  P is rounded to bf16 (beta through the
// sigmoid first), as launch_project rounds it, into a staging area in the
// fp32 work space, from which the prep takes its inputs instead of global
// memory; the prep then runs as in chunk_prep_kernel.
constexpr int kXStage = 8192 + 3 * 8192; // one K step: the x box and three W boxes

struct ProjCols {
    int q, k, v, b; // first column of the q, k, v parts of W_all and of its beta columns
    int ldw;        // row stride of W_all (elements)
};

// The staged bf16 rows (k and q [64][DK], v [64][d_vr]) keep each row's
// 16-byte chunks in the order chunk ^ (row % chunks per row), so that the
// 16-byte stores of eight consecutive rows (one row per thread) fall in
// different banks.
FW_DEV int staged_chunk(int row, int c8, int chunks) { return row * chunks + (c8 ^ (row & (chunks - 1))); }

// prep_load's registers, from the staged bf16 rows and beta [64].
template <int DK>
FW_DEV void prep_load_staged(const __nv_bfloat16 *kst, const __nv_bfloat16 *qst, const __nv_bfloat16 *vst,
                             const __nv_bfloat16 *bst, int Lc, int d_vr, int tid, PrepRegs<DK> &r) {
    using R = PrepRegs<DK>;
    static_assert(R::kHalfRows, "d_key <= 64");
    const int warp = tid >> 5, lane = tid & 31;
    const int hr = 16 * warp + ((lane & 7) | ((lane >> 4) << 3));
    const int t = hr & 63;
    const uint4 *src = reinterpret_cast<const uint4 *>(hr < 64 ? kst : qst);
#pragma unroll
    for (int c8 = 0; c8 < R::kRaw; ++c8)
        r.raw[c8] = t < Lc ? src[staged_chunk(t, c8, R::kRaw)] : make_uint4(0, 0, 0, 0);
    const int vcpr = d_vr / 8;
#pragma unroll
    for (int i = 0; i < R::kVChunks; ++i) {
        const int idx = tid + i * kPrepThreads, tt = idx / vcpr, j8 = idx % vcpr;
        r.vpre[i] = (idx < 64 * vcpr && tt < Lc) ? reinterpret_cast<const uint4 *>(vst)[staged_chunk(tt, j8, vcpr)]
                                                 : make_uint4(0, 0, 0, 0);
    }
    r.beta_raw = (tid < Lc && tid < 64) ? bst[tid] : __float2bfloat16_rn(0.f);
}

template <int DK, int NS>
__global__ void __launch_bounds__(kPrepThreads, 2)
    chunk_prep_x_kernel(PrepArgs g, const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                        int d_model, int H, ProjCols pc, const __nv_bfloat16 *W_all) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const PrepSmem m = prep_layout(smem, g.Dp);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + 32); // [NS] a stage's copies landed
    uint64_t *empty = full + NS;                                // [NS] a stage is read (2 MMA issuers + 2 beta warps)
    uint64_t *pdone = full + 2 * NS;                            // every projection MMA is done
    uint8_t *ring = smem + kPrepHead;
    float *wb = reinterpret_cast<float *>(ring + NS * kXStage); // w_beta's column of head h [d_model]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int t0 = c * g.C, Lc = min(g.C, g.L - t0);
    const int nk = d_model / 64;

    prep_init<false>(m, g.Dp, g.d_v, tid);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 4);
        }
        mbar_init(pdone, 2);
        fence_barrier_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tx)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tw)) : "memory");
    }
    griddep_wait(); // x and W_all may be, and the workspace may still be read by, the preceding kernel
    griddep_launch_dependents();
    W_all = after_wait(W_all);
    // the copies of K step i (thread 0: the ring's first stages go out before
    // anything else, the rest as the stages free up)
    const int row0 = b * g.L + t0; // x row of the chunk's first token
    auto issue = [&](int i) {
        const int s = i % NS;
        uint8_t *st = ring + s * kXStage;
        mbar_arrive_expect_tx(full + s, kXStage);
        tma_load_2d(st, &tx, 64 * i, row0, full + s);
        tma_load_2d(st + 8192, &tw, pc.q + h * DK, 64 * i, full + s);
        tma_load_2d(st + 16384, &tw, pc.k + h * DK, 64 * i, full + s);
        tma_load_2d(st + 24576, &tw, pc.v + h * g.d_vr, 64 * i, full + s);
    };
    if (tid == 0)
        for (int i = 0; i < min(NS, nk); ++i)
            issue(i);
    for (int j = tid; j < d_model; j += kPrepThreads)
        wb[j] = __bfloat162float(__ldcg(W_all + (size_t)j * pc.ldw + pc.b + h));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *m.slot;

    bool ok = true;
    float zb = 0.f; // beta's pre-activation of this thread's row (warps 4 and 5)
    if (warp == 0 && lane == 0) {          // producer: the rest of the copies
        int issued = min(NS, nk);
        for (int i = NS; i < nk; ++i) {
            if (!mbar_wait(empty + i % NS, (uint32_t)((i / NS - 1) & 1), g.status)) {
                ok = false;
                break;
            }
            issue(i);
            issued = i + 1;
        }
        // before the ring is reused or the CTA leaves, every copy issued has landed (bounded)
        for (int i = max(0, issued - NS); i < issued; ++i)
            mbar_wait(full + i % NS, (uint32_t)((i / NS) & 1), g.status);
    } else if ((warp == 1 || warp == 2) && lane == 0) { // warp 1: q | k, warp 2: v
        const uint32_t idesc = idesc_bf16(128, warp == 1 ? 128 : 64, 0, 1);
        const uint32_t acc = tm + (uint32_t)(128 * (warp - 1));
        for (int i = 0; i < nk; ++i) {
            const int s = i % NS;
            if (!mbar_wait(full + s, (uint32_t)((i / NS) & 1), g.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_u32(ring + s * kXStage);
            const uint32_t w = a + 8192u + (uint32_t)(warp - 1) * 16384u;
#pragma unroll
            for (int st = 0; st < 4; ++st)
                mma_bf16(acc, desc_sw128(a + kmajor_step(st, 128), 16, 1024),
                         desc_sw128(w + (uint32_t)st * 2048u, 8192, 1024), idesc, (i > 0 || st > 0) ? 1u : 0u);
            mma_commit(empty + s);
        }
        mma_commit(pdone);
    } else if (warp == 4 || warp == 5) {   // beta's pre-activation, one row of x per thread
        const int row = tid - 128;
        for (int i = 0; i < nk; ++i) {
            const int s = i % NS;
            if (!mbar_wait(full + s, (uint32_t)((i / NS) & 1), g.status)) {
                ok = false;
                break;
            }
            const uint8_t *xr = ring + s * kXStage + row * 128; // the box's row: 8 swizzled 16-byte chunks
            const float *w = wb + 64 * i;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float xv[8];
                unpack8(*reinterpret_cast<const uint4 *>(xr + ((c8 ^ (row & 7)) << 4)), xv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    zb = fmaf(xv[e], w[8 * c8 + e], zb);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty + s);
        }
    }
    __syncwarp();
    ok = mbar_wait(pdone, 0, g.status) && ok;
    tc_fence_after();
    if (__syncthreads_or(!ok)) {
        tc_fence_before();
        __syncthreads();
        if (warp == 0)
            tmem_dealloc(tm, prep_tmem_cols(g.Dp, g.d_v));
        return;
    }
    // P (rows = the chunk's tokens, lanes 0..63) to the bf16 staging area:
    // warps 0 and 1 the q | k columns, warps 4 and 5 the v | beta columns
    __nv_bfloat16 *kst = reinterpret_cast<__nv_bfloat16 *>(m.Am);
    __nv_bfloat16 *qst = kst + 64 * DK;
    __nv_bfloat16 *vst = qst + 64 * DK;
    __nv_bfloat16 *bst = vst + 64 * g.d_vr;
    if ((warp & 3) < 2) {
        const int row = 32 * (warp & 3) + lane, half = warp >> 2;
        const uint32_t lb = tmem_lane_base(warp);
        constexpr int KC = DK / 8;
        const int vcpr = g.d_vr / 8;
        if (half == 1)
            bst[row] = __float2bfloat16_rn(1.0f / (1.0f + expf(-zb)));
        for (int c0 = 0; c0 < (half ? 64 : 128); c0 += 64) { // four loads in flight, then one wait
            float p[64];
#pragma unroll
            for (int j = 0; j < 64; j += 16)
                tmem_ld16(tm + lb + (uint32_t)(128 * half + c0 + j), p + j);
            tmem_ld_wait();
#pragma unroll
            for (int e8 = 0; e8 < 64; e8 += 8) {
                const int col = c0 + e8; // first of 8 columns
                if (half == 0) {
                    if (col < DK)
                        reinterpret_cast<uint4 *>(qst)[staged_chunk(row, col / 8, KC)] = pack8(p + e8);
                    else if (col >= 64 && col - 64 < DK)
                        reinterpret_cast<uint4 *>(kst)[staged_chunk(row, (col - 64) / 8, KC)] = pack8(p + e8);
                } else if (col < g.d_vr) {
                    reinterpret_cast<uint4 *>(vst)[staged_chunk(row, col / 8, vcpr)] = pack8(p + e8);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    PrepRegs<DK> r;
    prep_load_staged<DK>(kst, qst, vst, bst, Lc, g.d_vr, tid, r);
    prep_compute<DK, false>(g, m, r, c, bh, 0, tid, false);
    if (warp == 0)
        tmem_dealloc(tm, prep_tmem_cols(g.Dp, g.d_v));
}

// ---------------------------------------------------------------------------
// 16-byte chunk holding columns j0 .. j0+7 of row `row` of an MN-major SW128
// operand tile whose rows are the contraction index and whose columns are
// value channels (64-column blocks `blk` bytes apart).
FW_DEV uint32_t vtile_chunk(int row, int j0, uint32_t blk) {
    return (uint32_t)(j0 >> 6) * blk + (uint32_t)row * 128u + ((uint32_t)(((j0 & 63) >> 3) ^ (row & 7)) << 4);
}

struct ScanArgs {
    const float *W0;
    float *Wf;
    const float *z0;
    float *zf;
    __nv_bfloat16 *y;
    const uint8_t *ws;
    const unsigned *flags; // ready flags when the records are being written meanwhile, else null
    int L, C, nch, d_v, d_vr, d_dot, Dp;
    unsigned *status;
};

// One CTA walks the chunks of one (batch, head) for DVB value channels, with
// NTH threads: thread t owns accumulator row t % 128 and DVB * 128 / NTH of
// the CTA's columns (16 or 32), worked 16 at a time.  NA = number of
// [W'; Q'] buffers (2: the image of chunk c + 2 is fetched as soon as MMA1
// has read chunk c's; 1: chunk c + 1's, into the same buffer).  NKB = number
// of K buffers (2: K images two chunks ahead; 1: the next K image is
// fetched as soon as MMA3 has read the current one).
// ZN = true (the normalised sum rule): the CTA's block is 16 value channels
// followed by the record's 16-channel normaliser block (channel d_vr holds
// the running z, its output the denominator z . phi(q)); DVB = 32, NTH = 128,
// and y is written as the ratio of the value columns to that denominator (0
// where it is 0).  d_v = the record's channel count, d_vr = the value
// channels of y, W0 and W_final; z0 / zf: the normaliser state in and out
// ([B,H,d_dot]).
// FUSED = true: the records are written by other CTAs of the same launch;
// thread 0 acquires chunk j's ready flag before anything of record j is read.
template <int DVB, int NTH, int NKB, int NA, bool ZN, bool FUSED>
FW_DEV void scan_walk(const ScanArgs &g, uint8_t *smem, int vblk, int64_t bh, int tid) {
    static_assert(!ZN || (DVB == 32 && NTH == 128), "the normalised form takes 16 value + 16 normaliser channels");
    constexpr int CPT = DVB * 128 / NTH;             // columns per thread
    static_assert(CPT % 16 == 0, "16 columns at a time");
    constexpr int DS = DVB < 32 ? 32 : DVB;          // TMEM columns per accumulator region
    constexpr int VB = (DVB + 63) / 64;              // 64-column blocks of the value tiles
    const float *W0 = g.W0;
    float *Wf = g.Wf;
    const float *z0 = g.z0;
    float *zf = g.zf;
    __nv_bfloat16 *y = g.y;
    const int L = g.L, C = g.C, nch = g.nch, d_v = g.d_v, d_vr = g.d_vr, d_dot = g.d_dot, Dp = g.Dp;
    unsigned *status = g.status;
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
    uint32_t *flag_ok = slot + 1;                     // FUSED: the acquiring thread's verdict

    const int warp = tid >> 5, row = tid & 127, col0 = (tid >> 7) * CPT;
    const int v0 = vblk * (ZN ? 16 : DVB);
    // record channel of the CTA's column j (column groups of 4 stay contiguous)
    auto chan = [&](int j) { return (ZN && j >= 16) ? d_vr + (j - 16) : v0 + j; };
    const int MB = Dp / 128;
    const uint32_t ncols = tmem_cols_pow2((2 + MB) * DS);
    const uint8_t *rec0 = g.ws + (size_t)bh * nch * rc.bytes;
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
    // W0 is the caller's and never written by the prep, which lets the
    // standalone scan start only after its own wait (so everything enqueued
    // before the prep has completed): it runs before the wait for the prep.
    for (int mb = 0; mb < MB; ++mb) {
        const int d = 128 * mb + row;
#pragma unroll
        for (int j0 = 0; j0 < CPT; j0 += 16) {
            const int jc = col0 + j0;
            float w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int jj = jc + j;
                if (ZN && jj >= 16)
                    w[j] = (jj == 16 && z0 && d < d_dot) ? z0[(size_t)bh * d_dot + d] : 0.f;
                else
                    w[j] = (W0 && d < d_dot) ? W0[((size_t)bh * d_vr + v0 + jj) * d_dot + d] : 0.f;
            }
            if (has_w0)
                tmem_st16(tS + (uint32_t)(mb * DS + jc) + lb, w);
            *reinterpret_cast<uint4 *>(st + vtile_chunk(d, jc, sblk)) = pack8(w);
            *reinterpret_cast<uint4 *>(st + vtile_chunk(d, jc + 8, sblk)) = pack8(w + 8);
        }
    }
    if (has_w0)
        tmem_st_wait();
    // Thread 0's bookkeeping of the bulk loads: images issued and images
    // waited for (its own waits).
    int a_issued = 0, a_waited = 0, k_issued = 0, k_waited = 0;
    // FUSED: thread kAcq (lane 0 of warp 3, which issues no MMA) acquires the
    // ready flags, while MMA1 runs: an acquire load holds back the thread's
    // later memory accesses until it returns, and warp 3 only waits there.
    // Its verdict goes to thread 0 through shared memory; the CTA barrier
    // after MMA1 orders the acquire before thread 0's bulk copies (which a
    // proxy fence then orders after it).
    constexpr int kAcq = 96;
    int acquired = 0; // thread kAcq: the flags of chunks 0 .. acquired - 1 are acquired
    const unsigned *fl = FUSED ? g.flags + (size_t)bh * nch : nullptr;
    auto acquire_to = [&](int cc) -> bool { // thread kAcq
        if constexpr (FUSED) {
            for (; acquired <= cc && acquired < nch; ++acquired)
                if (!flag_wait(fl + acquired, status))
                    return false;
        }
        return true;
    };
    auto fetch_a = [&](int j) { // image of chunk j into buffer j % NA (thread 0)
        uint64_t *b = bar_a + (NA == 2 ? (j & 1) : 0);
        mbar_arrive_expect_tx(b, a_bytes);
        bulk_g2s(NA == 2 && (j & 1) ? at1 : at0, rec0 + (size_t)j * rc.bytes + rc.a, a_bytes, b);
        ++a_issued;
    };
    auto fetch_k = [&](int j) {
        uint64_t *b = bar_k + (NKB == 2 ? (j & 1) : 0);
        mbar_arrive_expect_tx(b, k_bytes);
        bulk_g2s(NKB == 2 && (j & 1) ? kt1 : kt0, rec0 + (size_t)j * rc.bytes + rc.k, k_bytes, b);
        ++k_issued;
    };
    // On an early exit (a wait that gave up) thread 0 waits, bounded, for the
    // bulk loads still in flight, so that none lands after the CTA has left:
    // image j sits in buffer j % NA (j % NKB), in that buffer's phase j / NA.
    auto drain = [&]() {
        if (tid != 0)
            return;
        for (int j = a_waited; j < a_issued; ++j)
            mbar_wait(bar_a + (NA == 2 ? (j & 1) : 0), (uint32_t)((NA == 2 ? j >> 1 : j) & 1), status);
        for (int j = k_waited; j < k_issued; ++j)
            mbar_wait(bar_k + (NKB == 2 ? (j & 1) : 0), (uint32_t)((NKB == 2 ? j >> 1 : j) & 1), status);
    };
    const uint8_t *wsr = g.ws;
    if constexpr (!FUSED) {
        // the workspace records are the prep kernel's: wait for it to complete
        // (and let the next kernel on the stream start its set-up meanwhile)
        griddep_launch_dependents();
        griddep_wait();
        wsr = after_wait(wsr);
        rec0 = wsr + (size_t)bh * nch * rc.bytes;
    }
    bool ok = true;
    if constexpr (FUSED) { // the flags of the chunks the first loads read
        if (tid == kAcq)
            *flag_ok = acquire_to(NA == 2 || NKB == 2 ? 1 : 0) ? 1u : 0u;
        __syncthreads();
        if (tid == 0) {
            ok = *flag_ok != 0;
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
    }
    if (tid == 0) { // chunk 0's [W'; Q'] and the first K image(s)
        if (ok) {
            fetch_a(0);
            if (NA == 2 && nch > 1)
                fetch_a(1);
            fetch_k(0);
            if (NKB == 2 && nch > 1)
                fetch_k(1);
        }
    }
    fence_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) { // nothing in flight yet
        tc_fence_before();
        __syncthreads();
        if (warp == 0)
            tmem_dealloc(tm, ncols);
        return;
    }

    // U' (rows 0..63) or Y' (rows 64..127) of a chunk, [d_v/4][64][4] in the
    // record: each 16-byte load of a warp is one 512-byte run.  Chunk c + 1's
    // are loaded once MMA3 of chunk c may start (its flag acquired by then).
    float pre[CPT];
    auto load_pre = [&](int cc) {
        const float *src =
            (const float *)(rec0 + (size_t)cc * rc.bytes + (row < 64 ? rc.up : rc.yp)) + 4 * (row & 63);
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
            const float4 f = __ldcg(reinterpret_cast<const float4 *>(src + 64 * chan(col0 + j)));
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
        ok = mbar_wait(bar_a + ab, a_parity, status);
        if (tid == 0 && ok)
            ++a_waited;
        if (__syncthreads_or(!ok)) {
            drain();
            break;
        }

        // the flags of the chunks the loads after this MMA1 read (thread kAcq)
        if (FUSED && tid == kAcq)
            *flag_ok = acquire_to(c + (NA > NKB ? NA : NKB)) ? 1u : 0u;
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
            drain();
            break;
        }
        tc_fence_after();
        // this [W'; Q'] buffer is consumed: fetch a later chunk's at once
        // (thread 0, once the ready flags of the chunks the next loads read
        // are acquired): the image's load takes most of the time until the
        // next MMA1
        bool ok_f = true;
        if (tid == 0) {
            if constexpr (FUSED) {
                ok_f = *flag_ok != 0;
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            if (ok_f && c + NA < nch)
                fetch_a(c + NA);
        }
        {
            float d1[CPT], d1b[CPT];
#pragma unroll
            for (int j0 = 0; j0 < CPT; j0 += 16) { // every load in flight, then one wait
                tmem_ld16(tD1 + lb + (uint32_t)(col0 + j0), d1 + j0);
                tmem_ld16(tD1b + lb + (uint32_t)(col0 + j0), d1b + j0);
            }
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                d1[j] += d1b[j];
            if (row < 64) {                           // U = U' - W' S^T
#pragma unroll
                for (int j0 = 0; j0 < CPT; j0 += 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        d1[j0 + j] = pre[j0 + j] - d1[j0 + j];
                    *reinterpret_cast<uint4 *>(ut + vtile_chunk(row, col0 + j0, 8192u)) = pack8(d1 + j0);
                    *reinterpret_cast<uint4 *>(ut + vtile_chunk(row, col0 + j0 + 8, 8192u)) = pack8(d1 + j0 + 8);
                }
            } else if (row - 64 < Lc) {               // y = Y' + Q' S^T
#pragma unroll
                for (int j = 0; j < CPT; ++j)
                    d1[j] += pre[j];
                if constexpr (ZN) {                   // the ratio to the normaliser column
                    const float den = d1[16];
                    const float inv = den != 0.f ? 1.0f / den : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        d1[j] *= inv;
                }
                __nv_bfloat16 *dst = y + ((size_t)bh * L + t0 + (row - 64)) * d_vr + v0 + col0;
#pragma unroll
                for (int j0 = 0; j0 < (ZN ? 16 : CPT); j0 += 8)
                    *reinterpret_cast<uint4 *>(dst + j0) = pack8(d1 + j0);
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = ok_f && mbar_wait(bar_k + kb, k_parity, status);
        if (tid == 0 && ok)
            ++k_waited;
        if (__syncthreads_or(!ok)) {
            drain();
            break;
        }
        if (c + 1 < nch)
            load_pre(c + 1);

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
            drain();
            break;
        }
        tc_fence_after();
        if (tid == 0 && c + NKB < nch) // this K buffer is consumed: fetch a later chunk's
            fetch_k(c + NKB);
        for (int mb = 0; mb < MB; ++mb) {
            const int d = 128 * mb + row;
            float sv[CPT];
#pragma unroll
            for (int j0 = 0; j0 < CPT; j0 += 16) // every load in flight, then one wait
                tmem_ld16(tS + (uint32_t)(mb * DS + col0 + j0) + lb, sv + j0);
            tmem_ld_wait();
#pragma unroll
            for (int j0 = 0; j0 < CPT; j0 += 16) {
                const int jc = col0 + j0;
                if (c + 1 < nch) {
                    *reinterpret_cast<uint4 *>(st + vtile_chunk(d, jc, sblk)) = pack8(sv + j0);
                    *reinterpret_cast<uint4 *>(st + vtile_chunk(d, jc + 8, sblk)) = pack8(sv + j0 + 8);
                } else if (d < d_dot) {
                    if (ZN && jc >= 16) {             // the normaliser state: column 16
                        if (jc == 16 && zf && vblk == 0)
                            zf[(size_t)bh * d_dot + d] = sv[j0];
                    } else if (Wf) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            Wf[((size_t)bh * d_vr + v0 + jc + j) * d_dot + d] = sv[j0 + j];
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

template <int DVB, int NTH, int NKB, int NA, bool ZN>
__global__ void __launch_bounds__(NTH) chunk_scan_kernel(ScanArgs g) {
    extern __shared__ uint8_t smem_raw[];
    scan_walk<DVB, NTH, NKB, NA, ZN, false>(g, align1024(smem_raw), blockIdx.x, blockIdx.y, threadIdx.x);
}

// The whole forward in one launch: CTAs [0, nscan) walk the chunks of a
// (value block, batch*head) as chunk_scan_kernel does, the others prepare
// chunks as chunk_prep_kernel does, chunk-major (chunk c of every (b,h)
// before chunk c + 1 of any), so the walk finds its next record ready (or
// nearly so) while the rest of the records are still being prepared.  A
// record is handed over through its ready flag, which the caller zeroes
// before the launch.  The launch is cooperative, so every CTA is resident and
// a walk that waits on a flag always waits on a CTA that is running.
// Same arithmetic as the two kernels, bit for bit.
template <int DK, int DVB, int NTH, int NKB, int NA>
__global__ void __launch_bounds__(NTH, 1) chunk_fused_kernel(PrepArgs pa, ScanArgs sa, unsigned *flags, int nscan) {
    static_assert(NTH == kPrepThreads, "one block size for both roles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int tid = threadIdx.x;
    const int nvb = sa.d_v / DVB;
    if ((int)blockIdx.x < nscan) {
        scan_walk<DVB, NTH, NKB, NA, false, true>(sa, smem, (int)blockIdx.x % nvb, (int)blockIdx.x / nvb, tid);
        return;
    }
    const int BH = nscan / nvb;
    prep_jobs<DK, false>(pa, prep_layout(smem, pa.Dp), BH, (int)blockIdx.x - nscan, (int)gridDim.x - nscan, flags,
                         tid);
}

// ---------------------------------------------------------------- host side
size_t prep_smem(int Dp, int d_v) {
    const int VB = (d_v + 63) / 64;
    (void)VB; // the V tile (<= 16 KB) reuses the fp32 work space (37 KB)
    return (size_t)kPrepHead + 256 * Dp + 16384 + 8192 + (2 * 64 + 16) * LDS * 4 + 64 * 4 + 1024;
}

size_t scan_smem(int Dp, int dvb, int nkb, int na) {
    const int VB = (dvb + 63) / 64;
    return (size_t)na * 256 * Dp + (size_t)nkb * 128 * Dp + (size_t)VB * 128 * Dp + (size_t)VB * 8192 + 64 + 1024;
}

constexpr size_t kMaxSmem = 227 * 1024;

// Dynamic shared memory of a kernel, with the whole unified L1 / shared
// array given to shared memory (these kernels keep their data there and read
// global memory through L2), so that the occupancy the runtime reports is the
// one the kernel gets.
template <typename K> cudaError_t set_smem(K kern, size_t bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
}

// Prep CTAs resident per SM: shared memory, tensor memory (512 columns per
// SM) and registers (the kernel is built for two CTAs of 256 threads).
// Counted here: the runtime's occupancy query reports one CTA per SM for
// this kernel whatever its resources, while two do run at once.
cudaError_t prep_ctas_per_sm(int Dp, int d_v, int *per_sm) {
    int dev = 0, smem_sm = 0, rsv = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess)
        return e;
    const int by_smem = (int)((size_t)smem_sm / (prep_smem(Dp, d_v) + (size_t)rsv));
    const int by_tmem = 512 / (int)prep_tmem_cols(Dp, d_v);
    *per_sm = std::max(1, std::min(std::min(by_smem, by_tmem), 2));
    return cudaSuccess;
}

bool fits(int Dp, int d_v, int dvb) {
    return Dp <= kMaxDp && Dp + d_v <= 512 && scan_smem(Dp, dvb, 1, 1) <= kMaxSmem && prep_smem(Dp, d_v) <= kMaxSmem;
}

// Value channels per scan CTA and threads per scan CTA.  The walk over the
// chunks is serial, so the per-chunk latency decides: a tcgen05.mma costs
// about the same for any N up to 128, but the per-thread work between the
// MMAs (TMEM loads, the U and S tiles, y) grows with the columns a thread
// owns, so every thread owns 16 columns: 32 channels on 256 threads, or 16
// on 128 threads where d_v is not a multiple of 32.  (Measured with 128
// threads on the b4h8 L512 and nu = 3 L2048 workloads: 16 channels per CTA
// beat 32 and 64, scan 14.4 / 18.5 / 24.5 us and 80 / 96 / 141 us.)  The
// normalised sum rule takes 16 value + 16 normaliser channels on 128 threads.
bool wide_scan(int d_v) { return d_v % 32 == 0; }

// Two K buffers when they fit in shared memory, else one; then two [W'; Q']
// buffers when those fit as well.
int choose_nkb(int Dp, int dvb) { return scan_smem(Dp, dvb, 2, 1) <= kMaxSmem ? 2 : 1; }
int choose_na(int Dp, int dvb) { return scan_smem(Dp, dvb, choose_nkb(Dp, dvb), 2) <= kMaxSmem ? 2 : 1; }

PrepArgs prep_args(const void *q, const void *k, const void *v, const void *beta, uint8_t *ws, int L, int C,
                   int nch, int nu, int Dp, int d_v, int d_vr, float eps, unsigned *status) {
    PrepArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.beta = static_cast<const __nv_bfloat16 *>(beta);
    a.ws = ws;
    a.L = L;
    a.C = C;
    a.nch = nch;
    a.nu = nu;
    a.Dp = Dp;
    a.d_v = d_v;
    a.d_vr = d_vr;
    a.eps = eps;
    a.status = status;
    return a;
}

ScanArgs scan_args(const float *W0, float *Wf, const float *z0, float *zf, void *y, const uint8_t *ws,
                   const unsigned *flags, int L, int C, int nch, int d_v, int d_vr, int d_dot, int Dp,
                   unsigned *status) {
    ScanArgs a;
    a.W0 = W0;
    a.Wf = Wf;
    a.z0 = z0;
    a.zf = zf;
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.ws = ws;
    a.flags = flags;
    a.L = L;
    a.C = C;
    a.nch = nch;
    a.d_v = d_v;
    a.d_vr = d_vr;
    a.d_dot = d_dot;
    a.Dp = Dp;
    a.status = status;
    return a;
}

// One CTA per chunk where every chunk's CTA is resident at once; otherwise
// a persistent grid of as many CTAs as the GPU holds, each looping over
// chunks (same arithmetic per chunk).
template <int DK, bool SUM>
cudaError_t launch_prep(const PrepArgs &a, int BH, int num_sms, cudaStream_t st) {
    const size_t smem = prep_smem(a.Dp, a.d_v);
    int per_sm = 0;
    cudaError_t e = prep_ctas_per_sm(a.Dp, a.d_v, &per_sm);
    if (e != cudaSuccess)
        return e;
    const long long jobs = (long long)BH * a.nch, resident = (long long)per_sm * num_sms;
    if (num_sms > 0 && jobs > resident) {
        auto kern = chunk_prep_persistent_kernel<DK, SUM>;
        e = set_smem(kern, smem);
        if (e != cudaSuccess)
            return e;
        return launch_pdl(kern, dim3((unsigned)resident), dim3(kPrepThreads), smem, st, a, BH);
    }
    auto kern = chunk_prep_kernel<DK, SUM>;
    e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3((unsigned)a.nch, (unsigned)BH), dim3(kPrepThreads), smem, st, a);
}

template <int DVB, int NTH, int NKB, int NA, bool ZN>
cudaError_t launch_scan(const ScanArgs &a, int BH, cudaStream_t st) {
    const size_t smem = scan_smem(a.Dp, DVB, NKB, NA);
    auto kern = chunk_scan_kernel<DVB, NTH, NKB, NA, ZN>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    // programmatic dependent launch: the scan's CTAs may be scheduled while
    // the preceding kernel (the prep) finishes; they wait in griddep_wait
    // before reading its output
    const dim3 grid((unsigned)(ZN ? a.d_vr / 16 : a.d_v / DVB), (unsigned)BH);
    return launch_pdl(kern, grid, dim3(NTH), smem, st, a);
}

template <int DVB, int NTH, bool ZN>
cudaError_t launch_scan_bufs(const ScanArgs &a, int BH, cudaStream_t st) {
    if (choose_nkb(a.Dp, DVB) == 2) {
        if (choose_na(a.Dp, DVB) == 2)
            return launch_scan<DVB, NTH, 2, 2, ZN>(a, BH, st);
        return launch_scan<DVB, NTH, 2, 1, ZN>(a, BH, st);
    }
    return launch_scan<DVB, NTH, 1, 1, ZN>(a, BH, st);
}

// The single-launch forward (chunk_fused_kernel): nscan walking CTAs and
// the rest preparing, as many CTAs as the GPU holds at once.  Its plan (grid
// and walking CTAs), or cudaErrorNotSupported where the two kernels are the
// better choice: when the standalone prep covers every chunk in one wave
// (there is then no later wave to overlap with the walk), or when the
// walking CTAs alone would fill the GPU.
template <int DK, int NKB, int NA>
cudaError_t fused_plan(int BH, int nch, int Dp, int d_v, int num_sms, int *grid, int *nscan) {
    constexpr int DVB = 32, NTH = 256;
    if (nch < 2 || !wide_scan(d_v) || num_sms <= 0)
        return cudaErrorNotSupported;
    const long long jobs = (long long)BH * nch;
    {
        int prep_per_sm = 0;
        const cudaError_t e = prep_ctas_per_sm(Dp, d_v, &prep_per_sm);
        if (e != cudaSuccess)
            return e;
        if (jobs <= (long long)prep_per_sm * num_sms)
            return cudaErrorNotSupported;
    }
    const size_t smem = std::max(prep_smem(Dp, d_v), scan_smem(Dp, DVB, NKB, NA));
    auto kern = chunk_fused_kernel<DK, DVB, NTH, NKB, NA>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NTH, smem);
    if (e != cudaSuccess)
        return e;
    *nscan = BH * (d_v / DVB);
    const long long resident = (long long)per_sm * num_sms;
    if (resident <= *nscan)
        return cudaErrorNotSupported;
    *grid = (int)std::min(resident, (long long)*nscan + jobs);
    return cudaSuccess;
}

template <int DK, int NKB, int NA>
cudaError_t launch_fused(const PrepArgs &pa, const ScanArgs &sa, unsigned *flags, int BH, int num_sms,
                         cudaStream_t st) {
    constexpr int DVB = 32, NTH = 256;
    int grid = 0, nscan = 0;
    cudaError_t e = fused_plan<DK, NKB, NA>(BH, pa.nch, pa.Dp, pa.d_v, num_sms, &grid, &nscan);
    if (e != cudaSuccess)
        return e;
    const size_t smem = std::max(prep_smem(pa.Dp, pa.d_v), scan_smem(pa.Dp, DVB, NKB, NA));
    e = cudaMemsetAsync(flags, 0, (size_t)BH * pa.nch * sizeof(unsigned), st);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTH);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_fused_kernel<DK, DVB, NTH, NKB, NA>, pa, sa, flags, nscan);
}

template <int DK>
cudaError_t launch_fused_bufs(const PrepArgs &pa, const ScanArgs &sa, unsigned *flags, int BH, int num_sms,
                              cudaStream_t st) {
    if (choose_nkb(pa.Dp, 32) == 2) {
        if (choose_na(pa.Dp, 32) == 2)
            return launch_fused<DK, 2, 2>(pa, sa, flags, BH, num_sms, st);
        return launch_fused<DK, 2, 1>(pa, sa, flags, BH, num_sms, st);
    }
    return launch_fused<DK, 1, 1>(pa, sa, flags, BH, num_sms, st);
}

template <int DK>
cudaError_t fused_plan_bufs(int BH, int nch, int Dp, int d_v, int num_sms, int *grid, int *nscan) {
    if (choose_nkb(Dp, 32) == 2) {
        if (choose_na(Dp, 32) == 2)
            return fused_plan<DK, 2, 2>(BH, nch, Dp, d_v, num_sms, grid, nscan);
        return fused_plan<DK, 2, 1>(BH, nch, Dp, d_v, num_sms, grid, nscan);
    }
    return fused_plan<DK, 1, 1>(BH, nch, Dp, d_v, num_sms, grid, nscan);
}

size_t records_bytes(int BH, int nch, int Dp, int d_v) { return (size_t)BH * nch * record_layout(Dp, d_v).bytes; }

} // namespace

bool tc_forward_supported(int d_key, int nu, int d_v, int chunk) {
    if (!(d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128))
        return false;
    if (!(d_v == 16 || d_v == 32 || d_v == 64 || d_v == 128))
        return false;
    if (chunk < 1 || chunk > kTile)
        return false;
    return fits(padded_ddot(2 * d_key * nu), d_v, wide_scan(d_v) ? 32 : 16);
}

// The records, then one ready flag per chunk (the single-launch forward).
size_t tc_forward_workspace_bytes(int B, int H, int L, int d_key, int nu, int d_v, int chunk) {
    const int nch = (L + chunk - 1) / chunk;
    return records_bytes(B * H, nch, padded_ddot(2 * d_key * nu), d_v) + (size_t)B * H * nch * sizeof(unsigned);
}

namespace {

template <bool SUM>
cudaError_t prep_dispatch(const PrepArgs &a, int BH, int d_key, int num_sms, cudaStream_t st) {
    switch (d_key) {
    case 8: return launch_prep<8, SUM>(a, BH, num_sms, st);
    case 16: return launch_prep<16, SUM>(a, BH, num_sms, st);
    case 32: return launch_prep<32, SUM>(a, BH, num_sms, st);
    case 64: return launch_prep<64, SUM>(a, BH, num_sms, st);
    case 128: return launch_prep<128, SUM>(a, BH, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

// The scan of the delta rule or of the unnormalised sum rule: 16 channels
// per CTA (128 threads) where those CTAs fit on the GPU at once, else 32
// (256 threads: half as many CTAs for the same per-chunk time), and 64 (256
// threads, each with 32 columns) where even the 32-channel CTAs would take
// more than one wave: a chunk step's MMAs cost about the same for N = 64 and
// the read-outs double, so one wave of 64-channel CTAs beats two of 32
// (b16h8_l2048_nu3: 156 -> 118 us).  `wide` forces 32, as the single-launch
// forward uses, so that the standalone phases of a shape that forward takes
// give the same bits.
cudaError_t scan_dispatch(const ScanArgs &a, int BH, int num_sms, bool wide, cudaStream_t st) {
    if (!wide && a.d_v % 64 == 0 && (long long)BH * (a.d_v / 32) > num_sms)
        return launch_scan_bufs<64, 256, false>(a, BH, st);
    if (wide_scan(a.d_v) && (wide || (long long)BH * (a.d_v / 16) > num_sms))
        return launch_scan_bufs<32, 256, false>(a, BH, st);
    return launch_scan_bufs<16, 128, false>(a, BH, st);
}

// Kernels the bf16 forward enqueues for this shape: 1 where fused_plan
// accepts it, else 2.
cudaError_t forward_plan(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int num_sms, int *count) {
    const int nch = (L + chunk - 1) / chunk;
    const int Dp = padded_ddot(2 * d_key * nu);
    int grid = 0, nscan = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (d_key) {
    case 8: e = fused_plan_bufs<8>(B * H, nch, Dp, d_v, num_sms, &grid, &nscan); break;
    case 16: e = fused_plan_bufs<16>(B * H, nch, Dp, d_v, num_sms, &grid, &nscan); break;
    case 32: e = fused_plan_bufs<32>(B * H, nch, Dp, d_v, num_sms, &grid, &nscan); break;
    case 64: e = fused_plan_bufs<64>(B * H, nch, Dp, d_v, num_sms, &grid, &nscan); break;
    case 128: e = fused_plan_bufs<128>(B * H, nch, Dp, d_v, num_sms, &grid, &nscan); break;
    default: break;
    }
    if (e == cudaSuccess || e == cudaErrorNotSupported) {
        *count = e == cudaSuccess ? 1 : 2;
        return cudaSuccess;
    }
    return e;
}

} // namespace

cudaError_t tc_prepare_launch(const void *q, const void *k, const void *v, const void *beta, void *workspace,
                              int B, int H, int L, int d_key, int nu, int d_v, int chunk, float eps, int num_sms,
                              unsigned *status, cudaStream_t st) {
    const int nch = (L + chunk - 1) / chunk;
    const PrepArgs a = prep_args(q, k, v, beta, static_cast<uint8_t *>(workspace), L, chunk, nch, nu,
                                 padded_ddot(2 * d_key * nu), d_v, d_v, eps, status);
    return prep_dispatch<false>(a, B * H, d_key, num_sms, st);
}

cudaError_t tc_scan_launch(const void *workspace, const float *W0, float *W_final, void *y, int B, int H, int L,
                           int d_key, int nu, int d_v, int chunk, int num_sms, unsigned *status, cudaStream_t st) {
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const ScanArgs a = scan_args(W0, W_final, nullptr, nullptr, y, static_cast<const uint8_t *>(workspace), nullptr,
                                 L, chunk, nch, d_v, d_v, d_dot, padded_ddot(d_dot), status);
    int count = 0;
    const cudaError_t e = forward_plan(B, H, L, d_key, nu, d_v, chunk, num_sms, &count);
    if (e != cudaSuccess)
        return e;
    return scan_dispatch(a, B * H, num_sms, count == 1, st);
}

int tc_forward_kernel_count(int B, int H, int L, int d_key, int nu, int d_v, int chunk, int num_sms) {
    int count = 0;
    return forward_plan(B, H, L, d_key, nu, d_v, chunk, num_sms, &count) == cudaSuccess ? count : -1;
}

// One launch (chunk_fused_kernel) where fused_plan accepts the shape;
// otherwise the two kernels.  Both give the same bits.
cudaError_t tc_forward_launch(const void *q, const void *k, const void *v, const void *beta,
                              const float *W0, float *W_final, void *y, void *workspace, int B,
                              int H, int L, int d_key, int nu, int d_v, int chunk, float eps,
                              int num_sms, unsigned *status, cudaStream_t st) {
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const int Dp = padded_ddot(d_dot);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const PrepArgs pa = prep_args(q, k, v, beta, ws, L, chunk, nch, nu, Dp, d_v, d_v, eps, status);
    {
        unsigned *flags = reinterpret_cast<unsigned *>(ws + records_bytes(BH, nch, Dp, d_v));
        const ScanArgs sa = scan_args(W0, W_final, nullptr, nullptr, y, ws, flags, L, chunk, nch, d_v, d_v, d_dot,
                                      Dp, status);
        cudaError_t e = cudaErrorNotSupported;
        switch (d_key) {
        case 8: e = launch_fused_bufs<8>(pa, sa, flags, BH, num_sms, st); break;
        case 16: e = launch_fused_bufs<16>(pa, sa, flags, BH, num_sms, st); break;
        case 32: e = launch_fused_bufs<32>(pa, sa, flags, BH, num_sms, st); break;
        case 64: e = launch_fused_bufs<64>(pa, sa, flags, BH, num_sms, st); break;
        case 128: e = launch_fused_bufs<128>(pa, sa, flags, BH, num_sms, st); break;
        default: return cudaErrorInvalidValue;
        }
        if (e != cudaErrorNotSupported)
            return e;
    }
    const cudaError_t e = prep_dispatch<false>(pa, BH, d_key, num_sms, st);
    if (e != cudaSuccess)
        return e;
    const ScanArgs sa = scan_args(W0, W_final, nullptr, nullptr, y, ws, nullptr, L, chunk, nch, d_v, d_v, d_dot, Dp,
                                  status);
    return scan_dispatch(sa, BH, num_sms, false, st);
}

// ------------------------------------------------ the prep from x (projections folded in)
bool tc_prepare_x_supported(int d_key, int d_v) { return d_key <= 64 && d_v <= 64; }

namespace {

template <int DK, int NS>
cudaError_t launch_prep_x(const PrepArgs &a, const CUtensorMap &tx, const CUtensorMap &tw, int BH, int d_model,
                          int H, ProjCols pc, const __nv_bfloat16 *W_all, cudaStream_t st) {
    const size_t smem =
        std::max(prep_smem(a.Dp, a.d_v), (size_t)kPrepHead + (size_t)NS * kXStage + 4 * (size_t)d_model + 1024);
    auto kern = chunk_prep_x_kernel<DK, NS>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3((unsigned)a.nch, (unsigned)BH), dim3(kPrepThreads), smem, st, a, tx, tw, d_model,
                      H, pc, W_all);
}

} // namespace

template <int DK>
cudaError_t launch_prep_x_stages(const PrepArgs &a, const CUtensorMap &tx, const CUtensorMap &tw, int BH,
                                 int d_model, int H, ProjCols pc, const __nv_bfloat16 *W_all, int num_sms,
                                 cudaStream_t st) {
    // four stages in flight where every CTA has an SM to itself (the ring
    // then costs the second CTA per SM nothing), else two
    if ((long long)a.nch * BH <= num_sms)
        return launch_prep_x<DK, 4>(a, tx, tw, BH, d_model, H, pc, W_all, st);
    return launch_prep_x<DK, 2>(a, tx, tw, BH, d_model, H, pc, W_all, st);
}

cudaError_t tc_prepare_x_launch(const void *x, const void *W_all, int ldw, void *workspace, int B, int H, int L,
                                int d_model, int d_key, int nu, int d_v, int chunk, float eps, int num_sms,
                                unsigned *status, cudaStream_t st) {
    if (!tc_prepare_x_supported(d_key, d_v))
        return cudaErrorInvalidValue;
    const int N = H * (2 * d_key + d_v + 1);
    CUtensorMap tx, tw;
    cudaError_t e = make_bf16_map(&tx, x, B * L, d_model, d_model, 64);
    if (e == cudaSuccess)
        e = make_bf16_map(&tw, W_all, d_model, N, ldw, 64);
    if (e != cudaSuccess)
        return e;
    const int nch = (L + chunk - 1) / chunk;
    const PrepArgs a = prep_args(nullptr, nullptr, nullptr, nullptr, static_cast<uint8_t *>(workspace), L, chunk, nch,
                                 nu, padded_ddot(2 * d_key * nu), d_v, d_v, eps, status);
    const ProjCols pc = {0, H * d_key, 2 * H * d_key, H * (2 * d_key + d_v), ldw};
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(W_all);
    switch (d_key) {
    case 8: return launch_prep_x_stages<8>(a, tx, tw, B * H, d_model, H, pc, w, num_sms, st);
    case 16: return launch_prep_x_stages<16>(a, tx, tw, B * H, d_model, H, pc, w, num_sms, st);
    case 32: return launch_prep_x_stages<32>(a, tx, tw, B * H, d_model, H, pc, w, num_sms, st);
    case 64: return launch_prep_x_stages<64>(a, tx, tw, B * H, d_model, H, pc, w, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------ the sum rule (linear attention)
bool tc_linear_supported(int d_key, int nu, int d_v, int chunk, int normalize) {
    if (!(d_key == 8 || d_key == 16 || d_key == 32 || d_key == 64 || d_key == 128))
        return false;
    if (!(d_v == 16 || d_v == 32 || d_v == 64 || d_v == 128))
        return false;
    if (chunk < 1 || chunk > kTile)
        return false;
    return fits(padded_ddot(2 * d_key * nu), d_v + (normalize ? 16 : 0), normalize || wide_scan(d_v) ? 32 : 16);
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
    const int dv2 = d_v + (normalize ? 16 : 0);
    const int BH = B * H;
    const int nch = (L + chunk - 1) / chunk;
    const int d_dot = 2 * d_key * nu;
    const int Dp = padded_ddot(d_dot);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const PrepArgs pa = prep_args(q, k, v, nullptr, ws, L, chunk, nch, nu, Dp, dv2, d_v, eps, status);
    cudaError_t e = prep_dispatch<true>(pa, BH, d_key, num_sms, st);
    if (e != cudaSuccess)
        return e;
    if (normalize)
        return launch_scan_bufs<32, 128, true>(
            scan_args(W0, W_final, z0, z_final, y, ws, nullptr, L, chunk, nch, dv2, d_v, d_dot, Dp, status), BH, st);
    return scan_dispatch(scan_args(W0, W_final, nullptr, nullptr, y, ws, nullptr, L, chunk, nch, d_v, d_v, d_dot, Dp,
                                   status),
                         BH, num_sms, false, st);
}

} // namespace fw
