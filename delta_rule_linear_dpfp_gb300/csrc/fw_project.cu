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
// slice it finishes the tile at once.  With several, the slices of a tile
// are one thread-block cluster: every CTA stages its fp32 partial tile in
// its own shared memory and sends rows [r R, r R + R) of it to cluster rank
// r with one bulk copy into r's receive buffer (distributed shared memory,
// completion counted on r's mbarrier); CTA r then adds its rows of all the
// slices in slice order (the same sum on every run) and finishes them.  The
// receive buffers lie outside the TMA ring, so a slice sends as soon as its
// own tile is staged; the one cluster barrier (every CTA's mbarriers are
// initialised) comes before the wait for the preceding kernel.
// Finishing routes every 8 columns to their head in q, k, v (16-byte
// stores) or beta (sigmoid), or adds the bias and then the residual (fp32,
// optionally also a bf16 copy) or applies ReLU (bf16).
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
// SMs, into slices that bring the grid to about kTargetCtas CTAs, at most
// kMaxSlices (the portable cluster size): measured on the layer stack's
// GEMMs (M = 256), splitting every one of them beat splitting only the long
// (K = 2048) one by 13% per token (471 vs 540 us, with the slices then added
// by a separate kernel).
constexpr int kTargetCtas = 148;
constexpr int kMaxSlices = 8;
constexpr int kPartLd = 132; // fp32 row stride of a staged partial tile (16-byte stores 4-way at most)
// the staged partial tile over the ring (once it is drained), the rows
// received from the other slices after it, then the mbarriers
constexpr int kTileBytes = 128 * kPartLd * 4;
static_assert(kTileBytes <= kStages * kStageBytes, "the staged tile fits in the ring");
constexpr int kRxOff = kStages * kStageBytes;
constexpr int kBarOff = kRxOff + kTileBytes;
constexpr int kLnOff = kBarOff + 256; // the rows' LayerNorm statistics (a DenseLn A), 1 KB

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
    // kEpiBiasResid (or null): per output row and 128-column tile n0 / 128,
    // the (mean, sum of squared deviations) of the finished values, at
    // stats[m * (ldo / 128) + n0 / 128]: a later LayerNorm's statistics
    float2 *stats;
};

// Chan's combination of group a's (mean, M2) with group b's, of na and nb
// values: the statistics of the union.
FW_DEV void chan_combine(float &mean, float &m2, float na, float mb, float m2b, float nb) {
    const float d = mb - mean, n = na + nb;
    mean = mean + d * (nb / n);
    m2 = m2 + m2b + d * d * (na * nb / n);
}
// (mean, M2) of 8 values, two passes.
FW_DEV void stats8(const float (&v)[8], float &mean, float &m2) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        s += v[e];
    mean = s * 0.125f;
    m2 = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        m2 = fmaf(v[e] - mean, v[e] - mean, m2);
}

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
FW_DEV void bias_out(const GemmOut &o, const float *acc, int m, int n, float (&t8)[8]) {
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

// 16 columns of row m; with o.stats, the 8-column groups' statistics are
// folded into the row's running (mean, M2) over `cnt` values.
template <int EPI>
FW_DEV void finish16(const GemmOut &o, const float *acc, int m, int n, int N, float &mean, float &m2, float &cnt) {
#pragma unroll
    for (int h8 = 0; h8 < 16; h8 += 8) {
        if (n + h8 >= N)
            break;
        if (EPI == kEpiHeads) {
            heads_out(o, acc + h8, m, n + h8, N);
        } else {
            float t8[8];
            bias_out<EPI>(o, acc + h8, m, n + h8, t8);
            if (EPI == kEpiBiasResid && o.stats) {
                float mb, m2b;
                stats8(t8, mb, m2b);
                if (cnt == 0.f) {
                    mean = mb;
                    m2 = m2b;
                } else {
                    chan_combine(mean, m2, cnt, mb, m2b, 8.f);
                }
                cnt += 8.f;
            }
        }
    }
}


FW_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of this CTA's shared location `saddr` in cluster rank `rank`.
FW_DEV uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(saddr), "r"(rank));
    return ra;
}
// Bulk copy of `bytes` (a multiple of 16, both ends 16-byte aligned) from
// this CTA's shared memory to another CTA's of the cluster, completion
// counted in bytes on that CTA's mbarrier (dst and bar: cluster addresses).
FW_DEV void bulk_s2cluster(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(smem_u32(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// The finish of 8 columns n .. n + 7 of row m from the slices' sum, with
// the bias (bz) and residual (rz) loaded beforehand: the same arithmetic as
// bias_out.
template <int EPI>
FW_DEV void bias_finish(const GemmOut &o, const float *acc, const float (&bz)[8], const float (&rz)[8], int m, int n,
                        float (&t8)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
        t8[e] = acc[e] + bz[e];
    const size_t off = (size_t)m * o.ldo + n;
    if (EPI == kEpiBiasResid) {
        if (o.resid) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                t8[e] += rz[e];
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

// grid (M tiles, N tiles, SL K slices); K slice z covers K steps
// [z * per, min(nk, (z + 1) * per)) of 64 (none past nk: its partial tile is
// zero).  With SL > 1 the launch groups a tile's slices into one cluster
// (1, 1, SL), so slice z is the cluster's rank z.  w_early: the weights' copies
// of the first stages are issued before the wait for the preceding kernel
// (which then must not be one that writes W while this kernel may run: in
// the layer stack it is always one of this library's kernels, none of which
// writes a weight).  ln.x (or null): A is LayerNorm(x), formed by the CTA's
// threads (every K step of the slice staged at once: per <= 2), in place of
// A's TMA copies; tx: x's fp32 tensor map (128-row x 64-column boxes).
template <int EPI, int SL>
__global__ void __launch_bounds__(kProjThreads)
    gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                const __grid_constant__ CUtensorMap tx, int K, int M, int N, int per, GemmOut o, DenseLn ln,
                int w_early, unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = (uint64_t *)(smem + kBarOff); // [kStages] a stage's copies landed
    uint64_t *empty = full + kStages;              // [kStages] a stage's MMAs are done
    uint64_t *done = empty + kStages;              // every MMA is done
    uint64_t *rx = done + 1;                       // SL > 1: the other slices' rows have landed
    uint64_t *sent = rx + 1;                       // SL > 1: every rank has received this slice's rows
    uint64_t *xbar = sent + 1;                     // [2] ln.x: x's tile of stage i has landed
    uint32_t *slot = (uint32_t *)(xbar + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128, z = blockIdx.z;
    const int nk = K / 64, kb0 = z * per, nkl = max(0, min(nk, kb0 + per) - kb0);
    constexpr uint32_t kRowsBytes = (uint32_t)(128 / SL) * kPartLd * 4; // one rank's rows of a partial tile

    // a stage is full once its copies have landed and, where A is formed
    // here, every thread has stored its row of A
    const uint32_t stage_tx = ln.x ? 16384u : (uint32_t)kStageBytes;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, ln.x ? 1u + kProjThreads : 1u);
            mbar_init(empty + s, 1);
        }
        mbar_init(done, 1);
        mbar_init(rx, 1);
        mbar_init(sent, SL > 1 ? SL - 1 : 1);
        mbar_init(xbar, 1);
        mbar_init(xbar + 1, 1);
        fence_barrier_init();
        if (SL > 1) // armed before the cluster barrier that precedes any sender's copy
            mbar_arrive_expect_tx(rx, (uint32_t)(SL - 1) * kRowsBytes);
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ta)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tb)) : "memory");
    }
    if (warp == 0) {
        tmem_alloc(slot, 128);
        tmem_relinquish();
    }
    __syncthreads(); // the barriers are initialised
    if (SL > 1)
        cluster_sync(); // ... in every CTA of the cluster, before any copy or arrival reaches them
    griddep_launch_dependents();
    const int npre = w_early ? min(kStages, nkl) : 0;
    if (warp == 0 && lane == 0) // the weights of the first stages, before the wait
        for (int i = 0; i < npre; ++i) {
            uint8_t *b = smem + i * kStageBytes + 16384;
            const int k0 = 64 * (kb0 + i);
            mbar_arrive_expect_tx(full + i, stage_tx);
            tma_load_2d(b, &tb, n0, k0, full + i);
            tma_load_2d(b + 8192, &tb, n0 + 64, k0, full + i);
        }
    griddep_wait(); // A (and, without w_early, W) may be the preceding kernel's output
    o.bias = after_wait(o.bias);
    o.resid = after_wait(o.resid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;
    if (ln.x) {
        // A = LN(x) for every stage (at most two: per <= 2).  x's fp32 tile of
        // each stage (128 rows x 64 columns, 32 KB, unswizzled) comes by TMA
        // into the ring's stages 2 and 3, which two K steps leave free, while
        // each row's mean and 1 / sqrt(var + eps) are combined from its
        // 128-column parts (thread = row) into shared memory.  Then two rows
        // per warp instruction (16 lanes x 16 bytes each) are normalised and
        // stored in bf16 into the stage's K-major 128-byte-swizzled layout.
        const float2 *stats = after_wait(ln.stats);
        float *mst = reinterpret_cast<float *>(smem + kLnOff); // [128] means, then [128] 1 / sigma
        if (tid == 0)
            for (int i = 0; i < nkl; ++i) {
                mbar_arrive_expect_tx(xbar + i, 32768u);
                tma_load_2d(smem + (2 + i) * kStageBytes, &tx, 64 * (kb0 + i), m0, xbar + i);
            }
        {
            const int m = m0 + tid;
            float mean = 0.f, rstd = 0.f;
            if (m < M) { // every part's load in flight first (parts <= 8: K <= 1024)
                float2 sp[8];
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    sp[p] = p < ln.parts ? __ldcg(stats + (size_t)m * ln.parts + p) : make_float2(0.f, 0.f);
                mean = sp[0].x;
                float m2 = sp[0].y;
#pragma unroll
                for (int p = 1; p < 8; ++p)
                    if (p < ln.parts)
                        chan_combine(mean, m2, 128.f * p, sp[p].x, sp[p].y, 128.f);
                rstd = rsqrtf(m2 / (128.f * ln.parts) + ln.eps);
            }
            mst[tid] = mean;
            mst[128 + tid] = rstd;
        }
        __syncthreads();
        const int cq = lane & 15, rsel = lane >> 4; // the lane's 4 columns of a stage; which of the 2 rows
        for (int i = 0; i < nkl; ++i) {
            // (a timeout leaves this stage's A zero: the status word reports it)
            const bool xin = mbar_wait(xbar + i, 0, status);
            uint8_t *a = smem + i * kStageBytes;
            const float *xs = reinterpret_cast<const float *>(smem + (2 + i) * kStageBytes); // [128][64]
            const int k = 64 * (kb0 + i) + 4 * cq;
            float4 g = make_float4(1.f, 1.f, 1.f, 1.f), bb = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ln.gamma)
                g = __ldg(reinterpret_cast<const float4 *>(ln.gamma + k));
            if (ln.beta)
                bb = __ldg(reinterpret_cast<const float4 *>(ln.beta + k));
#pragma unroll 4
            for (int r = 0; r < 16; ++r) {
                const int row = 32 * warp + 2 * r + rsel;
                const float mu = mst[row], rs = mst[128 + row];
                const bool live = xin && m0 + row < M;
                const float4 xr = *reinterpret_cast<const float4 *>(xs + row * 64 + 4 * cq);
                const float v0 = live ? (xr.x - mu) * rs * g.x + bb.x : 0.f;
                const float v1 = live ? (xr.y - mu) * rs * g.y + bb.y : 0.f;
                const float v2 = live ? (xr.z - mu) * rs * g.z + bb.z : 0.f;
                const float v3 = live ? (xr.w - mu) * rs * g.w + bb.w : 0.f;
                *reinterpret_cast<uint2 *>(a + (uint32_t)row * 128u + ((uint32_t)((cq >> 1) ^ (row & 7)) << 4) +
                                           (uint32_t)(cq & 1) * 8u) = make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
            }
            fence_async_smem();
            mbar_arrive(full + i);
        }
    }

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
            if (i >= npre) {
                mbar_arrive_expect_tx(full + s, stage_tx);
                tma_load_2d(b, &tb, n0, k0, full + s);
                tma_load_2d(b + 8192, &tb, n0 + 64, k0, full + s);
            }
            if (!ln.x)
                tma_load_2d(a, &ta, k0, m0, full + s);
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
    const bool bad = __syncthreads_or(!ok);
    const int m = m0 + tid;
    const uint32_t lane_base = tmem_lane_base(warp);
    if constexpr (SL == 1) {
        float mu = 0.f, m2 = 0.f, cnt = 0.f; // the row's statistics (o.stats)
        if (!bad) {
            for (int c0 = 0; c0 < 128; c0 += 16) {
                float acc[16];
                tmem_ld16(tm + lane_base + (uint32_t)c0, acc);
                tmem_ld_wait();
                if (m < M && n0 + c0 < N)
                    finish16<EPI>(o, acc, m, n0 + c0, N, mu, m2, cnt);
            }
            if (EPI == kEpiBiasResid && o.stats && m < M)
                o.stats[(size_t)m * (o.ldo / 128) + n0 / 128] = make_float2(mu, m2);
        }
    } else {
        // Rank z finishes rows [z R, z R + R) of the tile; this thread the
        // 8-column group cg of rows z R + rr + 8 j, j < UPT.  Its bias and
        // residual are loaded first, to arrive while the partials are staged.
        constexpr int R = 128 / SL, UPT = R / 8;
        const int cg = tid & 15, rr = tid >> 4, n = n0 + 8 * cg;
        float bz[8], rz[UPT][8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            bz[e] = 0.f;
        if (EPI != kEpiHeads && o.bias && n < N)
            load8(o.bias + n, bz);
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
            const int mm = m0 + z * R + rr + 8 * j;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                rz[j][e] = 0.f;
            if (EPI == kEpiBiasResid && o.resid && mm < M && n < N)
                load8(o.resid + (size_t)mm * o.ldo + n, rz[j]);
        }
        // this slice's partial tile into shared memory, over the ring (every
        // copy has landed and every MMA is done; zero for a slice past K); a
        // CTA whose wait gave up still sends its rows and takes part in both
        // cluster barriers (the status word then reports the timeout)
        float *pt = reinterpret_cast<float *>(smem), *rxb = reinterpret_cast<float *>(smem + kRxOff);
        if (!bad)
            for (int c0 = 0; c0 < 128; c0 += 16) {
                float acc[16];
                if (nkl > 0) {
                    tmem_ld16(tm + lane_base + (uint32_t)c0, acc);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        acc[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(pt + tid * kPartLd + c0 + j) =
                        make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            }
        fence_async_smem(); // the staged tile, for the bulk copies that read it
        __syncthreads();
        // rows [r R, r R + R) of the staged tile to rank r, into its receive
        // buffer's slot z (R rows at stride kPartLd are one contiguous run)
        if (tid == 0) {
            const uint32_t rx_s = smem_u32(rx), slot_s = smem_u32(rxb + (size_t)z * R * kPartLd);
            for (int r = 0; r < SL; ++r)
                if (r != z)
                    bulk_s2cluster(cluster_addr(slot_s, (uint32_t)r), pt + (size_t)r * R * kPartLd, kRowsBytes,
                                   cluster_addr(rx_s, (uint32_t)r));
        }
        (void)mbar_wait(rx, 0, status); // the other slices' rows of this rank have landed
        // ... so their copies are done with the senders' tiles: tell each
        // sender (a relaxed arrival: it publishes no data, and a release
        // would hold the warp at a cluster-scope fence for about a microsecond)
        if (tid < SL && tid != z)
            asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                             cluster_addr(smem_u32(sent), (uint32_t)tid))
                         : "memory");
        // the sums in slice order: slice z's rows from the staged tile, the
        // others' from the receive buffer
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
            const int row = rr + 8 * j; // within this rank's R rows
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] = 0.f;
#pragma unroll
            for (int zz = 0; zz < SL; ++zz) {
                const float *src = zz == z ? pt + (size_t)(z * R + row) * kPartLd + 8 * cg
                                           : rxb + (size_t)(zz * R + row) * kPartLd + 8 * cg;
                const float4 a = *reinterpret_cast<const float4 *>(src);
                const float4 b = *reinterpret_cast<const float4 *>(src + 4);
                acc[0] += a.x;
                acc[1] += a.y;
                acc[2] += a.z;
                acc[3] += a.w;
                acc[4] += b.x;
                acc[5] += b.y;
                acc[6] += b.z;
                acc[7] += b.w;
            }
            const int mm = m0 + z * R + rr + 8 * j;
            float t8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (mm < M && n < N) {
                if (EPI == kEpiHeads)
                    heads_out(o, acc, mm, n, N);
                else
                    bias_finish<EPI>(o, acc, bz, rz[j], mm, n, t8);
            }
            if (EPI == kEpiBiasResid && o.stats) {
                // the row's 128 columns lie with the 16 lanes of this
                // half-warp: their groups combined pairwise, lane cg = 0's
                // result stored
                float mu, m2;
                stats8(t8, mu, m2);
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) {
                    const float mb = __shfl_xor_sync(0xffffffffu, mu, off);
                    const float m2b = __shfl_xor_sync(0xffffffffu, m2, off);
                    chan_combine(mu, m2, 8.f * off, mb, m2b, 8.f * off);
                }
                if (cg == 0 && mm < M)
                    o.stats[(size_t)mm * (o.ldo / 128) + n0 / 128] = make_float2(mu, m2);
            }
        }
        (void)mbar_wait(sent, 0, status); // every rank has this slice's rows: the staged tile is free
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, 128);
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

// A row-major fp32 matrix [rows, cols] with row stride ld (elements) seen as
// unswizzled boxes of box_rows x 64 columns (256-byte rows); out-of-range
// elements read as zero.
cudaError_t make_f32_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows) {
    EncodeTiled fn = encoder();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
    const int want = std::min(std::min(nk, kMaxSlices), (kTargetCtas + tiles - 1) / tiles);
    int sl = 1; // a power of two (the reduction's shape is compiled per slice count)
    while (2 * sl <= want)
        sl *= 2;
    return sl;
}

size_t project_smem_bytes() { return (size_t)kLnOff + 1024 + 1024; }

bool dense_ln_supported(int M, int N, int K) {
    const int nk = K / 64, sl = gemm_slices(M, N, K);
    // x's tiles fill the ring's stages 2 and 3; a row has at most 8 parts
    return K % 128 == 0 && K <= 1024 && (nk + sl - 1) / sl <= 2;
}

template <int EPI, int SL>
cudaError_t launch_gemm_sl(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tx, int K, int M, int N,
                           const GemmOut &o, const DenseLn &ln, bool w_early, unsigned *status, cudaStream_t st) {
    const size_t smem = project_smem_bytes();
    auto kern = gemm_kernel<EPI, SL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int nk = K / 64, per = (nk + SL - 1) / SL;
    // programmatic dependent launch, and the slices of a tile as one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + 127) / 128), (unsigned)((N + 127) / 128), (unsigned)SL);
    cfg.blockDim = dim3(kProjThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = (unsigned)SL;
    cfg.attrs = attr;
    cfg.numAttrs = SL > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tx, K, M, N, per, o, ln, w_early ? 1 : 0, status);
}

template <int EPI>
cudaError_t launch_gemm_t(const void *A, const void *W, int ldw, int K, int M, int N, const GemmOut &o,
                          const DenseLn &ln, bool w_early, unsigned *status, cudaStream_t st) {
    if (ln.x && !dense_ln_supported(M, N, K))
        return cudaErrorInvalidValue;
    if (o.stats && N % 128)
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb, tx;
    // (with ln.x, A's map is encoded but never read; without, x's map is A's)
    cudaError_t e = make_map(&ta, A, M, K, K, 128);
    if (e == cudaSuccess)
        e = make_map(&tb, W, K, N, ldw, 64);
    if (e == cudaSuccess)
        e = ln.x ? make_f32_map(&tx, ln.x, M, K, K, 128) : cudaSuccess;
    if (e != cudaSuccess)
        return e;
    if (!ln.x)
        tx = ta;
    switch (gemm_slices(M, N, K)) {
    case 1: return launch_gemm_sl<EPI, 1>(ta, tb, tx, K, M, N, o, ln, w_early, status, st);
    case 2: return launch_gemm_sl<EPI, 2>(ta, tb, tx, K, M, N, o, ln, w_early, status, st);
    case 4: return launch_gemm_sl<EPI, 4>(ta, tb, tx, K, M, N, o, ln, w_early, status, st);
    default: return launch_gemm_sl<EPI, 8>(ta, tb, tx, K, M, N, o, ln, w_early, status, st);
    }
}

cudaError_t launch_project(const void *x, const void *Wall, int ldw, void *q, void *k, void *v, void *beta, int B,
                           int L, int H, int d_key, int d_v, int d_model, bool w_early, unsigned *status,
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
    return launch_gemm_t<kEpiHeads>(x, Wall, ldw, d_model, M, N, o, DenseLn{}, w_early, status, st);
}

cudaError_t launch_dense(const void *A, const void *W, int K, int M, int N, const float *bias, const float *resid,
                         void *out, bool relu, void *out_bf16_copy, bool w_early, float2 *stats, const DenseLn *ln,
                         unsigned *status, cudaStream_t st) {
    GemmOut o = {};
    o.bias = bias;
    o.resid = resid;
    o.ldo = N;
    const DenseLn lnv = ln ? *ln : DenseLn{};
    if (relu) {
        o.out_bf16 = static_cast<__nv_bfloat16 *>(out);
        return launch_gemm_t<kEpiBiasRelu>(A, W, N, K, M, N, o, lnv, w_early, status, st);
    }
    o.out_f32 = static_cast<float *>(out);
    o.out_bf16 = static_cast<__nv_bfloat16 *>(out_bf16_copy);
    o.stats = stats;
    return launch_gemm_t<kEpiBiasResid>(A, W, N, K, M, N, o, lnv, w_early, status, st);
}

} // namespace fw
