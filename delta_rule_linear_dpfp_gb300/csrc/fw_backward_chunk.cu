// fw_backward_chunk.cu -- the chunk-parallel form of the delta-rule backward.
//
// The forward's chunk algebra (the WY/UT form of the recurrence of the Fast
// Weights Transformer guide, section "FastWeightsAttention: the new update
// rule"), for one chunk of C tokens that starts from the state S (d_v x d_dot):
//   A = strict_lower(diag(beta) K K^T),  M = (I + A)^-1,  T = M diag(beta),
//   X = V - K S^T,  U = T X,  P = tril_inclusive(Q K^T),
//   Y = Q S^T + P U,  S' = S + U^T K,
// with K, Q the chunk's phi(k), phi(q) rows.  Its transpose, given dY and the
// gradient dS' of the next chunk's start state:
//   dU = P^T dY + K dS'^T,  dX = T^T dU,  dS = dS' + dY^T Q - dX^T K,
//   dV = dX,  dT = dU X^T,  dP = tril_inclusive(dY U^T),
//   dA = strict_lower(-M^T (dT diag(beta)) M^T),  B = diag(beta) dA,
//   dQ = dY S + dP K,  dK = U dS' - dX S + dP^T Q + (B + B^T) K,
//   dbeta_i = sum_j M_ji dT_ji + sum_j dA_ij (K K^T)_ij,
// then the DPFP backward of the q and k rows.  The pages print no backward
// (the guide trains through its loop with autograd); this is the chain rule
// of the chunk algebra above, equal to the token-by-token chain rule.
//
// Kernels (fp32 on CUDA cores, deterministic summation orders):
//   chunk_prep   one CTA per (b,h, chunk): K K^T, P, M (blocked: forward
//                substitution inside 16 x 16 diagonal blocks, products
//                below them), T = M diag(beta), and
//                G = dY^T Q (the part of dS that does not depend on the scan);
//   scans        one launch, two independent kinds of CTA, each per (b,h,
//                16 value rows): the state scan (the chunk-start states S in
//                chunk order, kept for the gradient kernel, with X and U) and
//                the reverse scan (chunks in reverse: dS' kept per chunk, dU,
//                dX (= dV, written out), dS = dS' + G - dX^T K, and dW0 at
//                the end);
//   chunk_grad   one CTA per (b,h, chunk): dT, dP, dA, dbeta and the phi-space
//                gradients of q and k, written where the DPFP-backward kernel
//                of fw_backward.cu reads them.
// The two scans split the state by value rows: row r of S (and of dS) only
// meets column r of X, U, dX and dU.
//
// Every kernel is a sequence of phases separated by block barriers, and no
// thread keeps a value in registers across a barrier: each phase is a
// block-stride loop over its outputs.
#include "fw_common.cuh"
#include "fw_forward_tc.h"

#include <algorithm>
#include <type_traits>

namespace fw {

namespace {

constexpr int kCC = 64;        // chunk length
constexpr int kCT = 256;       // threads per CTA
constexpr int kCR = 16;        // value rows per scan CTA
constexpr int kSl = 32;        // width of a staged slice of a contraction dimension
constexpr int kLd = kCC + 1;   // row stride of a C x C tile read along rows and columns
constexpr int kLdP = kCC + 4;  // row stride of the dP tile (16-byte rows)
constexpr int kSd = kSl + 1;   // row stride of a staged slice
constexpr int kRd = kCR + 4;   // row stride of a C x 16 tile (16-byte rows)

FW_DEV float ldf(const float *p) { return __ldcg(p); }

FW_DEV float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Stage a rows x cols block of fp32 (cols a multiple of 4, every source row
// 16-byte aligned, source row stride lds floats) into shared memory (row
// stride ldd floats); rows at or past `valid` read as zero.  16-byte loads,
// four per thread in flight before the first store.
FW_DEV void stage4(float *dst, int ldd, const float *src, size_t lds, int rows, int valid, int cols, int tid,
                   int nt) {
    const int c4 = cols >> 2, n = rows * c4;
    for (int e0 = tid; e0 < n; e0 += 4 * nt) {
        float4 t[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nt, i = e / c4;
            t[u] = (e < n && i < valid) ? __ldcg(reinterpret_cast<const float4 *>(src + (size_t)i * lds) + e % c4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nt;
            if (e < n) {
                float *d = dst + (size_t)(e / c4) * ldd + (e % c4) * 4;
                d[0] = t[u].x;
                d[1] = t[u].y;
                d[2] = t[u].z;
                d[3] = t[u].w;
            }
        }
    }
}

// Stage a rows x cols block of T (source row stride lds elements) into
// shared memory as fp32 (row stride ldd); rows at or past `valid` read as
// zero.  Four loads per thread in flight before the first store.
template <typename T>
FW_DEV void stage1(float *dst, int ldd, const T *src, size_t lds, int rows, int valid, int cols, int tid, int nt) {
    const int n = rows * cols;
    for (int e0 = tid; e0 < n; e0 += 4 * nt) {
        float t[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nt, i = e / cols;
            t[u] = (e < n && i < valid) ? io<T>::load(src + (size_t)i * lds + e % cols) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nt;
            if (e < n)
                dst[(size_t)(e / cols) * ldd + e % cols] = t[u];
        }
    }
}

FW_DEV float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// ----------------------------------------------------------- chunk_prep
// Shared memory: ks, qs [C][kSd] (a slice of the chunk's K and Q rows),
// kk, pq, ms [C][kLd], dyv [C][dvp + 1] (dY, dvp = d_v rounded up to 8), bs [C].
template <typename T>
__global__ void __launch_bounds__(kCT)
    chunk_prep_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ beta,
                      const T *__restrict__ gy, float *__restrict__ Mb, float *__restrict__ Tb,
                      float *__restrict__ Pb, float *__restrict__ KKb, float *__restrict__ Gb, int L, int d_dot,
                      int d_v, int nC) {
    extern __shared__ float sm[];
    const int dvp = (d_v + 7) & ~7, yd = dvp + 1;
    float *ks = sm, *qs = ks + kCC * kSd, *kk = qs + kCC * kSd, *pq = kk + kCC * kLd, *ms = pq + kCC * kLd;
    float *dyv = ms + kCC * kLd, *bs = dyv + kCC * yd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, c = blockIdx.y;
    const int t0 = c * kCC, cl = min(kCC, L - t0);
    const size_t tok0 = (size_t)bh * L + t0;
    const size_t cc0 = ((size_t)bh * nC + c) * kCC * kCC;
    const size_t gs0 = ((size_t)bh * nC + c) * d_v;

    for (int i = tid; i < kCC; i += nt)
        bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
    for (int e = tid; e < kCC * kCC; e += nt) {
        kk[(e / kCC) * kLd + e % kCC] = 0.f;
        pq[(e / kCC) * kLd + e % kCC] = 0.f;
    }
    for (int e = tid; e < kCC * (dvp - d_v); e += nt)
        dyv[(e / (dvp - d_v)) * yd + d_v + e % (dvp - d_v)] = 0.f;
    stage1(dyv, yd, gy + tok0 * d_v, d_v, kCC, cl, d_v, tid, nt);
    __syncthreads();
    for (int s0 = 0; s0 < d_dot; s0 += kSl) {
        const int sw = min(kSl, d_dot - s0);
        stage4(ks, kSd, phk + tok0 * d_dot + s0, d_dot, kCC, cl, sw, tid, nt);
        stage4(qs, kSd, phq + tok0 * d_dot + s0, d_dot, kCC, cl, sw, tid, nt);
        __syncthreads();
        // K K^T and Q K^T: 256 tiles of 4 x 4 outputs, rows ty + 16a, columns tx + 16b
        for (int w = tid; w < 256; w += nt) {
            const int tx = w & 15, ty = w >> 4;
            float ak[4][4], aq[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    ak[a][b] = kk[(ty + 16 * a) * kLd + tx + 16 * b];
                    aq[a][b] = pq[(ty + 16 * a) * kLd + tx + 16 * b];
                }
            for (int j = 0; j < sw; ++j) {
                float ki[4], qi[4], kj[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    ki[a] = ks[(ty + 16 * a) * kSd + j];
                    qi[a] = qs[(ty + 16 * a) * kSd + j];
                    kj[a] = ks[(tx + 16 * a) * kSd + j];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        ak[a][b] = fmaf(ki[a], kj[b], ak[a][b]);
                        aq[a][b] = fmaf(qi[a], kj[b], aq[a][b]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    kk[(ty + 16 * a) * kLd + tx + 16 * b] = ak[a][b];
                    pq[(ty + 16 * a) * kLd + tx + 16 * b] = aq[a][b];
                }
        }
        // G = dY^T Q for this slice: slice column j = w & 31, rows rb .. rb + 7
        for (int w = tid; w < (dvp / 8) * 32; w += nt) {
            const int j = w & 31, rb = (w >> 5) * 8;
            if (j < sw) {
                float acc[8];
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    acc[a] = 0.f;
                for (int i = 0; i < cl; ++i) {
                    const float qv = qs[i * kSd + j];
#pragma unroll
                    for (int a = 0; a < 8; ++a)
                        acc[a] = fmaf(dyv[i * yd + rb + a], qv, acc[a]);
                }
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    if (rb + a < d_v)
                        Gb[(gs0 + rb + a) * d_dot + s0 + j] = acc[a];
            }
        }
        __syncthreads();
    }
    // K K^T and P out; A = strict_lower(diag(beta) K K^T) replaces Q K^T in pq
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        const float g = kk[i * kLd + j], p = pq[i * kLd + j];
        KKb[cc0 + e] = g;
        Pb[cc0 + e] = j <= i ? p : 0.f;
        pq[i * kLd + j] = j < i ? bs[i] * g : 0.f;
    }
    __syncthreads();
    // M = (I + A)^-1, unit lower, in blocks of kB: the diagonal blocks by
    // forward substitution (one thread per column), then the blocks below
    // the diagonal one block distance d at a time, from (I + A) M = I:
    //   M_IJ = -M_II Z_IJ,  Z_IJ = sum_{K=J}^{I-1} A_IK M_KJ  (I = J + d),
    // with Z in the dead K slice buffer.
    constexpr int kB = 16, kNB = kCC / kB;
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        if (i < j)
            ms[i * kLd + j] = 0.f;
    }
    for (int j = tid; j < kCC; j += nt) {
        const int bend = (j / kB + 1) * kB;
        ms[j * kLd + j] = 1.f;
        for (int i = j + 1; i < bend; ++i) {
            float acc = 0.f;
            for (int m = j; m < i; ++m)
                acc = fmaf(pq[i * kLd + m], ms[m * kLd + j], acc);
            ms[i * kLd + j] = -acc;
        }
    }
    __syncthreads();
    float *zb = ks; // (kNB - 1) blocks of kB x kB
    for (int d = 1; d < kNB; ++d) {
        const int nblk = kNB - d;
        for (int w = tid; w < nblk * kB * kB; w += nt) {
            const int J = w / (kB * kB), a = (w / kB) % kB, b = w % kB, I = J + d;
            float acc = 0.f;
            for (int m = J * kB; m < I * kB; ++m)
                acc = fmaf(pq[(I * kB + a) * kLd + m], ms[m * kLd + J * kB + b], acc);
            zb[w] = acc;
        }
        __syncthreads();
        for (int w = tid; w < nblk * kB * kB; w += nt) {
            const int J = w / (kB * kB), a = (w / kB) % kB, b = w % kB, I = J + d;
            float acc = 0.f;
            for (int c = 0; c < kB; ++c)
                acc = fmaf(ms[(I * kB + a) * kLd + I * kB + c], zb[J * kB * kB + c * kB + b], acc);
            ms[(I * kB + a) * kLd + J * kB + b] = -acc;
        }
        __syncthreads();
    }
    for (int e = tid; e < kCC * kCC; e += nt) {
        const float mv = ms[(e / kCC) * kLd + e % kCC];
        Mb[cc0 + e] = mv;
        Tb[cc0 + e] = mv * bs[e % kCC];
    }
}

// ----------------------------------------------------------- state_scan
// Shared memory: ss [kCR][d_dot + 4] (the CTA's rows of S), kc [C][d_dot + 4],
// tc [C][kLd] (T), xs, us [C][kRd].
template <typename T>
FW_DEV void state_scan(float *sm, const float *__restrict__ phk, const T *__restrict__ v, const float *__restrict__ W0,
                       const float *__restrict__ Tb, float *__restrict__ Sb, float *__restrict__ Xb,
                       float *__restrict__ Ub, int L, int d_dot, int d_v, int nC, int bh, int rb) {
    const int sd = d_dot + 4, d4 = d_dot >> 2;
    float *ss = sm, *kc = ss + kCR * sd, *tc = kc + kCC * sd, *xs = tc + kCC * kLd, *us = xs + kCC * kRd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int r0 = rb * kCR, R = min(kCR, d_v - r0);

    if (W0)
        stage4(ss, sd, W0 + ((size_t)bh * d_v + r0) * d_dot, d_dot, kCR, R, d_dot, tid, nt);
    else
        for (int e = tid; e < kCR * d_dot; e += nt)
            ss[(e / d_dot) * sd + e % d_dot] = 0.f;
    __syncthreads();
    for (int c = 0; c < nC; ++c) {
        const int t0 = c * kCC, cl = min(kCC, L - t0);
        const size_t tok0 = (size_t)bh * L + t0;
        const size_t st0 = ((size_t)bh * nC + c) * d_v;
        for (int e = tid; e < R * d_dot; e += nt) {
            const int r = e / d_dot, m = e % d_dot;
            Sb[(st0 + r0 + r) * d_dot + m] = ss[r * sd + m];
        }
        stage4(kc, sd, phk + tok0 * d_dot, d_dot, kCC, cl, d_dot, tid, nt);
        stage4(tc, kLd, Tb + ((size_t)bh * nC + c) * kCC * kCC, kCC, kCC, kCC, kCC, tid, nt);
        for (int e = tid; e < kCC * (kCR - R); e += nt)
            xs[(e / (kCR - R)) * kRd + R + e % (kCR - R)] = 0.f;
        stage1(xs, kRd, v + tok0 * d_v + r0, d_v, kCC, cl, R, tid, nt);
        __syncthreads();
        // X = V - K S^T: 256 tiles, row r = w & 15, tokens (w >> 4) + 16a
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
            float acc[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                acc[a] = 0.f;
            for (int m4 = 0; m4 < d4; ++m4) {
                const float4 s = lds4(ss + r * sd + 4 * m4);
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    acc[a] = dot4(lds4(kc + (i0 + 16 * a) * sd + 4 * m4), s, acc[a]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                const float x = xs[i * kRd + r] - acc[a];
                xs[i * kRd + r] = x;
                if (i < cl && r < R)
                    Xb[(tok0 + i) * d_v + r0 + r] = x;
            }
        }
        __syncthreads();
        // U = T X (T lower)
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                float acc = 0.f;
                for (int s = 0; s <= i; ++s)
                    acc = fmaf(tc[i * kLd + s], xs[s * kRd + r], acc);
                us[i * kRd + r] = acc;
                if (i < cl && r < R)
                    Ub[(tok0 + i) * d_v + r0 + r] = acc;
            }
        }
        __syncthreads();
        // S += U^T K: thread per (column m, half of the rows)
        for (int e = tid; e < 2 * d_dot; e += nt) {
            const int m = e % d_dot, rh = (e / d_dot) * (kCR / 2);
            float acc[kCR / 2];
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                acc[r] = ss[(rh + r) * sd + m];
            for (int i = 0; i < cl; ++i) {
                const float kv = kc[i * sd + m];
                const float4 u0 = lds4(us + i * kRd + rh), u1 = lds4(us + i * kRd + rh + 4);
                acc[0] = fmaf(u0.x, kv, acc[0]);
                acc[1] = fmaf(u0.y, kv, acc[1]);
                acc[2] = fmaf(u0.z, kv, acc[2]);
                acc[3] = fmaf(u0.w, kv, acc[3]);
                acc[4] = fmaf(u1.x, kv, acc[4]);
                acc[5] = fmaf(u1.y, kv, acc[5]);
                acc[6] = fmaf(u1.z, kv, acc[6]);
                acc[7] = fmaf(u1.w, kv, acc[7]);
            }
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                ss[(rh + r) * sd + m] = acc[r];
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ grad_scan
// Shared memory: ds [kCR][d_dot + 4] (the CTA's rows of dS), kc [C][d_dot + 4],
// tc, pc [C][kLd] (T and P), dys, dus, dxs [C][kRd].
template <typename T>
FW_DEV void grad_scan(float *sm, const float *__restrict__ phk, const T *__restrict__ gy,
                      const float *__restrict__ gWL, const float *__restrict__ Tb, const float *__restrict__ Pb,
                      const float *__restrict__ Gb, float *__restrict__ dSb, float *__restrict__ dXb,
                      float *__restrict__ dUb, T *__restrict__ gv, float *__restrict__ gW0, int L, int d_dot, int d_v,
                      int nC, int bh, int rb) {
    const int sd = d_dot + 4, d4 = d_dot >> 2;
    float *ds = sm, *kc = ds + kCR * sd, *tc = kc + kCC * sd, *pc = tc + kCC * kLd, *dys = pc + kCC * kLd;
    float *dus = dys + kCC * kRd, *dxs = dus + kCC * kRd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int r0 = rb * kCR, R = min(kCR, d_v - r0);

    if (gWL)
        stage4(ds, sd, gWL + ((size_t)bh * d_v + r0) * d_dot, d_dot, kCR, R, d_dot, tid, nt);
    else
        for (int e = tid; e < kCR * d_dot; e += nt)
            ds[(e / d_dot) * sd + e % d_dot] = 0.f;
    __syncthreads();
    for (int c = nC - 1; c >= 0; --c) {
        const int t0 = c * kCC, cl = min(kCC, L - t0);
        const size_t tok0 = (size_t)bh * L + t0;
        const size_t st0 = ((size_t)bh * nC + c) * d_v;
        const size_t cc0 = ((size_t)bh * nC + c) * kCC * kCC;
        for (int e = tid; e < R * d_dot; e += nt) {
            const int r = e / d_dot, m = e % d_dot;
            dSb[(st0 + r0 + r) * d_dot + m] = ds[r * sd + m];
        }
        stage4(kc, sd, phk + tok0 * d_dot, d_dot, kCC, cl, d_dot, tid, nt);
        stage4(tc, kLd, Tb + cc0, kCC, kCC, kCC, kCC, tid, nt);
        stage4(pc, kLd, Pb + cc0, kCC, kCC, kCC, kCC, tid, nt);
        for (int e = tid; e < kCC * (kCR - R); e += nt)
            dys[(e / (kCR - R)) * kRd + R + e % (kCR - R)] = 0.f;
        stage1(dys, kRd, gy + tok0 * d_v + r0, d_v, kCC, cl, R, tid, nt);
        __syncthreads();
        // dU = K dS'^T + P^T dY (P lower, so P_si is zero for s < i)
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
            float acc[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                acc[a] = 0.f;
            for (int m4 = 0; m4 < d4; ++m4) {
                const float4 s = lds4(ds + r * sd + 4 * m4);
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    acc[a] = dot4(lds4(kc + (i0 + 16 * a) * sd + 4 * m4), s, acc[a]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                for (int s = i; s < kCC; ++s)
                    acc[a] = fmaf(pc[s * kLd + i], dys[s * kRd + r], acc[a]);
                dus[i * kRd + r] = acc[a];
                if (i < cl && r < R)
                    dUb[(tok0 + i) * d_v + r0 + r] = acc[a];
            }
        }
        __syncthreads();
        // dX = T^T dU = dV
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                float acc = 0.f;
                for (int s = i; s < kCC; ++s)
                    acc = fmaf(tc[s * kLd + i], dus[s * kRd + r], acc);
                dxs[i * kRd + r] = acc;
                if (i < cl && r < R) {
                    dXb[(tok0 + i) * d_v + r0 + r] = acc;
                    io<T>::store(gv + (tok0 + i) * d_v + r0 + r, acc);
                }
            }
        }
        __syncthreads();
        // dS = dS' + G - dX^T K: thread per (column m, half of the rows)
        for (int e = tid; e < 2 * d_dot; e += nt) {
            const int m = e % d_dot, rh = (e / d_dot) * (kCR / 2);
            float acc[kCR / 2];
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                acc[r] = ds[(rh + r) * sd + m] + (rh + r < R ? ldf(Gb + (st0 + r0 + rh + r) * d_dot + m) : 0.f);
            for (int i = 0; i < cl; ++i) {
                const float kv = kc[i * sd + m];
                const float4 x0 = lds4(dxs + i * kRd + rh), x1 = lds4(dxs + i * kRd + rh + 4);
                acc[0] = fmaf(-x0.x, kv, acc[0]);
                acc[1] = fmaf(-x0.y, kv, acc[1]);
                acc[2] = fmaf(-x0.z, kv, acc[2]);
                acc[3] = fmaf(-x0.w, kv, acc[3]);
                acc[4] = fmaf(-x1.x, kv, acc[4]);
                acc[5] = fmaf(-x1.y, kv, acc[5]);
                acc[6] = fmaf(-x1.z, kv, acc[6]);
                acc[7] = fmaf(-x1.w, kv, acc[7]);
            }
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                ds[(rh + r) * sd + m] = acc[r];
        }
        __syncthreads();
    }
    if (gW0)
        for (int e = tid; e < R * d_dot; e += nt) {
            const int r = e / d_dot, m = e % d_dot;
            gW0[((size_t)bh * d_v + r0 + r) * d_dot + m] = ds[r * sd + m];
        }
}

// ----------------------------------------------------------------- scans
// The two scans do not depend on each other (the reverse scan needs T, P, G,
// K and dY, not S), so one launch runs both: blocks y < nRB scan the states,
// the others their gradients.
template <typename T>
__global__ void __launch_bounds__(kCT)
    scans_kernel(const float *__restrict__ phk, const T *__restrict__ v, const T *__restrict__ gy,
                 const float *__restrict__ W0, const float *__restrict__ gWL, const float *__restrict__ Tb,
                 const float *__restrict__ Pb, const float *__restrict__ Gb, float *__restrict__ Sb,
                 float *__restrict__ Xb, float *__restrict__ Ub, float *__restrict__ dSb, float *__restrict__ dXb,
                 float *__restrict__ dUb, T *__restrict__ gv, float *__restrict__ gW0, int L, int d_dot, int d_v,
                 int nC, int nRB) {
    extern __shared__ float sm[];
    if ((int)blockIdx.y < nRB)
        state_scan<T>(sm, phk, v, W0, Tb, Sb, Xb, Ub, L, d_dot, d_v, nC, blockIdx.x, blockIdx.y);
    else
        grad_scan<T>(sm, phk, gy, gWL, Tb, Pb, Gb, dSb, dXb, dUb, gv, gW0, L, d_dot, d_v, nC, blockIdx.x,
                     blockIdx.y - nRB);
}

// ------------------------------------------------------------ chunk_grad
// Shared memory: c1 (dT, then dA), c3 (M), c4 (M^T dT diag(beta), then
// B + B^T), each [C][kLd]; c2 (dP) [C][kLdP]; dys, uvs, dxs [C][d_v + 1]; a
// staging region (slices of dU and X, later of S, dS' [d_v][SW + 4] and K, Q
// [C][SW + 4]); bs, gb [C].  SW: the width of a feature slice (64 or 32).
template <int SW> __host__ __device__ constexpr int grad_stage_floats(int d_v) {
    return 2 * kCC * kSd > (2 * d_v + 2 * kCC) * (SW + 4) ? 2 * kCC * kSd : (2 * d_v + 2 * kCC) * (SW + 4);
}

template <typename T, int SW>
__global__ void __launch_bounds__(kCT)
    chunk_grad_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ beta,
                      const T *__restrict__ gy, const float *__restrict__ Sb, const float *__restrict__ dSb,
                      const float *__restrict__ Xb, const float *__restrict__ Ub, const float *__restrict__ dXb,
                      const float *__restrict__ dUb, const float *__restrict__ Mb, const float *__restrict__ KKb,
                      float *__restrict__ part, int L, int d_dot, int d_v, int nC) {
    constexpr int NCG = SW / 4, NTG = kCT / NCG, TPT = kCC / NTG, ld6 = SW + 4;
    extern __shared__ float sm[];
    const int vd = d_v + 1;
    const size_t pst = 2 * (size_t)d_dot + 4;
    float *c1 = sm, *c3 = c1 + kCC * kLd, *c4 = c3 + kCC * kLd, *c2 = c4 + kCC * kLd;
    float *dys = c2 + kCC * kLdP, *uvs = dys + kCC * vd, *dxs = uvs + kCC * vd, *stg = dxs + kCC * vd;
    float *bs = stg + grad_stage_floats<SW>(d_v), *gb = bs + kCC;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, c = blockIdx.y;
    const int t0 = c * kCC, cl = min(kCC, L - t0);
    const size_t tok0 = (size_t)bh * L + t0;
    const size_t cc0 = ((size_t)bh * nC + c) * kCC * kCC;
    const size_t st0 = ((size_t)bh * nC + c) * d_v;

    for (int i = tid; i < kCC; i += nt)
        bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
    stage1(dys, vd, gy + tok0 * d_v, d_v, kCC, cl, d_v, tid, nt);
    stage1(uvs, vd, Ub + tok0 * d_v, d_v, kCC, cl, d_v, tid, nt);
    stage1(dxs, vd, dXb + tok0 * d_v, d_v, kCC, cl, d_v, tid, nt);
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        c1[i * kLd + j] = 0.f;
        c2[i * kLdP + j] = 0.f;
    }
    __syncthreads();
    // dT = dU X^T and dY U^T, over slices of the value dimension
    float *dul = stg, *xl = stg + kCC * kSd;
    for (int r0 = 0; r0 < d_v; r0 += kSl) {
        const int rn = min(kSl, d_v - r0);
        stage1(dul, kSd, dUb + tok0 * d_v + r0, d_v, kCC, cl, rn, tid, nt);
        stage1(xl, kSd, Xb + tok0 * d_v + r0, d_v, kCC, cl, rn, tid, nt);
        __syncthreads();
        for (int w = tid; w < 256; w += nt) {
            const int tx = w & 15, ty = w >> 4;
            float at[4][4], ap[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    at[a][b] = c1[(ty + 16 * a) * kLd + tx + 16 * b];
                    ap[a][b] = c2[(ty + 16 * a) * kLdP + tx + 16 * b];
                }
            for (int j = 0; j < rn; ++j) {
                float du[4], xj[4], dy[4], uj[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    du[a] = dul[(ty + 16 * a) * kSd + j];
                    xj[a] = xl[(tx + 16 * a) * kSd + j];
                    dy[a] = dys[(ty + 16 * a) * vd + r0 + j];
                    uj[a] = uvs[(tx + 16 * a) * vd + r0 + j];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        at[a][b] = fmaf(du[a], xj[b], at[a][b]);
                        ap[a][b] = fmaf(dy[a], uj[b], ap[a][b]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    c1[(ty + 16 * a) * kLd + tx + 16 * b] = at[a][b];
                    c2[(ty + 16 * a) * kLdP + tx + 16 * b] = ap[a][b];
                }
        }
        __syncthreads();
    }
    // M in, K K^T into the staging region; dP = tril_inclusive(dY U^T)
    float *kks = stg;
    stage4(c3, kLd, Mb + cc0, kCC, kCC, kCC, kCC, tid, nt);
    stage4(kks, kLd, KKb + cc0, kCC, kCC, kCC, kCC, tid, nt);
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        if (j > i)
            c2[i * kLdP + j] = 0.f;
    }
    __syncthreads();
    // dbeta's first part, column sums of M * dT; c4 = M^T (dT diag(beta))
    for (int i = tid; i < kCC; i += nt) {
        float acc = 0.f;
        for (int j = i; j < kCC; ++j)
            acc = fmaf(c3[j * kLd + i], c1[j * kLd + i], acc);
        gb[i] = acc;
    }
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        float acc = 0.f;
        for (int s = i; s < kCC; ++s)
            acc = fmaf(c3[s * kLd + i], c1[s * kLd + j], acc);
        c4[i * kLd + j] = acc * bs[j];
    }
    __syncthreads();
    // dA = strict_lower(-c4 M^T), into c1
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        float acc = 0.f;
        if (j < i)
            for (int s = 0; s <= j; ++s)
                acc = fmaf(c4[i * kLd + s], c3[j * kLd + s], acc);
        c1[i * kLd + j] = -acc;
    }
    __syncthreads();
    // dbeta's second part, row sums of dA * K K^T; c4 = B + B^T, B = diag(beta) dA
    for (int i = tid; i < kCC; i += nt) {
        float acc = gb[i];
        for (int j = 0; j < i; ++j)
            acc = fmaf(c1[i * kLd + j], kks[i * kLd + j], acc);
        gb[i] = acc;
    }
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        c4[i * kLd + j] = bs[i] * c1[i * kLd + j] + bs[j] * c1[j * kLd + i];
    }
    __syncthreads();
    for (int i = tid; i < cl; i += nt)
        part[(tok0 + i) * pst + 2 * (size_t)d_dot] = gb[i];
    // dQ = dY S + dP K and dK = U dS' - dX S + dP^T Q + (B + B^T) K, over
    // slices of the feature dimension; a thread owns TPT tokens x 4 columns
    float *sl = stg, *dsl = sl + d_v * ld6, *kl = dsl + d_v * ld6, *ql = kl + kCC * ld6;
    for (int m0 = 0; m0 < d_dot; m0 += SW) {
        const int sw = min(SW, d_dot - m0);
        stage4(sl, ld6, Sb + st0 * d_dot + m0, d_dot, d_v, d_v, sw, tid, nt);
        stage4(dsl, ld6, dSb + st0 * d_dot + m0, d_dot, d_v, d_v, sw, tid, nt);
        stage4(kl, ld6, phk + tok0 * d_dot + m0, d_dot, kCC, cl, sw, tid, nt);
        stage4(ql, ld6, phq + tok0 * d_dot + m0, d_dot, kCC, cl, sw, tid, nt);
        __syncthreads();
        for (int w = tid; w < kCT; w += nt) {
            const int cg = w % NCG, i0 = (w / NCG) * TPT, j4 = 4 * cg;
            if (j4 < sw) {
                float aq[TPT][4], ak[TPT][4];
#pragma unroll
                for (int a = 0; a < TPT; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        aq[a][b] = ak[a][b] = 0.f;
                for (int r = 0; r < d_v; ++r) {
                    const float4 s = lds4(sl + r * ld6 + j4), d = lds4(dsl + r * ld6 + j4);
#pragma unroll
                    for (int a = 0; a < TPT; ++a) {
                        const float y = dys[(i0 + a) * vd + r], u = uvs[(i0 + a) * vd + r];
                        const float x = -dxs[(i0 + a) * vd + r];
                        aq[a][0] = fmaf(y, s.x, aq[a][0]);
                        aq[a][1] = fmaf(y, s.y, aq[a][1]);
                        aq[a][2] = fmaf(y, s.z, aq[a][2]);
                        aq[a][3] = fmaf(y, s.w, aq[a][3]);
                        ak[a][0] = fmaf(u, d.x, fmaf(x, s.x, ak[a][0]));
                        ak[a][1] = fmaf(u, d.y, fmaf(x, s.y, ak[a][1]));
                        ak[a][2] = fmaf(u, d.z, fmaf(x, s.z, ak[a][2]));
                        ak[a][3] = fmaf(u, d.w, fmaf(x, s.w, ak[a][3]));
                    }
                }
                for (int s = 0; s < cl; ++s) {
                    const float4 kv = lds4(kl + s * ld6 + j4), qv = lds4(ql + s * ld6 + j4);
#pragma unroll
                    for (int a = 0; a < TPT; ++a) {
                        const float p = c2[(i0 + a) * kLdP + s], pt = c2[s * kLdP + i0 + a];
                        const float b = c4[(i0 + a) * kLd + s];
                        aq[a][0] = fmaf(p, kv.x, aq[a][0]);
                        aq[a][1] = fmaf(p, kv.y, aq[a][1]);
                        aq[a][2] = fmaf(p, kv.z, aq[a][2]);
                        aq[a][3] = fmaf(p, kv.w, aq[a][3]);
                        ak[a][0] = fmaf(b, kv.x, fmaf(pt, qv.x, ak[a][0]));
                        ak[a][1] = fmaf(b, kv.y, fmaf(pt, qv.y, ak[a][1]));
                        ak[a][2] = fmaf(b, kv.z, fmaf(pt, qv.z, ak[a][2]));
                        ak[a][3] = fmaf(b, kv.w, fmaf(pt, qv.w, ak[a][3]));
                    }
                }
#pragma unroll
                for (int a = 0; a < TPT; ++a)
                    if (i0 + a < cl) {
                        float *dst = part + (tok0 + i0 + a) * pst + m0 + j4;
                        *reinterpret_cast<float4 *>(dst) = make_float4(aq[a][0], aq[a][1], aq[a][2], aq[a][3]);
                        *reinterpret_cast<float4 *>(dst + d_dot) = make_float4(ak[a][0], ak[a][1], ak[a][2], ak[a][3]);
                    }
            }
        }
        __syncthreads();
    }
}

size_t prep_smem(int d_v) {
    const size_t dvp = ((size_t)d_v + 7) & ~(size_t)7;
    return sizeof(float) * (2 * kCC * kSd + 3 * kCC * kLd + kCC * (dvp + 1) + kCC);
}
size_t scan_smem(int d_dot) {
    return sizeof(float) * ((size_t)(kCR + kCC) * (d_dot + 4) + kCC * kLd + 2 * kCC * kRd);
}
size_t gscan_smem(int d_dot) {
    return sizeof(float) * ((size_t)(kCR + kCC) * (d_dot + 4) + 2 * kCC * kLd + 3 * kCC * kRd);
}
template <int SW> size_t cgrad_smem(int d_v) {
    return sizeof(float) * (3 * kCC * kLd + kCC * kLdP + 3 * (size_t)kCC * (d_v + 1) + grad_stage_floats<SW>(d_v) +
                            2 * kCC);
}
constexpr size_t kSmemCap = (size_t)227 * 1024;

// Offsets (in floats) of the buffers after phi(k), phi(q) and the per-token
// gradient records inside the workspace.
struct ChunkLayout {
    size_t M, T, P, KK, G, S, dS, X, U, dX, dU, end;
};

ChunkLayout chunk_layout(int BH, int L, int d_dot, int d_v) {
    const size_t rows = (size_t)BH * L, nC = ((size_t)L + kCC - 1) / kCC, cc = (size_t)BH * nC * kCC * kCC;
    const size_t sts = (size_t)BH * nC * d_v * d_dot;
    ChunkLayout o;
    o.M = 0;
    o.T = o.M + cc;
    o.P = o.T + cc;
    o.KK = o.P + cc;
    o.G = o.KK + cc;
    o.S = o.G + sts;
    o.dS = o.S + sts;
    o.X = o.dS + sts;
    o.U = o.X + rows * d_v;
    o.dX = o.U + rows * d_v;
    o.dU = o.dX + rows * d_v;
    o.end = o.dU + rows * d_v;
    return o;
}

template <typename T>
cudaError_t launch_chunked_t(const float *phk, const float *phq, const void *v, const void *beta, const float *W0,
                             const void *gy, const float *gWL, void *gv, float *gW0, float *part, float *buf, int BH,
                             int L, int d_dot, int d_v, cudaStream_t st) {
    const int nC = (L + kCC - 1) / kCC, nRB = (d_v + kCR - 1) / kCR;
    const ChunkLayout o = chunk_layout(BH, L, d_dot, d_v);
    const T *vt = static_cast<const T *>(v), *bt = static_cast<const T *>(beta), *gyt = static_cast<const T *>(gy);
    const dim3 chunks((unsigned)BH, (unsigned)nC);
    cudaError_t e;
    {
        auto kern = chunk_prep_kernel<T>;
        const size_t smem = prep_smem(d_v);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kern<<<chunks, kCT, smem, st>>>(phk, phq, bt, gyt, buf + o.M, buf + o.T, buf + o.P, buf + o.KK, buf + o.G, L,
                                        d_dot, d_v, nC);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    {
        auto kern = scans_kernel<T>;
        const size_t smem = std::max(scan_smem(d_dot), gscan_smem(d_dot));
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kern<<<dim3((unsigned)BH, 2u * nRB), kCT, smem, st>>>(
            phk, vt, gyt, W0, gWL, buf + o.T, buf + o.P, buf + o.G, buf + o.S, buf + o.X, buf + o.U, buf + o.dS,
            buf + o.dX, buf + o.dU, static_cast<T *>(gv), gW0, L, d_dot, d_v, nC, nRB);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    const bool wide = cgrad_smem<64>(d_v) <= kSmemCap;
    auto kern = wide ? chunk_grad_kernel<T, 64> : chunk_grad_kernel<T, 32>;
    const size_t smem = wide ? cgrad_smem<64>(d_v) : cgrad_smem<32>(d_v);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kern<<<chunks, kCT, smem, st>>>(phk, phq, bt, gyt, buf + o.S, buf + o.dS, buf + o.X, buf + o.U, buf + o.dX,
                                    buf + o.dU, buf + o.M, buf + o.KK, part, L, d_dot, d_v, nC);
    return cudaGetLastError();
}

} // namespace

bool backward_chunked_supported(int d_key, int nu, int d_v, int L) {
    const int d_dot = 2 * d_key * nu;
    return d_dot <= 512 && d_v <= 128 && ((int64_t)L + kCC - 1) / kCC <= 65535 && prep_smem(d_v) <= kSmemCap &&
           scan_smem(d_dot) <= kSmemCap && gscan_smem(d_dot) <= kSmemCap && cgrad_smem<32>(d_v) <= kSmemCap;
}

size_t backward_chunked_buffer_floats(int BH, int L, int d_key, int nu, int d_v) {
    return chunk_layout(BH, L, 2 * d_key * nu, d_v).end;
}

cudaError_t launch_backward_chunked(const float *phk, const float *phq, const void *v, const void *beta,
                                    const float *W0, const void *gy, const float *gWL, void *gv, float *gW0,
                                    float *part, float *buf, int BH, int L, int d_dot, int d_v, int bf16,
                                    cudaStream_t st) {
    if (bf16)
        return launch_chunked_t<__nv_bfloat16>(phk, phq, v, beta, W0, gy, gWL, gv, gW0, part, buf, BH, L, d_dot, d_v,
                                               st);
    return launch_chunked_t<float>(phk, phq, v, beta, W0, gy, gWL, gv, gW0, part, buf, BH, L, d_dot, d_v, st);
}

} // namespace fw
