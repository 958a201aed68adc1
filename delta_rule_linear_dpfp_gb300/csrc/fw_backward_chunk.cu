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
//   chunk_prep   one CTA per (b,h, chunk): K K^T, P, and M by forward
//                substitution, column by column;
//   state_scan   one CTA per (b,h, 16 value rows): the chunk-start states S
//                in chunk order (kept for the gradient kernel), X and U;
//   grad_scan    the same split, chunks in reverse: dS' kept per chunk, dU,
//                dX (= dV, written out), and dW0 at the end;
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

constexpr int kCC = 64;       // chunk length
constexpr int kCT = 256;      // threads per CTA
constexpr int kCR = 16;       // value rows per scan CTA
constexpr int kSl = 32;       // width of a staged slice of a contraction dimension
constexpr int kLd = kCC + 1;  // row stride of a C x C tile in shared memory
constexpr int kSd = kSl + 1;  // row stride of a staged slice
constexpr int kRd = kCR + 1;  // row stride of a C x 16 tile

FW_DEV float ldf(const float *p) { return __ldcg(p); }

// ----------------------------------------------------------- chunk_prep
// Shared memory: ks, qs [C][kSd] (a slice of the chunk's K and Q rows),
// kk, pq, ms [C][kLd], bs [C].
template <typename T>
__global__ void __launch_bounds__(kCT)
    chunk_prep_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ beta,
                      float *__restrict__ Mb, float *__restrict__ Pb, float *__restrict__ KKb, int L, int d_dot,
                      int nC) {
    extern __shared__ float sm[];
    float *ks = sm, *qs = ks + kCC * kSd, *kk = qs + kCC * kSd, *pq = kk + kCC * kLd, *ms = pq + kCC * kLd;
    float *bs = ms + kCC * kLd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, c = blockIdx.y;
    const int t0 = c * kCC, cl = min(kCC, L - t0);
    const size_t tok0 = (size_t)bh * L + t0;
    const size_t cc0 = ((size_t)bh * nC + c) * kCC * kCC;

    for (int i = tid; i < kCC; i += nt)
        bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
    for (int e = tid; e < kCC * kCC; e += nt) {
        kk[(e / kCC) * kLd + e % kCC] = 0.f;
        pq[(e / kCC) * kLd + e % kCC] = 0.f;
    }
    __syncthreads();
    for (int s0 = 0; s0 < d_dot; s0 += kSl) {
        for (int e = tid; e < kCC * kSl; e += nt) {
            const int i = e / kSl, j = e % kSl;
            const bool in = i < cl && s0 + j < d_dot;
            ks[i * kSd + j] = in ? ldf(phk + (tok0 + i) * d_dot + s0 + j) : 0.f;
            qs[i * kSd + j] = in ? ldf(phq + (tok0 + i) * d_dot + s0 + j) : 0.f;
        }
        __syncthreads();
        // 256 tiles of 4 x 4 outputs: rows ty + 16a, columns tx + 16b
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
            for (int j = 0; j < kSl; ++j) {
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
    // M = (I + A)^-1, unit lower: column j by forward substitution
    for (int j = tid; j < kCC; j += nt) {
        for (int i = 0; i < j; ++i)
            ms[i * kLd + j] = 0.f;
        ms[j * kLd + j] = 1.f;
        for (int i = j + 1; i < kCC; ++i) {
            float acc = 0.f;
            for (int m = j; m < i; ++m)
                acc = fmaf(pq[i * kLd + m], ms[m * kLd + j], acc);
            ms[i * kLd + j] = -acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < kCC * kCC; e += nt)
        Mb[cc0 + e] = ms[(e / kCC) * kLd + e % kCC];
}

// ----------------------------------------------------------- state_scan
// Shared memory: ss [kCR][d_dot + 1] (the CTA's rows of S), kc [C][d_dot + 1],
// mc [C][kLd], xs, us [C][kRd], bs [C].
template <typename T>
__global__ void __launch_bounds__(kCT)
    state_scan_kernel(const float *__restrict__ phk, const T *__restrict__ v, const T *__restrict__ beta,
                      const float *__restrict__ W0, const float *__restrict__ Mb, float *__restrict__ Sb,
                      float *__restrict__ Xb, float *__restrict__ Ub, int L, int d_dot, int d_v, int nC) {
    extern __shared__ float sm[];
    const int sd = d_dot + 1;
    float *ss = sm, *kc = ss + kCR * sd, *mc = kc + kCC * sd, *xs = mc + kCC * kLd, *us = xs + kCC * kRd;
    float *bs = us + kCC * kRd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, r0 = blockIdx.y * kCR, R = min(kCR, d_v - r0);

    for (int e = tid; e < kCR * d_dot; e += nt) {
        const int r = e / d_dot, m = e % d_dot;
        ss[r * sd + m] = (r < R && W0) ? ldf(W0 + ((size_t)bh * d_v + r0 + r) * d_dot + m) : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < nC; ++c) {
        const int t0 = c * kCC, cl = min(kCC, L - t0);
        const size_t tok0 = (size_t)bh * L + t0;
        const size_t st0 = ((size_t)bh * nC + c) * d_v;
        for (int e = tid; e < R * d_dot; e += nt) {
            const int r = e / d_dot, m = e % d_dot;
            Sb[(st0 + r0 + r) * d_dot + m] = ss[r * sd + m];
        }
        for (int e = tid; e < kCC * d_dot; e += nt) {
            const int i = e / d_dot, m = e % d_dot;
            kc[i * sd + m] = i < cl ? ldf(phk + (tok0 + i) * d_dot + m) : 0.f;
        }
        for (int e = tid; e < kCC * kCC; e += nt)
            mc[(e / kCC) * kLd + e % kCC] = ldf(Mb + ((size_t)bh * nC + c) * kCC * kCC + e);
        for (int e = tid; e < kCC * kCR; e += nt) {
            const int i = e / kCR, r = e % kCR;
            xs[i * kRd + r] = (i < cl && r < R) ? io<T>::load(v + (tok0 + i) * d_v + r0 + r) : 0.f;
        }
        for (int i = tid; i < kCC; i += nt)
            bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
        __syncthreads();
        // X = V - K S^T: 256 tiles, row r = w & 15, tokens (w >> 4) + 16a
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
            float acc[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                acc[a] = xs[(i0 + 16 * a) * kRd + r];
            for (int m = 0; m < d_dot; ++m) {
                const float s = ss[r * sd + m];
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    acc[a] = fmaf(-kc[(i0 + 16 * a) * sd + m], s, acc[a]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                xs[i * kRd + r] = acc[a];
                if (i < cl && r < R)
                    Xb[(tok0 + i) * d_v + r0 + r] = acc[a];
            }
        }
        __syncthreads();
        // U = M diag(beta) X (M unit lower)
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                float acc = 0.f;
                for (int s = 0; s <= i; ++s)
                    acc = fmaf(mc[i * kLd + s] * bs[s], xs[s * kRd + r], acc);
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
#pragma unroll
                for (int r = 0; r < kCR / 2; ++r)
                    acc[r] = fmaf(us[i * kRd + rh + r], kv, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                ss[(rh + r) * sd + m] = acc[r];
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ grad_scan
// Shared memory: ds [kCR][d_dot + 1] (the CTA's rows of dS), kc [C][d_dot + 1],
// mc, pc [C][kLd], dys, dus, dxs [C][kRd], bs [C].
template <typename T>
__global__ void __launch_bounds__(kCT)
    grad_scan_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ beta,
                     const T *__restrict__ gy, const float *__restrict__ gWL, const float *__restrict__ Mb,
                     const float *__restrict__ Pb, float *__restrict__ dSb, float *__restrict__ dXb,
                     float *__restrict__ dUb, T *__restrict__ gv, float *__restrict__ gW0, int L, int d_dot, int d_v,
                     int nC) {
    extern __shared__ float sm[];
    const int sd = d_dot + 1;
    float *ds = sm, *kc = ds + kCR * sd, *mc = kc + kCC * sd, *pc = mc + kCC * kLd, *dys = pc + kCC * kLd;
    float *dus = dys + kCC * kRd, *dxs = dus + kCC * kRd, *bs = dxs + kCC * kRd;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, r0 = blockIdx.y * kCR, R = min(kCR, d_v - r0);

    for (int e = tid; e < kCR * d_dot; e += nt) {
        const int r = e / d_dot, m = e % d_dot;
        ds[r * sd + m] = (r < R && gWL) ? ldf(gWL + ((size_t)bh * d_v + r0 + r) * d_dot + m) : 0.f;
    }
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
        for (int e = tid; e < kCC * d_dot; e += nt) {
            const int i = e / d_dot, m = e % d_dot;
            kc[i * sd + m] = i < cl ? ldf(phk + (tok0 + i) * d_dot + m) : 0.f;
        }
        for (int e = tid; e < kCC * kCC; e += nt) {
            mc[(e / kCC) * kLd + e % kCC] = ldf(Mb + cc0 + e);
            pc[(e / kCC) * kLd + e % kCC] = ldf(Pb + cc0 + e);
        }
        for (int e = tid; e < kCC * kCR; e += nt) {
            const int i = e / kCR, r = e % kCR;
            dys[i * kRd + r] = (i < cl && r < R) ? io<T>::load(gy + (tok0 + i) * d_v + r0 + r) : 0.f;
        }
        for (int i = tid; i < kCC; i += nt)
            bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
        __syncthreads();
        // dU = P^T dY + K dS'^T (P lower, so P_si is zero for s < i)
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
            float acc[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                acc[a] = 0.f;
            for (int m = 0; m < d_dot; ++m) {
                const float s = ds[r * sd + m];
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    acc[a] = fmaf(kc[(i0 + 16 * a) * sd + m], s, acc[a]);
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
        // dX = diag(beta) M^T dU = dV
        for (int w = tid; w < 256; w += nt) {
            const int r = w & 15, i0 = w >> 4;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + 16 * a;
                float acc = 0.f;
                for (int s = i; s < kCC; ++s)
                    acc = fmaf(mc[s * kLd + i], dus[s * kRd + r], acc);
                acc *= bs[i];
                dxs[i * kRd + r] = acc;
                if (i < cl && r < R) {
                    dXb[(tok0 + i) * d_v + r0 + r] = acc;
                    io<T>::store(gv + (tok0 + i) * d_v + r0 + r, acc);
                }
            }
        }
        __syncthreads();
        // dS = dS' + dY^T Q - dX^T K: thread per (column m, half of the rows)
        for (int e = tid; e < 2 * d_dot; e += nt) {
            const int m = e % d_dot, rh = (e / d_dot) * (kCR / 2);
            float acc[kCR / 2];
#pragma unroll
            for (int r = 0; r < kCR / 2; ++r)
                acc[r] = ds[(rh + r) * sd + m];
            for (int i = 0; i < cl; ++i) {
                const float qv = ldf(phq + (tok0 + i) * d_dot + m), kv = kc[i * sd + m];
#pragma unroll
                for (int r = 0; r < kCR / 2; ++r)
                    acc[r] = fmaf(dys[i * kRd + rh + r], qv, fmaf(-dxs[i * kRd + rh + r], kv, acc[r]));
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

// ------------------------------------------------------------ chunk_grad
// Shared memory: c1 (dT, then dA), c2 (dP), c3 (M), c4 (M^T dT diag(beta),
// then B + B^T), each [C][kLd]; dys, uvs, dxs [C][d_v + 1]; a staging region
// of 2 d_v kSd + 2 C kSd floats (slices of dU and X, later of S, dS', K, Q);
// bs, gb [C].
template <typename T>
__global__ void __launch_bounds__(kCT)
    chunk_grad_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ beta,
                      const T *__restrict__ gy, const float *__restrict__ Sb, const float *__restrict__ dSb,
                      const float *__restrict__ Xb, const float *__restrict__ Ub, const float *__restrict__ dXb,
                      const float *__restrict__ dUb, const float *__restrict__ Mb, const float *__restrict__ KKb,
                      float *__restrict__ part, int L, int d_dot, int d_v, int nC) {
    extern __shared__ float sm[];
    const int vd = d_v + 1;
    const size_t pst = 2 * (size_t)d_dot + 4;
    float *c1 = sm, *c2 = c1 + kCC * kLd, *c3 = c2 + kCC * kLd, *c4 = c3 + kCC * kLd;
    float *dys = c4 + kCC * kLd, *uvs = dys + kCC * vd, *dxs = uvs + kCC * vd, *stg = dxs + kCC * vd;
    float *bs = stg + 2 * d_v * kSd + 2 * kCC * kSd, *gb = bs + kCC;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, c = blockIdx.y;
    const int t0 = c * kCC, cl = min(kCC, L - t0);
    const size_t tok0 = (size_t)bh * L + t0;
    const size_t cc0 = ((size_t)bh * nC + c) * kCC * kCC;
    const size_t st0 = ((size_t)bh * nC + c) * d_v;

    for (int i = tid; i < kCC; i += nt)
        bs[i] = i < cl ? io<T>::load(beta + tok0 + i) : 0.f;
    for (int e = tid; e < kCC * d_v; e += nt) {
        const int i = e / d_v, r = e % d_v;
        const bool in = i < cl;
        dys[i * vd + r] = in ? io<T>::load(gy + (tok0 + i) * d_v + r) : 0.f;
        uvs[i * vd + r] = in ? ldf(Ub + (tok0 + i) * d_v + r) : 0.f;
        dxs[i * vd + r] = in ? ldf(dXb + (tok0 + i) * d_v + r) : 0.f;
    }
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        c1[i * kLd + j] = 0.f;
        c2[i * kLd + j] = 0.f;
        c3[i * kLd + j] = ldf(Mb + cc0 + e);
    }
    __syncthreads();
    // dT = dU X^T and dY U^T, over slices of the value dimension
    float *dul = stg, *xl = stg + kCC * kSd;
    for (int r0 = 0; r0 < d_v; r0 += kSl) {
        for (int e = tid; e < kCC * kSl; e += nt) {
            const int i = e / kSl, j = e % kSl;
            const bool in = i < cl && r0 + j < d_v;
            dul[i * kSd + j] = in ? ldf(dUb + (tok0 + i) * d_v + r0 + j) : 0.f;
            xl[i * kSd + j] = in ? ldf(Xb + (tok0 + i) * d_v + r0 + j) : 0.f;
        }
        __syncthreads();
        const int rn = min(kSl, d_v - r0);
        for (int w = tid; w < 256; w += nt) {
            const int tx = w & 15, ty = w >> 4;
            float at[4][4], ap[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    at[a][b] = c1[(ty + 16 * a) * kLd + tx + 16 * b];
                    ap[a][b] = c2[(ty + 16 * a) * kLd + tx + 16 * b];
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
                    c2[(ty + 16 * a) * kLd + tx + 16 * b] = ap[a][b];
                }
        }
        __syncthreads();
    }
    // dP = tril_inclusive(dY U^T); dbeta's first part, column sums of M * dT
    for (int e = tid; e < kCC * kCC; e += nt) {
        const int i = e / kCC, j = e % kCC;
        if (j > i)
            c2[i * kLd + j] = 0.f;
    }
    for (int i = tid; i < kCC; i += nt) {
        float acc = 0.f;
        for (int j = i; j < kCC; ++j)
            acc = fmaf(c3[j * kLd + i], c1[j * kLd + i], acc);
        gb[i] = acc;
    }
    __syncthreads();
    // c4 = M^T (dT diag(beta))
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
            acc = fmaf(c1[i * kLd + j], ldf(KKb + cc0 + (size_t)i * kCC + j), acc);
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
    // slices of the feature dimension
    float *sl = stg, *dsl = sl + d_v * kSd, *kl = dsl + d_v * kSd, *ql = kl + kCC * kSd;
    for (int m0 = 0; m0 < d_dot; m0 += kSl) {
        for (int e = tid; e < d_v * kSl; e += nt) {
            const int r = e / kSl, j = e % kSl;
            const bool in = m0 + j < d_dot;
            sl[r * kSd + j] = in ? ldf(Sb + (st0 + r) * d_dot + m0 + j) : 0.f;
            dsl[r * kSd + j] = in ? ldf(dSb + (st0 + r) * d_dot + m0 + j) : 0.f;
        }
        for (int e = tid; e < kCC * kSl; e += nt) {
            const int i = e / kSl, j = e % kSl;
            const bool in = i < cl && m0 + j < d_dot;
            kl[i * kSd + j] = in ? ldf(phk + (tok0 + i) * d_dot + m0 + j) : 0.f;
            ql[i * kSd + j] = in ? ldf(phq + (tok0 + i) * d_dot + m0 + j) : 0.f;
        }
        __syncthreads();
        // 256 tiles: slice column j = w & 31, tokens (w >> 5) + 8a
        for (int w = tid; w < 256; w += nt) {
            const int j = w & 31, i0 = w >> 5;
            float aq[8], ak[8];
#pragma unroll
            for (int a = 0; a < 8; ++a)
                aq[a] = ak[a] = 0.f;
            for (int r = 0; r < d_v; ++r) {
                const float s = sl[r * kSd + j], dsv = dsl[r * kSd + j];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int i = i0 + 8 * a;
                    aq[a] = fmaf(dys[i * vd + r], s, aq[a]);
                    ak[a] = fmaf(uvs[i * vd + r], dsv, fmaf(-dxs[i * vd + r], s, ak[a]));
                }
            }
            for (int s = 0; s < kCC; ++s) {
                const float kv = kl[s * kSd + j], qv = ql[s * kSd + j];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int i = i0 + 8 * a;
                    aq[a] = fmaf(c2[i * kLd + s], kv, aq[a]);
                    ak[a] = fmaf(c2[s * kLd + i], qv, fmaf(c4[i * kLd + s], kv, ak[a]));
                }
            }
            if (m0 + j < d_dot)
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int i = i0 + 8 * a;
                    if (i < cl) {
                        part[(tok0 + i) * pst + m0 + j] = aq[a];
                        part[(tok0 + i) * pst + d_dot + m0 + j] = ak[a];
                    }
                }
        }
        __syncthreads();
    }
}

size_t prep_smem() { return sizeof(float) * (2 * kCC * kSd + 3 * kCC * kLd + kCC); }
size_t scan_smem(int d_dot) {
    return sizeof(float) * ((size_t)(kCR + kCC) * (d_dot + 1) + kCC * kLd + 2 * kCC * kRd + kCC);
}
size_t gscan_smem(int d_dot) {
    return sizeof(float) * ((size_t)(kCR + kCC) * (d_dot + 1) + 2 * kCC * kLd + 3 * kCC * kRd + kCC);
}
size_t cgrad_smem(int d_v) {
    return sizeof(float) * (4 * kCC * kLd + 3 * (size_t)kCC * (d_v + 1) + 2 * (size_t)d_v * kSd + 2 * kCC * kSd +
                            2 * kCC);
}

// Offsets (in floats) of the buffers after phi(k), phi(q) and the per-token
// gradient records inside the workspace.
struct ChunkLayout {
    size_t M, P, KK, S, dS, X, U, dX, dU, end;
};

ChunkLayout chunk_layout(int BH, int L, int d_dot, int d_v) {
    const size_t rows = (size_t)BH * L, nC = ((size_t)L + kCC - 1) / kCC, cc = (size_t)BH * nC * kCC * kCC;
    const size_t sts = (size_t)BH * nC * d_v * d_dot;
    ChunkLayout o;
    o.M = 0;
    o.P = o.M + cc;
    o.KK = o.P + cc;
    o.S = o.KK + cc;
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
    cudaError_t e;
    {
        auto kern = chunk_prep_kernel<T>;
        const size_t smem = prep_smem();
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kern<<<dim3((unsigned)BH, (unsigned)nC), kCT, smem, st>>>(phk, phq, bt, buf + o.M, buf + o.P, buf + o.KK, L,
                                                                  d_dot, nC);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    {
        auto kern = state_scan_kernel<T>;
        const size_t smem = scan_smem(d_dot);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kern<<<dim3((unsigned)BH, (unsigned)nRB), kCT, smem, st>>>(phk, vt, bt, W0, buf + o.M, buf + o.S, buf + o.X,
                                                                   buf + o.U, L, d_dot, d_v, nC);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    {
        auto kern = grad_scan_kernel<T>;
        const size_t smem = gscan_smem(d_dot);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kern<<<dim3((unsigned)BH, (unsigned)nRB), kCT, smem, st>>>(phk, phq, bt, gyt, gWL, buf + o.M, buf + o.P,
                                                                   buf + o.dS, buf + o.dX, buf + o.dU,
                                                                   static_cast<T *>(gv), gW0, L, d_dot, d_v, nC);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    auto kern = chunk_grad_kernel<T>;
    const size_t smem = cgrad_smem(d_v);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kern<<<dim3((unsigned)BH, (unsigned)nC), kCT, smem, st>>>(phk, phq, bt, gyt, buf + o.S, buf + o.dS, buf + o.X,
                                                              buf + o.U, buf + o.dX, buf + o.dU, buf + o.M,
                                                              buf + o.KK, part, L, d_dot, d_v, nC);
    return cudaGetLastError();
}

} // namespace

bool backward_chunked_supported(int d_key, int nu, int d_v, int L) {
    const int d_dot = 2 * d_key * nu;
    const size_t cap = (size_t)227 * 1024;
    return d_dot <= 512 && d_v <= 128 && (L + kCC - 1) / kCC <= 65535 && scan_smem(d_dot) <= cap &&
           gscan_smem(d_dot) <= cap && cgrad_smem(d_v) <= cap;
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
