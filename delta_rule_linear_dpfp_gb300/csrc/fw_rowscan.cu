// fw_rowscan.cu -- the token-serial delta rule on CUDA cores, fp32 throughout.
//
// Serves fw_delta_forward with fp32 I/O: the exact-arithmetic path (fp32
// FMA, no tensor cores), token by token.
//
// Method (Fast Weights Transformer guide, section "FastWeightsAttention: the
// new update rule" and its forward-pass loop): per token t,
//   vbar = W phi(k_t);  W += beta_t (v_t - vbar) phi(k_t)^T;  y_t = W phi(q_t).
// Each row of W evolves on its own (row r only needs v_t[r]), so the work is
// split over (batch, head, block of 16 rows): one warp owns two rows, each
// lane holds every 32nd entry of a row in registers for the whole sequence,
// and the two dot products per token are warp reductions.  phi(k_t) and
// phi(q_t) for a tile of tokens are built in shared memory by the DPFP
// definition (x = ReLU([k,-k]); block i: x[j] * x[(j - i) mod 2*d_key];
// divide by sum + eps) once per CTA.
#include "fw_common.cuh"

namespace fw {

namespace {

constexpr int kRowsPerWarp = 2;
constexpr int kWarps = 8;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;

template <typename T, int NPL>
__global__ void __launch_bounds__(256)
    rowscan_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   const T *__restrict__ beta, const float *W0, float *Wout, T *__restrict__ y,
                   int L, int d_key, int nu, int d_v, int tt, float eps) {
    constexpr int DD = 32 * NPL; // padded d_dot held per row
    extern __shared__ float smem[];
    const int n = 2 * d_key;
    const int d_dot = n * nu;
    float *xs = smem;                         // [kWarps][n]
    float *pk = xs + kWarps * n;              // [tt][DD]
    float *pq = pk + tt * DD;                 // [tt][DD]
    float *bt = pq + tt * DD;                 // [tt]
    float *vt = bt + tt;                      // [tt][kRowsPerCta]
    float *yt = vt + tt * kRowsPerCta;        // [tt][kRowsPerCta]

    const int nrb = (d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t bh = blockIdx.x / nrb;
    const int r0 = (blockIdx.x % nrb) * kRowsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // state rows in registers: S[j][e] = W[r][lane + 32 e]
    float S[kRowsPerWarp][NPL];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const int r = r0 + warp + kWarps * j;
        const float *src = W0 ? W0 + (bh * d_v + r) * (int64_t)d_dot : nullptr;
#pragma unroll
        for (int e = 0; e < NPL; ++e) {
            const int m = lane + 32 * e;
            S[j][e] = (src && r < d_v && m < d_dot) ? src[m] : 0.f;
        }
    }

    for (int t0 = 0; t0 < L; t0 += tt) {
        const int nt = min(tt, L - t0);
        // phi(k) and phi(q) of the tile, one (token, key-or-query) per warp
        for (int task = warp; task < 2 * nt; task += kWarps) {
            const int which = task / nt, tok = task % nt;
            const T *src = (which ? q : k) + (bh * L + t0 + tok) * (int64_t)d_key;
            float *x = xs + warp * n;
            for (int j = lane; j < d_key; j += 32) {
                const float a = io<T>::load(src + j);
                x[j] = fmaxf(a, 0.f);
                x[d_key + j] = fmaxf(-a, 0.f);
            }
            __syncwarp();
            float *dst = (which ? pq : pk) + tok * DD;
            float s = 0.f;
            for (int m = lane; m < DD; m += 32) {
                float p = 0.f;
                if (m < d_dot) {
                    const int i = m / n + 1, jj = m % n;
                    p = x[jj] * x[(jj - i + n) % n];
                }
                dst[m] = p;
                s += p;
            }
            s = warp_sum(s);
            const float denom = s + eps;
            for (int m = lane; m < DD; m += 32)
                dst[m] = __fdiv_rn(dst[m], denom);
            __syncwarp();
        }
        for (int i = threadIdx.x; i < nt; i += blockDim.x)
            bt[i] = io<T>::load(beta + bh * L + t0 + i);
        for (int i = threadIdx.x; i < nt * kRowsPerCta; i += blockDim.x) {
            const int tok = i / kRowsPerCta, rr = i % kRowsPerCta;
            vt[i] = (r0 + rr < d_v) ? io<T>::load(v + (bh * L + t0 + tok) * (int64_t)d_v + r0 + rr) : 0.f;
        }
        __syncthreads();

        for (int tok = 0; tok < nt; ++tok) {
            const float *fk = pk + tok * DD;
            const float *fq = pq + tok * DD;
            float kv[NPL], qv[NPL];
#pragma unroll
            for (int e = 0; e < NPL; ++e) {
                kv[e] = fk[lane + 32 * e];
                qv[e] = fq[lane + 32 * e];
            }
            const float b = bt[tok];
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                const int rr = warp + kWarps * j;
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < NPL; ++e)
                    acc = fmaf(S[j][e], kv[e], acc);
                const float vbar = warp_sum(acc);              // retrieve with W_{t-1}
                const float u = b * (vt[tok * kRowsPerCta + rr] - vbar);
                float o = 0.f;
#pragma unroll
                for (int e = 0; e < NPL; ++e) {
                    S[j][e] = fmaf(u, kv[e], S[j][e]);          // write
                    o = fmaf(S[j][e], qv[e], o);                // read with W_t
                }
                o = warp_sum(o);
                if (lane == 0)
                    yt[tok * kRowsPerCta + rr] = o;
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nt * kRowsPerCta; i += blockDim.x) {
            const int tok = i / kRowsPerCta, rr = i % kRowsPerCta;
            if (r0 + rr < d_v)
                io<T>::store(y + (bh * L + t0 + tok) * (int64_t)d_v + r0 + rr, yt[i]);
        }
        __syncthreads();
    }

    if (Wout) {
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            const int r = r0 + warp + kWarps * j;
            if (r < d_v) {
                float *dst = Wout + (bh * d_v + r) * (int64_t)d_dot;
#pragma unroll
                for (int e = 0; e < NPL; ++e) {
                    const int m = lane + 32 * e;
                    if (m < d_dot)
                        dst[m] = S[j][e];
                }
            }
        }
    }
}

template <typename T, int NPL>
cudaError_t launch_rowscan_t(const void *q, const void *k, const void *v, const void *beta,
                             const float *W0, float *Wout, void *y, int BH, int L, int d_key,
                             int nu, int d_v, float eps, cudaStream_t st) {
    constexpr int DD = 32 * NPL;
    // tokens per tile: phi tiles of at most ~64 KB, between 1 and 32 tokens
    int tt = (64 * 1024) / (2 * DD * 4);
    tt = tt < 1 ? 1 : (tt > 32 ? 32 : tt);
    if (tt > L)
        tt = L;
    const size_t smem = sizeof(float) * ((size_t)kWarps * 2 * d_key + 2 * (size_t)tt * DD + tt +
                                         2 * (size_t)tt * kRowsPerCta);
    auto kern = rowscan_kernel<T, NPL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int nrb = (d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t grid = (int64_t)BH * nrb;
    kern<<<(unsigned)grid, 256, smem, st>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                                           static_cast<const T *>(v), static_cast<const T *>(beta),
                                           W0, Wout, static_cast<T *>(y), L, d_key, nu, d_v, tt, eps);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rowscan_dt(const void *q, const void *k, const void *v, const void *beta,
                              const float *W0, float *Wout, void *y, int BH, int L, int d_key,
                              int nu, int d_v, float eps, cudaStream_t st) {
    const int d_dot = 2 * d_key * nu;
    if (d_dot <= 32)
        return launch_rowscan_t<T, 1>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 64)
        return launch_rowscan_t<T, 2>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 128)
        return launch_rowscan_t<T, 4>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 256)
        return launch_rowscan_t<T, 8>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 384)
        return launch_rowscan_t<T, 12>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 512)
        return launch_rowscan_t<T, 16>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    if (d_dot <= 1024)
        return launch_rowscan_t<T, 32>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
    return cudaErrorInvalidValue;
}

} // namespace

// Host launcher for the token-serial path (arguments validated by the caller).
// W0 may be null (zeros); Wout may be null (not written); W0 == Wout is allowed.
cudaError_t launch_rowscan(const void *q, const void *k, const void *v, const void *beta,
                           const float *W0, float *Wout, void *y, int BH, int L, int d_key, int nu,
                           int d_v, int bf16, float eps, cudaStream_t st) {
    if (bf16)
        return launch_rowscan_dt<__nv_bfloat16>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v,
                                                eps, st);
    return launch_rowscan_dt<float>(q, k, v, beta, W0, Wout, y, BH, L, d_key, nu, d_v, eps, st);
}

} // namespace fw

