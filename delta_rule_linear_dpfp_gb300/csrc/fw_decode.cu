// fw_decode.cu -- K3, the decode step: one new token per (batch, head)
// against a persistent fp32 state W [B, H, d_v, d_dot], updated in place.
//
// Method (Fast Weights Transformer guide, sections "token_wise variant" and
// "FastWeightsAttention: the new update rule"): for each row r of W,
//   vbar_r = W[r] . phi(k),  u_r = beta (v_r - vbar_r),  W[r] += u_r phi(k),
//   y_r = W_new[r] . phi(q) = W[r] . phi(q) + u_r (phi(k) . phi(q)).
// The second form of y lets both dot products come from the same read of the
// row, so every element of W is read once and written once: the step is
// bound by HBM bandwidth (2 * d_v * d_dot * 4 bytes per head-token).
//
// Mapping: one CTA of 8 warps per (batch*head, block of 64 rows).  Warps 0-1
// build phi(k) and phi(q) in shared memory with the shuffle DPFP of the
// standalone kernel while every warp already has its first row in flight;
// then each warp streams 8 rows (rows warp, warp + 8, ...), loading the next
// row before it computes the current one.  A lane holds float4 chunks
// lane, lane + 32, ... of a row, so each load and store instruction of a
// warp covers 512 contiguous bytes.
#include "fw_dpfp.cuh"

namespace fw {

namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 8;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

template <int DK, typename T, int NQ>
__global__ void __launch_bounds__(256)
    decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                  const T *__restrict__ beta, float *__restrict__ W, T *__restrict__ y, int nu,
                  int d_v, float eps) {
    constexpr int G = DK / 4, RPW = 32 / G, N2 = 2 * DK;
    constexpr int DD = 128 * NQ; // padded d_dot held per row (NQ float4 per lane)
    __shared__ __align__(16) float phk[DD];
    __shared__ __align__(16) float phq[DD];
    __shared__ float vsh[kRowsPerCta];
    __shared__ float ysh[kRowsPerCta];
    __shared__ float kq_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrb = (d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t bh = blockIdx.x / nrb;
    const int r0 = (blockIdx.x % nrb) * kRowsPerCta;
    const int d_dot = N2 * nu;

    auto row_ptr = [&](int j) { return W + (bh * d_v + r0 + warp + kWarps * j) * (int64_t)d_dot; };
    auto row_ok = [&](int j) { return r0 + warp + kWarps * j < d_v; };
    auto load_row = [&](int j, float4 (&w)[NQ]) {
        const float4 *src = reinterpret_cast<const float4 *>(row_ptr(j));
#pragma unroll
        for (int e = 0; e < NQ; ++e) {
            const int m4 = lane + 32 * e;
            w[e] = (row_ok(j) && 4 * m4 < d_dot) ? __ldcs(src + m4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };

    griddep_launch_dependents();
    // the CTA's rows into L2 while the preceding kernel still runs (a
    // prefetch, so safe even if that kernel writes W: L2 is the point of
    // coherence, and the loads below come after the wait)
    if (tid == 0) {
        const int nr = min(kRowsPerCta, d_v - r0);
        l2_prefetch(W + (bh * d_v + r0) * (int64_t)d_dot, (uint32_t)(nr * d_dot * 4));
    }
    griddep_wait(); // q, k, v, beta or W may be the preceding kernel's output: no load before this
    q = after_wait(q);
    k = after_wait(k);
    v = after_wait(v);
    beta = after_wait(beta);
    W = after_wait(W);
    const float b = io<T>::load(beta + bh);
    float4 cur[NQ];
    load_row(0, cur); // first row in flight while phi is built

    for (int i = tid; i < DD; i += blockDim.x) {
        phk[i] = 0.f;
        phq[i] = 0.f;
    }
    if (tid < kRowsPerCta)
        vsh[tid] = r0 + tid < d_v ? io<T>::load(v + bh * d_v + r0 + tid) : 0.f;
    __syncthreads();
    // phi(k) (row 0) and phi(q) (row 1) with the shuffle DPFP
    if (warp * RPW < 2) {
        const int g = lane % G, base_lane = lane - g;
        const int rr = warp * RPW + lane / G; // 0: key, 1: query, >= 2: idle rows
        const bool valid = rr < 2;
        const T *src = (rr == 1 ? q : k) + bh * DK;
        float x[8];
        dpfp_load_x<G>(src, g, valid, x);
        float *dst = rr == 1 ? phq : phk;
        dpfp_row_emit<G, 4>(x, g, base_lane, nu, eps, [&](int i, float (&p)[8]) {
            if (valid) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[(i - 1) * N2 + 8 * g + c] = p[c];
            }
        });
    }
    __syncthreads();
    if (warp == 0) {
        float acc = 0.f;
        for (int m = lane; m < d_dot; m += 32)
            acc = fmaf(phk[m], phq[m], acc);
        acc = warp_sum(acc);
        if (lane == 0)
            kq_sh = acc;
    }
    float4 fk[NQ], fq[NQ];
#pragma unroll
    for (int e = 0; e < NQ; ++e) {
        fk[e] = reinterpret_cast<const float4 *>(phk)[lane + 32 * e];
        fq[e] = reinterpret_cast<const float4 *>(phq)[lane + 32 * e];
    }
    __syncthreads();
    const float kq = kq_sh;

    for (int j = 0; j < kRowsPerWarp; ++j) {
        float4 nxt[NQ];
        if (j + 1 < kRowsPerWarp)
            load_row(j + 1, nxt);
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < NQ; ++e) {
            sk = fmaf(cur[e].x, fk[e].x, fmaf(cur[e].y, fk[e].y, fmaf(cur[e].z, fk[e].z, fmaf(cur[e].w, fk[e].w, sk))));
            sq = fmaf(cur[e].x, fq[e].x, fmaf(cur[e].y, fq[e].y, fmaf(cur[e].z, fq[e].z, fmaf(cur[e].w, fq[e].w, sq))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        const int rr = warp + kWarps * j;
        const float u = b * (vsh[rr] - sk);
        if (row_ok(j)) {
            float4 *dst = reinterpret_cast<float4 *>(row_ptr(j));
#pragma unroll
            for (int e = 0; e < NQ; ++e) {
                const int m4 = lane + 32 * e;
                if (4 * m4 < d_dot) {
                    float4 w = cur[e];
                    w.x = fmaf(u, fk[e].x, w.x);
                    w.y = fmaf(u, fk[e].y, w.y);
                    w.z = fmaf(u, fk[e].z, w.z);
                    w.w = fmaf(u, fk[e].w, w.w);
                    __stcs(dst + m4, w);
                }
            }
            if (lane == 0)
                ysh[rr] = fmaf(u, kq, sq);
        }
        if (j + 1 < kRowsPerWarp) {
#pragma unroll
            for (int e = 0; e < NQ; ++e)
                cur[e] = nxt[e];
        }
    }
    __syncthreads();
    if (tid < kRowsPerCta && r0 + tid < d_v)
        io<T>::store(y + bh * d_v + r0 + tid, ysh[tid]);
}

template <int DK, typename T>
cudaError_t launch_decode_t(const void *q, const void *k, const void *v, const void *beta, float *W,
                            void *y, int BH, int nu, int d_v, float eps, cudaStream_t st) {
    const int d_dot = 2 * DK * nu;
    const int nrb = (d_v + kRowsPerCta - 1) / kRowsPerCta;
    const dim3 grid((unsigned)((int64_t)BH * nrb));
    const T *qq = static_cast<const T *>(q), *kk = static_cast<const T *>(k), *vv = static_cast<const T *>(v),
            *bb = static_cast<const T *>(beta);
    T *yy = static_cast<T *>(y);
    if (d_dot <= 128)
        return launch_pdl(decode_kernel<DK, T, 1>, grid, dim3(256), 0, st, qq, kk, vv, bb, W, yy, nu, d_v, eps);
    else if (d_dot <= 256)
        return launch_pdl(decode_kernel<DK, T, 2>, grid, dim3(256), 0, st, qq, kk, vv, bb, W, yy, nu, d_v, eps);
    else if (d_dot <= 512)
        return launch_pdl(decode_kernel<DK, T, 4>, grid, dim3(256), 0, st, qq, kk, vv, bb, W, yy, nu, d_v, eps);
    else if (d_dot <= 1024)
        return launch_pdl(decode_kernel<DK, T, 8>, grid, dim3(256), 0, st, qq, kk, vv, bb, W, yy, nu, d_v, eps);
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_decode_dt(const void *q, const void *k, const void *v, const void *beta, float *W,
                             void *y, int BH, int d_key, int nu, int d_v, float eps, cudaStream_t st) {
    switch (d_key) {
    case 8: return launch_decode_t<8, T>(q, k, v, beta, W, y, BH, nu, d_v, eps, st);
    case 16: return launch_decode_t<16, T>(q, k, v, beta, W, y, BH, nu, d_v, eps, st);
    case 32: return launch_decode_t<32, T>(q, k, v, beta, W, y, BH, nu, d_v, eps, st);
    case 64: return launch_decode_t<64, T>(q, k, v, beta, W, y, BH, nu, d_v, eps, st);
    case 128: return launch_decode_t<128, T>(q, k, v, beta, W, y, BH, nu, d_v, eps, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

// Host launcher (arguments validated by the caller).
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *beta, float *W,
                          void *y, int BH, int d_key, int nu, int d_v, int bf16, float eps,
                          int num_sms, cudaStream_t st) {
    (void)num_sms;
    if (bf16)
        return launch_decode_dt<__nv_bfloat16>(q, k, v, beta, W, y, BH, d_key, nu, d_v, eps, st);
    return launch_decode_dt<float>(q, k, v, beta, W, y, BH, d_key, nu, d_v, eps, st);
}

} // namespace fw
