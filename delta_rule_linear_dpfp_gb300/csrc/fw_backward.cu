// fw_backward.cu -- the backward of the delta-rule layer core: gradients of
// q, k, v, beta and the initial state W0 given those of y and W_final.
//
// Method: the chain rule applied to the recurrence of the Fast Weights
// Transformer guide (section "FastWeightsAttention: the new update rule":
// a = W_{t-1} phi(k_t), u = beta_t (v_t - a), W_t = W_{t-1} + u phi(k_t)^T,
// y_t = W_t phi(q_t)) in reverse token order; the pages print no backward
// (the guide trains through the loop with autograd).  With gW the gradient
// of the state carried back from later tokens, per token t from L to 1:
//   gW += gy_t phi(q_t)^T;  g_phi(q_t) = W_t^T gy_t;  gu = gW phi(k_t);
//   gbeta_t = gu . (v_t - a);  gv_t = beta_t gu;
//   g_phi(k_t) = gW^T u - W_{t-1}^T (beta_t gu);  gW -= (beta_t gu) phi(k_t)^T,
// then through the DPFP map (quotient rule of the normalisation, both
// factors of each rolled product, the two ReLU halves of [k, -k]).
//
// Mapping: one CTA of 512 threads per (batch, head); W and gW stay in shared
// memory in fp32 for the whole sequence.  A forward sweep keeps u_t for every
// token (global scratch, d_v floats per token); the reverse sweep steps W
// back exactly as the forward stepped it up (W_{t-1} = W_t - u_t phi(k_t)^T,
// one rounding per element and token).  Row dot products take one warp per
// row, column sums one thread per column (deterministic order), updates one
// thread per element; one warp builds phi of a row, one warp takes the DPFP
// backward.  fp32 arithmetic on CUDA cores throughout: the token loop is
// serial, so this kernel is latency-bound.
#include "fw_common.cuh"
#include "fw_forward_tc.h"

namespace fw {

namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;

// phi of one row (d_key raw values) by one warp: x = ReLU([k, -k]) into xs,
// phi into ph.  Block i of phi holds x[j] * x[(j - i) mod n].
template <typename T>
FW_DEV void dpfp_warp(const T *src, float *xs, float *ph, int d_key, int nu, float eps, int lane) {
    const int n = 2 * d_key, d_dot = n * nu;
    for (int j = lane; j < d_key; j += 32) {
        const float kv = io<T>::load(src + j);
        xs[j] = fmaxf(kv, 0.f);
        xs[d_key + j] = fmaxf(-kv, 0.f);
    }
    __syncwarp();
    float s = 0.f;
    for (int m = lane; m < d_dot; m += 32) {
        const int i = m / n + 1, j = m - (i - 1) * n;
        const float p = xs[j] * xs[(j - i + n) % n];
        ph[m] = p;
        s += p;
    }
    s = warp_sum(s);
    const float inv = 1.0f / (s + eps);
    for (int m = lane; m < d_dot; m += 32)
        ph[m] *= inv;
    __syncwarp();
}

// The DPFP backward of one row by one warp: given g = dL/dphi (shared), the
// raw row src, writes dL/dk to dst.  xs: scratch of 2 d_key floats.
template <typename T>
FW_DEV void dpfp_backward_warp(const T *src, const float *g, float *xs, T *dst, int d_key, int nu, float eps,
                               int lane) {
    const int n = 2 * d_key, d_dot = n * nu;
    for (int j = lane; j < d_key; j += 32) {
        const float kv = io<T>::load(src + j);
        xs[j] = fmaxf(kv, 0.f);
        xs[d_key + j] = fmaxf(-kv, 0.f);
    }
    __syncwarp();
    float s = 0.f, gp = 0.f; // sum of the products, g . products
    for (int m = lane; m < d_dot; m += 32) {
        const int i = m / n + 1, j = m - (i - 1) * n;
        const float p = xs[j] * xs[(j - i + n) % n];
        s += p;
        gp = fmaf(g[m], p, gp);
    }
    s = warp_sum(s);
    gp = warp_sum(gp);
    const float c1 = 1.0f / (s + eps), c2 = gp * c1 * c1; // d phi_m / d p_l = delta_ml c1 - p_m c1^2
    for (int j = lane; j < d_key; j += 32) {
        float gx[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) { // x[j] (from k) and x[d_key + j] (from -k)
            const int jj = j + h * d_key;
            for (int i = 1; i <= nu; ++i) {
                const int lo = (jj - i + n) % n, hi = (jj + i) % n;
                // x[jj] is the left factor of product (i, jj) and the rolled
                // factor of product (i, jj + i)
                gx[h] = fmaf(g[(i - 1) * n + jj] * c1 - c2, xs[lo], gx[h]);
                gx[h] = fmaf(g[(i - 1) * n + hi] * c1 - c2, xs[hi], gx[h]);
            }
        }
        const float kv = io<T>::load(src + j);
        io<T>::store(dst + j, (kv > 0.f ? gx[0] : 0.f) - (kv < 0.f ? gx[1] : 0.f));
    }
    __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    delta_backward_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                          const T *__restrict__ beta, const float *__restrict__ W0, const T *__restrict__ gy,
                          const float *__restrict__ gWL, T *__restrict__ gq, T *__restrict__ gk, T *__restrict__ gv,
                          T *__restrict__ gbeta, float *__restrict__ gW0, float *__restrict__ us, int L, int d_key,
                          int nu, int d_v, float eps) {
    extern __shared__ float sm[];
    const int d_dot = 2 * d_key * nu, n = 2 * d_key;
    const int nel = d_v * d_dot;
    float *W = sm;                 // [d_v][d_dot] the state W_t
    float *G = W + nel;            // [d_v][d_dot] dL/dW_t
    float *pk = G + nel;           // phi(k_t)
    float *pq = pk + d_dot;        // phi(q_t)
    float *gpq = pq + d_dot;       // dL/dphi(q_t)
    float *gpk = gpq + d_dot;      // dL/dphi(k_t)
    float *gyv = gpk + d_dot;      // gy_t
    float *vv = gyv + d_v;         // v_t
    float *uu = vv + d_v;          // u_t
    float *gu = uu + d_v;          // dL/du_t, then beta_t dL/du_t
    float *aa = gu + d_v;          // W_{t-1} phi(k_t)
    float *xk = aa + d_v;          // x of k_t (one warp's scratch)
    float *xq = xk + n;            // x of q_t
    float *sc = xq + n;            // scalars: [0] beta_t

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = blockIdx.x;
    const T *qb = q + bh * L * d_key, *kb = k + bh * L * d_key, *vb = v + bh * L * d_v, *bb = beta + bh * L;
    const T *gyb = gy + bh * L * d_v;
    float *ub = us + bh * L * d_v;

    griddep_launch_dependents();
    griddep_wait();
    for (int e = tid; e < nel; e += kBwdThreads) {
        W[e] = W0 ? W0[bh * nel + e] : 0.f;
        G[e] = gWL ? gWL[bh * nel + e] : 0.f;
    }
    // ---- forward sweep: keep u_t
    for (int t = 0; t < L; ++t) {
        __syncthreads();
        if (warp == 0)
            dpfp_warp(kb + (int64_t)t * d_key, xk, pk, d_key, nu, eps, lane);
        else if (warp == 1) {
            for (int r = lane; r < d_v; r += 32)
                vv[r] = io<T>::load(vb + (int64_t)t * d_v + r);
            if (lane == 0)
                sc[0] = io<T>::load(bb + t);
        }
        __syncthreads();
        for (int r = warp; r < d_v; r += kBwdWarps) { // a = W_{t-1} phi(k), u = beta (v - a)
            float acc = 0.f;
            for (int m = lane; m < d_dot; m += 32)
                acc = fmaf(W[r * d_dot + m], pk[m], acc);
            acc = warp_sum(acc);
            if (lane == 0) {
                const float u = sc[0] * (vv[r] - acc);
                uu[r] = u;
                ub[(int64_t)t * d_v + r] = u;
            }
        }
        __syncthreads();
        for (int e = tid; e < nel; e += kBwdThreads) // W_t = W_{t-1} + u phi(k)^T
            W[e] = fmaf(uu[e / d_dot], pk[e % d_dot], W[e]);
    }
    // ---- reverse sweep
    for (int t = L - 1; t >= 0; --t) {
        __syncthreads();
        if (warp == 0)
            dpfp_warp(kb + (int64_t)t * d_key, xk, pk, d_key, nu, eps, lane);
        else if (warp == 1)
            dpfp_warp(qb + (int64_t)t * d_key, xq, pq, d_key, nu, eps, lane);
        else if (warp == 2) {
            for (int r = lane; r < d_v; r += 32) {
                gyv[r] = io<T>::load(gyb + (int64_t)t * d_v + r);
                vv[r] = io<T>::load(vb + (int64_t)t * d_v + r);
                uu[r] = ub[(int64_t)t * d_v + r];
            }
            if (lane == 0)
                sc[0] = io<T>::load(bb + t);
        }
        __syncthreads();
        for (int m = tid; m < d_dot; m += kBwdThreads) { // g_phi(q) = W_t^T gy
            float acc = 0.f;
            for (int r = 0; r < d_v; ++r)
                acc = fmaf(W[r * d_dot + m], gyv[r], acc);
            gpq[m] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nel; e += kBwdThreads) { // gW += gy phi(q)^T; W_{t-1} = W_t - u phi(k)^T
            const int r = e / d_dot, m = e - r * d_dot;
            G[e] = fmaf(gyv[r], pq[m], G[e]);
            W[e] = fmaf(-uu[r], pk[m], W[e]);
        }
        __syncthreads();
        for (int r = warp; r < d_v; r += kBwdWarps) { // gu = gW phi(k), a = W_{t-1} phi(k)
            float g = 0.f, a = 0.f;
            for (int m = lane; m < d_dot; m += 32) {
                g = fmaf(G[r * d_dot + m], pk[m], g);
                a = fmaf(W[r * d_dot + m], pk[m], a);
            }
            g = warp_sum(g);
            a = warp_sum(a);
            if (lane == 0) {
                gu[r] = g;
                aa[r] = a;
            }
        }
        __syncthreads();
        const float bt = sc[0];
        if (warp == 0) { // gbeta = gu . (v - a)
            float acc = 0.f;
            for (int r = lane; r < d_v; r += 32)
                acc = fmaf(gu[r], vv[r] - aa[r], acc);
            acc = warp_sum(acc);
            if (lane == 0)
                io<T>::store(gbeta + bh * L + t, acc);
        }
        __syncthreads();
        for (int r = tid; r < d_v; r += kBwdThreads) { // gv = beta gu; keep e = beta gu
            gu[r] *= bt;
            io<T>::store(gv + (bh * L + t) * d_v + r, gu[r]);
        }
        __syncthreads();
        for (int m = tid; m < d_dot; m += kBwdThreads) { // g_phi(k) = gW^T u - W_{t-1}^T e
            float acc = 0.f;
            for (int r = 0; r < d_v; ++r)
                acc = fmaf(G[r * d_dot + m], uu[r], fmaf(-W[r * d_dot + m], gu[r], acc));
            gpk[m] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nel; e += kBwdThreads) { // gW_{t-1} = gW - e phi(k)^T
            const int r = e / d_dot, m = e - r * d_dot;
            G[e] = fmaf(-gu[r], pk[m], G[e]);
        }
        if (warp == kBwdWarps - 1)
            dpfp_backward_warp(qb + (int64_t)t * d_key, gpq, xq, gq + (bh * L + t) * d_key, d_key, nu, eps, lane);
        else if (warp == kBwdWarps - 2)
            dpfp_backward_warp(kb + (int64_t)t * d_key, gpk, xk, gk + (bh * L + t) * d_key, d_key, nu, eps, lane);
    }
    __syncthreads();
    if (gW0)
        for (int e = tid; e < nel; e += kBwdThreads)
            gW0[bh * nel + e] = G[e];
}

template <typename T>
cudaError_t launch_backward_t(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                              const void *gy, const float *gWL, void *gq, void *gk, void *gv, void *gbeta,
                              float *gW0, float *us, int BH, int L, int d_key, int nu, int d_v, float eps,
                              cudaStream_t st) {
    const size_t smem = backward_smem_bytes(d_key, nu, d_v);
    auto kern = delta_backward_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3((unsigned)BH), dim3(kBwdThreads), smem, st, static_cast<const T *>(q),
                      static_cast<const T *>(k), static_cast<const T *>(v), static_cast<const T *>(beta), W0,
                      static_cast<const T *>(gy), gWL, static_cast<T *>(gq), static_cast<T *>(gk),
                      static_cast<T *>(gv), static_cast<T *>(gbeta), gW0, us, L, d_key, nu, d_v, eps);
}

} // namespace

// Shared memory of one CTA: W and gW, six vectors, the x scratch, scalars.
size_t backward_smem_bytes(int d_key, int nu, int d_v) {
    const size_t d_dot = (size_t)2 * d_key * nu;
    return sizeof(float) * (2 * (size_t)d_v * d_dot + 4 * d_dot + 5 * (size_t)d_v + 4 * (size_t)d_key + 8);
}

cudaError_t launch_backward(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                            const void *gy, const float *gWL, void *gq, void *gk, void *gv, void *gbeta,
                            float *gW0, float *scratch, int BH, int L, int d_key, int nu, int d_v, int bf16,
                            float eps, cudaStream_t st) {
    if (bf16)
        return launch_backward_t<__nv_bfloat16>(q, k, v, beta, W0, gy, gWL, gq, gk, gv, gbeta, gW0, scratch, BH, L,
                                                d_key, nu, d_v, eps, st);
    return launch_backward_t<float>(q, k, v, beta, W0, gy, gWL, gq, gk, gv, gbeta, gW0, scratch, BH, L, d_key, nu,
                                    d_v, eps, st);
}

} // namespace fw
