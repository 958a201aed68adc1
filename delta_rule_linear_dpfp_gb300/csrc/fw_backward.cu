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
// Mapping.  The rows of W are independent in both sweeps except for three
// sums over rows per token (g_phi(q), g_phi(k), gbeta), which only feed the
// outputs.  So the state is split by rows: one CTA of 256 threads per
// (batch, head) and block of up to 16 rows keeps those rows of W and gW in
// shared memory (fp32) for the whole sequence and writes, per token, its
// partial sums over its rows; a second kernel adds the blocks' partials in
// block order (deterministic) and takes the DPFP backward of q and k, one
// warp per token.  phi(k_t) and phi(q_t) of every token are made first by
// the DPFP kernel (fp32, in the scratch), so the serial token loop only
// stages them.  The forward sweep keeps u_t for every token (global
// scratch); the reverse sweep steps W back exactly as the forward stepped it
// up (W_{t-1} = W_t - u_t phi(k_t)^T, one rounding per element and token).
// Row dot products take one warp per row, column sums one thread per column
// (deterministic order), updates one thread per 4 elements.  fp32 arithmetic on
// CUDA cores throughout: the token loop is serial, so the first kernel is
// latency-bound, and the split multiplies the CTAs that hide that latency.
#include "fw_common.cuh"
#include "fw_forward_tc.h"

#include <algorithm>
#include <type_traits>

namespace fw {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdRows = 16;  // rows of W per CTA

// The DPFP backward of one row by one warp: given g = dL/dphi and the raw row
// kr (both in shared memory), writes dL/dk to dst.  xs: scratch of 2 d_key.
template <typename T>
FW_DEV void dpfp_backward_warp(const float *kr, const float *g, float *xs, T *dst, int d_key, int nu, float eps,
                               int lane) {
    const int n = 2 * d_key, d_dot = n * nu;
    for (int j = lane; j < d_key; j += 32) {
        const float kv = kr[j];
        xs[j] = fmaxf(kv, 0.f);
        xs[d_key + j] = fmaxf(-kv, 0.f);
    }
    __syncwarp();
    float s = 0.f, gp = 0.f; // sum of the products, g . products
    int i = lane / n + 1, j = lane - (i - 1) * n;
    for (int m = lane; m < d_dot; m += 32) {
        const int src = j - i < 0 ? j - i + n : j - i;
        const float p = xs[j] * xs[src];
        s += p;
        gp = fmaf(g[m], p, gp);
        for (j += 32; j >= n; j -= n)
            ++i;
    }
    s = warp_sum(s);
    gp = warp_sum(gp);
    const float c1 = 1.0f / (s + eps), c2 = gp * c1 * c1; // d phi_m / d p_l = delta_ml c1 - p_m c1^2
    for (int j0 = lane; j0 < d_key; j0 += 32) {
        float gx[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) { // x[j0] (from k) and x[d_key + j0] (from -k)
            const int jj = j0 + h * d_key;
            for (int ii = 1; ii <= nu; ++ii) {
                const int lo = jj - ii < 0 ? jj - ii + n : jj - ii, hi = jj + ii >= n ? jj + ii - n : jj + ii;
                // x[jj] is the left factor of product (ii, jj) and the rolled
                // factor of product (ii, jj + ii)
                gx[h] = fmaf(g[(ii - 1) * n + jj] * c1 - c2, xs[lo], gx[h]);
                gx[h] = fmaf(g[(ii - 1) * n + hi] * c1 - c2, xs[hi], gx[h]);
            }
        }
        const float kv = kr[j0];
        io<T>::store(dst + j0, (kv > 0.f ? gx[0] : 0.f) - (kv < 0.f ? gx[1] : 0.f));
    }
    __syncwarp();
}

// f(e4, r, m4) for the float4 groups e4 = r * d_dot / 4 + m4 this thread
// owns (e4 = tid, tid + 256, ...); d_dot % 4 == 0.
template <typename F>
FW_DEV void for_groups(int nel, int d_dot, int tid, F f) {
    const int g = d_dot / 4, ng = nel / 4;
    const int dr = kBwdThreads / g, dm = kBwdThreads - dr * g;
    int r = tid / g, m4 = tid - r * g;
    for (int e4 = tid; e4 < ng; e4 += kBwdThreads) {
        f(e4, r, m4);
        r += dr;
        m4 += dm;
        if (m4 >= g) {
            m4 -= g;
            ++r;
        }
    }
}

FW_DEV float4 fma4(float s, float4 x, float4 y) {
    return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}

// Row dot products a = A[r] . p and, with HAS_B, b = B[r] . p for every row,
// then fin(r, a, b) on lane 0 of the warp that owns the row; warp w takes
// rows w and w + 8 (rows <= 16).
template <bool HAS_B, typename F>
FW_DEV void row_dots_fin(const float *A, const float *B, const float *p, int rows, int d_dot, int warp, int lane,
                         F fin) {
    constexpr int kMaxRows = (kBwdRows + kBwdWarps - 1) / kBwdWarps;
    float sa[kMaxRows], sb[kMaxRows];
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
        sa[i] = 0.f;
        sb[i] = 0.f;
    }
    for (int m = 4 * lane; m < d_dot; m += 128) { // d_dot % 4 == 0, 16-byte aligned rows and p
        const float4 pm = *reinterpret_cast<const float4 *>(p + m);
#pragma unroll
        for (int i = 0; i < kMaxRows; ++i) {
            const int r = warp + kBwdWarps * i;
            if (r < rows) {
                const float4 x = *reinterpret_cast<const float4 *>(A + r * d_dot + m);
                sa[i] = fmaf(x.x, pm.x, fmaf(x.y, pm.y, fmaf(x.z, pm.z, fmaf(x.w, pm.w, sa[i]))));
                if (HAS_B) {
                    const float4 y = *reinterpret_cast<const float4 *>(B + r * d_dot + m);
                    sb[i] = fmaf(y.x, pm.x, fmaf(y.y, pm.y, fmaf(y.z, pm.z, fmaf(y.w, pm.w, sb[i]))));
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < kMaxRows; ++i) {
            sa[i] += __shfl_xor_sync(0xffffffffu, sa[i], o);
            if (HAS_B)
                sb[i] += __shfl_xor_sync(0xffffffffu, sb[i], o);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kMaxRows; ++i) {
            const int r = warp + kBwdWarps * i;
            if (r < rows)
                fin(r, sa[i], sb[i]);
        }
    }
}

// Sum over the d_v rows of a[r][m] * b[r] (plus c[r][m] * d[r] when c is
// given) for column m: four independent accumulators.
FW_DEV float col_sum(const float *a, const float *b, const float *c, const float *d, int m, int d_v, int d_dot) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int r = 0;
    for (; r + 4 <= d_v; r += 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[e] = fmaf(a[(r + e) * d_dot + m], b[r + e], acc[e]);
            if (c)
                acc[e] = fmaf(c[(r + e) * d_dot + m], d[r + e], acc[e]);
        }
    }
    for (; r < d_v; ++r) {
        acc[0] = fmaf(a[r * d_dot + m], b[r], acc[0]);
        if (c)
            acc[0] = fmaf(c[r * d_dot + m], d[r], acc[0]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Block z of rows [r0, r0 + R) of one (batch, head).  phk, phq: phi(k),
// phi(q) of every token ([BH, L, d_dot] fp32, made by the DPFP kernel
// beforehand).  part: [blocks][BH][L][2 d_dot + 4]: per token this block's
// sums over its rows of g_phi(q) (first d_dot), g_phi(k) (next d_dot) and
// gbeta (at 2 d_dot).
// NH: staged entries per thread, the least with 256 NH >= 2 d_dot + 3 R + 1
// (each token's staging costs NH loads and stores per thread).
template <typename T, int NH>
__global__ void __launch_bounds__(kBwdThreads, 1)
    delta_backward_kernel(const float *__restrict__ phk, const float *__restrict__ phq, const T *__restrict__ v,
                          const T *__restrict__ beta, const float *__restrict__ W0, const T *__restrict__ gy,
                          const float *__restrict__ gWL, T *__restrict__ gv, float *__restrict__ gW0,
                          float *__restrict__ us, float *__restrict__ part, int L, int d_dot, int d_v) {
    extern __shared__ float sm[];
    const int r0 = blockIdx.y * kBwdRows, R = min(kBwdRows, d_v - r0);
    const int nel = R * d_dot;
    const int64_t BH = gridDim.x, bh = blockIdx.x;
    const size_t pst = 2 * (size_t)d_dot + 4; // floats per token in part
    // one token's inputs, staged: phi(k), phi(q) (d_dot each), v, gy, u (R each), beta
    const int ntok = 2 * d_dot + 3 * R + 1, sstr = (ntok + 3) & ~3; // slot stride keeps phi 16-byte aligned
    float *W = sm;                 // [R][d_dot] rows r0.. of the state W_t
    float *G = W + nel;            // [R][d_dot] the same rows of dL/dW_t
    float *gu = G + nel;           // dL/du_t, then beta_t dL/du_t
    float *aa = gu + kBwdRows;     // W_{t-1} phi(k_t), then -beta_t dL/du_t
    float *gbr = aa + kBwdRows;    // per row: dL/du_t (v_t - W_{t-1} phi(k_t)), the terms of gbeta
    float *stg = gbr + kBwdRows;   // [2][sstr] staged token inputs (double-buffered)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *pkb = phk + bh * L * d_dot, *pqb = phq + bh * L * d_dot;
    const T *vb = v + bh * L * d_v + r0, *bb = beta + bh * L, *gyb = gy + bh * L * d_v + r0;
    float *ub = us + bh * L * d_v + r0;
    float *pb = part + ((size_t)blockIdx.y * BH + bh) * L * pst;

    // Thread tid loads entries tid, tid + 256, ... of token t's staged vector
    // into registers; they are stored to shared memory one token later, so
    // the load latency hides behind the current token's work.
    auto fetch = [&](int t, bool reverse, float (&x)[NH]) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const int e = tid + h * kBwdThreads;
            float val = 0.f;
            if (t >= 0 && t < L && e < ntok) {
                if (e < d_dot)
                    val = __ldcg(pkb + (int64_t)t * d_dot + e);
                else if (e < 2 * d_dot)
                    val = reverse ? __ldcg(pqb + (int64_t)t * d_dot + e - d_dot) : 0.f;
                else if (e < 2 * d_dot + R)
                    val = io<T>::load(vb + (int64_t)t * d_v + e - 2 * d_dot);
                else if (e < 2 * d_dot + 2 * R)
                    val = reverse ? io<T>::load(gyb + (int64_t)t * d_v + e - 2 * d_dot - R) : 0.f;
                else if (e < 2 * d_dot + 3 * R)
                    val = reverse ? __ldcg(ub + (int64_t)t * d_v + e - 2 * d_dot - 2 * R) : 0.f;
                else
                    val = io<T>::load(bb + t);
            }
            x[h] = val;
        }
    };
    auto stage = [&](int t, const float (&x)[NH]) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const int e = tid + h * kBwdThreads;
            if (e < ntok)
                stg[(t & 1) * sstr + e] = x[h];
        }
    };

    griddep_launch_dependents();
    griddep_wait();
    pkb = after_wait(pkb);
    pqb = after_wait(pqb);
    vb = after_wait(vb);
    bb = after_wait(bb);
    gyb = after_wait(gyb);
    ub = after_wait(ub);
    W0 = after_wait(W0);
    gWL = after_wait(gWL);
    const size_t wofs = (size_t)bh * d_v * d_dot + (size_t)r0 * d_dot; // this block's rows in W0, gW
    for (int e = tid; e < nel; e += kBwdThreads) {
        W[e] = W0 ? __ldcg(W0 + wofs + e) : 0.f;
        G[e] = gWL ? __ldcg(gWL + wofs + e) : 0.f;
    }
    float nxt[NH];
    // ---- forward sweep: keep u_t
    fetch(0, false, nxt);
    stage(0, nxt);
    for (int t = 0; t < L; ++t) {
        fetch(t + 1, false, nxt);
        const float *pk = stg + (t & 1) * sstr, *tv = pk + 2 * d_dot;
        __syncthreads(); // token t's inputs were staged by every thread at the end of the previous step
        const float bt = pk[ntok - 1];
        row_dots_fin<false>(W, nullptr, pk, R, d_dot, warp, lane, [&](int r, float a, float) { // u = beta (v - W_{t-1} phi(k))
            const float u = bt * (tv[r] - a);
            gu[r] = u;
            ub[(int64_t)t * d_v + r] = u;
        });
        __syncthreads();
        for_groups(nel, d_dot, tid, [&](int e4, int r, int m4) { // W_t = W_{t-1} + u phi(k)^T
            float4 *w = reinterpret_cast<float4 *>(W) + e4;
            *w = fma4(gu[r], reinterpret_cast<const float4 *>(pk)[m4], *w);
        });
        stage(t + 1, nxt);
    }
    __syncthreads(); // the u_t written above are read back below by other threads
    // ---- reverse sweep
    fetch(L - 1, true, nxt);
    stage(L - 1, nxt);
    for (int t = L - 1; t >= 0; --t) {
        fetch(t - 1, true, nxt);
        const float *pk = stg + (t & 1) * sstr, *pq = pk + d_dot, *tv = pq + d_dot, *tg = tv + R, *tu = tg + R;
        float *pt = pb + (size_t)t * pst;
        __syncthreads(); // token t's inputs were staged by every thread at the end of the previous step
        const float bt = pk[ntok - 1];
        for (int m = tid; m < d_dot; m += kBwdThreads) // this block's share of g_phi(q) = W_t^T gy
            pt[m] = col_sum(W, tg, nullptr, nullptr, m, R, d_dot);
        __syncthreads(); // W_t read above before it is stepped back below
        for_groups(nel, d_dot, tid, [&](int e4, int r, int m4) { // gW += gy phi(q)^T; W_{t-1} = W_t - u phi(k)^T
            float4 *g = reinterpret_cast<float4 *>(G) + e4, *w = reinterpret_cast<float4 *>(W) + e4;
            *g = fma4(tg[r], reinterpret_cast<const float4 *>(pq)[m4], *g);
            *w = fma4(-tu[r], reinterpret_cast<const float4 *>(pk)[m4], *w);
        });
        __syncthreads();
        // g = gW phi(k), a = W_{t-1} phi(k); gv = beta g; keep e = beta g (and -e) and g (v - a)
        row_dots_fin<true>(G, W, pk, R, d_dot, warp, lane, [&](int r, float g, float a) {
            gu[r] = g * bt;
            aa[r] = -g * bt;
            gbr[r] = g * (tv[r] - a);
            io<T>::store(gv + (bh * L + t) * d_v + r0 + r, g * bt);
        });
        __syncthreads();
        for (int m = tid; m < d_dot; m += kBwdThreads) // this block's share of g_phi(k) = gW^T u - W_{t-1}^T e
            pt[d_dot + m] = col_sum(G, tu, W, aa, m, R, d_dot);
        if (warp == 0) { // and of gbeta (R <= 32 rows, one lane each, a fixed order)
            const float acc = warp_sum(lane < R ? gbr[lane] : 0.f);
            if (lane == 0)
                pt[2 * d_dot] = acc;
        }
        __syncthreads();
        for_groups(nel, d_dot, tid, [&](int e4, int r, int m4) { // gW_{t-1} = gW - e phi(k)^T
            float4 *g = reinterpret_cast<float4 *>(G) + e4;
            *g = fma4(-gu[r], reinterpret_cast<const float4 *>(pk)[m4], *g);
        });
        if (t > 0)
            stage(t - 1, nxt);
    }
    __syncthreads();
    if (gW0)
        for (int e = tid; e < nel; e += kBwdThreads)
            gW0[wofs + e] = G[e];
}

// The blocks' partial sums added in block order, then the DPFP backward of
// q_t and k_t and gbeta_t: one warp per (batch, head, token).
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
    backward_finish_kernel(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ part,
                           T *__restrict__ gq, T *__restrict__ gk, T *__restrict__ gbeta, int64_t rows, int blocks,
                           int d_key, int nu, float eps) {
    extern __shared__ float sm[];
    const int d_dot = 2 * d_key * nu, n = 2 * d_key;
    const size_t pst = 2 * (size_t)d_dot + 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *ws = sm + (size_t)warp * (2 * d_dot + 2 * d_key + 2 * n);
    float *gpq = ws, *gpk = gpq + d_dot, *kr = gpk + d_dot, *qr = kr + d_key, *xs = qr + d_key; // xs: 2 n
    griddep_launch_dependents();
    griddep_wait(); // the partial sums are the preceding kernel's
    q = after_wait(q);
    k = after_wait(k);
    part = after_wait(part);
    for (int64_t row = (int64_t)blockIdx.x * kBwdWarps + warp; row < rows; row += (int64_t)gridDim.x * kBwdWarps) {
        for (int j = lane; j < d_key; j += 32) {
            kr[j] = io<T>::load(k + row * d_key + j);
            qr[j] = io<T>::load(q + row * d_key + j);
        }
        for (int m = lane; m < 2 * d_dot + 1; m += 32) {
            float acc = 0.f;
            for (int z = 0; z < blocks; ++z)
                acc += __ldcg(part + ((size_t)z * rows + row) * pst + m);
            if (m < 2 * d_dot)
                gpq[m] = acc; // gpk follows gpq contiguously
            else
                io<T>::store(gbeta + row, acc);
        }
        __syncwarp();
        dpfp_backward_warp(qr, gpq, xs, gq + row * d_key, d_key, nu, eps, lane);
        dpfp_backward_warp(kr, gpk, xs + n, gk + row * d_key, d_key, nu, eps, lane);
        __syncwarp();
    }
}

template <typename T>
cudaError_t launch_backward_t(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                              const void *gy, const float *gWL, void *gq, void *gk, void *gv, void *gbeta,
                              float *gW0, float *scratch, int BH, int L, int d_key, int nu, int d_v, float eps,
                              int num_sms, cudaStream_t st) {
    const bool chunked = backward_chunked_supported(d_key, nu, d_v, L);
    const int blocks = chunked ? 1 : (d_v + kBwdRows - 1) / kBwdRows, d_dot = 2 * d_key * nu;
    const int64_t rows = (int64_t)BH * L;
    const size_t pst = 2 * (size_t)d_dot + 4;
    float *us = chunked ? nullptr : scratch;
    float *phk = chunked ? scratch : us + (size_t)rows * d_v, *phq = phk + (size_t)rows * d_dot;
    float *part = phq + (size_t)rows * d_dot;
    const int bf16 = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    cudaError_t e = launch_dpfp(k, phk, rows, d_key, nu, bf16, 0, eps, num_sms, st);
    if (e == cudaSuccess)
        e = launch_dpfp(q, phq, rows, d_key, nu, bf16, 0, eps, num_sms, st);
    if (e != cudaSuccess)
        return e;
    if (chunked) {
        e = launch_backward_chunked(phk, phq, v, beta, W0, gy, gWL, gv, gW0, part, part + (size_t)rows * pst, BH, L,
                                    d_dot, d_v, bf16, st);
        if (e != cudaSuccess)
            return e;
    } else {
        const size_t smem = backward_smem_bytes(d_key, nu, d_v);
        const int ntok = 2 * d_dot + 3 * std::min(d_v, kBwdRows) + 1;
        auto kern = ntok <= kBwdThreads       ? delta_backward_kernel<T, 1>
                    : ntok <= 2 * kBwdThreads ? delta_backward_kernel<T, 2>
                    : ntok <= 3 * kBwdThreads ? delta_backward_kernel<T, 3>
                    : ntok <= 5 * kBwdThreads ? delta_backward_kernel<T, 5>
                                              : delta_backward_kernel<T, 9>; // d_dot <= 1024
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        e = launch_pdl(kern, dim3((unsigned)BH, (unsigned)blocks), dim3(kBwdThreads), smem, st, (const float *)phk,
                       (const float *)phq, static_cast<const T *>(v), static_cast<const T *>(beta), W0,
                       static_cast<const T *>(gy), gWL, static_cast<T *>(gv), gW0, us, part, L, d_dot, d_v);
        if (e != cudaSuccess)
            return e;
    }
    const size_t fsmem = sizeof(float) * kBwdWarps * (2 * (size_t)d_dot + 6 * (size_t)d_key);
    auto fin = backward_finish_kernel<T>;
    e = cudaFuncSetAttribute(fin, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = (unsigned)std::min<int64_t>((rows + kBwdWarps - 1) / kBwdWarps, 4096);
    return launch_pdl(fin, dim3(grid), dim3(kBwdThreads), fsmem, st, static_cast<const T *>(q),
                      static_cast<const T *>(k), (const float *)part, static_cast<T *>(gq), static_cast<T *>(gk),
                      static_cast<T *>(gbeta), rows, blocks, d_key, nu, eps);
}

} // namespace

// Shared memory of one CTA of the first kernel: its rows of W and gW, three
// row vectors and two staged copies of one token's inputs.
size_t backward_smem_bytes(int d_key, int nu, int d_v) {
    const size_t d_dot = (size_t)2 * d_key * nu, R = std::min(d_v, kBwdRows);
    const size_t ntok = 2 * d_dot + 3 * R + 1, sstr = (ntok + 3) & ~(size_t)3;
    return sizeof(float) * (2 * R * d_dot + 3 * (size_t)kBwdRows + 2 * sstr);
}

// Global scratch: u_t for every token and row, phi(k_t) and phi(q_t) for
// every token, then the row blocks' partial sums per token.
size_t backward_workspace_bytes(int BH, int L, int d_key, int nu, int d_v) {
    const size_t d_dot = (size_t)2 * d_key * nu, rows = (size_t)BH * L;
    if (backward_chunked_supported(d_key, nu, d_v, L))
        return sizeof(float) * (2 * rows * d_dot + rows * (2 * d_dot + 4) +
                                backward_chunked_buffer_floats(BH, L, d_key, nu, d_v));
    const size_t blocks = (d_v + kBwdRows - 1) / kBwdRows;
    return sizeof(float) * (rows * d_v + 2 * rows * d_dot + blocks * rows * (2 * d_dot + 4));
}

cudaError_t launch_backward(const void *q, const void *k, const void *v, const void *beta, const float *W0,
                            const void *gy, const float *gWL, void *gq, void *gk, void *gv, void *gbeta,
                            float *gW0, float *scratch, int BH, int L, int d_key, int nu, int d_v, int bf16,
                            float eps, int num_sms, cudaStream_t st) {
    if (bf16)
        return launch_backward_t<__nv_bfloat16>(q, k, v, beta, W0, gy, gWL, gq, gk, gv, gbeta, gW0, scratch, BH, L,
                                                d_key, nu, d_v, eps, num_sms, st);
    return launch_backward_t<float>(q, k, v, beta, W0, gy, gWL, gq, gk, gv, gbeta, gW0, scratch, BH, L, d_key, nu,
                                    d_v, eps, num_sms, st);
}

} // namespace fw
