// fw_dpfp.cu -- K1: the DPFP feature map with its sum-normalisation in one
// pass over HBM.
//
// Method (Fast Weights Transformer guide, section "DPFP: projection formula
// and hyper-parameters", the normalisation formula and the DPFP source shown
// with it): x = ReLU([k, -k]) of length n = 2*d_key; block i (i = 1..nu) of
// phi holds x[j] * x[(j - i) mod n] (torch.roll(shifts=i) convention);
// phi /= (sum(phi) + eps).
//
// Mapping: G = d_key/4 lanes own one row; lane g of a row group holds the 8
// consecutive entries x[8g .. 8g+7] in registers (lanes g < G/2 build them
// from k, the others from -k, each with one 16- or 32-byte load).  For a
// shift i = 8*qs + r the rolled entry needed at x[8g + c] sits in lane
// g - qs (or g - qs - 1) of the same row group at register (c - r) mod 8;
// r is dispatched to a compile-time case so every register index stays
// static and the roll costs 8 warp shuffles per block.  The products are
// summed (reduced over the G lanes with xor shuffles), scaled by one
// reciprocal of (sum + eps) per row and written 8 per lane with 16-byte
// stores; for nu <= 3 they stay in registers between the two steps, beyond
// that they are recomputed.
#include "fw_dpfp.cuh"

namespace fw {

namespace {

// Products of up to NUC blocks stay in registers between the sum and the
// output (dpfp_row_emit); larger nu recomputes them.
constexpr int NUC = 3;
constexpr int kBlocksPerSM = 4; // resident CTAs of 256 threads (__launch_bounds__ below)

// The 8 raw input values behind one lane's entries of x, as loaded (the
// load is issued one row ahead of its use, so only the registers travel).
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 u;
    FW_DEV void load(const __nv_bfloat16 *p, bool valid) {
        u = valid ? __ldcg(reinterpret_cast<const uint4 *>(p)) : make_uint4(0, 0, 0, 0);
    }
    FW_DEV void widen(float (&o)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    FW_DEV void load(const float *p, bool valid) {
        a = valid ? __ldcg(reinterpret_cast<const float4 *>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
        b = valid ? __ldcg(reinterpret_cast<const float4 *>(p) + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    FW_DEV void widen(float (&o)[8]) const {
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
};

// A persistent grid (kBlocksPerSM CTAs per SM, one wave): each warp walks
// its rows RPW at a time with a grid stride, and the next rows' input is
// loaded before the current rows are worked on, so the load latency is paid
// once per warp rather than once per row.  Launched with programmatic
// dependent launch (its set-up overlaps the tail of the preceding kernel).
template <int DK, typename Tin, typename Tout>
__global__ void __launch_bounds__(256, kBlocksPerSM) dpfp_kernel(const Tin *__restrict__ xin, Tout *__restrict__ out,
                                                              int64_t rows, int nu, float eps) {
    constexpr int G = DK / 4;         // lanes per row
    constexpr int RPW = 32 / G;       // rows per warp
    constexpr int N = 2 * DK;         // length of [k, -k]
    const int lane = threadIdx.x & 31;
    const int g = lane % G;
    const int base_lane = lane - g;
    const bool neg = g >= G / 2;      // lanes of the second half hold ReLU(-k)
    const int koff = 8 * (g % (G / 2));
    const int64_t d_dot = (int64_t)N * nu;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    // this warp's first rows are pulled into L2 while the preceding kernel
    // finishes (a prefetch is safe before the wait: see l2_prefetch)
    if (lane == 0 && wid * RPW < rows) {
        const int64_t n = rows - wid * RPW < RPW ? rows - wid * RPW : RPW;
        if ((DK * sizeof(Tin)) % 16 == 0)
            l2_prefetch(xin + wid * RPW * DK, (uint32_t)(n * DK * sizeof(Tin)));
    }
    griddep_launch_dependents();
    griddep_wait(); // x may be the preceding kernel's output
    xin = after_wait(xin);
    Raw8<Tin> cur;
    {
        const int64_t row = wid * RPW + lane / G;
        cur.load(xin + (row < rows ? row : 0) * DK + koff, row < rows);
    }
    for (; wid * RPW < rows; wid += warps_total) {
        const int64_t row = wid * RPW + lane / G;
        const bool valid = row < rows;
        Raw8<Tin> nxt;
        {
            const int64_t nrow = row + warps_total * RPW;
            nxt.load(xin + (nrow < rows ? nrow : 0) * DK + koff, nrow < rows);
        }
        float x[8];
        cur.widen(x);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            x[e] = fmaxf(neg ? -x[e] : x[e], 0.f);
        Tout *orow = out + row * d_dot + 8 * g;
        dpfp_row_emit<G, NUC>(x, g, base_lane, nu, eps, [&](int i, float (&p)[8]) {
            if (valid)
                store8(orow + (int64_t)(i - 1) * N, p);
        });
        cur = nxt;
    }
}

template <int DK, typename Tin, typename Tout>
cudaError_t launch_dpfp_t(const void *x, void *phi, int64_t rows, int nu, float eps, int num_sms,
                          cudaStream_t stream) {
    constexpr int RPW = 32 / (DK / 4);
    const int64_t warps = (rows + RPW - 1) / RPW;
    int64_t blocks = (warps + 7) / 8;
    const int64_t cap = (int64_t)num_sms * kBlocksPerSM;
    if (blocks > cap)
        blocks = cap;
    return launch_pdl(dpfp_kernel<DK, Tin, Tout>, dim3((unsigned)blocks), dim3(256), 0, stream,
                      static_cast<const Tin *>(x), static_cast<Tout *>(phi), rows, nu, eps);
}

template <int DK>
cudaError_t launch_dpfp_dk(const void *x, void *phi, int64_t rows, int nu, int in_bf16, int out_bf16,
                           float eps, int num_sms, cudaStream_t st) {
    if (in_bf16 && out_bf16)
        return launch_dpfp_t<DK, __nv_bfloat16, __nv_bfloat16>(x, phi, rows, nu, eps, num_sms, st);
    if (in_bf16)
        return launch_dpfp_t<DK, __nv_bfloat16, float>(x, phi, rows, nu, eps, num_sms, st);
    if (out_bf16)
        return launch_dpfp_t<DK, float, __nv_bfloat16>(x, phi, rows, nu, eps, num_sms, st);
    return launch_dpfp_t<DK, float, float>(x, phi, rows, nu, eps, num_sms, st);
}

} // namespace

// Host launcher; arguments were validated by the caller.
cudaError_t launch_dpfp(const void *x, void *phi, int64_t rows, int d_key, int nu, int in_bf16,
                        int out_bf16, float eps, int num_sms, cudaStream_t st) {
    switch (d_key) {
    case 8: return launch_dpfp_dk<8>(x, phi, rows, nu, in_bf16, out_bf16, eps, num_sms, st);
    case 16: return launch_dpfp_dk<16>(x, phi, rows, nu, in_bf16, out_bf16, eps, num_sms, st);
    case 32: return launch_dpfp_dk<32>(x, phi, rows, nu, in_bf16, out_bf16, eps, num_sms, st);
    case 64: return launch_dpfp_dk<64>(x, phi, rows, nu, in_bf16, out_bf16, eps, num_sms, st);
    case 128: return launch_dpfp_dk<128>(x, phi, rows, nu, in_bf16, out_bf16, eps, num_sms, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace fw
