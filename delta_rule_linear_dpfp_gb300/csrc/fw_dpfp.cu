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
// stores; for nu <= 4 they stay in registers between the two steps, beyond
// that they are recomputed.
#include "fw_dpfp.cuh"

namespace fw {

namespace {

// Products of up to NUC blocks stay in registers between the sum and the
// output (dpfp_row_emit); larger nu recomputes them.
constexpr int NUC = 3;

template <int DK, typename Tin, typename Tout>
__global__ void __launch_bounds__(256, 4) dpfp_kernel(const Tin *__restrict__ xin, Tout *__restrict__ out,
                                                   int64_t rows, int nu, float eps) {
    constexpr int G = DK / 4;         // lanes per row
    constexpr int RPW = 32 / G;       // rows per warp
    constexpr int N = 2 * DK;         // length of [k, -k]
    const int lane = threadIdx.x & 31;
    const int g = lane % G;
    const int base_lane = lane - g;
    const int64_t d_dot = (int64_t)N * nu;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (; wid * RPW < rows; wid += warps_total) {
        const int64_t row = wid * RPW + lane / G;
        const bool valid = row < rows;
        float x[8];
        dpfp_load_x<G>(xin + (valid ? row : 0) * DK, g, valid, x);
        Tout *orow = out + row * d_dot + 8 * g;
        dpfp_row_emit<G, NUC>(x, g, base_lane, nu, eps, [&](int i, float (&p)[8]) {
            if (valid)
                store8(orow + (int64_t)(i - 1) * N, p);
        });
    }
}

template <int DK, typename Tin, typename Tout>
cudaError_t launch_dpfp_t(const void *x, void *phi, int64_t rows, int nu, float eps, int num_sms,
                          cudaStream_t stream) {
    constexpr int RPW = 32 / (DK / 4);
    const int64_t warps = (rows + RPW - 1) / RPW;
    int64_t blocks = (warps + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap)
        blocks = cap;
    dpfp_kernel<DK, Tin, Tout><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const Tin *>(x), static_cast<Tout *>(phi), rows, nu, eps);
    return cudaGetLastError();
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
