// fw_dpfp.cuh -- the register/shuffle form of the DPFP roll shared by the
// standalone DPFP kernel and the prologue of the chunked forward.
//
// A row of x = ReLU([k, -k]) (n = 2*d_key entries) is held by G = d_key/4
// consecutive lanes of a warp, lane g holding x[8g .. 8g+7].  Block i of phi
// needs x[j] * x[(j - i) mod n] (torch.roll(shifts=i) convention, Fast
// Weights Transformer guide, DPFP source).  For i = 8*qs + R the rolled entry
// at position 8g + c lives in lane g - qs (c >= R) or g - qs - 1 (c < R) of
// the same row group, register (c - R) mod 8; R is a template argument so
// that every register index is static.
#pragma once

#include "fw_common.cuh"

namespace fw {

// Products x[8g+c] * x[(8g+c-i) mod n] for c = 0..7 with i = 8*qs + R.
template <int G, int R>
FW_DEV void dpfp_block(const float (&x)[8], float (&p)[8], int g, int base_lane, int qs) {
    const int src0 = base_lane + ((g - qs) % G + G) % G;     // holds x[8(g-qs) + .]
    const int src1 = base_lane + ((g - qs - 1) % G + G) % G; // holds x[8(g-qs-1) + .]
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float rolled;
        if (c >= R)
            rolled = __shfl_sync(0xffffffffu, x[c - R], src0);
        else
            rolled = __shfl_sync(0xffffffffu, x[c - R + 8], src1);
        p[c] = x[c] * rolled;
    }
}

template <int G>
FW_DEV void dpfp_block_dispatch(const float (&x)[8], float (&p)[8], int g, int base_lane, int i) {
    const int qs = i >> 3;
    switch (i & 7) {
    case 0: dpfp_block<G, 0>(x, p, g, base_lane, qs); break;
    case 1: dpfp_block<G, 1>(x, p, g, base_lane, qs); break;
    case 2: dpfp_block<G, 2>(x, p, g, base_lane, qs); break;
    case 3: dpfp_block<G, 3>(x, p, g, base_lane, qs); break;
    case 4: dpfp_block<G, 4>(x, p, g, base_lane, qs); break;
    case 5: dpfp_block<G, 5>(x, p, g, base_lane, qs); break;
    case 6: dpfp_block<G, 6>(x, p, g, base_lane, qs); break;
    default: dpfp_block<G, 7>(x, p, g, base_lane, qs); break;
    }
}

// The 8 raw key values behind this lane's entries of x (row `src`, d_key =
// 4*G elements), zeros when valid = false.
template <int G, typename T>
FW_DEV void dpfp_load_raw(const T *src, int g, bool valid, float (&kv)[8]) {
    if (valid) {
        load8(src + 8 * (g % (G / 2)), kv);
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            kv[c] = 0.f;
    }
}

// Load the 8 entries of x this lane owns from row `src` (d_key = 4*G
// elements): lanes g < G/2 take ReLU(k), the others ReLU(-k).  valid = false
// gives zeros (a padded row).
template <int G, typename T>
FW_DEV void dpfp_load_x(const T *src, int g, bool valid, float (&x)[8]) {
    float kv[8];
    if (valid) {
        load8(src + 8 * (g % (G / 2)), kv);
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            kv[c] = 0.f;
    }
    const bool neg = g >= G / 2;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        x[c] = fmaxf(neg ? -kv[c] : kv[c], 0.f);
}

// Sum of every phi product of the row (all nu blocks), reduced over the G
// lanes of the row group: the DPFP normaliser before eps.
template <int G>
FW_DEV float dpfp_row_sum(const float (&x)[8], int g, int base_lane, int nu) {
    float s = 0.f;
    for (int i = 1; i <= nu; ++i) {
        float p[8];
        dpfp_block_dispatch<G>(x, p, g, base_lane, i);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            s += p[c];
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// phi of one row, normalised, handed block by block to emit(i, p) with
// i = 1..nu and p[8] this lane's 8 entries of block i (already divided by
// sum + eps).  For nu <= NUC the products stay in registers between the sum
// and the output; beyond that they are recomputed.
template <int G, int NUC, typename Emit>
FW_DEV void dpfp_row_emit(const float (&x)[8], int g, int base_lane, int nu, float eps, Emit emit) {
    if (nu <= NUC) {
        float p[NUC][8];
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NUC; ++i) {
            if (i < nu) {
                dpfp_block_dispatch<G>(x, p[i], g, base_lane, i + 1); // i is static once unrolled
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    s += p[i][c];
            }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        const float inv = 1.0f / (s + eps);
#pragma unroll
        for (int i = 0; i < NUC; ++i) {
            if (i < nu) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    p[i][c] *= inv;
                emit(i + 1, p[i]);
            }
        }
    } else {
        const float inv = 1.0f / (dpfp_row_sum<G>(x, g, base_lane, nu) + eps);
        for (int i = 1; i <= nu; ++i) {
            float p[8];
            dpfp_block_dispatch<G>(x, p, g, base_lane, i);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                p[c] *= inv;
            emit(i, p);
        }
    }
}

} // namespace fw
