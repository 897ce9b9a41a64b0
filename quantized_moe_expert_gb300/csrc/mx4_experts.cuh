// MXFP4 routed experts with 8-bit activations.
//
// The weights are OCP microscaling MXFP4: E2M1 elements with one E8M0 scale per
// 32 consecutive weights of a row, w = 2^(s - 127) * e2m1(c) ("Running DeepSeek
// V4 Flash on an RTX 5080 ...", model list: the MXFP4 GGUF keeps DeepSeek's
// released MXFP4 routed-expert weights; decode runs them on Q8 activations).
// Every routed-expert product first quantises its input per 32 values:
// d = amax / 127 and q = x / d rounded to the nearest integer (ties to even),
// both in binary32; the product uses d * q. That covers the token rows x and
// the SwiGLU rows h before the down product.
//
// Layout (repacked at create from the 17-byte blocks): per row and 32-weight
// block, the 16 code bytes as one uint4 (weight i at byte i/2, even weight in
// the low nibble) in `codes` [rows][K/32], the scale bytes in `scale`
// [rows][K/32].
//
// One launch per product over (distinct expert, 8 rows): a warp owns a row,
// each lane a stride of 32-weight blocks, for the expert's token rows in chunks
// of up to 8; the lane decodes a block once per chunk and multiplies it with
// every row of the chunk.
#pragma once

#include "common.cuh"

namespace ds4 {

constexpr int kMx4Bytes = 17;

// E8M0 scale 2^(s - 127); s = 0 is the binary32 subnormal 2^-127, s = 255 NaN.
__device__ __forceinline__ float e8m0_value(unsigned s) {
    return __uint_as_float(s == 0u ? 0x00400000u : s == 255u ? 0x7FC00000u : s << 23);
}

// Canonical 17-byte blocks -> codes and scales (one thread per block).
__global__ void repack_mx4_kernel(const uint8_t *__restrict__ src, int64_t nblocks, uint4 *__restrict__ codes,
                                  uint8_t *__restrict__ scale) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks)
        return;
    const uint8_t *b = src + i * kMx4Bytes;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
        w[k] = (uint32_t)b[4 * k] | (uint32_t)b[4 * k + 1] << 8 | (uint32_t)b[4 * k + 2] << 16 |
               (uint32_t)b[4 * k + 3] << 24;
    codes[i] = make_uint4(w[0], w[1], w[2], w[3]);
    scale[i] = b[16];
}

// Q8 activation blocks, dequantised: out[i] = d * q_i for the 32-value block of
// i. One thread per value; a warp is one block (n is a multiple of 32).
// src is bf16 (src_bf16) or fp32.
__global__ void act_q8_kernel(const void *__restrict__ src, int src_bf16, int64_t n, float *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i - (threadIdx.x & 31) >= n) // whole warps past the end
        return;
    const float v = i < n ? (src_bf16 ? bf16_to_f32(static_cast<const uint16_t *>(src)[i])
                                      : static_cast<const float *>(src)[i])
                          : 0.f;
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float d = amax / 127.0f; // IEEE division: the build does not use fast math
    const float q = d > 0.f ? rintf(v / d) : 0.f;
    if (i < n)
        out[i] = d * q;
}

// E2M1 value of the low nibble of c (a multiple of 0.5 in [-6, 6]).
__device__ __forceinline__ float e2m1_value(unsigned c) {
    const float m = 0.5f * (float)((kE2M1Twice >> (4u * (c & 7u))) & 15u);
    return (c & 8u) ? -m : m;
}

// out[pos][r] for the expert-grouped rows pos of distinct expert u, r in the
// expert's M rows: the MXFP4 product of matrix A (or SwiGLU of gate/up when
// GATEUP) with activation rows act[row_of(pos)][0..Kd).
// GATEUP: A = gate, B = up, act rows are tokens perm[pos] / K, out = h (fp32);
// else A = down, act rows are grouped positions, out = ye.
// NT: rows of the expert handled together (the launch's bound on an expert's
// rows, 1, 2, 4 or 8; more are taken in chunks of NT). A lane first loads the
// codes and scales of up to kMx4LaneBlocks of its blocks, then multiplies.
constexpr int kMx4LaneBlocks = 4;

template <bool GATEUP, int NT>
__global__ void __launch_bounds__(256) mx4_product_kernel(Mx4Mat A, Mx4Mat B, const float *__restrict__ act,
                                                          const int32_t *__restrict__ uexp,
                                                          const int32_t *__restrict__ uoff,
                                                          const int32_t *__restrict__ nuniq,
                                                          const int32_t *__restrict__ perm, int K, int M, int Kd,
                                                          float *__restrict__ out) {
    const int u = blockIdx.y;
    if (u >= __ldg(nuniq))
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= M)
        return;
    const int e = __ldg(uexp + u);
    const int p0 = __ldg(uoff + u), p1 = __ldg(uoff + u + 1);
    const int nb = Kd / 32;
    const int64_t row = ((int64_t)e * M + r) * nb;
    for (int c0 = p0; c0 < p1; c0 += NT) {
        const int n = p1 - c0 < NT ? p1 - c0 : NT;
        const float *arow[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int pos = c0 + (t < n ? t : 0);
            const int64_t ar = GATEUP ? __ldg(perm + pos) / K : pos;
            arow[t] = act + ar * Kd;
        }
        float ga[NT], ua[NT];
#pragma unroll
        for (int t = 0; t < NT; t++)
            ga[t] = ua[t] = 0.f;
        for (int b0 = lane; b0 < nb; b0 += 32 * kMx4LaneBlocks) {
            uint4 ca[kMx4LaneBlocks], cb[kMx4LaneBlocks];
            unsigned sa[kMx4LaneBlocks], sb[kMx4LaneBlocks];
#pragma unroll
            for (int j = 0; j < kMx4LaneBlocks; j++) {
                const int b = b0 + 32 * j;
                ca[j] = cb[j] = make_uint4(0, 0, 0, 0);
                sa[j] = sb[j] = 0;
                if (b < nb) {
                    ca[j] = __ldg(A.codes + row + b);
                    sa[j] = __ldg(A.scale + row + b);
                    if (GATEUP) {
                        cb[j] = __ldg(B.codes + row + b);
                        sb[j] = __ldg(B.scale + row + b);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kMx4LaneBlocks; j++) {
                const int b = b0 + 32 * j;
                if (b < nb) {
                    const uint32_t wa[4] = {ca[j].x, ca[j].y, ca[j].z, ca[j].w};
                    const uint32_t wb[4] = {cb[j].x, cb[j].y, cb[j].z, cb[j].w};
                    float pa[NT], pb[NT];
#pragma unroll
                    for (int t = 0; t < NT; t++)
                        pa[t] = pb[t] = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; q++) { // 8 weights per code word
                        float va[8], vb[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            va[i] = e2m1_value(wa[q] >> (4 * i));
                            vb[i] = GATEUP ? e2m1_value(wb[q] >> (4 * i)) : 0.f;
                        }
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            if (t < n) {
                                const float4 x0 = __ldg(reinterpret_cast<const float4 *>(arow[t] + b * 32 + 8 * q));
                                const float4 x1 =
                                    __ldg(reinterpret_cast<const float4 *>(arow[t] + b * 32 + 8 * q + 4));
                                const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                                for (int i = 0; i < 8; i++) {
                                    pa[t] = fmaf(va[i], xv[i], pa[t]);
                                    if (GATEUP)
                                        pb[t] = fmaf(vb[i], xv[i], pb[t]);
                                }
                            }
                        }
                    }
                    const float Xa = e8m0_value(sa[j]), Xb = GATEUP ? e8m0_value(sb[j]) : 0.f;
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        ga[t] = fmaf(Xa, pa[t], ga[t]);
                        if (GATEUP)
                            ua[t] = fmaf(Xb, pb[t], ua[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const float g = warp_sum(ga[t]);
            const float uu = GATEUP ? warp_sum(ua[t]) : 0.f;
            if (lane == 0 && t < n)
                out[(int64_t)(c0 + t) * M + r] = GATEUP ? silu(g) * uu : g;
        }
    }
}

} // namespace ds4
