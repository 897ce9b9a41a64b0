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

// Canonical 17-byte blocks [rows][K/32] -> the prefill GEMM's tile records
// (Mx4Tile). One thread per (row, 32-weight block).
__global__ void repack_mx4_tile_kernel(const uint8_t *__restrict__ src, int64_t rows, int nb,
                                       uint8_t *__restrict__ rec) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * nb)
        return;
    const int64_t row = i / nb;
    const int kb = (int)(i % nb);
    const int64_t rt = row >> 7;
    const int r = (int)(row & 127), ks = kb >> 1, half = kb & 1;
    const uint8_t *b = src + i * kMx4Bytes;
    uint8_t *dst = rec + (rt * (nb / 2) + ks) * kMx4TileRec;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
        w[k] = (uint32_t)b[4 * k] | (uint32_t)b[4 * k + 1] << 8 | (uint32_t)b[4 * k + 2] << 16 |
               (uint32_t)b[4 * k + 3] << 24;
    reinterpret_cast<uint4 *>(dst)[half * 128 + r] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[2 * 128 * 16 + 2 * r + half] = b[16];
}

// The OCP MX conversion of one value v of a 32-value block whose largest
// magnitude is amax: X = 2^(floor(log2 amax) - 2), clamped to the E8M0 range
// (amax = 0 or subnormal: 2^-127), and the E2M1 value nearest to v / X (ties to
// the even code, magnitude saturating at 6, sign kept: -0 for small negatives).
// Returns X * e2m1 as binary16 bits: exact while X lies in [2^-23, 2^13] (every
// block whose amax is in [2^-21, 2^16)); beyond that the binary16 value
// underflows or overflows.
__device__ __forceinline__ uint16_t fp4_grid_f16(float v, float amax) {
    const int ef = (int)(__float_as_uint(amax) >> 23); // biased exponent of amax >= 0
    const int sb = ef == 0 ? 0 : min(254, max(0, ef - 2));
    const float inv = sb == 254 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(254 - sb) << 23);
    const float X = sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)sb << 23);
    const float r = fabsf(v) * inv; // exact: a power of two (r < 8)
    const float m = r <= 0.25f  ? 0.f
                    : r < 0.75f ? 0.5f
                    : r <= 1.25f ? 1.f
                    : r < 1.75f ? 1.5f
                    : r <= 2.5f ? 2.f
                    : r < 3.5f  ? 3.f
                    : r <= 5.f  ? 4.f
                                : 6.f;
    return __half_as_ushort(__float2half_rn(copysignf(m * X, v)));
}

// FP4 activation rows for the MXFP4 prefill: bf16 x [n] -> binary16 values on
// the FP4 grid (fp4_grid_f16 per 32-value block). A thread per 8 values, four
// consecutive lanes per block (n is a multiple of 32, both arrays 16-byte
// aligned).
__global__ void act_fp4_kernel(const uint16_t *x, int64_t n, uint16_t *out) {
    pdl_launch_next();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i - (threadIdx.x & 31) >= n / 8) // whole warps past the end
        return;
    float v[8];
    uint32_t mb = 0u; // the largest magnitude's bits (a NaN ranks above every number)
    if (i < n / 8) {
        const uint4 w = reinterpret_cast<const uint4 *>(x)[i];
        const uint32_t p[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            v[2 * j] = bf16_to_f32(p[j] & 0xFFFFu);
            v[2 * j + 1] = bf16_to_f32(p[j] >> 16);
        }
#pragma unroll
        for (int j = 0; j < 8; j++)
            mb = max(mb, __float_as_uint(fabsf(v[j])));
    }
    // the block's four lanes (a block never straddles lanes of two warps)
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
    const float m = __uint_as_float(mb);
    if (i < n / 8) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; j++)
            o[j] = (uint32_t)fp4_grid_f16(v[2 * j], m) | ((uint32_t)fp4_grid_f16(v[2 * j + 1], m) << 16);
        reinterpret_cast<uint4 *>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Q8 activation blocks: per 32 values d = amax / 127 and q_i = x_i / d
// rounded to the nearest integer (ties to even), both IEEE binary32 (the build
// has no fast-math flags). One thread per value, a warp per block (n is a
// multiple of 32); codes to q, block scales to d. src is bf16 (src_bf16) or fp32.
__global__ void act_q8_kernel(const void *src, int src_bf16, int64_t n, int8_t *q,
                              float *d) {
    pdl_launch_next();
    pdl_wait();
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
    const float db = amax / 127.0f;
    if (i < n) {
        q[i] = (int8_t)(db > 0.f ? rintf(v / db) : 0.f);
        if ((threadIdx.x & 31) == 0)
            d[i / 32] = db;
    }
}

// Four consecutive E2M1 codes (the nibbles of the low 16 bits of h) as signed
// int8 lanes of 2 * e2m1: the magnitude by a byte permute of the table
// 0, 1, 2, 3, 4, 6, 8, 12; the sign as a byte mask M (0x00 / 0xFF) by a second
// permute that picks byte 0 (0x00) for a clear sign bit and replicates the top
// bit of byte 4 (0x80) for a set one. Returns the magnitudes; M in *neg.
__device__ __forceinline__ uint32_t e2m1x4_twice(uint32_t h, uint32_t *neg) {
    const uint32_t mag = __byte_perm(0x03020100u, 0x0C080604u, h & 0x7777u);
    const uint32_t s = h & 0x8888u;
    uint32_t m; // prmt's generic mode: a selector nibble with bit 3 set replicates the byte's sign bit
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m) : "r"(0u), "r"(0x80u), "r"(s | (s >> 1)));
    *neg = m;
    return mag;
}

// out[pos][r] for the expert-grouped rows pos of distinct expert u, r in the
// expert's M rows: the MXFP4 product of matrix A (or SwiGLU of gate/up when
// GATEUP) with Q8 activation rows (codes aq [rows][Kd], scales ad [rows][Kd/32]).
// GATEUP: A = gate, B = up, activation rows are tokens perm[pos] / K, out = h
// (fp32); else A = down, rows are grouped positions, out = ye.
// Per 32-weight block and activation row the sum of 2 e2m1(c_i) q_i is exact in
// int32 (two dp4a per 4 weights: all magnitudes, minus twice the negative
// ones), then scaled once by X d / 2 in fp32.
// NT: rows of the expert handled together (1, 2, 4 or 8; more in chunks).
constexpr int kMx4LaneBlocks = 4;

template <bool GATEUP, int NT>
__global__ void __launch_bounds__(256) mx4_product_kernel(Mx4Mat A, Mx4Mat B, const int8_t *aq,
                                                          const float *ad,
                                                          const int32_t *uexp,
                                                          const int32_t *uoff,
                                                          const int32_t *nuniq,
                                                          const int32_t *perm, int K, int M, int Kd,
                                                          float *out) {
    pdl_launch_next();
    pdl_wait();
    const int u = blockIdx.y;
    if (u >= *nuniq)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= M)
        return;
    const int e = uexp[u];
    const int p0 = uoff[u], p1 = uoff[u + 1];
    const int nb = Kd / 32;
    const int64_t row = ((int64_t)e * M + r) * nb;
    for (int c0 = p0; c0 < p1; c0 += NT) {
        const int n = p1 - c0 < NT ? p1 - c0 : NT;
        int64_t arow[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int pos = c0 + (t < n ? t : 0);
            arow[t] = GATEUP ? perm[pos] / K : pos;
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
                    // weights 8q+4h .. 8q+4h+3 are the nibbles of half h of code word q
                    uint32_t ma[8], na[8], mb[8], nbm[8];
                    const uint32_t wa[4] = {ca[j].x, ca[j].y, ca[j].z, ca[j].w};
                    const uint32_t wb[4] = {cb[j].x, cb[j].y, cb[j].z, cb[j].w};
#pragma unroll
                    for (int q = 0; q < 4; q++)
#pragma unroll
                        for (int hh = 0; hh < 2; hh++) {
                            ma[2 * q + hh] = e2m1x4_twice(wa[q] >> (16 * hh), &na[2 * q + hh]);
                            na[2 * q + hh] &= ma[2 * q + hh];
                            if (GATEUP) {
                                mb[2 * q + hh] = e2m1x4_twice(wb[q] >> (16 * hh), &nbm[2 * q + hh]);
                                nbm[2 * q + hh] &= mb[2 * q + hh];
                            }
                        }
                    const float Xa = 0.5f * e8m0_value(sa[j]), Xb = GATEUP ? 0.5f * e8m0_value(sb[j]) : 0.f;
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        if (t < n) {
                            const int4 *qp = reinterpret_cast<const int4 *>(aq + arow[t] * Kd + b * 32);
                            const int4 q0 = qp[0], q1 = qp[1];
                            const int qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                            int sa_ = 0, sn = 0, sbm = 0, snb = 0;
#pragma unroll
                            for (int m = 0; m < 8; m++) {
                                sa_ = __dp4a((int)ma[m], qw[m], sa_);
                                sn = __dp4a((int)na[m], qw[m], sn);
                                if (GATEUP) {
                                    sbm = __dp4a((int)mb[m], qw[m], sbm);
                                    snb = __dp4a((int)nbm[m], qw[m], snb);
                                }
                            }
                            const float dt = ad[arow[t] * (Kd / 32) + b];
                            ga[t] = fmaf(Xa * dt, (float)(sa_ - 2 * sn), ga[t]);
                            if (GATEUP)
                                ua[t] = fmaf(Xb * dt, (float)(sbm - 2 * snb), ua[t]);
                        }
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
