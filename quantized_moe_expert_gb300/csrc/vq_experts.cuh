// VQ routed experts: every 8 consecutive weights of a row are one codeword of
// a per-layer codebook times one gain per row, w[r, 8j .. 8j+7] = g_r *
// C[idx[r, j]] ("YoungAi - DeepSeek V4.1 Flash on one DGX Spark", section
// 4.1). The codebook holds 2^12 or 2^13 codewords of 8 FP8 E4M3 values and is
// shared by all experts and the three matrices; indices are 12-bit fields,
// least significant bit first, the rows of one expert matrix back to back;
// 13-bit layers add a bit plane holding bit 12 of every index. Gains are
// binary16. Activations are used as they are (bf16 x, fp32 SwiGLU rows).
//
// Kernel: persistent over (distinct expert, 8 rows); the CTA loads the
// codebook into shared memory once. A warp owns a row; lane l takes groups of
// 8 indices (96 bits = 3 aligned words, 64 weights), decodes the codewords
// with the hardware E4M3 -> f16x2 conversion, and multiplies them with up to
// NT activation rows in fp32; the row gain scales the sum once.
#pragma once

#include "common.cuh"

namespace ds4 {

// Two E4M3 values (low byte first) -> two floats, by the hardware conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    uint32_t h2;
    asm("{ .reg .b16 t;\n\t"
        "cvt.u16.u32 t, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, t; }"
        : "=r"(h2)
        : "r"(two));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// The index stream of one matrix (all experts) -> the prefill GEMM's tile
// records (VqTile). One thread per (row of all experts, 256-column block):
// 48 bytes of indices and, for 13-bit layers, 4 bytes of bit plane.
__global__ void repack_vq_tile_kernel(const uint32_t *__restrict__ stream, const uint8_t *__restrict__ plane,
                                      int64_t rows, int k, uint8_t *__restrict__ rec) {
    const int nkb = k / 256;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * nkb)
        return;
    const int64_t grow = i / nkb;
    const int kb = (int)(i % nkb);
    const int64_t g0 = grow * (k / 8) + 32 * kb; // first index of the piece (in the whole matrix's stream)
    const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(stream) + g0 * 3 / 2);
    uint8_t *dst = rec + ((grow >> 7) * nkb + kb) * kVqTileRec;
    const int r = (int)(grow & 127);
#pragma unroll
    for (int c = 0; c < 3; c++)
        reinterpret_cast<uint4 *>(dst)[c * 128 + r] = src[c];
    reinterpret_cast<uint32_t *>(dst + 3 * 128 * 16)[r] =
        plane ? *reinterpret_cast<const uint32_t *>(plane + g0 / 8) : 0u;
}

// A bf16 pair -> the binary16 pair, round to nearest, magnitudes beyond the
// largest finite binary16 saturating to it.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(v & 0xFFFF0000u)), "f"(__uint_as_float(v << 16)));
    return r;
}

// bf16 -> binary16 (bf16x2_to_f16x2_sat; x for the VQ tensor-core form and for
// the shared expert's tensor-core GEMMs). A thread per 8 values: n is a
// multiple of 8 and both arrays 16-byte aligned.
__global__ void bf16_to_f16_kernel(const uint16_t *x, int64_t n, uint16_t *out) {
    pdl_launch_next();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n / 8) {
        const uint4 v = reinterpret_cast<const uint4 *>(x)[i];
        reinterpret_cast<uint4 *>(out)[i] = make_uint4(bf16x2_to_f16x2_sat(v.x), bf16x2_to_f16x2_sat(v.y),
                                                       bf16x2_to_f16x2_sat(v.z), bf16x2_to_f16x2_sat(v.w));
    }
}

// B rows of the VQ tensor-core form's routed gate/up in expert-grouped order,
// as binary16: xp[pos] = bf16x2_to_f16x2_sat(x[perm[pos] / K]); one CTA per row,
// 8 values per thread (H a multiple of 8, both arrays 16-byte aligned).
__global__ void gather_rows_f16_kernel(const uint16_t *x, const int32_t *perm, int K, int H, uint16_t *xp) {
    pdl_launch_next();
    pdl_wait();
    const int pos = blockIdx.x;
    const int t = perm[pos] / K;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H);
    uint4 *dst = reinterpret_cast<uint4 *>(xp + (int64_t)pos * H);
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
        const uint4 v = src[c];
        dst[c] = make_uint4(bf16x2_to_f16x2_sat(v.x), bf16x2_to_f16x2_sat(v.y), bf16x2_to_f16x2_sat(v.z),
                            bf16x2_to_f16x2_sat(v.w));
    }
}

// bf16 rows -> fp32 (exact). A thread per 8 values: n is a multiple of 8 and
// both arrays 16-byte aligned.
__global__ void widen_bf16_kernel(const uint16_t *x, int64_t n, float *out) {
    pdl_launch_next();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n / 8) {
        const uint4 v = reinterpret_cast<const uint4 *>(x)[i];
        float4 *o = reinterpret_cast<float4 *>(out) + 2 * i;
        o[0] = make_float4(bf16_to_f32(v.x & 0xFFFFu), bf16_to_f32(v.x >> 16), bf16_to_f32(v.y & 0xFFFFu),
                           bf16_to_f32(v.y >> 16));
        o[1] = make_float4(bf16_to_f32(v.z & 0xFFFFu), bf16_to_f32(v.z >> 16), bf16_to_f32(v.w & 0xFFFFu),
                           bf16_to_f32(v.w >> 16));
    }
}

// out[pos][r] for the expert-grouped rows pos of each distinct expert and r in
// its M rows: the VQ product of A (or SwiGLU of gate A and up B when GATEUP)
// with activation rows act[row_of(pos)][0..Kd). GATEUP: act rows are tokens
// perm[pos] / K; else grouped positions. The launch's dynamic shared memory
// holds the codebook (entries << 3 bytes).
template <bool GATEUP, int NT>
__global__ void __launch_bounds__(256) vq_product_kernel(VqMat A, VqMat B, const uint8_t *codebook,
                                                         int entries, const float *act,
                                                         const int32_t *uexp,
                                                         const int32_t *uoff,
                                                         const int32_t *nuniq,
                                                         const int32_t *perm, int K, int M, int Kd,
                                                         int ubound, float *out) {
    extern __shared__ __align__(16) uint8_t cb_smem[];
    pdl_launch_next();
    { // the codebook is the layer's own: loaded while the predecessor in the stream finishes
        const uint4 *src = reinterpret_cast<const uint4 *>(codebook);
        uint4 *dst = reinterpret_cast<uint4 *>(cb_smem);
        for (int i = threadIdx.x; i < entries / 2; i += blockDim.x)
            dst[i] = __ldg(src + i);
    }
    pdl_wait();
    __syncthreads();
    const uint2 *cb = reinterpret_cast<const uint2 *>(cb_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nu = *nuniq;
    const int groups = (M + 7) / 8;
    const int ngrp = Kd / 64; // 8-index groups per row
    const int64_t row_words = (int64_t)Kd * 3 / 64;
    for (int w = blockIdx.x; w < ubound * groups; w += gridDim.x) {
        const int u = w / groups;
        if (u >= nu)
            break; // work items are ordered by distinct expert
        const int r = (w - u * groups) * 8 + warp;
        if (r >= M)
            continue;
        const int e = uexp[u];
        const int p0 = uoff[u], p1 = uoff[u + 1];
        const int64_t er = (int64_t)e * M + r; // row within the whole matrix
        const uint32_t *sa = A.stream + er * row_words;
        const uint32_t *sb = B.stream + er * row_words;
        const uint8_t *pa = A.plane ? A.plane + er * (Kd / 64) : nullptr;
        const uint8_t *pb = B.plane ? B.plane + er * (Kd / 64) : nullptr;
        const float ga_row = __half2float(__ushort_as_half(__ldg(A.gain + er)));
        const float gb_row = GATEUP ? __half2float(__ushort_as_half(__ldg(B.gain + er))) : 0.f;
        for (int c0 = p0; c0 < p1; c0 += NT) {
            const int n = p1 - c0 < NT ? p1 - c0 : NT;
            const float *arow[NT];
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const int pos = c0 + (t < n ? t : 0);
                const int64_t ar = GATEUP ? perm[pos] / K : pos;
                arow[t] = act + ar * Kd;
            }
            float acc_a[NT], acc_b[NT];
#pragma unroll
            for (int t = 0; t < NT; t++)
                acc_a[t] = acc_b[t] = 0.f;
            for (int g = lane; g < ngrp; g += 32) {
                uint32_t wa[4], wb[4];
#pragma unroll
                for (int q = 0; q < 3; q++) {
                    wa[q] = __ldg(sa + 3 * g + q);
                    wb[q] = GATEUP ? __ldg(sb + 3 * g + q) : 0u;
                }
                wa[3] = wb[3] = 0u;
                const unsigned hia = pa ? __ldg(pa + g) : 0u;
                const unsigned hib = (GATEUP && pb) ? __ldg(pb + g) : 0u;
#pragma unroll
                for (int i = 0; i < 8; i++) { // index i of the group: bits 12i .. 12i+11
                    const int word = (12 * i) >> 5, off = (12 * i) & 31;
                    const unsigned ia = (__funnelshift_r(wa[word], wa[word + 1], off) & 0xFFFu) |
                                        (((hia >> i) & 1u) << 12);
                    const uint2 ca = cb[ia];
                    float va[8], vb[8];
                    {
                        const float2 v0 = e4m3x2_to_float2(ca.x), v1 = e4m3x2_to_float2(ca.x >> 16);
                        const float2 v2 = e4m3x2_to_float2(ca.y), v3 = e4m3x2_to_float2(ca.y >> 16);
                        va[0] = v0.x, va[1] = v0.y, va[2] = v1.x, va[3] = v1.y;
                        va[4] = v2.x, va[5] = v2.y, va[6] = v3.x, va[7] = v3.y;
                    }
                    if (GATEUP) {
                        const unsigned ib = (__funnelshift_r(wb[word], wb[word + 1], off) & 0xFFFu) |
                                            (((hib >> i) & 1u) << 12);
                        const uint2 cbv = cb[ib];
                        const float2 v0 = e4m3x2_to_float2(cbv.x), v1 = e4m3x2_to_float2(cbv.x >> 16);
                        const float2 v2 = e4m3x2_to_float2(cbv.y), v3 = e4m3x2_to_float2(cbv.y >> 16);
                        vb[0] = v0.x, vb[1] = v0.y, vb[2] = v1.x, vb[3] = v1.y;
                        vb[4] = v2.x, vb[5] = v2.y, vb[6] = v3.x, vb[7] = v3.y;
                    }
                    const int col = 64 * g + 8 * i;
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        if (t < n) {
                            const float4 x0 = *reinterpret_cast<const float4 *>(arow[t] + col);
                            const float4 x1 = *reinterpret_cast<const float4 *>(arow[t] + col + 4);
                            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int m = 0; m < 8; m++) {
                                acc_a[t] = fmaf(va[m], xv[m], acc_a[t]);
                                if (GATEUP)
                                    acc_b[t] = fmaf(vb[m], xv[m], acc_b[t]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const float a = ga_row * warp_sum(acc_a[t]);
                const float b = GATEUP ? gb_row * warp_sum(acc_b[t]) : 0.f;
                if (lane == 0 && t < n)
                    out[(int64_t)(c0 + t) * M + r] = GATEUP ? silu(a) * b : a;
            }
        }
    }
}

} // namespace ds4
