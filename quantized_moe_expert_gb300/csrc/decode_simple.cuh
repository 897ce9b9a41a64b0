// Warp-per-row dequant-GEMV kernels: the plain reference schedule of the
// expert stage. Every 2-bit weight is expanded on the fly from the block
// fields, w = d * sc * q - dmin * m, using the sub-block factorisation
//   sum_i w_i x_i = d * sc * sum_i q_i x_i - dmin * m * sum_i x_i
// over each 16-weight sub-block; accumulation is fp32.
#pragma once

#include "common.cuh"

namespace ds4 {

// Dot of 2-bit row `row` of m with the fp32 vector x (K = m.nb * 256 entries).
// xs: per-16 sums of x, or nullptr to form them on the fly. Warp-collective;
// every lane returns the full sum. Lane l handles 64-column chunks l, l+32, ...
__device__ __forceinline__ float dot_q2_row(const Q2Mat &m, int64_t row, const float *__restrict__ x,
                                            const float *__restrict__ xs, int lane) {
    const int nb = m.nb;
    const uint8_t *qs = m.qs + row * nb * 64;
    const uint8_t *sc = m.sc + row * nb * 16;
    const uint32_t *dm = m.dm + row * nb;
    float acc = 0.f;
    for (int c = lane; c < nb * 4; c += 32) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(qs) + c);
        const uint32_t scw = __ldg(reinterpret_cast<const uint32_t *>(sc) + c);
        const uint32_t dmw = __ldg(dm + (c >> 2));
        const float d = f16_to_f32(dmw), dmin = f16_to_f32(dmw >> 16);
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int s = 0; s < 4; s++) {
            const int col0 = c * 64 + s * 16;
            const float4 *xv = reinterpret_cast<const float4 *>(x + col0);
            float xx[16];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float4 v = __ldg(xv + j);
                xx[4 * j] = v.x;
                xx[4 * j + 1] = v.y;
                xx[4 * j + 2] = v.z;
                xx[4 * j + 3] = v.w;
            }
            float sqx = 0.f, sx = 0.f;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                sqx = fmaf((float)((words[s] >> (2 * i)) & 3u), xx[i], sqx);
                sx += xx[i];
            }
            if (xs)
                sx = __ldg(xs + (col0 >> 4));
            const uint32_t b = (scw >> (8 * s)) & 0xFFu;
            acc += d * (float)(b & 15u) * sqx - dmin * (float)(b >> 4) * sx;
        }
    }
    return warp_sum(acc);
}

// Dot of 8-bit row `row` with x (K = m.k). Lane l handles 16-column chunks.
__device__ __forceinline__ float dot_q8_row(const Q8Mat &m, int64_t row, const float *__restrict__ x, int lane) {
    const int K = m.k;
    const int8_t *qs = m.qs + row * K;
    const uint16_t *d = m.d + row * (K / 32);
    float acc = 0.f;
    for (int c = lane; c < K / 16; c += 32) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(qs) + c);
        const float dd = f16_to_f32(__ldg(d + (c >> 1)));
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
        const float4 *xv = reinterpret_cast<const float4 *>(x + c * 16);
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float4 v = __ldg(xv + j);
            const uint32_t wd = words[j];
            part = fmaf((float)(int8_t)(wd & 0xFF), v.x, part);
            part = fmaf((float)(int8_t)((wd >> 8) & 0xFF), v.y, part);
            part = fmaf((float)(int8_t)((wd >> 16) & 0xFF), v.z, part);
            part = fmaf((float)(int8_t)(wd >> 24), v.w, part);
        }
        acc = fmaf(dd, part, acc);
    }
    return warp_sum(acc);
}

constexpr int kRowsPerCta = 8; // one warp per row

// h[pos][i] = silu(gate_e[i] . x_t) * (up_e[i] . x_t) for every pair position
// pos of distinct expert `slot` (grid.y), rows i of grid.x.
__global__ void simple_gateup_q2_kernel(LayerDev L, Scratch S) {
    const int slot = blockIdx.y;
    if (slot >= *S.nuniq)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kRowsPerCta + warp;
    if (i >= L.I)
        return;
    const int e = S.uexp[slot];
    const int64_t row = (int64_t)e * L.I + i;
    for (int pos = S.uoff[slot]; pos < S.uoff[slot + 1]; pos++) {
        const int t = S.perm[pos] / L.K;
        const float *x = S.x32 + (int64_t)t * L.H;
        const float *xs = S.xsum + (int64_t)t * (L.H / 16);
        const float g = dot_q2_row(L.gate, row, x, xs, lane);
        const float u = dot_q2_row(L.up, row, x, xs, lane);
        if (lane == 0)
            S.h[(int64_t)pos * L.I + i] = silu(g) * u;
    }
}

// ye[pos][j] = down_e[j] . h[pos]
__global__ void simple_down_q2_kernel(LayerDev L, Scratch S) {
    const int slot = blockIdx.y;
    if (slot >= *S.nuniq)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * kRowsPerCta + warp;
    if (j >= L.H)
        return;
    const int e = S.uexp[slot];
    const int64_t row = (int64_t)e * L.H + j;
    for (int pos = S.uoff[slot]; pos < S.uoff[slot + 1]; pos++) {
        const float v = dot_q2_row(L.down, row, S.h + (int64_t)pos * L.I, nullptr, lane);
        if (lane == 0)
            S.ye[(int64_t)pos * L.H + j] = v;
    }
}

// Shared expert, every token: hsh[t][i], then ysh[t][j].
__global__ void simple_gateup_q8_kernel(LayerDev L, Scratch S, int T) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kRowsPerCta + warp;
    if (i >= L.Ish)
        return;
    for (int t = 0; t < T; t++) {
        const float *x = S.x32 + (int64_t)t * L.H;
        const float g = dot_q8_row(L.sh_gate, i, x, lane);
        const float u = dot_q8_row(L.sh_up, i, x, lane);
        if (lane == 0)
            S.hsh[(int64_t)t * L.Ish + i] = silu(g) * u;
    }
}

__global__ void simple_down_q8_kernel(LayerDev L, Scratch S, int T) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * kRowsPerCta + warp;
    if (j >= L.H)
        return;
    for (int t = 0; t < T; t++) {
        const float v = dot_q8_row(L.sh_down, j, S.hsh + (int64_t)t * L.Ish, lane);
        if (lane == 0)
            S.ysh[(int64_t)t * L.H + j] = v;
    }
}

// y[t][j] = sum_k w[t][k] * ye[inv[t*K+k]][j] + ysh[t][j], summed in k order
// and then the shared term, so the result does not depend on the schedule.
__global__ void combine_kernel(const float *__restrict__ ye, const float *__restrict__ ysh,
                               const float *__restrict__ w, const int32_t *__restrict__ inv, int T, int H, int K,
                               float *__restrict__ y) {
    const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = (int64_t)T * H / 4;
    if (i4 >= n4)
        return;
    const int t = (int)((i4 * 4) / H);
    const int j = (int)((i4 * 4) % H);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; k++) {
        const float wk = w[(int64_t)t * K + k];
        const float4 v = *reinterpret_cast<const float4 *>(ye + (int64_t)inv[(int64_t)t * K + k] * H + j);
        acc.x = fmaf(wk, v.x, acc.x);
        acc.y = fmaf(wk, v.y, acc.y);
        acc.z = fmaf(wk, v.z, acc.z);
        acc.w = fmaf(wk, v.w, acc.w);
    }
    if (ysh) {
        const float4 s = *reinterpret_cast<const float4 *>(ysh + (int64_t)t * H + j);
        acc.x += s.x;
        acc.y += s.y;
        acc.z += s.z;
        acc.w += s.w;
    }
    *reinterpret_cast<float4 *>(y + (int64_t)t * H + j) = acc;
}

} // namespace ds4
