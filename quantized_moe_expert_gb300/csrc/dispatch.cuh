// Token-to-expert grouping: per-expert counts, their exclusive scan, the list
// of distinct experts, and a stable permutation of the (token, k) pairs into
// expert-grouped order (pairs of one expert keep ascending pair index), so the
// grouping is deterministic. Grouping the rows by distinct expert lets each
// chosen expert's weights be read once for all the rows that picked it, the
// batching the verify-batch expert kernel of "YoungAi - DeepSeek V4.1 Flash on
// one DGX Spark", section 4.4, is built on. The prefill path's weighted
// combine, which reads the grouped outputs back in token order, sits at the end.
#pragma once

#include "common.cuh"

namespace ds4 {

__global__ void dispatch_count_kernel(int32_t *__restrict__ idx, int npairs, int E, int32_t *__restrict__ counts,
                                      unsigned *__restrict__ status) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= npairs)
        return;
    int e = idx[p];
    if (e < 0 || e >= E) {
        atomicOr(status, kErrIndex);
        e = e < 0 ? 0 : E - 1;
        idx[p] = e;
    }
    atomicAdd(counts + e, 1);
}

// One block of 1024 threads; E <= 1024.
__global__ void dispatch_scan_kernel(const int32_t *__restrict__ counts, int E, int npairs,
                                     int32_t *__restrict__ offsets, int32_t *__restrict__ uexp,
                                     int32_t *__restrict__ uoff, int32_t *__restrict__ nuniq) {
    __shared__ int32_t sc[1024];
    __shared__ int32_t sf[1024];
    const int e = threadIdx.x;
    const int c = e < E ? counts[e] : 0;
    sc[e] = c;
    sf[e] = c > 0;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive Hillis-Steele scans
        int a = e >= o ? sc[e - o] : 0;
        int b = e >= o ? sf[e - o] : 0;
        __syncthreads();
        sc[e] += a;
        sf[e] += b;
        __syncthreads();
    }
    if (e < E) {
        offsets[e] = sc[e] - c;
        if (c > 0) {
            uexp[sf[e] - 1] = e;
            uoff[sf[e] - 1] = sc[e] - c;
        }
    }
    if (e == 0) {
        int n = sf[1023];
        *nuniq = n;
        uoff[n] = npairs;
        offsets[E] = npairs;
    }
}

// One block of 256 threads per expert: walk the pairs in order and give each
// pair routed to this expert its stable rank.
__global__ void dispatch_place_kernel(const int32_t *__restrict__ idx, int npairs, const int32_t *__restrict__ counts,
                                      const int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                                      int32_t *__restrict__ inv) {
    const int e = blockIdx.x;
    if (counts[e] == 0)
        return;
    __shared__ int32_t warp_tot[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int base = offsets[e];
    for (int p0 = 0; p0 < npairs; p0 += 256) {
        const int p = p0 + threadIdx.x;
        const bool hit = p < npairs && idx[p] == e;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
        if (lane == 0)
            warp_tot[warp] = __popc(m);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < 8; w++) {
            before += w < warp ? warp_tot[w] : 0;
            total += warp_tot[w];
        }
        if (hit) {
            const int pos = base + before + __popc(m & ((1u << lane) - 1u));
            perm[pos] = p;
            inv[p] = pos;
        }
        base += total;
        __syncthreads();
    }
}

// The prefill path's combine, after its grouped GEMMs.
// y[t][j] = sum_k w[t][k] * (g[e][j] * ye[inv[t*K+k]][j]) + ysh[t][j], e =
// idx[t*K+k], summed in k order and then the shared term, so the result does
// not depend on the schedule. g: [E][H] per-expert down gains, or nullptr (1).
__global__ void combine_kernel(const float *ye, const float *ysh,
                               const float *w, const int32_t *inv,
                               const int32_t *idx, const float *g, int T, int H, int K,
                               float *y) {
    pdl_launch_next();
    pdl_wait();
    const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = (int64_t)T * H / 4;
    if (i4 >= n4)
        return;
    const int t = (int)((i4 * 4) / H);
    const int j = (int)((i4 * 4) % H);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; k++) {
        const float wk = w[(int64_t)t * K + k];
        float4 v = *reinterpret_cast<const float4 *>(ye + (int64_t)inv[(int64_t)t * K + k] * H + j);
        if (g) {
            const float4 s = __ldg(reinterpret_cast<const float4 *>(g + (int64_t)idx[(int64_t)t * K + k] * H + j));
            v.x *= s.x;
            v.y *= s.y;
            v.z *= s.z;
            v.w *= s.w;
        }
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
