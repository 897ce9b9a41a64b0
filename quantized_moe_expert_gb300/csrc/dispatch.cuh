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

// The grouping in one block of 1024 threads for any number of pairs P (E <= 1024):
// warp w owns the w-th of 32 contiguous chunks of the pairs.
//   0. with stage_idx, the block first copies idx into shared memory (every
//      thread's loads in flight at once), so the two walks below do not wait
//      on a global load per step;
//   1. each warp counts its chunk's pairs per expert in its own row of a
//      shared-memory histogram [32][E] (dynamic shared memory: 128 E bytes,
//      then 4 P bytes of staged indices);
//   2. per expert: the total over the rows, the exclusive scan over experts
//      (offsets), the distinct experts, and per row the first grouped position
//      of that warp's pairs of the expert (the expert's offset plus the counts
//      of the lower rows), written over the histogram;
//   3. each warp walks its chunk again, 32 pairs at a time in pair order: the
//      lanes of one expert (match_any) take consecutive positions in lane
//      order from the warp's cursor, which the lowest of them then advances.
// Pairs of one expert keep ascending pair index (chunks, steps and lanes in
// order). Out-of-range indices are clamped and reported (kErrIndex).
__global__ void __launch_bounds__(1024) group_kernel(int32_t *idx, int P, int E, bool stage_idx, int32_t *counts,
                                                     int32_t *offsets, int32_t *uexp, int32_t *uoff, int32_t *nuniq,
                                                     int32_t *perm, int32_t *inv, unsigned *status) {
    pdl_launch_next();
    pdl_wait();
    extern __shared__ int32_t hist[]; // [32][E], then (stage_idx) the P indices
    __shared__ int32_t sc[1024], sf[1024];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += 1024)
        hist[i] = 0;
    int32_t *ix = idx; // where the walks read the (clamped) indices
    if (stage_idx) {
        ix = hist + 32 * E;
        for (int p = tid; p < P; p += 1024) {
            int e = idx[p];
            if (e < 0 || e >= E) {
                atomicOr(status, kErrIndex);
                e = e < 0 ? 0 : E - 1;
                idx[p] = e;
            }
            ix[p] = e;
        }
    }
    __syncthreads();
    const int chunk = (P + 31) / 32;
    const int p_begin = min(P, warp * chunk), p_end = min(P, p_begin + chunk);
    int32_t *row = hist + warp * E;
    for (int p = p_begin + lane; p < p_end; p += 32) {
        int e = ix[p];
        if (e < 0 || e >= E) { // unstaged indices only: the staging clamped its copies
            atomicOr(status, kErrIndex);
            e = e < 0 ? 0 : E - 1;
            idx[p] = e;
        }
        atomicAdd(row + e, 1);
    }
    __syncthreads();
    int c = 0;
    if (tid < E)
        for (int w = 0; w < 32; w++)
            c += hist[w * E + tid];
    sc[tid] = c;
    sf[tid] = c > 0;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive Hillis-Steele scans
        const int a = tid >= o ? sc[tid - o] : 0;
        const int b = tid >= o ? sf[tid - o] : 0;
        __syncthreads();
        sc[tid] += a;
        sf[tid] += b;
        __syncthreads();
    }
    const int nu = sf[1023];
    if (tid < E) {
        const int off = sc[tid] - c;
        counts[tid] = c;
        offsets[tid] = off;
        if (c > 0) {
            uexp[sf[tid] - 1] = tid;
            uoff[sf[tid] - 1] = off;
        }
        int run = off;
        for (int w = 0; w < 32; w++) {
            const int n = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += n;
        }
    }
    if (tid == 0) {
        *nuniq = nu;
        uoff[nu] = P;
        offsets[E] = P;
    }
    __syncthreads();
    for (int p0 = p_begin; p0 < p_end; p0 += 32) { // warp-uniform bounds
        const int p = p0 + lane;
        const int e = p < p_end ? ix[p] : -1; // clamped in step 0 or 1 (by this lane, unstaged)
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        const int leader = __ffs(m) - 1;
        const int base = __shfl_sync(0xFFFFFFFFu, e >= 0 && lane == leader ? row[e] : 0, leader);
        if (e >= 0) {
            const int pos = base + __popc(m & ((1u << lane) - 1u));
            perm[pos] = p;
            inv[p] = pos;
        }
        __syncwarp();
        if (e >= 0 && lane == leader)
            row[e] = base + __popc(m);
        __syncwarp();
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
    // every pair's row loaded first (up to kMaxTopK loads in flight), then summed in k order
    float wk[kMaxTopK];
    float4 v[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; k++) {
        if (k < K) {
            wk[k] = w[(int64_t)t * K + k];
            v[k] = *reinterpret_cast<const float4 *>(ye + (int64_t)inv[(int64_t)t * K + k] * H + j);
        }
    }
    if (g) {
#pragma unroll
        for (int k = 0; k < kMaxTopK; k++) {
            if (k < K) {
                const float4 s =
                    __ldg(reinterpret_cast<const float4 *>(g + (int64_t)idx[(int64_t)t * K + k] * H + j));
                v[k].x *= s.x;
                v[k].y *= s.y;
                v[k].z *= s.z;
                v[k].w *= s.w;
            }
        }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kMaxTopK; k++) {
        if (k < K) {
            acc.x = fmaf(wk[k], v[k].x, acc.x);
            acc.y = fmaf(wk[k], v[k].y, acc.y);
            acc.z = fmaf(wk[k], v[k].z, acc.z);
            acc.w = fmaf(wk[k], v[k].w, acc.w);
        }
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
