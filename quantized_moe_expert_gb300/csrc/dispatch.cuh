// Token-to-expert grouping: per-expert counts, their exclusive scan, the list
// of distinct experts, and a stable permutation of the (token, k) pairs into
// expert-grouped order (pairs of one expert keep ascending pair index), so the
// grouping is deterministic. The batched-union idea - one dispatch per distinct
// expert for all rows that chose it - is the verify-batch expert kernel of
// "YoungAi - DeepSeek V4.1 Flash on one DGX Spark", section 4.4 ("a persistent
// expert kernel over (unique expert x rows) that reads each chosen expert's
// bits once").
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

} // namespace ds4
