// Router: fp32 logits, sigmoid scores, exact top-k and renormalised weights.
//
// Scores are sigmoids of the logits; a per-expert bias, when present, is added
// to the selection score only ("YoungAi - DeepSeek V4.1 Flash on one DGX
// Spark", section 3: "selection score += delta-b", mixing weights untouched).
// The top-k is exact on the fp32 selection score with equal scores resolved
// towards the lower expert index, and the weights are the chosen sigmoid
// scores divided by their sum.
#pragma once

#include "common.cuh"
#include "frag_layout.cuh"
#include "tile_gemv.cuh"

namespace ds4 {

// x bf16 [T][H] -> x32 fp32 [T][H] and xsum [T][H/16]. One thread per
// 16-element sub-block: two 16-byte loads, four 16-byte stores, one sum.
__global__ void prep_x_kernel(const uint16_t *__restrict__ x, int T, int H, float *__restrict__ x32,
                              float *__restrict__ xsum) {
    const int64_t nsub = (int64_t)T * (H / 16);
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nsub)
        return;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + i * 16);
    uint4 a = src[0], b = src[1];
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
#pragma unroll
    for (int j = 0; j < 16; j++)
        s += v[j];
    float4 *dst = reinterpret_cast<float4 *>(x32 + i * 16);
#pragma unroll
    for (int j = 0; j < 4; j++)
        dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    xsum[i] = s;
}

// logits[t][e] = sum_h x32[t][h] * Wr[e][h]. One warp per (expert, tile of up
// to 8 tokens); each lane strides the row with 16-byte loads and keeps one
// partial per token, then the warp reduces.
constexpr int kRouterTok = 8;

__global__ void router_logits_kernel(const float *__restrict__ x32, int T, int H, const float *__restrict__ wr,
                                     int E, float *__restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + warp;
    const int t0 = blockIdx.y * kRouterTok;
    if (e >= E)
        return;
    const int nt = min(kRouterTok, T - t0);
    float acc[kRouterTok];
#pragma unroll
    for (int t = 0; t < kRouterTok; t++)
        acc[t] = 0.f;
    const float4 *row = reinterpret_cast<const float4 *>(wr + (int64_t)e * H);
    for (int c = lane; c < H / 4; c += 32) {
        float4 wv = __ldg(row + c);
#pragma unroll
        for (int t = 0; t < kRouterTok; t++) {
            if (t < nt) {
                float4 xv = __ldg(reinterpret_cast<const float4 *>(x32 + (int64_t)(t0 + t) * H) + c);
                acc[t] = fmaf(wv.x, xv.x, acc[t]);
                acc[t] = fmaf(wv.y, xv.y, acc[t]);
                acc[t] = fmaf(wv.z, xv.z, acc[t]);
                acc[t] = fmaf(wv.w, xv.w, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kRouterTok; t++) {
        float v = warp_sum(acc[t]);
        if (lane == 0 && t < nt)
            logits[(int64_t)(t0 + t) * E + e] = v;
    }
}

// Router logits for up to 64 tokens as column-slice partials on CUDA cores:
// part[s][t][e] = sum over the 256 columns k of slice s of x[t][k] Wr[e][k],
// plain fp32 FMAs in ascending k (the selection kernel adds the slices in
// order, so the logits do not depend on the schedule). Block (expert tile of
// 32, slice s): the slice's 32 router rows and TT token rows (bf16 -> fp32)
// in shared memory; thread (ex, tk) accumulates experts ex + 8 i, tokens
// tk + 16 j over 16-byte loads. With xq given, the blocks of expert tile 0
// also write the slice's tokens in the 2-bit GEMV's activation layout (x 4^-p,
// permuted) and their 16-column sums (bf16 hi + lo), as the batch path needs.
constexpr int kRtExperts = 32, kRtSlice = 256, kRtThreads = 128, kRtPitch = kRtSlice + 4;
constexpr int kRtMaxT = 64;

__host__ __device__ constexpr int router_tile_smem(int TT) { return (kRtExperts + TT) * kRtPitch * 4; }

template <int TT>
__global__ void __launch_bounds__(kRtThreads) router_tile_kernel(const uint16_t *x, int T, int H,
                                                                 const float *wr, int E,
                                                                 float *part, uint16_t *xq,
                                                                 uint16_t *xsums, unsigned *status) {
    pdl_launch_next();
    pdl_wait();
    extern __shared__ __align__(16) float rt_sm[];
    __shared__ alignas(8) uint64_t wbar;
    float *Ws = rt_sm;                          // [32][kRtPitch]
    float *Xs = rt_sm + kRtExperts * kRtPitch;  // [TT][kRtPitch]
    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kRtExperts, s = blockIdx.y, k0 = s * kRtSlice;
    const int nrows = min(kRtExperts, E - e0);
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&wbar));
    // the router rows' slice: one 1 KB bulk copy per row (warp 0), rows beyond E zeroed
    if (tid < 32) {
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"((unsigned)nrows * kRtSlice * 4u)
                         : "memory");
        }
        __syncwarp();
        if (tid < nrows)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    static_cast<uint32_t>(__cvta_generic_to_shared(Ws + tid * kRtPitch))),
                "l"(wr + (int64_t)(e0 + tid) * H + k0), "r"((unsigned)kRtSlice * 4u), "r"(bar)
                : "memory");
    }
    for (int f = nrows * (kRtSlice / 4) + tid; f < kRtExperts * (kRtSlice / 4); f += kRtThreads)
        *reinterpret_cast<float4 *>(Ws + (f / (kRtSlice / 4)) * kRtPitch + 4 * (f % (kRtSlice / 4))) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    // the token rows' slice, bf16 -> fp32 (every load of a thread in flight at once)
    constexpr int NX = TT * (kRtSlice / 8) / kRtThreads;
    uint4 xv[NX];
#pragma unroll
    for (int i = 0; i < NX; i++) {
        const int f = tid + i * kRtThreads, t = f / (kRtSlice / 8), c8 = f % (kRtSlice / 8);
        xv[i] = t < T ? reinterpret_cast<const uint4 *>(x + (int64_t)t * H + k0)[c8] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < NX; i++) {
        const int f = tid + i * kRtThreads, t = f / (kRtSlice / 8), c8 = f % (kRtSlice / 8);
        const uint4 v = xv[i];
        float *d = Xs + t * kRtPitch + 8 * c8;
        *reinterpret_cast<float4 *>(d) = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
        *reinterpret_cast<float4 *>(d + 4) =
            make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                        __uint_as_float(v.w & 0xFFFF0000u));
    }
    __syncthreads();
    {
        // bounded wait for the rows (1 s; on time-out the logits of this block are garbage and the
        // status word says so)
        uint64_t t0 = 0;
        for (unsigned it = 0;; it++) {
            uint32_t done;
            asm volatile("{\n\t.reg .pred p;\n\t"
                         "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(done)
                         : "r"(bar)
                         : "memory");
            if (done)
                break;
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (it == 0) {
                t0 = now;
            } else if (now - t0 > 1000000000ull) {
                if (tid == 0)
                    atomicOr(status, kErrTimeout);
                break;
            }
        }
    }
    if (xq && blockIdx.x == 0) {
        // one thread per (token, 16-column sub-block j) of this 256-column block s
        for (int f = tid; f < T * 16; f += kRtThreads) {
            const int t = f >> 4, j = f & 15, kappa = j >> 3;
            const float *v = Xs + t * kRtPitch + 16 * j;
            uint16_t *xt = xq + (int64_t)t * H;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 16; c++) {
                sum += v[c];
                const float sv = v[c] * (1.0f / (float)(1 << (2 * q2_p(c, kappa)))); // exact: power of two
                xt[q2_act_index(k0 + 16 * j + c)] = (uint16_t)f32_to_bf16_bits(sv);
            }
            const uint32_t hi = f32_to_bf16_bits(sum);
            const uint32_t lo = f32_to_bf16_bits(sum - __uint_as_float(hi << 16));
            uint16_t *st = xsums + (int64_t)t * (H / 8);
            st[q2_sum_index(s, j, 0)] = (uint16_t)hi;
            st[q2_sum_index(s, j, 1)] = (uint16_t)lo;
        }
    }
    constexpr int NJ = TT / 16;
    const int ex = tid & 7, tk = tid >> 3;
    float acc[4][NJ];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < NJ; j++)
            acc[i][j] = 0.f;
    for (int k = 0; k < kRtSlice; k += 4) {
        float4 w4[4], x4[NJ];
#pragma unroll
        for (int i = 0; i < 4; i++)
            w4[i] = *reinterpret_cast<const float4 *>(Ws + (ex + 8 * i) * kRtPitch + k);
#pragma unroll
        for (int j = 0; j < NJ; j++)
            x4[j] = *reinterpret_cast<const float4 *>(Xs + (tk + 16 * j) * kRtPitch + k);
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                acc[i][j] = fmaf(w4[i].x, x4[j].x, acc[i][j]);
                acc[i][j] = fmaf(w4[i].y, x4[j].y, acc[i][j]);
                acc[i][j] = fmaf(w4[i].z, x4[j].z, acc[i][j]);
                acc[i][j] = fmaf(w4[i].w, x4[j].w, acc[i][j]);
            }
    }
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int t = tk + 16 * j;
        if (t >= T)
            continue;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int e = e0 + ex + 8 * i;
            if (e < E)
                part[((int64_t)s * T + t) * E + e] = acc[i][j];
        }
    }
}

// One warp per token: selection scores into shared memory, then K+1 rounds of
// a warp-wide arg-max ordered by (score desc, index asc). Round K+1 only
// yields the runner-up score for the near-tie gap.
// Selection scores within this distance of the approximate (K+1)-th best are
// recomputed exactly before the decision when the logits came from the
// tensor-core GEMM (its fp32 accumulation order leaves scores up to ~5e-6 off
// a plain dot product; the margin is 4x that).
constexpr float kRefineMargin = 2e-5f;
constexpr int kSelectThreads = 128; // one block per token
constexpr int kSelectSmemPerExpert = 16;

// Warp-wide: the K (+1) best selection keys (sel_key) by K+1 rounds of a
// warp arg-max (larger key first, equal keys by lower index). Consumes keys
// (a chosen expert's key becomes 0). kth / next: the scores of the K-th and
// (K+1)-th choice (NaN for a NaN score).
__device__ __forceinline__ void select_rounds(unsigned *keys, const float *score, int E, int K,
                                              float (&chosen_s)[kMaxTopK], int (&chosen_e)[kMaxTopK], float &kth,
                                              float &next, int lane) {
    kth = 0.f;
    next = -INFINITY;
    const int rounds = K < E ? K + 1 : K;
    for (int r = 0; r < rounds; r++) {
        // every round has an untaken expert (K < E, or r < K = E), whose key is >= 1
        unsigned bk = 0u;
        int be = 0x7FFFFFFF;
        for (int e = lane; e < E; e += 32) { // ascending e: strict > keeps the lower index
            const unsigned k = keys[e];
            if (k > bk) {
                bk = k;
                be = e;
            }
        }
        const unsigned gk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int ge = (int)__reduce_min_sync(0xFFFFFFFFu, bk == gk ? (unsigned)be : 0xFFFFFFFFu);
        const float gv = sel_key_value(gk);
        if (r < K) {
            chosen_e[r] = ge;
            chosen_s[r] = score[ge];
            if (r == K - 1)
                kth = gv;
            if (lane == (ge & 31))
                keys[ge] = 0u;
            __syncwarp();
        } else {
            next = gv;
        }
    }
}

// One block of kSelectThreads per token; the logits are the sum of nsplit
// partial arrays split_stride floats apart. x_refine/wr/H: when x_refine is
// given, the logits are approximate and every expert whose selection score is
// within kRefineMargin of the (K+1)-th best gets its logit recomputed as an
// fp32 dot product of x (bf16) and its router row (the block's warps share
// the candidates) before the final decision.
// Shared memory: 2 * E floats + 2 * E ints (kSelectSmemPerExpert bytes per expert).
__global__ void router_select_kernel(const float *logits, const float *bias, int T,
                                     int E, int K, int32_t *idx, float *w,
                                     float *gap, float *sel_out,
                                     const uint16_t *x_refine, const float *wr, int H,
                                     int nsplit, int64_t split_stride) {
    pdl_launch_next();
    pdl_wait();
    extern __shared__ float smem[];
    __shared__ int ncand;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    if (t >= T)
        return;
    float *sel = smem;
    float *score = sel + E;
    int *cand = reinterpret_cast<int *>(score + E);
    unsigned *keys = reinterpret_cast<unsigned *>(cand + E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const float *lp = logits + (int64_t)t * E + e;
        float l = lp[0];
        // partial logits of a K split, added in order (eight loads in flight at a time)
        int q = 1;
        for (; q + 8 <= nsplit; q += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; i++)
                v[i] = lp[(q + i) * split_stride];
#pragma unroll
            for (int i = 0; i < 8; i++)
                l += v[i];
        }
        for (; q < nsplit; q++)
            l += lp[q * split_stride];
        float s = sigmoid(l);
        score[e] = s;
        sel[e] = bias ? s + bias[e] : s;
        keys[e] = sel_key(sel[e]);
    }
    __syncthreads();
    float chosen_s[kMaxTopK];
    int chosen_e[kMaxTopK];
    float kth, next;
    if (x_refine) {
        if (warp == 0) {
            select_rounds(keys, score, E, K, chosen_s, chosen_e, kth, next, lane);
            const float thr = (K < E ? next : kth) - kRefineMargin; // NaN: no candidate
            int n = 0;
            for (int e0 = 0; e0 < E; e0 += 32) {
                const int e = e0 + lane;
                const float v = e < E ? sel[e] : -INFINITY;
                const unsigned m = __ballot_sync(0xFFFFFFFFu, v >= thr);
                if (v >= thr)
                    cand[n + __popc(m & ((1u << lane) - 1u))] = e;
                n += __popc(m);
            }
            if (lane == 0)
                ncand = n;
        }
        __syncthreads();
        const uint2 *xr = reinterpret_cast<const uint2 *>(x_refine + (int64_t)t * H);
        for (int c = warp; c < ncand; c += blockDim.x / 32) {
            const int e = cand[c];
            const float4 *row = reinterpret_cast<const float4 *>(wr + (int64_t)e * H);
            float acc = 0.f;
            for (int q = lane; q < H / 4; q += 32) {
                const float4 v = __ldg(row + q);
                const uint2 xb = __ldg(xr + q);
                acc = fmaf(__uint_as_float(xb.x << 16), v.x, acc);
                acc = fmaf(__uint_as_float(xb.x & 0xFFFF0000u), v.y, acc);
                acc = fmaf(__uint_as_float(xb.y << 16), v.z, acc);
                acc = fmaf(__uint_as_float(xb.y & 0xFFFF0000u), v.w, acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) {
                const float s = sigmoid(acc);
                score[e] = s;
                sel[e] = bias ? s + bias[e] : s;
            }
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sel_out)
            sel_out[(int64_t)t * E + e] = sel[e];
        keys[e] = sel_key(sel[e]);
    }
    __syncthreads();
    if (warp != 0)
        return;
    select_rounds(keys, score, E, K, chosen_s, chosen_e, kth, next, lane);
    if (lane == 0) {
        float total = 0.f;
        for (int k = 0; k < K; k++)
            total += chosen_s[k];
        for (int k = 0; k < K; k++) {
            idx[(int64_t)t * K + k] = chosen_e[k];
            w[(int64_t)t * K + k] = total > 0.f ? chosen_s[k] / total : 1.0f / K;
        }
        if (gap)
            gap[t] = K < E ? kth - next : INFINITY;
    }
}

} // namespace ds4
