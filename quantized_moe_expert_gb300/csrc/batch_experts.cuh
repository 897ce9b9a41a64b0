// Batch path for 2-bit layers, up to 64 tokens per call: the expert products
// run as persistent kernels (one CTA per SM) over items (slot, row tile). For
// the routed experts a slot is a distinct expert with up to kBatchCols of its
// (token, k) pairs, i.e. the 8 columns of one mma.sync; for the shared expert
// a group of up to 8 tokens. Each CTA takes a contiguous range of items, keeps
// a ring of stages of tile records in flight (bulk copies; an 8-bit item spans
// several stages, each a range of columns) and holds the activation rows of its
// current slot; per stage the 16 warps run the tile GEMVs of tile_gemv.cuh
// (exact products, fp32 accumulation, the decode path's arithmetic) and after
// an item's last stage the CTA writes its results. Every routed expert's
// weights are read once for all the rows that chose it (an expert with more
// than kBatchCols pairs once per group of them): the batching of the
// verify-batch expert kernel of "YoungAi - DeepSeek V4.1 Flash on one DGX
// Spark", section 4.4. No CTA waits on another; every wait on a copy is bounded.
#pragma once

#include "common.cuh"
#include "frag_layout.cuh"
#include "tile_gemv.cuh"

namespace ds4 {

constexpr int kBatchCols = 8;  // pairs per virtual slot: the MMA's columns
constexpr int kBatchMaxT = 64; // tokens per call of the batch path
// Warp roles of a batch CTA: 16 compute warps, a producer warp (its lane 0
// issues every copy), 2 epilogue warps; they meet only at mbarriers. 19 warps
// leave 96 registers a thread (at most 5 warps on each of the 4 schedulers).
constexpr int kBatchComputeWarps = 16;
constexpr int kBatchProducerWarp = kBatchComputeWarps;
constexpr int kBatchEpiWarps = 2;
constexpr int kBatchEpiThreads = 32 * kBatchEpiWarps;
constexpr int kBatchThreads = 32 * (kBatchComputeWarps + 1 + kBatchEpiWarps);
constexpr int kPartPitch = 20; // floats per (warp, matrix, column) run of 16 row sums: 20 avoids bank conflicts
constexpr uint64_t kBatchWaitNs = 1000000000ull; // 1 s: far beyond any legitimate wait
constexpr int kBatchStageCap = 48 << 10; // most bytes of one 8-bit stage
// Relative cost of a routed and a shared item (a 16-row tile pair over all
// columns, or four 16-row tiles), for splitting the items over the CTAs.
constexpr int kBatchCostRouted = 2, kBatchCostShared = 3;
// Up to this many tokens one launch per product runs both kinds of items.
constexpr int kBatchMergeMaxT = 4;

// Each product kernel (gate/up, down) runs two kinds of items: first the
// routed experts' (2-bit; a slot is a distinct expert with up to kBatchCols
// of its pairs), then the shared expert's (8-bit; a slot is a group of up to
// kBatchCols tokens).
enum BatchKind : int { kRouted = 0, kShared = 1 };
// Which kinds a product kernel runs (KINDS): bit 0 routed, bit 1 shared.
constexpr int kBatchRouted = 1, kBatchShared = 2, kBatchBoth = 3;

struct BatchArgs {
    int H, I, K, Ish, T;
    Q2Frag gate, up, down;
    Q8Frag sh_gate, sh_up, sh_down;
    const uint16_t *x;       // [T][H] bf16 token rows
    const uint16_t *xq;      // [T][H] bf16 x * 4^-p in the permuted layout
    const uint16_t *xsums;   // [T][H/8] the 16-column sums of x, bf16 hi and lo
    uint16_t *hq_hi, *hq_lo; // [P][I] SwiGLU rows as a bf16 hi + lo pair, permuted, by grouped position
    uint16_t *hsums;         // [P][I/8]
    float *ye;               // [P][H] routed expert outputs by grouped position
    uint16_t *hs_hi, *hs_lo; // [T][Ish] shared SwiGLU rows as a binary16 hi + lo pair
    float *ysh;              // [T][H] shared expert output
    const int4 *vslot;       // {expert, first grouped position, pairs, 0}
    const int32_t *nvslot;
    const int32_t *perm;     // grouped position -> pair t * K + k
    int nstage;              // stages in each CTA's ring
    int chunk;               // columns per stage of the 8-bit products
    int skip_signal;         // test hook: CTA 0's producer issues nothing for its first stage, so that
                             // stage's bounded waits run out (kErrTimeout) and every role stops
    unsigned *status;
};

// x bf16 [T][H] -> the 2-bit GEMV's activation layout (x 4^-p, permuted) and
// the 16-column sums (bf16 hi + lo), for calls whose router did not write them.
// One thread per 16-column sub-block.
__global__ void batch_prep_x_kernel(const uint16_t *x, int T, int H, uint16_t *xq,
                                    uint16_t *xsums) {
    pdl_launch_next();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int nsub = H / 16;
    if (i >= (int64_t)T * nsub)
        return;
    const int t = (int)(i / nsub), j = (int)(i % nsub);
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H + 16 * j);
    const uint4 p0 = src[0], p1 = src[1];
    const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const int kappa = (j & 15) >> 3;
    uint16_t *xt = xq + (int64_t)t * H;
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 16; c++) {
        const float v = __uint_as_float(c & 1 ? wv[c >> 1] & 0xFFFF0000u : wv[c >> 1] << 16);
        sum += v;
        const float sv = v * (1.0f / (float)(1 << (2 * q2_p(c, kappa)))); // exact: power of two
        xt[q2_act_index(16 * j + c)] = (uint16_t)f32_to_bf16_bits(sv);
    }
    const uint32_t hi = f32_to_bf16_bits(sum);
    const uint32_t lo = f32_to_bf16_bits(sum - __uint_as_float(hi << 16));
    uint16_t *st = xsums + (int64_t)t * (H / 8);
    st[q2_sum_index(j >> 4, j & 15, 0)] = (uint16_t)hi;
    st[q2_sum_index(j >> 4, j & 15, 1)] = (uint16_t)lo;
}

// The grouping of the batch path in one block of 1024 threads (at most 1024
// pairs, E <= 1024): per-expert counts, their exclusive scan, the distinct
// experts, the stable expert-grouped order of the pairs (perm, and inv its
// inverse: pairs of one expert keep ascending pair index) and the virtual
// slots (distinct expert u with n pairs gives ceil(n / kBatchCols) slots of
// consecutive grouped positions). Out-of-range indices are clamped and
// reported (kErrIndex). The same results as group_kernel, the grouping of
// larger calls.
__global__ void __launch_bounds__(1024) batch_group_kernel(int32_t *idx, int P, int E,
                                                           int32_t *counts, int32_t *offsets,
                                                           int32_t *uexp, int32_t *uoff,
                                                           int32_t *nuniq, int32_t *perm,
                                                           int32_t *inv, int4 *vslot,
                                                           int32_t *nvslot, unsigned *status) {
    pdl_launch_next();
    pdl_wait();
    __shared__ int32_t cnt[1024], sc[1024], sf[1024], cur[1024], ue[1024], uo[1025];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    cnt[tid] = 0;
    __syncthreads();
    int e = -1;
    if (tid < P) {
        e = idx[tid];
        if (e < 0 || e >= E) {
            atomicOr(status, kErrIndex);
            e = e < 0 ? 0 : E - 1;
            idx[tid] = e;
        }
        atomicAdd(cnt + e, 1);
    }
    __syncthreads();
    const int c = cnt[tid]; // tid as an expert index (0 beyond E)
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
        counts[tid] = c;
        offsets[tid] = sc[tid] - c;
        cur[tid] = sc[tid] - c;
        if (c > 0) {
            uexp[sf[tid] - 1] = tid;
            uoff[sf[tid] - 1] = sc[tid] - c;
            ue[sf[tid] - 1] = tid;
            uo[sf[tid] - 1] = sc[tid] - c;
        }
    }
    if (tid == 0) {
        *nuniq = nu;
        uoff[nu] = P;
        uo[nu] = P;
        offsets[E] = P;
    }
    __syncthreads();
    // stable placement: the warps take their 32 pairs in turn; within a warp the
    // lanes of one expert are ranked by lane
    const int nwarps = (P + 31) / 32;
    for (int w = 0; w < nwarps; w++) {
        if (warp == w) {
            const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
            const int leader = __ffs(m) - 1;
            int base = 0;
            if (e >= 0 && lane == leader) {
                base = cur[e];
                cur[e] = base + __popc(m);
            }
            base = __shfl_sync(0xFFFFFFFFu, base, leader);
            if (e >= 0) {
                const int pos = base + __popc(m & ((1u << lane) - 1u));
                perm[pos] = tid;
                inv[tid] = pos;
            }
        }
        __syncthreads();
    }
    // virtual slots of the distinct experts, in grouped order
    int ns_u = 0, first = 0, npairs = 0, eu = 0;
    if (tid < nu) {
        eu = ue[tid];
        first = uo[tid];
        npairs = uo[tid + 1] - first;
        ns_u = (npairs + kBatchCols - 1) / kBatchCols;
    }
    sc[tid] = ns_u; // (every earlier read of sc is behind the placement loop's barriers)
    __syncthreads();
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int a = tid >= o ? sc[tid - o] : 0;
        __syncthreads();
        sc[tid] += a;
        __syncthreads();
    }
    const int base = sc[tid] - ns_u;
    for (int i = 0; i < ns_u; i++)
        vslot[base + i] = make_int4(eu, first + i * kBatchCols, min(kBatchCols, npairs - i * kBatchCols), 0);
    if (tid == 1023)
        *nvslot = sc[1023];
}

// Shared memory of a batch CTA for one product (gate/up or DOWN): the ring of
// stages (routed: an item's whole 2-bit records; shared: `chunk` columns of an
// item's 8-bit records), the slot's activation rows (hi, and lo for down) and,
// for routed slots, their sub-block sums, each row padded by 32 bytes, the
// compute warps' partial sums of one item, the barriers (full and empty per
// stage; activations full and empty; partial sums full and empty) and the
// abort flag.
struct BatchPlan {
    int K2, nb2, mat2, stage2;                  // routed: columns, 256-blocks, a tile's records, an item's stage
    int K8, chunk8, nsub8, nblk8, mat8, stage8; // shared: columns, per stage, stages per item, 32-blocks per stage,
                                                // a tile's records in a stage, a stage
    int stage_bytes, nstage;
    int act_pitch, sum_pitch;
    int oact, olo, osum, opart, obar, oflag, total;
    __host__ __device__ BatchPlan(bool down, int H, int I, int Ish, int chunk, int ns) {
        const int tiles = down ? 4 : 2;
        K2 = down ? I : H;
        nb2 = K2 / 256;
        mat2 = nb2 * kQ2Rec;
        stage2 = tiles * mat2;
        K8 = Ish > 0 ? (down ? Ish : H) : 0;
        chunk8 = Ish > 0 ? chunk : 32;
        nsub8 = K8 / chunk8;
        nblk8 = chunk8 / 32;
        mat8 = nblk8 * kQ8Rec;
        stage8 = Ish > 0 ? tiles * mat8 : 0;
        stage_bytes = stage2 > stage8 ? stage2 : stage8;
        nstage = ns;
        const int kmax = K2 > K8 ? K2 : K8;
        act_pitch = 2 * kmax + 32; // 32: the 8-byte loads of rows g = 0..3 (one half-warp) hit distinct banks
        sum_pitch = K2 / 4 + 32;
        oact = ns * stage_bytes;
        olo = oact + kBatchCols * act_pitch;
        osum = olo + (down ? kBatchCols * act_pitch : 0);
        opart = osum + kBatchCols * sum_pitch;
        obar = opart + kBatchComputeWarps * 2 * kBatchCols * kPartPitch * (int)sizeof(float);
        oflag = obar + 8 * (2 * ns + 4);
        total = oflag + 16;
    }
};

// Position in a CTA's item range: kind, slot within the kind, row tile.
struct BatchCursor {
    int kind, v, tile;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One try_wait: the thread may sleep up to kBatchSuspendNs for the phase to
// complete, so a waiting warp issues few instructions.
constexpr unsigned kBatchSuspendNs = 20000;
__device__ __forceinline__ bool batch_try(uint64_t *bar, unsigned parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_addr(bar)), "r"(parity), "r"(kBatchSuspendNs)
                 : "memory");
    return done != 0;
}

// Bounded wait for phase `parity` of a barrier. false if the CTA's abort flag
// is set or the wait ran out (which sets the flag and the status word's
// kErrTimeout), so that every role of the CTA stops within one poll.
__device__ __forceinline__ bool batch_wait(uint64_t *bar, unsigned parity, volatile int *abort, unsigned *status) {
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        if (batch_try(bar, parity))
            return true;
        if ((it & 3) == 0) {
            if (*abort)
                return false;
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (it == 0) {
                t0 = now;
            } else if (now - t0 > kBatchWaitNs) {
                *abort = 1;
                atomicOr(status, kErrTimeout);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: the producer's last look at its
// own copies before the CTA leaves.
__device__ __forceinline__ void batch_drain(uint64_t *bar, unsigned parity) {
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        if (batch_try(bar, parity))
            return;
        if ((it & 3) == 0) {
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (it == 0)
                t0 = now;
            else if (now - t0 > kBatchWaitNs)
                return;
        }
    }
}

__device__ __forceinline__ void batch_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void batch_expect(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void batch_copy(uint8_t *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// One product over the items of this CTA. Gate/up items: rows 16 tile ..
// 16 tile + 15 of gate and up; the SwiGLU rows go to the down product's
// activation layout (routed: by grouped position, permuted, bf16 hi + lo and
// sums; shared: by token, binary16 hi + lo). Down items: rows 64 tile ..
// 64 tile + 63 (compute warps 0-7 the first two 16-row tiles, warps 8-15 the
// other two), into ye (routed, by grouped position) or ysh (shared, by token).
//
// The items are split over the CTAs in contiguous ranges of equal cost.
// Roles: the producer streams the
// stages of the CTA's items through the ring (waiting for a slot's release by
// all compute warps) and loads a slot's activation rows once every compute
// warp is done with the previous slot's; each compute warp runs its share of
// every stage as soon as it lands and leaves its partial sums of an item for
// the epilogue warps, which reduce them and write the results while the next
// item computes.
template <bool DOWN, int KINDS>
__global__ void __launch_bounds__(kBatchThreads, 1) batch_product_kernel(const BatchArgs a) {
    pdl_launch_next();
    pdl_wait();
    extern __shared__ __align__(128) uint8_t sm[];
    const BatchPlan pl(DOWN, a.H, a.I, a.Ish, a.chunk, a.nstage);
    const int ns = pl.nstage;
    uint64_t *const full = reinterpret_cast<uint64_t *>(sm + pl.obar); // [ns]
    uint64_t *const empty = full + ns;                                 // [ns]
    uint64_t *const act_full = empty + ns;
    uint64_t *const act_empty = act_full + 1;
    uint64_t *const part_full = act_full + 2;
    uint64_t *const part_empty = act_full + 3;
    volatile int *const abort = reinterpret_cast<volatile int *>(sm + pl.oflag);
    float *const part = reinterpret_cast<float *>(sm + pl.opart); // [warp][matrix][column][kPartPitch]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // items: routed (nslot2 slots x ntiles2), then shared (nslot8 token groups x ntiles8)
    const int ntiles2 = DOWN ? a.H / 64 : a.I / 16;
    const int ntiles8 = DOWN ? a.H / 64 : a.Ish / 16;
    const int nslot2 = (KINDS & kBatchRouted) ? *a.nvslot : 0;
    const int nslot8 = (KINDS & kBatchShared) && a.Ish > 0 ? (a.T + kBatchCols - 1) / kBatchCols : 0;
    // the item kind at a cursor (known at compile time unless the kernel runs both)
    auto routed = [&](const BatchCursor &c) {
        return KINDS == kBatchRouted ? true : KINDS == kBatchShared ? false : c.kind == kRouted;
    };
    const int nsub8 = pl.nsub8;
    const int64_t R = (int64_t)nslot2 * ntiles2, S8 = (int64_t)nslot8 * ntiles8;
    // cost units of the product: a routed item kBatchCostRouted, a shared item kBatchCostShared
    // (their measured times: both are bound by the tile GEMV's instruction issue)
    const int64_t R2 = R * kBatchCostRouted, U = R2 + S8 * kBatchCostShared;
    // the first item that starts at or after unit u
    auto item_at = [&](int64_t u) {
        return u <= R2 ? (u + kBatchCostRouted - 1) / kBatchCostRouted
                       : R + (u - R2 + kBatchCostShared - 1) / kBatchCostShared;
    };
    const int64_t i0 = item_at(U * blockIdx.x / gridDim.x);
    const int cnt = (int)(item_at(U * (blockIdx.x + 1) / gridDim.x) - i0);
    if (cnt <= 0)
        return;
    const int64_t tile_bytes2 = (int64_t)pl.nb2 * kQ2Rec; // a 2-bit tile's records over all K2
    const BatchCursor c0 = i0 < R ? BatchCursor{kRouted, (int)(i0 / ntiles2), (int)(i0 % ntiles2)}
                                  : BatchCursor{kShared, (int)((i0 - R) / ntiles8), (int)((i0 - R) % ntiles8)};
    auto step = [&](BatchCursor &c) {
        if (routed(c)) {
            if (++c.tile == ntiles2) {
                c.tile = 0;
                if (++c.v == nslot2 && KINDS == kBatchBoth) {
                    c.kind = kShared;
                    c.v = 0;
                }
            }
        } else if (++c.tile == ntiles8) {
            c.tile = 0;
            c.v++;
        }
    };
    auto slot_id = [&](const BatchCursor &c) { return routed(c) ? c.v : nslot2 + c.v; };
    // first grouped position (routed) or token (shared) of the cursor's slot, and its columns
    auto slot_cols = [&](const BatchCursor &c, int &p0, int &n) {
        if (routed(c)) {
            const int4 vs = a.vslot[c.v];
            p0 = vs.y;
            n = vs.z;
        } else {
            p0 = kBatchCols * c.v;
            n = min(kBatchCols, a.T - p0);
        }
    };

    if (tid == 0) {
        for (int s = 0; s < ns; s++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(full + s)) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(empty + s)),
                         "r"(kBatchComputeWarps)
                         : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(act_full)) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(act_empty)), "r"(kBatchComputeWarps)
                     : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(part_full)), "r"(kBatchComputeWarps)
                     : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(part_empty)), "r"(kBatchEpiWarps)
                     : "memory");
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kBatchProducerWarp) {
        if (lane != 0)
            return;
        int issued = 0, k = -1, cur = -1;
        BatchCursor c = c0;
        bool ok = true;
        for (int li = 0; li < cnt && ok; li++, step(c)) {
            const int nsub = routed(c) ? 1 : nsub8;
            for (int sub = 0; sub < nsub; sub++) {
                const int q = issued;
                if (q >= ns && !batch_wait(empty + q % ns, (unsigned)(q / ns - 1) & 1u, abort, a.status)) {
                    ok = false;
                    break;
                }
                uint64_t *bar = full + q % ns;
                uint8_t *dst = sm + (q % ns) * pl.stage_bytes;
                if (a.skip_signal && blockIdx.x == 0 && q == 0) {
                    // nothing arrives on this stage's barrier
                } else if (routed(c)) {
                    const int64_t e = a.vslot[c.v].x;
                    batch_expect(bar, (unsigned)(DOWN ? 4 : 2) * pl.mat2);
                    if (DOWN) {
                        batch_copy(dst, a.down.rec + (e * (a.H / 16) + 4 * c.tile) * tile_bytes2,
                                   (unsigned)(4 * pl.mat2), bar);
                    } else {
                        const int64_t gt = e * (a.I / 16) + c.tile;
                        batch_copy(dst, a.gate.rec + gt * tile_bytes2, (unsigned)pl.mat2, bar);
                        batch_copy(dst + pl.mat2, a.up.rec + gt * tile_bytes2, (unsigned)pl.mat2, bar);
                    }
                } else {
                    const int64_t nbq = pl.K8 / 32, b0 = (int64_t)sub * pl.nblk8;
                    batch_expect(bar, (unsigned)(DOWN ? 4 : 2) * pl.mat8);
                    if (DOWN) {
                        for (int m = 0; m < 4; m++)
                            batch_copy(dst + m * pl.mat8, a.sh_down.rec + ((4 * c.tile + m) * nbq + b0) * kQ8Rec,
                                       (unsigned)pl.mat8, bar);
                    } else {
                        batch_copy(dst, a.sh_gate.rec + (c.tile * nbq + b0) * kQ8Rec, (unsigned)pl.mat8, bar);
                        batch_copy(dst + pl.mat8, a.sh_up.rec + (c.tile * nbq + b0) * kQ8Rec, (unsigned)pl.mat8, bar);
                    }
                }
                issued = q + 1;
                if (sub == 0 && slot_id(c) != cur) { // the first stage of a new slot: its activation rows
                    cur = slot_id(c);
                    if (k >= 0 && !batch_wait(act_empty, (unsigned)k & 1u, abort, a.status)) {
                        ok = false;
                        break;
                    }
                    k++;
                    int p0, n;
                    slot_cols(c, p0, n);
                    const bool rt = routed(c);
                    const int K = rt ? pl.K2 : pl.K8;
                    const unsigned row_bytes = (DOWN ? 4u : 2u) * K + (rt ? K / 4 : 0);
                    batch_expect(act_full, (unsigned)n * row_bytes);
                    for (int col = 0; col < n; col++) {
                        const int64_t pos = p0 + col;
                        const uint16_t *hi, *lo = nullptr, *sums = nullptr;
                        if (rt && !DOWN) {
                            const int t = a.perm[pos] / a.K;
                            hi = a.xq + (int64_t)t * K;
                            sums = a.xsums + (int64_t)t * (K / 8);
                        } else if (rt) {
                            hi = a.hq_hi + pos * K;
                            lo = a.hq_lo + pos * K;
                            sums = a.hsums + pos * (K / 8);
                        } else if (!DOWN) {
                            hi = a.x + pos * K;
                        } else {
                            hi = a.hs_hi + pos * K;
                            lo = a.hs_lo + pos * K;
                        }
                        batch_copy(sm + pl.oact + col * pl.act_pitch, hi, 2 * K, act_full);
                        if (DOWN)
                            batch_copy(sm + pl.olo + col * pl.act_pitch, lo, 2 * K, act_full);
                        if (rt)
                            batch_copy(sm + pl.osum + col * pl.sum_pitch, sums, K / 4, act_full);
                    }
                }
            }
        }
        // the copies still owned by the ring and the last activation load land before the CTA leaves
        for (int q = issued - ns > 0 ? issued - ns : 0; q < issued; q++)
            batch_drain(full + q % ns, (unsigned)(q / ns) & 1u);
        if (k >= 0)
            batch_drain(act_full, (unsigned)k & 1u);
        return;
    }

    if (warp > kBatchProducerWarp) { // epilogue warps: thread et of kBatchEpiThreads
        const int et = (warp - kBatchProducerWarp - 1) * 32 + lane;
        int cur = -1, p0 = 0, n = 0;
        BatchCursor c = c0;
        for (int li = 0; li < cnt; li++, step(c)) {
            if (slot_id(c) != cur) {
                slot_cols(c, p0, n);
                cur = slot_id(c);
            }
            if (!batch_wait(part_full, (unsigned)li & 1u, abort, a.status))
                return;
            const int tile = c.tile;
            if (DOWN) {
                // output o = (col, m, r): row 64 tile + 16 m + r of column col, summed over its group's warps
                float *dst = routed(c) ? a.ye : a.ysh;
#pragma unroll
                for (int k4 = 0; k4 < 16 * 4 * kBatchCols / kBatchEpiThreads; k4++) {
                    const int o = et + kBatchEpiThreads * k4;
                    const int col = o >> 6, m = (o >> 4) & 3, r = o & 15;
                    if (col < n) {
                        float acc = 0.f;
#pragma unroll
                        for (int w = 8 * (m >> 1); w < 8 * (m >> 1) + 8; w++)
                            acc += part[((w * 2 + (m & 1)) * kBatchCols + col) * kPartPitch + r];
                        dst[(int64_t)(p0 + col) * a.H + 64 * tile + 16 * m + r] = acc;
                    }
                }
            } else {
#pragma unroll
                for (int k2 = 0; k2 < 16 * kBatchCols / kBatchEpiThreads; k2++) {
                    const int col = (et >> 4) + (kBatchEpiThreads / 16) * k2, r = et & 15;
                    float hv = 0.f;
                    if (col < n) {
                        float gs = 0.f, us = 0.f;
#pragma unroll
                        for (int w = 0; w < kBatchComputeWarps; w++) {
                            gs += part[((w * 2) * kBatchCols + col) * kPartPitch + r];
                            us += part[((w * 2 + 1) * kBatchCols + col) * kPartPitch + r];
                        }
                        hv = silu(gs) * us;
                    }
                    if (!routed(c)) {
                        if (col < n) {
                            const __half hi = __float2half_rn(hv);
                            const __half lo = __float2half_rn(hv - __half2float(hi));
                            const int64_t o = (int64_t)(p0 + col) * a.Ish + 16 * tile + r;
                            a.hs_hi[o] = __half_as_ushort(hi);
                            a.hs_lo[o] = __half_as_ushort(lo);
                        }
                    } else {
                        // row r of the tile is column k = 16 tile + r of the down matrix: position r
                        // of its sub-block j = tile % 16 in block tile / 16
                        const int blk = tile >> 4, j = tile & 15;
                        float hs = 0.f;
                        if (col < n) {
                            const int e2 = 2 * q2_p(r, j >> 3);
                            const float hp = hv * (1.0f / (float)(1 << e2)); // exact: power of two
                            const uint32_t h1 = f32_to_bf16_bits(hp);
                            const float h1f = __uint_as_float(h1 << 16);
                            const uint32_t h2 = f32_to_bf16_bits(hp - h1f);
                            const float h2f = __uint_as_float(h2 << 16);
                            const int64_t o = (int64_t)(p0 + col) * a.I + q2_act_index(tile * 16 + r);
                            a.hq_hi[o] = (uint16_t)h1;
                            a.hq_lo[o] = (uint16_t)h2;
                            hs = (h1f + h2f) * (float)(1 << e2); // the value the down product sees
                        }
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1) // over the 16 rows: one sub-block of the down columns
                            hs += __shfl_xor_sync(0xFFFFFFFFu, hs, o);
                        if (col < n && r == 0) {
                            const uint32_t h1 = f32_to_bf16_bits(hs);
                            const uint32_t h2 = f32_to_bf16_bits(hs - __uint_as_float(h1 << 16));
                            uint16_t *so = a.hsums + (int64_t)(p0 + col) * (a.I / 8);
                            so[q2_sum_index(blk, j, 0)] = (uint16_t)h1;
                            so[q2_sum_index(blk, j, 1)] = (uint16_t)h2;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                batch_arrive(part_empty);
        }
        return;
    }

    // compute warps
    const int g = lane >> 2, tig = lane & 3;
    const int grp = warp >> 3, wl = warp & 7; // down products: tile pair, warp within it
    int cur = -1, k = -1, n = 0, q = 0;
    BatchCursor c = c0;
    for (int li = 0; li < cnt; li++) {
        if (slot_id(c) != cur) {
            int p0;
            slot_cols(c, p0, n);
            cur = slot_id(c);
            k++;
            if (!batch_wait(act_full, (unsigned)k & 1u, abort, a.status))
                return;
        }
        const int col = g < n ? g : 0; // this lane's MMA column (a repeated row is discarded)
        const uint8_t *xrow = sm + pl.oact + col * pl.act_pitch;
        const uint8_t *lrow = sm + pl.olo + col * pl.act_pitch;
        const uint8_t *srow = sm + pl.osum + col * pl.sum_pitch;
        float out[2][2][2] = {};
        const int nsub = routed(c) ? 1 : nsub8;
        for (int sub = 0; sub < nsub; sub++, q++) {
            if (!batch_wait(full + q % ns, (unsigned)(q / ns) & 1u, abort, a.status))
                return;
            const uint8_t *stage = sm + (q % ns) * pl.stage_bytes;
            if (routed(c)) {
                const int nb = pl.nb2;
                if (DOWN) {
                    const uint8_t *rec[2] = {stage + (2 * grp) * pl.mat2, stage + (2 * grp + 1) * pl.mat2};
                    q2_gemv<2, true>(rec, xrow, lrow, srow, nb * wl / 8, nb * (wl + 1) / 8, lane, out);
                } else {
                    const uint8_t *rec[2] = {stage, stage + pl.mat2};
                    q2_gemv<2, false>(rec, xrow, xrow, srow, nb * warp / kBatchComputeWarps,
                                      nb * (warp + 1) / kBatchComputeWarps, lane, out);
                }
            } else {
                const int nb = pl.nblk8;
                const int off = 2 * sub * pl.chunk8;
                if (DOWN) {
                    const uint8_t *rec[2] = {stage + (2 * grp) * pl.mat8, stage + (2 * grp + 1) * pl.mat8};
                    q8_gemv<2, true, false>(rec, xrow + off, lrow + off, nb * wl / 8, nb * (wl + 1) / 8, lane, out);
                } else {
                    const uint8_t *rec[2] = {stage, stage + pl.mat8};
                    q8_gemv<2, false, true>(rec, xrow + off, xrow + off, nb * warp / kBatchComputeWarps,
                                            nb * (warp + 1) / kBatchComputeWarps, lane, out);
                }
            }
            __syncwarp();
            if (lane == 0)
                batch_arrive(empty + q % ns);
        }
        step(c);
        if (li + 1 < cnt && slot_id(c) != cur) { // done with this slot's activation rows
            __syncwarp();
            if (lane == 0)
                batch_arrive(act_empty);
        }
        if (li > 0 && !batch_wait(part_empty, (unsigned)(li - 1) & 1u, abort, a.status))
            return;
#pragma unroll
        for (int m = 0; m < 2; m++)
#pragma unroll
            for (int cc = 0; cc < 2; cc++) {
                const int cl = 2 * tig + cc;
                part[((warp * 2 + m) * kBatchCols + cl) * kPartPitch + g] = out[m][0][cc];
                part[((warp * 2 + m) * kBatchCols + cl) * kPartPitch + g + 8] = out[m][1][cc];
            }
        __syncwarp();
        if (lane == 0)
            batch_arrive(part_full);
    }
}

} // namespace ds4
