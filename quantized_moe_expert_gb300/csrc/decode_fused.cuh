// Decode path (T <= 8 tokens per launch): one persistent cooperative kernel.
//
// Each CTA is a producer warp, eight consumer warps and a publisher warp. The
// consumers hand each finished job to the publisher, which makes it visible
// GPU-wide (a release on the job's count, the output-tile arrivals and
// combines), so that no GPU-scope fence or atomic stalls the math. The producer warp
// pulls jobs from a global queue (an atomic counter) and streams each job's
// weight tiles and activation rows into a ring of shared-memory stages with
// bulk asynchronous copies (cp.async.bulk completing on an mbarrier; its lanes
// issue a stage's copies side by side); the
// consumer warps multiply them on the tensor cores (mma.sync, see the layouts
// in frag_layout.cuh) and release the stage. Two CTAs per SM, each with three
// 33 KB stages, keep up to 198 KB per SM in flight, independent of registers.
//
// Jobs are numbered so that each depends only on jobs with smaller numbers,
// and a CTA takes its jobs in increasing order (its first job is its own
// index, the rest come from the queue), so the oldest unfinished job can
// always run: the queue cannot deadlock as long as all CTAs are resident,
// which the cooperative launch guarantees. The queue, in order:
//
//   SEL  one job, the first job of CTA 0, run by its consumers at once: the
//        activations in the 2-bit MMA's layout; then, as the router rows
//        arrive, per-token sigmoid, exact top-k, weights and the
//        distinct-expert grouping; publishes one record per distinct expert
//        (waits for all R jobs)
//   R    one or two router rows: fp32 logits for all T tokens, each stored
//        with the launch's epoch in the same 64-bit word (the value is its
//        own completion flag); read straight from global memory by the
//        consumers (a CTA's first job at once, later ones on a descriptor-only
//        stage)
//   SGU  shared expert, one 16-row tile of gate and up: h_sh = silu(g) * u
//   GU   (distinct expert, 16-row tile of I): gate and up, h = silu(g) * u,
//        stored as a bf16 hi/lo pair in the down MMA's activation layout
//   SD   shared expert down, one 16-row tile of H (waits: all SGU)
//   D    (distinct expert, 32-row tile of H): down projection (waits: that
//        expert's GU tiles); the last of the experts' contributions to a tile
//        combines it once all SD jobs are done: y = sum_k w_k ye_k + ysh, in
//        fixed order
// The shared expert's gate/up jobs sit between the router and the routed jobs
// so that they stream while the routing is computed and published.
// The producer of a GU or D job polls that expert's routing record (epoch-
// tagged, so the poll and the lookup are one load) and then issues the
// weight copies; the weight loads of a job never wait for its data
// dependencies, only its consumers do, so loads overlap those waits.
//
// This follows the pages' decode engine in spirit - routed experts and the
// shared expert proceed side by side ("YoungAi - DeepSeek V4.1 Flash on one
// DGX Spark", section 4.4, "Side stream"), each distinct expert's bits are read
// once for all rows that chose it (same section, verify batch), and work
// starts on data that does not depend on its producer (same section,
// "Programmatic dependent launch") - but as one kernel with fine-grained
// dependencies instead of a chain of launches.
//
// Every wait is bounded (kWaitNs of %globaltimer); a wait that runs out sets
// kErrTimeout in the status word and an abort flag that makes every CTA drain
// its ring and leave.
#pragma once

#include "common.cuh"
#include "frag_layout.cuh"
#include "tile_gemv.cuh"

namespace ds4 {

constexpr int kDecodeT = 8;             // tokens per launch
constexpr int kMaxSlots = 64;           // distinct experts per launch <= 8 tokens * top-8
constexpr uint64_t kWaitNs = 500000000; // 0.5 s
constexpr int kRing = 3;                // shared-memory stages per CTA (two CTAs per SM)
constexpr int kSlotBytes = 33792;       // bytes per stage
constexpr int kConsumerWarps = 8;
// the selection job's keys ([T][E]) fit its stage buffer, the bias ([E]) the
// reduction buffer (E <= 1024)
static_assert(4 * kDecodeT * 1024 <= kSlotBytes, "selection scratch");
constexpr int kPubQ = 4; // publication tasks in flight (consumers -> publisher warp)
// consumers, the producer warp and the publisher warp
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 2);

// Control words (zeroed at create; every launch leaves them zeroed again).
enum : int {
    kCtlJobNext = 0,
    kCtlSguDone = 3,
    kCtlFinished = 4,
    kCtlAbort = 5,
    kCtlSdDone = 6,
    kCtlGuDone = 8,              // [kMaxSlots]
    kCtlTileCnt = 8 + kMaxSlots, // [H / 32]
};

// Where the selection reads its logits and writes its results.
struct SelIO {
    const unsigned long long *lgt;
    unsigned epoch;
    int32_t *idx;
    float *w, *gap;
    int32_t *inv, *counts, *nuniq;
    unsigned long long *srec;
};

struct DecodeArgs {
    int H, I, E, K, Ish;
    const float *router_w, *router_bias;
    Q2Frag gate, up, down;
    Q8Frag sh_gate, sh_up, sh_down;
    const uint16_t *x; // [T][H] bf16
    int T;
    float *y;                  // [T][H]
    const int32_t *forced_idx; // [T][K] or nullptr
    const float *forced_w;
    unsigned epoch;
    unsigned long long *lgt;  // [8][E] router logits: fp32 bits | epoch << 32
    unsigned long long *srec; // [kMaxSlots][2] routing record of each distinct-expert slot (| epoch << 32)
    int32_t *idx;    // [8][K]
    float *w;        // [8][K]
    float *gap;      // [8]
    int32_t *counts; // [E]
    int32_t *nuniq, *inv;
    uint16_t *xq;            // [8][H] bf16 x * 4^-p, permuted (q2_act_index)
    uint16_t *xsums;         // [8][H/8] bf16 hi and lo of each 16-column sum of x (q2_sum_index)
    uint16_t *hq_hi, *hq_lo; // [64][I] SwiGLU rows h * 4^-p as a bf16 hi + lo pair, permuted
    uint16_t *hsums;         // [64][I/8] the 16-column sums of h, hi and lo
    uint16_t *hs_hi, *hs_lo; // [8][Ish] binary16 shared h as hi + lo
    float *ye;               // [64][H]
    float *ysh;              // [8][H]
    unsigned *ctl;
    unsigned *status;
    SelIO io; // the selection's inputs and outputs (the buffers above)
    const float *gain; // [E][H] per-expert down gains (the kernel built with GAIN), or nullptr
};

enum JobType : int { kJobEnd = 0, kJobR, kJobSgu, kJobSel, kJobGu, kJobSd, kJobD };
enum PubKind : int { kPubSignal = 0, kPubTile, kPubEnd };

// What the producer tells the consumers about one stage.
struct StageDesc {
    int type;
    int a0;         // R: expert row; GU/D: distinct-expert slot; SGU/SD: tile
    int tile;       // GU/D: 16-row tile within the expert
    int sub, nsub;  // sub-stage index and count of the job
    int c0, W;      // column range [c0, c0 + W) of this sub-stage
    int ntok, tp;   // tokens of the job and their count padded to 1, 2, 4 or 8
    int nuniq;      // distinct experts of this launch (GU, SD, D)
    int pos[kDecodeT]; // pair position of each token column (GU, D outputs)
    int tok[kDecodeT]; // token of each column
    int oq[2];      // byte offsets of the matrix pieces (runs of records, frag_layout.cuh)
    int oact, olo, ooff, osum; // activation pieces
    int act_pitch, sub_pitch;  // bytes per token row of the hi/lo and off/sum pieces
};

struct DecodeSmem {
    alignas(128) uint8_t ring[kRing][kSlotBytes];
    StageDesc desc[kRing];
    alignas(8) uint64_t full[kRing];
    alignas(8) uint64_t empty[kRing];
    // per-warp partial sums of the job being finished
    alignas(16) float part[kConsumerWarps][2][16][kDecodeT];
                                                 // (the selection job: the router bias)
    // publication tasks: what the publisher warp makes visible GPU-wide after a job
    struct PubTask {
        unsigned *ctr; // the job count to increase, or the tile counter
        int kind;      // kPubSignal, kPubTile, kPubEnd
        int tile, nuniq;
    } pub[kPubQ];
    float cw[kDecodeT * kMaxTopK];   // publisher: routing weights of the tile being combined
    int cinv[kDecodeT * kMaxTopK];   // and the positions of their pairs
    alignas(8) uint64_t pub_full[kPubQ];
    alignas(8) uint64_t pub_empty[kPubQ];
    int sel_idx[kDecodeT][kMaxTopK];
    unsigned bitmap[32];
    int word_prefix[32];
    int slot_cnt[kMaxSlots];
    int pair_at[kMaxSlots]; // grouping: the pair at each expert-grouped position
    unsigned rec[2][kMaxSlots]; // grouping: the slot records before publication
    int sel_flag[2];            // selection: give-up decision of thread 0, double-buffered by poll round
    // the producer's next stage, built before its ring slot is free
    StageDesc pdesc;
    // the routing records of this launch (raw words), cached by the producer
    unsigned rcache[kMaxSlots][2];
    // the producer's list of bulk copies for the stage it is building
    const void *pc_src[40];
    unsigned pc_bytes[40];
    unsigned pc_dst[40];
    int cexp[kDecodeT * kMaxTopK]; // publisher, with down gains: the experts of the tile's pairs
};
static_assert(sizeof(DecodeSmem::part) >= 4 * 1024, "router bias staging");


// ---- small PTX helpers --------------------------------------------------------

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// A routing record of one distinct-expert slot: word 0 = expert | first pair
// position << 11 | token count << 18 | distinct experts << 22, word 1 = the
// tokens of its pairs, 3 bits each in pair order; both | epoch << 32.
struct SlotRec {
    int e, p0, ntok, nuniq;
    unsigned toks;
};

__device__ __forceinline__ SlotRec unpack_slot(unsigned w0, unsigned w1) {
    SlotRec r;
    r.e = (int)(w0 & 0x7FFu);
    r.p0 = (int)((w0 >> 11) & 0x7Fu);
    r.ntok = (int)((w0 >> 18) & 0xFu);
    r.nuniq = (int)((w0 >> 22) & 0x7Fu);
    r.toks = w1;
    return r;
}


__device__ __forceinline__ float nib_to_f(uint32_t n) { return __uint_as_float(0x4B000000u | n) - 8388608.0f; }

__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *p >= target (or == target when eq): acquire polls with a
// short sleep between them. Returns false after kWaitNs or when another CTA
// aborted.
__device__ bool wait_counter(const DecodeArgs &a, const unsigned *p, unsigned target, bool eq) {
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        const unsigned v = ld_acquire(p);
        if (eq ? v == target : v >= target)
            return true;
        if ((it & 63) == 0) {
            if (ld_relaxed(a.ctl + kCtlAbort))
                return false;
            const uint64_t now = globaltimer();
            if (it == 0)
                t0 = now;
            else if (now - t0 > kWaitNs) {
                atomicOr(a.status, kErrTimeout);
                atomicExch(a.ctl + kCtlAbort, 1u);
                return false;
            }
        }
        __nanosleep(128);
    }
}

// ---- mbarrier, bulk copy and barrier helpers ------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait for the completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_wait(const DecodeArgs &a, uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255) == 0) {
            const uint64_t now = globaltimer();
            if (it == 0)
                t0 = now;
            else if (now - t0 > kWaitNs) {
                atomicOr(a.status, kErrTimeout);
                atomicExch(a.ctl + kCtlAbort, 1u);
                return false;
            }
        }
        __nanosleep(32);
    }
}

// Global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Barrier of the eight consumer warps (the producer warp does not take part).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ---- tensor-core tile GEMV over one stage -----------------------------------------
//
// 2-bit matrices (layout in frag_layout.cuh): a warp takes whole 256-column
// blocks of the stage; per block and matrix it turns the sub-block scales of
// its two rows and four sub-blocks into bf16 multipliers once, then runs 16
// MMAs whose A registers are one LOP3 and one packed FMA each (sc q 4^p,
// exact), and two MMAs for the min term. The 8 MMA columns are the job's
// tokens (padded columns repeat token 0 and are ignored). At the end of a
// block, out[m][rho][col] (row g + 8 rho, token 2 tig + col) gains
// d D - dmin Dm.

template <int TP> __device__ __forceinline__ int srow(const StageDesc &d, int t) { return t < d.ntok ? t : 0; }

// NMAT 2-bit matrices of the stage sharing the activations; SPLIT: the
// activations are a bf16 hi + lo pair (both multiplied by the same A). Warp w
// takes its share of the stage's 256-column blocks.
template <int NMAT, bool SPLIT>
__device__ __forceinline__ void q2_stage(const uint8_t *sl, const StageDesc &d, int warp, int lane,
                                         float (&out)[2][2][2]) {
    const int nb = d.W >> 8;
    const int t = (lane >> 2) < d.ntok ? (lane >> 2) : 0; // this lane's B column's token
    const uint8_t *rec[NMAT];
#pragma unroll
    for (int m = 0; m < NMAT; m++)
        rec[m] = sl + d.oq[m];
    q2_gemv<NMAT, SPLIT>(rec, sl + d.oact + t * d.act_pitch, sl + d.olo + t * d.act_pitch,
                         sl + d.osum + t * d.sub_pitch, nb * warp / kConsumerWarps, nb * (warp + 1) / kConsumerWarps,
                         lane, out);
}

// Partial sums of a 2-bit job (q2_stage's layout: each (row, token) in one
// lane) into the warp's slot of the job's reduction buffer.
__device__ __forceinline__ void store_part_q2(DecodeSmem &sm, int warp, int lane, const float (&out)[2][2][2], int ntok) {
    const int g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int m = 0; m < 2; m++)
#pragma unroll
        for (int col = 0; col < 2; col++) {
            const int t = 2 * tig + col;
            if (t < ntok) {
                sm.part[warp][m][g][t] = out[m][0][col];
                sm.part[warp][m][g + 8][t] = out[m][1][col];
            }
        }
}

// 8-bit matrices: A = the codes as exact binary16 integers, B = binary16
// activations (FROM_BF16: the stage holds bf16 rows, converted here); each slot
// of an accumulator tile is one 32-column block (one scale).
template <int TP, int NMAT, bool SPLIT, bool FROM_BF16>
__device__ __forceinline__ void q8_stage(const uint8_t *sl, const StageDesc &d, int warp, int lane,
                                         float (&out)[2][2][2]) {
    constexpr int S = 8 / TP;
    const int g = lane >> 2, tig = lane & 3;
    const int bs = g / TP, bt = g % TP;
    const int n0 = 2 * tig, n1 = 2 * tig + 1;
    const int s0 = n0 / TP, s1 = n1 / TP;
    const int nbq = d.W >> 5;
    const int bb = nbq * warp / kConsumerWarps, be = nbq * (warp + 1) / kConsumerWarps;
    const uint32_t *act = reinterpret_cast<const uint32_t *>(sl + d.oact + srow<TP>(d, bt) * d.act_pitch);
    const uint32_t *act_lo = reinterpret_cast<const uint32_t *>(sl + d.olo + srow<TP>(d, bt) * d.act_pitch);
    for (int base = bb; base < be; base += S) {
        float D[NMAT][4], D2[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int i = 0; i < 4; i++)
                D[m][i] = D2[m][i] = 0.f;
#pragma unroll
        for (int sl2 = 0; sl2 < S; sl2++) {
            const int bq = base + sl2;
            if (bq < be) {
                uint4 q[NMAT];
#pragma unroll
                for (int m = 0; m < NMAT; m++)
                    q[m] = reinterpret_cast<const uint4 *>(sl + d.oq[m] + bq * kQ8Rec)[lane];
                const bool on = bs == sl2;
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int col = bq * 32 + 16 * c + 2 * tig;
                    uint32_t b0 = on ? act[col >> 1] : 0u, b1 = on ? act[(col + 8) >> 1] : 0u;
                    if (FROM_BF16) {
                        b0 = bf16x2_to_f16x2(b0);
                        b1 = bf16x2_to_f16x2(b1);
                    }
                    uint32_t c0 = 0, c1 = 0;
                    if (SPLIT) {
                        c0 = on ? act_lo[col >> 1] : 0u;
                        c1 = on ? act_lo[(col + 8) >> 1] : 0u;
                    }
#pragma unroll
                    for (int m = 0; m < NMAT; m++) {
                        const uint32_t vg = c ? q[m].z : q[m].x, vg8 = c ? q[m].w : q[m].y;
                        const uint32_t a0 = hsub2_1152(prmt(vg, 0x64646464u, 0x4140u));
                        const uint32_t a1 = hsub2_1152(prmt(vg8, 0x64646464u, 0x4140u));
                        const uint32_t a2 = hsub2_1152(prmt(vg, 0x64646464u, 0x4342u));
                        const uint32_t a3 = hsub2_1152(prmt(vg8, 0x64646464u, 0x4342u));
                        if (SPLIT) {
                            mma_f16(D[m], a0, a1, a2, a3, b0, b1);
                            mma_f16(D2[m], a0, a1, a2, a3, c0, c1);
                        } else {
                            mma_f16(c ? D2[m] : D[m], a0, a1, a2, a3, b0, b1);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int i = 0; i < 4; i++)
                D[m][i] += D2[m][i];
        const int bqa = base + s0, bqb = base + s1;
#pragma unroll
        for (int m = 0; m < NMAT; m++) {
            const uint8_t *rm = sl + d.oq[m] + kQ8RecD; // scale entries of block 0's record
            if (bqa < be) {
                const uint32_t dw = reinterpret_cast<const uint32_t *>(rm + bqa * kQ8Rec)[g];
                out[m][0][0] = fmaf(f16_to_f32(dw), D[m][0], out[m][0][0]);
                out[m][1][0] = fmaf(f16_to_f32(dw >> 16), D[m][2], out[m][1][0]);
            }
            if (bqb < be) {
                const uint32_t dw = reinterpret_cast<const uint32_t *>(rm + bqb * kQ8Rec)[g];
                out[m][0][1] = fmaf(f16_to_f32(dw), D[m][1], out[m][0][1]);
                out[m][1][1] = fmaf(f16_to_f32(dw >> 16), D[m][3], out[m][1][1]);
            }
        }
    }
}

// Combine the lanes that hold the same (row, token) at the end of a job.
template <int TP, int NMAT> __device__ __forceinline__ void reduce_out(float (&out)[2][2][2]) {
#pragma unroll
    for (int m = 0; m < NMAT; m++)
#pragma unroll
        for (int r = 0; r < 2; r++) {
            if (TP == 1) {
                out[m][r][0] += out[m][r][1];
                out[m][r][1] = 0.f;
            }
#pragma unroll
            for (int col = 0; col < 2; col++) {
                float v = out[m][r][col];
                if (TP <= 2) {
                    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                } else if (TP == 4) {
                    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                }
                out[m][r][col] = v;
            }
        }
}

// Lanes holding final (row, token) values and the token of each of their columns.
template <int TP> __device__ __forceinline__ bool tile_owner(int lane) {
    const int tig = lane & 3;
    return TP <= 2 ? tig == 0 : (TP == 4 ? tig < 2 : true);
}

template <int TP, int NMAT>
__device__ __forceinline__ void store_part(DecodeSmem &sm, int warp, int lane, const float (&out)[2][2][2]) {
    if (!tile_owner<TP>(lane))
        return;
    const int g = lane >> 2;
#pragma unroll
    for (int m = 0; m < NMAT; m++)
#pragma unroll
        for (int col = 0; col < 2; col++) {
            if (TP == 1 && col == 1)
                continue;
            const int t = (2 * (lane & 3) + col) % TP;
            sm.part[warp][m][g][t] = out[m][0][col];
            sm.part[warp][m][g + 8][t] = out[m][1][col];
        }
}

// Router rows a0 .. a0 + nrows - 1 (nrows <= 2, and nrows * T <= 8) for all T
// tokens, straight from global memory by the consumer threads (no stage):
// thread i takes float4 columns i, i + 256, ... of each row, all its loads in
// flight together; the warps' partial sums are added in warp order, and each
// logit is stored with the launch's epoch in the same 64-bit word (the value
// is its own completion flag). Ends with a consumer barrier.
__device__ void router_rows(const DecodeArgs &a, DecodeSmem &sm, int a0, int nrows, int warp, int lane) {
    const int T = a.T, n4 = a.H / 4;
    float acc[kDecodeT]; // index 4 r + t with two rows (T <= 4), else t
#pragma unroll
    for (int i = 0; i < kDecodeT; i++)
        acc[i] = 0.f;
#pragma unroll 4
    for (int q = threadIdx.x; q < n4; q += 32 * kConsumerWarps) {
        float4 wv[2];
#pragma unroll
        for (int r = 0; r < 2; r++)
            wv[r] = r < nrows ? __ldg(reinterpret_cast<const float4 *>(a.router_w + (int64_t)(a0 + r) * a.H) + q)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < kDecodeT; t++) {
            if (t < T) {
                const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(a.x + (int64_t)t * a.H) + q);
                const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xFFFF0000u);
                const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xFFFF0000u);
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    if (r < nrows && 4 * r + t < kDecodeT) {
                        float &cc = acc[4 * r + t];
                        cc = fmaf(wv[r].x, x0, cc);
                        cc = fmaf(wv[r].y, x1, cc);
                        cc = fmaf(wv[r].z, x2, cc);
                        cc = fmaf(wv[r].w, x3, cc);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kDecodeT; i++) {
        const int t = nrows == 2 ? (i & 3) : i; // row i >> 2 (two rows) or 0
        if (t < T) {
            const float v = warp_sum(acc[i]);
            if (lane == 0)
                sm.part[warp][0][0][i] = v;
        }
    }
    consumer_sync();
    {
        const int i = threadIdx.x, r = nrows == 2 ? i >> 2 : 0, t = nrows == 2 ? (i & 3) : i;
        if (i < kDecodeT && t < T && r < nrows) {
            float v = 0.f;
            for (int w = 0; w < kConsumerWarps; w++)
                v += sm.part[w][0][0][i];
            st_relaxed_u64(a.lgt + t * a.E + a0 + r, (unsigned long long)a.epoch << 32 | __float_as_uint(v));
        }
    }
    consumer_sync(); // the reduction buffer is read before the next job writes it
}

// Top-k of token t by one warp from the selection keys keys[e] (shared
// memory, e < E). Each expert is the 64-bit value key << 32 | ~e (larger key
// first, then lower index; all distinct, and above 0 since keys of untaken
// experts are >= 1). Lane l keeps the best K+1 of its experts l, l + 32, ...
// sorted in registers; each round the warp takes the largest head by two warp
// reductions and the owning lane shifts its list. One round more than K gives
// the (K+1)-th score for the near-tie gap.
__device__ __forceinline__ void select_token(const DecodeArgs &a, const SelIO &io, DecodeSmem &sm, unsigned *keys,
                                             int t, int lane) {
    const int E = a.E, K = a.K;
    constexpr int R = kMaxTopK + 1;
    uint64_t top[R];
#pragma unroll
    for (int i = 0; i < R; i++)
        top[i] = 0ull;
    for (int e = lane; e < E; e += 32) {
        uint64_t v = (uint64_t)keys[e] << 32 | (0xFFFFFFFFu - (unsigned)e);
#pragma unroll
        for (int i = 0; i < R; i++) { // insertion into the descending list
            const uint64_t hi = top[i] > v ? top[i] : v;
            v = top[i] > v ? v : top[i];
            top[i] = hi;
        }
    }
    int chosen = 0;
    unsigned chosen_key = 0u;
    float kth = 0.f, next = -INFINITY;
    const int rounds = K < E ? K + 1 : K;
    for (int r = 0; r < rounds; r++) {
        const unsigned hk = (unsigned)(top[0] >> 32);
        const unsigned gk = __reduce_max_sync(0xFFFFFFFFu, hk);
        const unsigned gl = __reduce_max_sync(0xFFFFFFFFu, hk == gk ? (unsigned)top[0] : 0u);
        const int be = (int)(0xFFFFFFFFu - gl); // < E: every round has a candidate
        const float bv = sel_key_value(gk);
        if (r < K) {
            if (lane == r) {
                chosen = be;
                chosen_key = gk;
            }
            if (r == K - 1)
                kth = bv;
            if (hk == gk && (unsigned)top[0] == gl) { // this lane's head was taken
#pragma unroll
                for (int i = 0; i + 1 < R; i++)
                    top[i] = top[i + 1];
                top[R - 1] = 0ull;
            }
        } else {
            next = bv;
        }
    }
    // weights: the chosen experts' sigmoid scores, renormalised in selection
    // order. Without a bias the selection key is the score itself; with one,
    // the score is recomputed from the logit with the same function.
    float sc = 0.f;
    if (lane < K) {
        if (a.router_bias)
            sc = sigmoid(__uint_as_float((unsigned)ld_relaxed_u64(io.lgt + t * E + chosen)));
        else
            sc = sel_key_value(chosen_key);
    }
    float total = 0.f;
    for (int r = 0; r < K; r++)
        total += __shfl_sync(0xFFFFFFFFu, sc, r);
    if (lane < K) {
        sm.sel_idx[t][lane] = chosen;
        io.idx[t * K + lane] = chosen;
        io.w[t * K + lane] = total > 0.f ? sc / total : 1.0f / K;
    }
    if (lane == 0)
        io.gap[t] = K < E ? kth - next : INFINITY;
}

// Work of the selection job that needs no router output (all consumer
// threads, before the wait for the router rows): the activations in the
// 2-bit GEMV's permuted layout (x 4^-p, exact) with their 16-column sums as a
// bf16 hi + lo pair, zeroed expert counts, and the router bias staged into
// shared memory (the reduction buffer, free during the selection job).
__device__ void select_prepare(const DecodeArgs &a, float *bias) {
    const int T = a.T, E = a.E, H = a.H;
    // thread i takes sub-blocks i, i + 256, ... of every token
    const int nsub = H / 16;
    for (int t = 0; t < T; t++)
    for (int j = threadIdx.x; j < nsub; j += 32 * kConsumerWarps) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)t * H + 16 * j);
        const uint4 p0 = __ldg(src), p1 = __ldg(src + 1);
        const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        const int kappa = (j & 15) >> 3;
        uint16_t *xt = a.xq + (int64_t)t * H;
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
        uint16_t *st = a.xsums + (int64_t)t * (H / 8);
        st[q2_sum_index(j >> 4, j & 15, 0)] = (uint16_t)hi;
        st[q2_sum_index(j >> 4, j & 15, 1)] = (uint16_t)lo;
    }
    for (int e = threadIdx.x; e < E; e += 32 * kConsumerWarps) {
        a.counts[e] = 0;
        if (!a.forced_idx)
            bias[e] = a.router_bias ? __ldg(a.router_bias + e) : 0.f;
    }
}

// Per-token selection as the router rows arrive: every consumer thread polls
// its share of the epoch-tagged logits until all are present (bounded),
// turning each into its selection key in the job's stage buffer; exact top-k
// (warp t takes token t); then the grouping, computed in shared memory, and
// one routing record per distinct-expert slot, published after a fence.
// Returns false if the wait for the router rows gave up.
__device__ __forceinline__ bool job_select(const DecodeArgs &a, const SelIO &io, DecodeSmem &sm, float *scratch,
                                           int warp, int lane) {
    const int T = a.T, E = a.E, K = a.K;
    unsigned *keys = reinterpret_cast<unsigned *>(scratch);
    if (!a.forced_idx) {
        const float *bias = &sm.part[0][0][0][0];
        const int n = T * E;
        constexpr int kStride = 32 * kConsumerWarps;
        // thread i owns entries i, i + 256, ... (at most 32 of them: T E <= 8192);
        // the expert of entry q (q mod E) is followed incrementally
        unsigned pending = 0u;
        for (int u = 0, q = threadIdx.x; q < n; u++, q += kStride)
            pending |= 1u << u;
        const int e0 = (int)threadIdx.x % E;
        uint64_t t0 = 0;
        for (unsigned it = 0;; it++) {
            unsigned still = 0u;
            int e = e0;
            // one or two tokens: at most two entries per thread, one at a time
            if (T <= 2) {
                for (int u = 0, q = threadIdx.x; q < n; u++, q += kStride) {
                    const int eq = e;
                    e += kStride;
                    while (e >= E)
                        e -= E;
                    if (!(pending >> u & 1u))
                        continue;
                    const unsigned long long v = ld_relaxed_u64(io.lgt + q);
                    if ((unsigned)(v >> 32) != io.epoch) {
                        still |= 1u << u;
                        continue;
                    }
                    const float sg = sigmoid(__uint_as_float((unsigned)v));
                    keys[q] = sel_key(a.router_bias ? sg + bias[eq] : sg);
                }
            }
            // more tokens: eight entries' loads in flight at a time
            for (int u0 = 0, q0 = threadIdx.x; T > 2 && q0 < n; u0 += 8, q0 += 8 * kStride) {
                unsigned long long v[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int q = q0 + i * kStride;
                    v[i] = (q < n && (pending >> (u0 + i) & 1u)) ? ld_relaxed_u64(io.lgt + q) : 0ull;
                }
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int q = q0 + i * kStride, u = u0 + i;
                    const int eq = e;
                    e += kStride;
                    while (e >= E)
                        e -= E;
                    if (q >= n || !(pending >> u & 1u))
                        continue;
                    if ((unsigned)(v[i] >> 32) != io.epoch) {
                        still |= 1u << u;
                        continue;
                    }
                    const float sg = sigmoid(__uint_as_float((unsigned)v[i]));
                    keys[q] = sel_key(a.router_bias ? sg + bias[eq] : sg);
                }
            }
            pending = still;
            // bounded: thread 0 decides for everyone; the flag of round it is
            // rewritten only two barriers later, after every thread has read it
            if (threadIdx.x == 0) {
                int give_up = 0;
                if ((it & 15) == 0) {
                    const uint64_t now = globaltimer();
                    if (it == 0)
                        t0 = now;
                    else if (now - t0 > kWaitNs) {
                        atomicOr(a.status, kErrTimeout);
                        atomicExch(a.ctl + kCtlAbort, 1u);
                        give_up = 1;
                    } else if (ld_relaxed(a.ctl + kCtlAbort)) {
                        give_up = 1;
                    }
                }
                sm.sel_flag[it & 1] = give_up;
            }
            int all_done;
            asm volatile("{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
                         "bar.red.and.pred q, 1, 256, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
                         : "=r"(all_done)
                         : "r"(pending)
                         : "memory");
            if (all_done)
                break;
            if (sm.sel_flag[it & 1])
                return false;
            __nanosleep(64);
        }
    }
    if (warp < T) {
        const int t = warp;
        if (a.forced_idx) {
            int e = -1 - lane; // lanes >= K hold distinct non-experts
            if (lane < K) {
                e = a.forced_idx[t * K + lane];
                if (e < 0 || e >= E) {
                    atomicOr(a.status, kErrIndex);
                    e = e < 0 ? 0 : E - 1;
                }
            }
            // a token's experts must be distinct (each expert's job holds at most
            // one column per token): a repeated one is replaced, in lane order,
            // by the smallest index the row does not hold, and reported
            for (int r = 1; r < K; r++) {
                const int er = __shfl_sync(0xFFFFFFFFu, e, r);
                const bool dup = __ballot_sync(0xFFFFFFFFu, lane < r && e == er) != 0u;
                if (dup) {
                    int c = 0;
                    while (__ballot_sync(0xFFFFFFFFu, e == c) != 0u)
                        c++; // ends below E: the row holds K <= E experts
                    if (lane == r)
                        e = c;
                    if (lane == 0)
                        atomicOr(a.status, kErrIndex);
                }
            }
            if (lane < K) {
                sm.sel_idx[t][lane] = e;
                a.idx[t * K + lane] = e;
                a.w[t * K + lane] = a.forced_w[t * K + lane];
            }
        } else {
            select_token(a, io, sm, keys + t * E, t, lane);
        }
    }
    if (threadIdx.x < 32)
        sm.bitmap[threadIdx.x] = 0;
    consumer_sync();
    // grouping (warp 0): distinct experts in ascending order, the pairs of each
    // in pair order. P <= 64 pairs: lane l owns pairs l and l + 32.
    const int P = T * K;
    // pair p = t K + k: t by a multiply-shift, exact for p < 64 and K <= 8
    const unsigned kmagic = (65536u + (unsigned)K - 1u) / (unsigned)K;
    auto tok_of_pair = [&](int p) -> int { return (int)(((unsigned)p * kmagic) >> 16); };
    if (T == 1) {
        // one token: its K experts are distinct; the slot of the k-th chosen
        // expert is its rank among them (ascending expert index, as for more
        // tokens), holding its single pair at that position
        if (warp == 0) {
            const int e = lane < K ? sm.sel_idx[0][lane] : 0x7FFFFFFF;
            int rank = 0;
            for (int j = 0; j < K; j++)
                rank += __shfl_sync(0xFFFFFFFFu, e, j) < e ? 1 : 0;
            if (lane < K) {
                io.inv[lane] = rank;
                atomicAdd(io.counts + e, 1);
                sm.rec[0][rank] = (unsigned)e | (unsigned)rank << 11 | 1u << 18 | (unsigned)K << 22;
                sm.rec[1][rank] = 0u; // token 0
            }
            if (lane == 0)
                *io.nuniq = K;
        }
    } else if (warp == 0) {
        int pe[2];
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int p = lane + 32 * h;
            const int pt = tok_of_pair(p);
            pe[h] = p < P ? sm.sel_idx[pt][p - pt * K] : -1;
            if (pe[h] >= 0)
                atomicOr(&sm.bitmap[pe[h] >> 5], 1u << (pe[h] & 31));
        }
        __syncwarp();
        const unsigned bits = sm.bitmap[lane];
        int incl = __popc(bits);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += v;
        }
        const int nu = __shfl_sync(0xFFFFFFFFu, incl, 31);
        sm.word_prefix[lane] = incl - __popc(bits);
        __syncwarp();
        int slot[2], rank[2];
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int e = pe[h];
            slot[h] = e >= 0 ? sm.word_prefix[e >> 5] + __popc(sm.bitmap[e >> 5] & ((1u << (e & 31)) - 1u)) : 0;
        }
        // rank of a pair among the earlier pairs of its expert: lanes holding the
        // same expert in the same half, plus (second half) the first half's count
        const unsigned lt = (1u << lane) - 1u;
        const unsigned m0 = __match_any_sync(0xFFFFFFFFu, pe[0]);
        const unsigned m1 = __match_any_sync(0xFFFFFFFFu, pe[1]);
        rank[0] = __popc(m0 & lt);
        if (lane < kMaxSlots / 2)
            sm.slot_cnt[lane] = sm.slot_cnt[lane + 32] = 0;
        __syncwarp();
        if (pe[0] >= 0 && rank[0] == 0)
            sm.slot_cnt[slot[0]] = __popc(m0);
        __syncwarp();
        rank[1] = pe[1] >= 0 ? sm.slot_cnt[slot[1]] + __popc(m1 & lt) : 0;
        __syncwarp();
        // pairs per slot: the rank-0 pair of each expert counts its pairs
        if (lane < kMaxSlots / 2)
            sm.slot_cnt[lane] = sm.slot_cnt[lane + 32] = 0;
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; h++)
            if (pe[h] >= 0)
                atomicAdd(&sm.slot_cnt[slot[h]], 1);
        __syncwarp();
        // exclusive scan of the (<= 64) slot counts: lane l sums slots 2l, 2l+1
        const int c0 = sm.slot_cnt[2 * lane], c1 = sm.slot_cnt[2 * lane + 1];
        int pair_incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, pair_incl, o);
            if (lane >= o)
                pair_incl += v;
        }
        const int base = pair_incl - c0 - c1;
        __syncwarp();
        sm.slot_cnt[2 * lane] = base;
        sm.slot_cnt[2 * lane + 1] = base + c0;
        __syncwarp();
        if (lane == 0)
            *io.nuniq = nu;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int p = lane + 32 * h, e = pe[h];
            if (e >= 0) {
                const int pos = sm.slot_cnt[slot[h]] + rank[h];
                io.inv[p] = pos;
                sm.pair_at[pos] = p;
                atomicAdd(io.counts + e, 1);
            }
        }
        __syncwarp();
        // records of slots 2 lane and 2 lane + 1 (slot expert from any of its pairs)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int sl = 2 * lane + h;
            unsigned w0 = (unsigned)nu << 22, w1 = 0u;
            if (sl < nu) {
                const int p0 = sm.slot_cnt[sl], p1 = sl + 1 < nu ? sm.slot_cnt[sl + 1] : P;
                const int pf = sm.pair_at[p0], tf = tok_of_pair(pf);
                w0 |= (unsigned)sm.sel_idx[tf][pf - tf * K] | (unsigned)p0 << 11 | (unsigned)(p1 - p0) << 18;
                for (int i = 0; i < p1 - p0; i++)
                    w1 |= (unsigned)tok_of_pair(sm.pair_at[p0 + i]) << (3 * i);
            }
            if (sl < kMaxSlots) {
                sm.rec[0][sl] = w0;
                sm.rec[1][sl] = w1;
            }
        }
    }
    // Everything the later jobs read (pre-scaled activations, routing outputs,
    // inverse positions) is written; each writer fences, then warp 0 publishes
    // the slot records. A reader that sees a record's epoch sees all of it.
    __threadfence();
    consumer_sync();
    if (warp == 0) {
        const unsigned long long tag = (unsigned long long)io.epoch << 32;
        const int umax = T * K < E ? T * K : E;
        for (int sl = lane; sl < umax; sl += 32) {
            st_relaxed_u64(io.srec + 2 * sl, tag | sm.rec[0][sl]);
            st_relaxed_u64(io.srec + 2 * sl + 1, tag | sm.rec[1][sl]);
        }
    }
    return true;
}

// ---- job space ---------------------------------------------------------------------

struct JobSpace {
    int nR, rows, nSGU, nSD, tilesI, tilesD, Umax;
    int oR, oSGU, oSD, oGU, oD, total;
};

// Job order: SEL, R, SGU, GU, SD, D. The selection is CTA 0's first
// job, so its consumers are idle and waiting when the last router row lands;
// the router rows are the first jobs of the next CTAs (two rows per job while
// both rows' accumulators fit, so that the router is one round of jobs); the
// shared expert's gate/up jobs follow, so that they fill the time in which
// the routing is computed and published. The shared down jobs wait for all of
// those: placed after the routed gate/up jobs they find them done, instead of
// holding CTAs that the routed experts need the moment the routing lands.
__host__ __device__ __forceinline__ JobSpace job_space(int E, int I, int H, int Ish, int T, int K, bool forced) {
    JobSpace s;
    s.rows = T <= 4 ? 2 : 1; // router rows per job: rows * T accumulators per lane (<= 8)
    s.nR = forced ? 0 : (E + s.rows - 1) / s.rows;
    s.nSGU = Ish > 0 ? Ish / 16 : 0;
    s.nSD = Ish > 0 ? H / 16 : 0;
    s.tilesI = I / 16; // GU: one 16-row tile of gate and up
    s.tilesD = H / 32; // D: two 16-row tiles of down
    s.Umax = (T * K < E) ? T * K : E;
    s.oR = 1;
    s.oSGU = s.oR + s.nR;
    s.oGU = s.oSGU + s.nSGU;
    s.oSD = s.oGU + s.Umax * s.tilesI;
    s.oD = s.oSD + s.nSD;
    s.total = s.oD + s.Umax * s.tilesD;
    return s;
}

__device__ __forceinline__ JobSpace job_space(const DecodeArgs &a) {
    return job_space(a.E, a.I, a.H, a.Ish, a.T, a.K, a.forced_idx != nullptr);
}

__device__ __forceinline__ int pad_tp(int n) { return n <= 1 ? 1 : (n <= 2 ? 2 : (n <= 4 ? 4 : 8)); }

// Widest stage W (a multiple of 256 dividing K) whose bytes, at per_col_x16
// sixteenths of a byte per column, fit one ring slot.
__device__ __forceinline__ int pick_w(int K, int per_col_x16) {
    const int nb = K / 256;
    for (int m = nb; m >= 1; m--)
        if (nb % m == 0 && (int64_t)256 * m * per_col_x16 <= (int64_t)16 * kSlotBytes)
            return 256 * m;
    return 256;
}

// Bytes of a 2-bit stage of W columns: two matrices' records, and per token
// the activation rows (hi and lo when split) and their sums, each row padded
// by 16 bytes so that the token rows of a warp's loads fall in different banks.
__device__ __forceinline__ int q2_stage_bytes(int W, int ntok, bool split) {
    return 2 * (W / 256) * kQ2Rec + ntok * ((2 * W + 16) * (split ? 2 : 1) + W / 4 + 16);
}

// Widest such stage (a multiple of 256 dividing K) that fits one ring slot.
__device__ __forceinline__ int pick_w_q2(int K, int ntok, bool split) {
    const int nb = K / 256;
    for (int m = nb; m >= 1; m--)
        if (nb % m == 0 && q2_stage_bytes(256 * m, ntok, split) <= kSlotBytes)
            return 256 * m;
    return 256;
}

// ---- producer (the last warp, all lanes in lockstep) ------------------------------------

// Lays out one stage: put() places a piece that the bulk copies bring in;
// reserve() only sets space aside for a piece the consumers fill themselves
// after their dependency wait (data other CTAs are still producing).
struct StageWriter {
    DecodeSmem &sm;
    int slot = -1; // ring slot, set once claimed
    // Most pieces of one stage: a D stage with 8 tokens has 3 weight pieces and
    // 4 activation pieces per token (hi, lo, offsets, sums) = 35.
    static constexpr int kMaxPieces = 40;
    unsigned off = 0; // layout offset
    unsigned tx = 0;  // bytes brought in by bulk copies
    const void **src;
    unsigned *bytes;
    unsigned *dst;
    int np = 0;
    bool overflow = false;
    __device__ explicit StageWriter(DecodeSmem &s) : sm(s), src(s.pc_src), bytes(s.pc_bytes), dst(s.pc_dst) {}
    __device__ int put(const void *p, unsigned n) {
        const int o = (int)off;
        if (np == kMaxPieces) { // cannot happen with the stage shapes above; never write past the arrays
            overflow = true;
            off += n;
            return o;
        }
        src[np] = p;
        bytes[np] = n;
        dst[np] = off;
        np++;
        off += n;
        tx += n;
        return o;
    }
    // leave n bytes of the stage unwritten (padding)
    __device__ void skip(unsigned n) { off += n; }
    int nindep = -1; // pieces before this index need no dependency wait
    // Pieces put after this call are data other CTAs of this launch are still
    // producing: issue() copies them only after the dependency is met.
    __device__ void dependent_from_here() { nindep = np; }
    // Expect every byte, copy the weights, then (if the stage has dependent
    // pieces) wait for *dep >= target and copy the rest. Returns false if the
    // wait gave up; the stage is then never completed and the consumers drain.
    // Run by the whole producer warp in lockstep (every lane built the same
    // piece list): lane 0 arrives, and lane i issues piece i, so one warp
    // instruction issues up to 32 copies.
    __device__ bool issue(const DecodeArgs &a, const unsigned *dep, unsigned target) {
        const int lane = threadIdx.x & 31;
        uint64_t *bar = &sm.full[slot];
        __syncwarp(); // every lane's writes of the stage description precede the arrival
        if (overflow && lane == 0)
            atomicOr(a.status, kErrInternal);
        if (tx == 0) {
            if (lane == 0)
                mbar_arrive(bar);
            return true;
        }
        if (lane == 0)
            mbar_arrive_tx(bar, tx);
        __syncwarp();
        const int split = nindep < 0 ? np : nindep;
        for (int i = lane; i < split; i += 32)
            bulk_g2s(sm.ring[slot] + dst[i], src[i], bytes[i], bar);
        if (split < np) {
            if (dep && !wait_counter(a, dep, target, false))
                return false;
            // the data was written through the generic proxy by other CTAs; the
            // bulk copies read it through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            for (int i = split + lane; i < np; i += 32)
                bulk_g2s(sm.ring[slot] + dst[i], src[i], bytes[i], bar);
        }
        return true;
    }
};

// The routing record of distinct-expert slot `sl`, polled until it carries this
// launch's epoch (bounded); raw words out.
__device__ bool wait_slot(const DecodeArgs &a, int sl, unsigned &w0, unsigned &w1) {
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        const unsigned long long v0 = ld_acquire_u64(a.srec + 2 * sl);
        const unsigned long long v1 = ld_acquire_u64(a.srec + 2 * sl + 1);
        if ((unsigned)(v0 >> 32) == a.epoch && (unsigned)(v1 >> 32) == a.epoch) {
            w0 = (unsigned)v0;
            w1 = (unsigned)v1;
            return true;
        }
        if ((it & 63) == 0) {
            if (ld_relaxed(a.ctl + kCtlAbort))
                return false;
            const uint64_t now = globaltimer();
            if (it == 0)
                t0 = now;
            else if (now - t0 > kWaitNs) {
                atomicOr(a.status, kErrTimeout);
                atomicExch(a.ctl + kCtlAbort, 1u);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// Every routing record of the launch into shared memory (the selection
// publishes them together): lane l polls slots l, l + 32 (the whole producer
// warp). The acquires order the later bulk copies of data the selection wrote
// before publishing. Returns false if a wait gave up.
__device__ bool load_records(const DecodeArgs &a, const JobSpace &js, DecodeSmem &sm) {
    bool good = true;
    for (int sl = threadIdx.x & 31; sl < js.Umax && good; sl += 32) {
        unsigned w0 = 0, w1 = 0;
        good = wait_slot(a, sl, w0, w1);
        sm.rcache[sl][0] = w0;
        sm.rcache[sl][1] = w1;
    }
    good = __all_sync(0xFFFFFFFFu, good);
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return good;
}

template <bool GAIN> __device__ void producer(const DecodeArgs &a, DecodeSmem &sm, const JobSpace &js) {
    const int lane = threadIdx.x & 31;
    unsigned n = 0;        // stages issued so far
    bool have_recs = false; // the launch's routing records are in sm.rcache
    // claim the next ring slot (waits until the consumers released it)
    auto claim = [&](int &slot) -> bool {
        slot = (int)(n % kRing);
        return mbar_wait(a, &sm.empty[slot], ((n / kRing) & 1u) ^ 1u);
    };
    bool ok = true;
    // the first job of each CTA is its own index; later ones come from the queue.
    // Lane 0 starts the atomic; its value is read (broadcast to the warp, which
    // runs this loop in lockstep) only once the current job's stages are issued,
    // so the round trip overlaps that work.
    auto start_claim = [&]() -> unsigned {
        unsigned v = 0;
        if (lane == 0)
            v = ld_relaxed(a.ctl + kCtlAbort) ? (unsigned)js.total
                                               : gridDim.x + atomicAdd(a.ctl + kCtlJobNext, 1u);
        return v;
    };
    // The consumers run the CTA's first job at once when it needs no stage (the
    // selection, router rows). Behind the selection the CTA takes no job before
    // the routing is published (a router row queued behind it would never run).
    int j_next = (int)blockIdx.x;
    if (j_next == 0) {
        ok = load_records(a, js, sm);
        have_recs = ok;
    }
    if (ok && j_next < js.oSGU)
        j_next = (int)__shfl_sync(0xFFFFFFFFu, start_claim(), 0);
    while (ok) {
        const int j = j_next;
        if (j >= js.total)
            break;
        const unsigned v_next = start_claim(); // the job after this one
        int type, a0 = 0, tile = 0, ntok = a.T, K = a.H, per16 = 0, nu = 0;
        int pos[kDecodeT], tok[kDecodeT]; // (compile-time indices only: registers)
#pragma unroll
        for (int i = 0; i < kDecodeT; i++)
            pos[i] = tok[i] = i < a.T ? i : 0;
        if (j < js.oSGU) { // router rows from the queue: the consumers read them directly
            type = kJobR;
            a0 = (j - js.oR) * js.rows;
            tile = a.E - a0 < js.rows ? a.E - a0 : js.rows; // rows of this job
        } else if (j < js.oGU) {
            type = kJobSgu;
            a0 = j - js.oSGU;
            per16 = 2 * 16 * 17 + 16 * 2 * a.T; // two 8-bit tiles (17/16 B per column each) + bf16 x rows
        } else if (j < js.oSD) {
            type = kJobGu;
            a0 = (j - js.oGU) / js.tilesI;
            tile = (j - js.oGU) % js.tilesI;
        } else if (j < js.oD) {
            type = kJobSd;
            a0 = j - js.oSD;
            K = a.Ish;
            per16 = 16 * 17 + 16 * 4 * a.T; // one 8-bit tile + binary16 hi and lo rows
        } else {
            type = kJobD;
            a0 = (j - js.oD) / js.tilesD;
            tile = (j - js.oD) % js.tilesD;
            K = a.I;
        }
        int e = 0;
        SlotRec rec{};
        if ((type == kJobGu || type == kJobD)) {
            if (!have_recs) {
                if (!load_records(a, js, sm))
                    break;
                have_recs = true;
            }
            rec = unpack_slot(sm.rcache[a0][0], sm.rcache[a0][1]);
            nu = rec.nuniq;
            if (a0 >= nu) { // fewer distinct experts than the bound
                j_next = (int)__shfl_sync(0xFFFFFFFFu, v_next, 0);
                continue;
            }
            e = rec.e;
            ntok = rec.ntok;
            if constexpr (GAIN) {
                // the gains of this job's 32 output rows (one 128-byte line), read by the
                // tile's combine: on their way to L2 long before it
                if (type == kJobD && lane == 0)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.gain + (int64_t)e * a.H + tile * 32));
            }
#pragma unroll
            for (int i = 0; i < kDecodeT; i++) {
                const int ii = i < ntok ? i : 0;
                pos[i] = rec.p0 + ii;
                tok[i] = (int)((rec.toks >> (3 * ii)) & 7u);
            }
        }
        const int W = type == kJobR                        ? 0
                      : (type == kJobGu || type == kJobD) ? pick_w_q2(K, ntok, type == kJobD)
                                                          : pick_w(K, per16);
        const int nsub = type == kJobR ? 1 : K / W;
        for (int sub = 0; sub < nsub && ok; sub++) {
            // the stage is described and its copies listed before its slot is free
            StageDesc &d = sm.pdesc;
            d.type = type;
            d.a0 = a0;
            d.tile = tile;
            d.sub = sub;
            d.nsub = nsub;
            d.c0 = sub * W;
            d.W = W;
            d.ntok = ntok;
            d.tp = pad_tp(ntok);
            d.nuniq = nu;
            for (int i = 0; i < kDecodeT; i++) {
                d.pos[i] = pos[i];
                d.tok[i] = tok[i];
            }
            StageWriter sw(sm);
            const int c0 = sub * W;
            // token of the job's column t (routed jobs: from the routing record)
            auto tok_of = [&](int t) -> int {
                return (type == kJobGu || type == kJobD) ? (int)((rec.toks >> (3 * t)) & 7u) : t;
            };
            if (type == kJobSgu) {
                const Q8Frag *M[2] = {&a.sh_gate, &a.sh_up};
                for (int m = 0; m < 2; m++) {
                    const int64_t u = (int64_t)a0 * M[m]->nbq + c0 / 32;
                    d.oq[m] = sw.put(M[m]->rec + u * kQ8Rec, (unsigned)(W / 32) * kQ8Rec);
                }
                d.act_pitch = 2 * W;
                d.oact = (int)sw.off;
                for (int t = 0; t < a.T; t++)
                    sw.put(a.x + (int64_t)t * a.H + c0, 2u * W);
            } else if (type == kJobSd) {
                const int64_t u = (int64_t)a0 * a.sh_down.nbq + c0 / 32;
                d.oq[0] = sw.put(a.sh_down.rec + u * kQ8Rec, (unsigned)(W / 32) * kQ8Rec);
                d.act_pitch = 2 * W;
                sw.dependent_from_here(); // h of the shared expert: written by the SGU jobs
                d.oact = (int)sw.off;
                for (int t = 0; t < a.T; t++)
                    sw.put(a.hs_hi + (int64_t)t * a.Ish + c0, 2u * W);
                d.olo = (int)sw.off;
                for (int t = 0; t < a.T; t++)
                    sw.put(a.hs_lo + (int64_t)t * a.Ish + c0, 2u * W);
            } else if (type == kJobGu || type == kJobD) {
                // GU: gate and up tile `tile`; D: down tiles 2 tile and 2 tile + 1
                const Q2Frag *M[2] = {type == kJobGu ? &a.gate : &a.down, type == kJobGu ? &a.up : &a.down};
                const int rows_per_e = type == kJobGu ? a.I : a.H;
                for (int m = 0; m < 2; m++) {
                    const int64_t gt = (int64_t)e * (rows_per_e / 16) + (type == kJobGu ? tile : 2 * tile + m);
                    const int64_t u = gt * (M[m]->nkc / 2) + c0 / 256; // first record of the stage
                    d.oq[m] = sw.put(M[m]->rec + u * kQ2Rec, (unsigned)(W / 256) * kQ2Rec);
                }
                // activation rows in the permuted layout: a block of 256 columns is 512
                // contiguous bytes of a row, its 16 sums (hi, lo) 64 bytes
                d.act_pitch = 2 * W + 16;
                d.sub_pitch = W / 4 + 16;
                if (type == kJobGu) {
                    // x rows were written by the selection job, which completed before the
                    // routing was published: safe to copy now
                    d.oact = (int)sw.off;
                    for (int t = 0; t < ntok; t++) {
                        sw.put(a.xq + (int64_t)tok_of(t) * K + c0, 2u * W);
                        sw.skip(16);
                    }
                    d.olo = d.oact;
                    d.osum = (int)sw.off;
                    for (int t = 0; t < ntok; t++) {
                        sw.put(a.xsums + (int64_t)tok_of(t) * (K / 8) + c0 / 8, (unsigned)W / 4u);
                        sw.skip(16);
                    }
                } else {
                    // h rows of this expert: written by its GU jobs
                    sw.dependent_from_here();
                    d.oact = (int)sw.off;
                    for (int t = 0; t < ntok; t++) {
                        sw.put(a.hq_hi + (int64_t)(rec.p0 + t) * K + c0, 2u * W);
                        sw.skip(16);
                    }
                    d.olo = (int)sw.off;
                    for (int t = 0; t < ntok; t++) {
                        sw.put(a.hq_lo + (int64_t)(rec.p0 + t) * K + c0, 2u * W);
                        sw.skip(16);
                    }
                    d.osum = (int)sw.off;
                    for (int t = 0; t < ntok; t++) {
                        sw.put(a.hsums + (int64_t)(rec.p0 + t) * (K / 8) + c0 / 8, (unsigned)W / 4u);
                        sw.skip(16);
                    }
                }
            }
            const unsigned *dep = type == kJobD ? a.ctl + kCtlGuDone + a0 : a.ctl + kCtlSguDone;
            const unsigned target = type == kJobD ? (unsigned)js.tilesI : (unsigned)js.nSGU;
            int slot;
            if (!claim(slot)) {
                ok = false;
                break;
            }
            {
                int *to = reinterpret_cast<int *>(&sm.desc[slot]);
                const int *from = reinterpret_cast<const int *>(&sm.pdesc);
                for (int i = lane; i < (int)(sizeof(StageDesc) / sizeof(int)); i += 32)
                    to[i] = from[i];
            }
            sw.slot = slot;
            n++;
            if (!sw.issue(a, dep, target)) {
                ok = false;
                break;
            }
        }
        j_next = (int)__shfl_sync(0xFFFFFFFFu, v_next, 0);
    }
    // end of this CTA's jobs
    int slot;
    if (claim(slot)) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            sm.desc[slot].type = kJobEnd;
            mbar_arrive(&sm.full[slot]);
        }
    }
}

// ---- consumers (warps 0..7) ----------------------------------------------------------

// y for 32 rows (tile ti) and all tokens, in fixed order: sum over k, then
// shared. The publisher warp, one row per lane: the routing weights and pair
// positions of all tokens go through shared memory in one round trip, then
// the expert outputs of two tokens at a time.
template <bool GAIN> __device__ void combine_tile(const DecodeArgs &a, DecodeSmem &sm, int ti, int lane) {
    const int P = a.T * a.K;
    for (int p = lane; p < P; p += 32) {
        sm.cw[p] = __ldcg(a.w + p);
        sm.cinv[p] = __ldcg(a.inv + p);
        if constexpr (GAIN)
            sm.cexp[p] = __ldcg(a.idx + p);
    }
    __syncwarp();
    const int col = ti * 32 + lane;
    for (int t0 = 0; t0 < a.T; t0 += 2) {
        float ye[2][kMaxTopK], sh[2];
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int t = t0 + u < a.T ? t0 + u : t0;
#pragma unroll
            for (int k = 0; k < kMaxTopK; k++)
                if (k < a.K)
                    ye[u][k] = __ldcg(a.ye + (int64_t)sm.cinv[t * a.K + k] * a.H + col);
            sh[u] = a.Ish > 0 ? __ldcg(a.ysh + (int64_t)t * a.H + col) : 0.f;
            if constexpr (GAIN) {
#pragma unroll
                for (int k = 0; k < kMaxTopK; k++)
                    if (k < a.K)
                        ye[u][k] *= __ldg(a.gain + (int64_t)sm.cexp[t * a.K + k] * a.H + col);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int t = t0 + u;
            if (t < a.T) {
                float v = 0.f;
#pragma unroll
                for (int k = 0; k < kMaxTopK; k++)
                    if (k < a.K)
                        v = fmaf(sm.cw[t * a.K + k], ye[u][k], v);
                if (a.Ish > 0)
                    v += sh[u];
                a.y[(int64_t)t * a.H + col] = v;
            }
        }
    }
}

// Consumer thread 0, after the consumers' barrier that follows a job's result
// writes: hand the job's publication to the publisher warp (a job count to
// increase, or a D job's arrival at its 32-row output tile). The mbarrier
// arrival orders the job's writes before the publisher's GPU-scope release.
// Returns false if the wait for a free task slot gave up.
__device__ bool publish(const DecodeArgs &a, DecodeSmem &sm, unsigned &npub, int kind, unsigned *ctr, int tile,
                        int nuniq) {
    const int s = (int)(npub % kPubQ);
    if (!mbar_wait(a, &sm.pub_empty[s], ((npub / kPubQ) & 1u) ^ 1u))
        return false;
    sm.pub[s].ctr = ctr;
    sm.pub[s].kind = kind;
    sm.pub[s].tile = tile;
    sm.pub[s].nuniq = nuniq;
    mbar_arrive(&sm.pub_full[s]);
    npub++;
    return true;
}

// The publisher warp: makes each job's results visible GPU-wide (one release
// reduction on its count) off the consumers' path; for a D job, counts its
// contribution to the 32-row tile, and the last of the nuniq contributions
// combines the tile once the shared expert's down rows are complete (those
// jobs precede every D job in the queue, so the wait ends).
template <bool GAIN> __device__ void publisher(const DecodeArgs &a, const JobSpace &js, DecodeSmem &sm, int lane) {
    for (unsigned k = 0;; k++) {
        const int s = (int)(k % kPubQ);
        if (!mbar_wait(a, &sm.pub_full[s], (k / kPubQ) & 1u))
            return;
        const int kind = sm.pub[s].kind;
        if (kind == kPubEnd)
            return;
        unsigned *ctr = sm.pub[s].ctr;
        const int tile = sm.pub[s].tile, nuniq = sm.pub[s].nuniq;
        if (kind == kPubSignal) {
            if (lane == 0)
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        } else {
            unsigned last = 0;
            if (lane == 0) {
                __threadfence();
                const unsigned old = atomicAdd(ctr, 1u);
                last = old + 1 == (unsigned)nuniq;
                if (last) {
                    __threadfence();
                    *ctr = 0; // ready for the next launch
                    if (js.nSD > 0 && !wait_counter(a, a.ctl + kCtlSdDone, (unsigned)js.nSD, false))
                        last = 0;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, last, 0))
                combine_tile<GAIN>(a, sm, tile, lane);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.pub_empty[s]);
    }
}

template <int TP> struct JobOps {
    static __device__ void stage(const DecodeArgs &a, const uint8_t *sl, const StageDesc &d, int warp, int lane,
                                 float (&out)[2][2][2]) {
        switch (d.type) {
        case kJobSgu: q8_stage<TP, 2, false, true>(sl, d, warp, lane, out); break;
        case kJobSd: q8_stage<TP, 1, true, false>(sl, d, warp, lane, out); break;
        default: break; // the 2-bit jobs do not depend on the token count (q2_stage)
        }
    }
    // End of a job: combine the warps' partial sums (barrier 1), write the
    // results, barrier 2, then publish (thread 0 / warp 0, without a barrier).
    static __device__ void finish(const DecodeArgs &a, const JobSpace &js, DecodeSmem &sm, const StageDesc &d,
                                  int warp, int lane, float (&out)[2][2][2], unsigned &npub) {
        const int tid = threadIdx.x;
        auto &P = sm.part;
        if (d.type == kJobGu || d.type == kJobD) {
            store_part_q2(sm, warp, lane, out, d.ntok);
        } else if (d.type != kJobSd) {
            reduce_out<TP, 2>(out);
            store_part<TP, 2>(sm, warp, lane, out);
        } else {
            reduce_out<TP, 1>(out);
            store_part<TP, 1>(sm, warp, lane, out);
        }
        consumer_sync();
        if (d.type == kJobSgu) {
            if (tid < 16 * a.T) {
                const int r = tid & 15, t = tid >> 4;
                float gs = 0.f, us = 0.f;
                for (int w = 0; w < kConsumerWarps; w++) {
                    gs += P[w][0][r][t];
                    us += P[w][1][r][t];
                }
                const float hv = silu(gs) * us;
                const __half hi = __float2half_rn(hv);
                const __half lo = __float2half_rn(hv - __half2float(hi));
                const int64_t o = (int64_t)t * a.Ish + d.a0 * 16 + r;
                a.hs_hi[o] = __half_as_ushort(hi);
                a.hs_lo[o] = __half_as_ushort(lo);
            }
            consumer_sync();
            if (tid == 0)
                publish(a, sm, npub, kPubSignal, a.ctl + kCtlSguDone, 0, 0);
        } else if (d.type == kJobGu) {
            // row r of the tile is column k = 16 tile + r of the down matrix: position
            // r of its sub-block j = tile % 16 in block tile / 16
            const int t = tid >> 4, r = tid & 15;
            const int blk = d.tile >> 4, j = d.tile & 15;
            float hs = 0.f;
            if (t < d.ntok) {
                float gs = 0.f, us = 0.f;
                for (int w = 0; w < kConsumerWarps; w++) {
                    gs += P[w][0][r][t];
                    us += P[w][1][r][t];
                }
                const float hv = silu(gs) * us;
                const int e2 = 2 * q2_p(r, j >> 3);
                const float hp = hv * (1.0f / (float)(1 << e2)); // exact: power of two
                const uint32_t hi = f32_to_bf16_bits(hp);
                const float hif = __uint_as_float(hi << 16);
                const uint32_t lo = f32_to_bf16_bits(hp - hif);
                const float lof = __uint_as_float(lo << 16);
                const int64_t o = (int64_t)d.pos[t] * a.I + q2_act_index(d.tile * 16 + r);
                a.hq_hi[o] = (uint16_t)hi;
                a.hq_lo[o] = (uint16_t)lo;
                hs = (hif + lof) * (float)(1 << e2); // the value the down product sees
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) // over the 16 rows: one sub-block of the down columns
                hs += __shfl_xor_sync(0xFFFFFFFFu, hs, o);
            if (t < d.ntok && r == 0) {
                const uint32_t hi = f32_to_bf16_bits(hs);
                const uint32_t lo = f32_to_bf16_bits(hs - __uint_as_float(hi << 16));
                uint16_t *st = a.hsums + (int64_t)d.pos[t] * (a.I / 8);
                st[q2_sum_index(blk, j, 0)] = (uint16_t)hi;
                st[q2_sum_index(blk, j, 1)] = (uint16_t)lo;
            }
            consumer_sync();
            if (tid == 0)
                publish(a, sm, npub, kPubSignal, a.ctl + kCtlGuDone + d.a0, 0, 0);
        } else if (d.type == kJobSd) {
            if (tid < 16 * a.T) {
                const int r = tid & 15, t = tid >> 4;
                float v = 0.f;
                for (int w = 0; w < kConsumerWarps; w++)
                    v += P[w][0][r][t];
                a.ysh[(int64_t)t * a.H + d.a0 * 16 + r] = v;
            }
            consumer_sync();
            if (tid == 0)
                publish(a, sm, npub, kPubSignal, a.ctl + kCtlSdDone, 0, 0);
        } else { // kJobD: rows 32 tile + 16 m + r
            const int t = tid >> 4, r = tid & 15;
            if (t < d.ntok) {
#pragma unroll
                for (int m = 0; m < 2; m++) {
                    float v = 0.f;
                    for (int w = 0; w < kConsumerWarps; w++)
                        v += P[w][m][r][t];
                    a.ye[(int64_t)d.pos[t] * a.H + d.tile * 32 + 16 * m + r] = v;
                }
            }
            consumer_sync();
            if (tid == 0)
                publish(a, sm, npub, kPubTile, a.ctl + kCtlTileCnt + d.tile, d.tile, d.nuniq);
        }
    }
};

// Dispatch on the job's padded token count; a kernel built for at most TPM
// tokens per job holds only the variants it can meet (smaller code, fewer
// registers for the small batches).
template <int TPM>
__device__ __forceinline__ void stage_tp(int tp, const DecodeArgs &a, const uint8_t *sl, const StageDesc &d,
                                         int warp, int lane, float (&out)[2][2][2]) {
    if (TPM == 1 || tp == 1)
        JobOps<1>::stage(a, sl, d, warp, lane, out);
    else if (TPM == 2 || tp == 2)
        JobOps<(TPM >= 2 ? 2 : 1)>::stage(a, sl, d, warp, lane, out);
    else if (TPM == 4 || tp == 4)
        JobOps<(TPM >= 4 ? 4 : 1)>::stage(a, sl, d, warp, lane, out);
    else
        JobOps<TPM>::stage(a, sl, d, warp, lane, out);
}

template <int TPM>
__device__ __forceinline__ void finish_tp(int tp, const DecodeArgs &a, const JobSpace &js, DecodeSmem &sm,
                                          const StageDesc &d, int warp, int lane, float (&out)[2][2][2],
                                          unsigned &npub) {
    if (TPM == 1 || tp == 1)
        JobOps<1>::finish(a, js, sm, d, warp, lane, out, npub);
    else if (TPM == 2 || tp == 2)
        JobOps<(TPM >= 2 ? 2 : 1)>::finish(a, js, sm, d, warp, lane, out, npub);
    else if (TPM == 4 || tp == 4)
        JobOps<(TPM >= 4 ? 4 : 1)>::finish(a, js, sm, d, warp, lane, out, npub);
    else
        JobOps<TPM>::finish(a, js, sm, d, warp, lane, out, npub);
}

template <int TPM> __device__ void consumer(const DecodeArgs &a, DecodeSmem &sm, const JobSpace &js, int warp, int lane) {
    unsigned n = 0, npub = 0;
    float out[2][2][2];
    bool alive = true; // false after a failed dependency wait: drain the ring without computing
    // The CTA's first job is its own index and needs no stage: the selection
    // (its keys in ring slot 0, which the producer leaves alone until the
    // routing is published) or router rows run at once.
    {
        const int j0 = (int)blockIdx.x;
        if (j0 == 0) {
            select_prepare(a, &sm.part[0][0][0][0]);
            if (threadIdx.x < kDecodeT * kMaxTopK)
                (&sm.sel_idx[0][0])[threadIdx.x] = 0;
            consumer_sync();
            alive = job_select(a, a.io, sm, reinterpret_cast<float *>(sm.ring[0]), warp, lane);
        } else if (j0 < js.oSGU) {
            const int a0 = (j0 - js.oR) * js.rows;
            router_rows(a, sm, a0, a.E - a0 < js.rows ? a.E - a0 : js.rows, warp, lane);
        }
    }
    while (true) {
        const int slot = (int)(n % kRing);
        if (!mbar_wait(a, &sm.full[slot], (n / kRing) & 1u))
            break;
        const StageDesc &d = sm.desc[slot];
        const int type = d.type;
        if (type == kJobEnd)
            break;
        if (d.sub == 0) {
#pragma unroll
            for (int i = 0; i < 8; i++)
                (&out[0][0][0])[i] = 0.f;
        }
        if (alive) {
            if (type == kJobR)
                router_rows(a, sm, d.a0, d.tile, warp, lane);
            else if (type == kJobGu)
                q2_stage<2, false>(sm.ring[slot], d, warp, lane, out);
            else if (type == kJobD)
                q2_stage<2, true>(sm.ring[slot], d, warp, lane, out);
            else
                stage_tp<TPM>(d.tp, a, sm.ring[slot], d, warp, lane, out);
        }
        const bool last = d.sub == d.nsub - 1;
        if (last && alive) {
            if (type != kJobR) // (router rows end in router_rows)
                finish_tp<TPM>(d.tp, a, js, sm, d, warp, lane, out, npub);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.empty[slot]);
        n++;
    }
    // every job's publication is queued: tell the publisher warp to stop
    if (threadIdx.x == 0)
        publish(a, sm, npub, kPubEnd, nullptr, 0, 0);
}

// TPM: the largest padded token count of a job in this launch (1, 2, 4 or 8).
template <int TPM, bool GAIN = false>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_fused_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t dsmem[];
    DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>(dsmem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; i++) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumerWarps);
        }
        for (int i = 0; i < kPubQ; i++) {
            mbar_init(&sm.pub_full[i], 1);
            mbar_init(&sm.pub_empty[i], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const JobSpace js = job_space(a);
    if (warp == kConsumerWarps) {
        producer<GAIN>(a, sm, js);
    } else if (warp == kConsumerWarps + 1) {
        publisher<GAIN>(a, js, sm, lane);
    } else {
        consumer<TPM>(a, sm, js, warp, lane);
    }
    // the last CTA out resets the counters for the next launch
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(a.ctl + kCtlFinished, 1u);
        if (done + 1 == gridDim.x) {
            __threadfence();
            if (!ld_acquire(a.ctl + kCtlAbort)) {
                a.ctl[kCtlJobNext] = 0;
                a.ctl[kCtlSguDone] = 0;
                a.ctl[kCtlSdDone] = 0;
                for (int s = 0; s < kMaxSlots; s++)
                    a.ctl[kCtlGuDone + s] = 0;
                __threadfence();
                a.ctl[kCtlFinished] = 0;
            }
        }
    }
}

} // namespace ds4
