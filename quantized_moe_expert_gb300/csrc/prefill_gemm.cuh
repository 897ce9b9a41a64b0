// Prefill expert stage: grouped GEMMs on the 5th-generation tensor cores with
// the quantised weights expanded to bf16 on the fly.
//
// For a batch of many tokens the routed layer is a dense contraction per
// expert ("a grouped GEMM that dequantizes tiles into shared memory as bf16",
// the prefill design of the routed-MoE layer): expert e's gate/up rows times
// the activations of the tokens routed to e, SwiGLU, then the down rows times
// those SwiGLU rows. One kernel template serves the GEMMs of the layer:
//
//   routed gate/up   A = 2-bit gate and up rows of e,  B = e's token rows (x,
//                    gathered into expert-grouped order beforehand),
//                    out = bf16 silu(g) * u in expert-grouped order
//   routed down      A = 2-bit down rows of e,         B = those bf16 rows,
//                    out = fp32 expert outputs in expert-grouped order
//   shared gate/up   A = 8-bit shared gate and up,     B = every x row (binary16),
//                    out = binary16 silu(g) * u
//   shared down      A = 8-bit shared down,            B = those binary16 rows
//   router logits    A = bf16 parts of the router,     B = every x row (K = 3H)
//
// A tile is (group of <= 128 B rows, 128-row m-tile of the expert's matrix):
// D[128 x n] = A[128 x K] * B[n x K]^T, the weights on the M side. The kernel
// is persistent (one CTA per SM, tiles dealt round robin) and warp
// specialised:
//   1 warp      loader: one lane streams each tile's quantised rows, one
//               256-weight block (2-bit) or 64-column step (8-bit, bf16) at
//               a time, into a shared-memory raw ring with bulk copies, and
//               each K step's B rows with a 2D tensor copy (128-byte swizzle,
//               box height 16..128 rows by the tile's n) into the B ring;
//   8 warps     producers: read their row of the raw block from shared
//               memory, expand it to bf16 and write it straight into TMEM
//               with tcgen05.st (A operand stages: row r of the tile is TMEM
//               lane r, bf16 pairs along the columns);
//   2 warps     one lane each issues tcgen05.mma (A from TMEM, B from shared
//               memory, M=128, N = n rounded up to 16, K=16) into its own
//               accumulator - gate and up, or, with one matrix, the partial
//               sums of even and odd K steps - and commits stage releases and
//               finished accumulators to mbarriers (the first also owns the
//               TMEM allocation, all 512 columns). Two issuers keep the
//               tensor core busy where one thread's issue rate would not;
//   4 warps     epilogue: tcgen05.ld the finished accumulators (warp w reads
//               TMEM lanes 32 (w % 4) ..), apply SwiGLU or add the partial
//               sums, store.
// The expanded weights never pass through shared memory, whose bandwidth
// would otherwise bound the small-n tiles. TMEM columns [0, 256) hold the
// two accumulators as two 128-column slots: a tile with n <= 64 uses one
// (so its epilogue overlaps the next tile's MMAs), a wider tile uses both.
// Columns [256, 512) hold the A stages. Every mbarrier wait is bounded; a
// wait that runs out sets the timeout bit of the status word and every role
// of the CTA stops.
//
// 2-bit expansion. For a 16-weight sub-block with scale sc, min m and the
// block's d, dmin: w = (d sc) q - (dmin m). S = d sc and C = dmin m are exact
// in fp32 and rounded once to bf16; each pair of codes becomes an exact bf16
// pair q through a magic-number OR and one packed fma, and a second packed
// fma gives round_bf16(q S - C). 8-bit expansion (binary16 operands: the
// MMA takes both operands in one type, so the shared expert's x and SwiGLU
// rows are binary16 too): each pair of codes becomes the exact binary16 pair q
// through a byte permute under a magic exponent and one packed subtraction,
// and one packed multiply by the block's binary16 scale d gives
// round_f16(d q).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "mx4_experts.cuh"
#include "umma.cuh"

namespace ds4 {
namespace pf {

constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull; // 1 s: far beyond any legitimate wait
constexpr int kBoxes = 4;                   // B box heights 16, 32, 64, 128 rows

enum { kFmtQ2 = 0, kFmtQ8 = 1, kFmtBF16 = 2, kFmtMx4 = 3, kFmtVq = 4 };
// Epilogues: SwiGLU -> bf16 rows; fp32 rows; SwiGLU -> binary16 rows on the FP4
// grid (each 32-row block of a token column is one MX block: the epilogue
// warp's 32 lanes).
// SwiGLU -> binary16 rows, saturating (the down-product operand of the VQ form
// and of the 8-bit shared expert).
enum { kEpiSwiGLU = 0, kEpiF32 = 1, kEpiSwiGLUFp4 = 2, kEpiSwiGLUF16 = 3 };

// Tensor maps of one B matrix (bf16 rows, 128-byte swizzle, box 64 columns x
// 16 << i rows); passed by value as a grid constant.
struct BMaps {
    CUtensorMap m[kBoxes];
};

// Routed tile groups: {expert, first row of the group in B and out, rows, 0}.
struct Args {
    Q2Mat q2[2];
    Q8Mat q8[2];
    BfMat bf[1];
    Mx4Tile mx4[2];
    VqTile vq[2];
    const uint16_t *rgain[2]; // VQ: binary16 gain of every row (all experts) of the A matrices
    const uint8_t *codebook;  // VQ: 2^vq_bits codewords of 8 E4M3 bytes
    int vq_bits;
    int M;                 // rows of one expert's matrix (output features)
    int Kd;                // reduction length
    const int4 *groups;    // routed groups (ignored when dense_n > 0)
    const int32_t *ngroups;
    int dense_n;           // > 0: one dense group of dense_n rows, in n-tiles
    int b_kwrap;           // > 0: B column of reduction index k is k % b_kwrap
    void *out;             // bf16 (SwiGLU) or fp32 rows [group row][ldo]
    int ldo;
    int ksplit;            // > 1: each tile is split over K into ksplit partial tiles (fp32 output
    int64_t out_kstride;   // only), partial s written at out + s * out_kstride
    unsigned *status;
};

#ifndef DS4_PF_PROD_WARPS
#define DS4_PF_PROD_WARPS 8
#endif

template <int FMT, int NA> struct Cfg {
    static constexpr int kProdWarps = DS4_PF_PROD_WARPS; // 8 or 16
    static constexpr int kProdThreads = 32 * kProdWarps;
    static constexpr int kLoadWarp = kProdWarps;           // one loader warp
    static constexpr int kMmaWarp = kProdWarps + 1;        // two issuer warps
    static constexpr int kEpiWarp0 = kProdWarps + 3;       // four epilogue warps
    static constexpr int kThreads = 32 * (kProdWarps + 1 + 2 + 4);
    static constexpr int kNMax = 128;                      // B rows per tile
    static constexpr int kPart = NA * 128 * 64 / kProdThreads; // weights per producer thread per K step
    static constexpr int kPartsPerMat = 64 / kPart;
    static constexpr int kStages = NA == 2 ? 4 : 8;        // A (TMEM) and B (smem) ring depth
    static constexpr int kACols = NA * kTileK / 2;         // TMEM columns of one A stage
    // K steps per raw block: a loader that issues a raw block every K step would bound the kernel
    static constexpr int kSPB = FMT == kFmtQ2 || FMT == kFmtMx4 || FMT == kFmtVq ? 4 : FMT == kFmtQ8 ? 2 : 1;
    static constexpr int kRawMat = FMT == kFmtQ2   ? 8192 + 2048 + 512
                                   : FMT == kFmtQ8 ? 2 * (8192 + 512)
                                   : FMT == kFmtMx4 ? 4 * kMx4TileRec
                                   : FMT == kFmtVq  ? kVqTileRec
                                                    : 16384;
    static constexpr int kRaw = 4;                         // raw ring depth (blocks)
    static constexpr int kBBytes = kNMax * kTileK * 2;     // one B stage
    static constexpr int kRawOffset = kStages * kBBytes;
    static constexpr int kCbOffset = kRawOffset + kRaw * NA * kRawMat; // VQ: the codebook (13-bit size)
    static constexpr int kCbBytes = FMT == kFmtVq ? 8 << 13 : 0;
    static constexpr int kBarOffset = kCbOffset + kCbBytes;
    static constexpr int kSmemBytes = kBarOffset + 512 + 1024; // + barriers + alignment slack
    static_assert(256 + kStages * kACols <= (int)kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// ---- PTX helpers --------------------------------------------------------------

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(umma::smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(umma::smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(umma::smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait for the phase of the given parity. Gives up (false) when the
// CTA's abort flag is raised or after kWaitNs, raising the flag and the
// status bit itself in the latter case.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, volatile unsigned *abort,
                                          unsigned *status) {
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = 0;
    for (unsigned it = 0;; it++) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63) == 0) {
            if (*abort)
                return false;
            const uint64_t now = globaltimer();
            if (it == 0)
                t0 = now;
            else if (now - t0 > kWaitNs) {
                atomicOr(status, kErrTimeout);
                *abort = 1u;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(umma::smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(umma::smem_addr(bar))
                 : "memory");
}

// 2D tensor copy of the box at (x, y) (x = column, a multiple of 8) into shared memory.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3}], [%4];" ::"r"(dst),
                 "l"(map), "r"(x), "r"(y), "r"(umma::smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lop3_or(uint32_t v, uint32_t mask, uint32_t magic) {
    uint32_t r; // (v & mask) | magic
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(magic));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Warp-wide: 32 lanes x 16 columns of TMEM from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// One thread: D[tmem] (+)= A[tmem] * B[smem]^T for one K=16 step.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       bool accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
                 : "memory");
}

// {lo, hi} rounded to bf16, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- quantised row data of one producer thread ----------------------------------
//
// Producer warp w writes TMEM lanes 32 (w % 4) .. + 31, so thread (w, lane)
// owns tile row r = 32 (w % 4) + lane. Unit u = w / 4 picks the part of every
// 64-column K step the thread expands: with two matrices (gate/up) all of
// matrix u, with one matrix the 32-column half u. The thread reads its row's
// share of a raw block from shared memory, where the loader put the block's
// tile-layout pieces (consecutive rows adjacent, so a warp's reads are
// conflict-free).

template <int P> struct RawQ2 { // one 256-weight block, P/16 quarters of 4 sub-blocks each
    uint4 c[P / 16];
    uint32_t sc[P / 16];
    uint32_t dm;
};

template <int P> struct RawQ8 { // two 64-column K steps, per step P weights (one or two 32-weight blocks)
    uint4 c[2][P / 16];
    uint32_t d[2][P > 32 ? 2 : 1];
};

template <int P> struct RawBF { // one 64-column K step: P bf16 of the row
    uint4 c[P / 8];
};

template <int P> struct RawVq { // one 256-column block of the row: 32 indices (48 bytes), plane bits
    uint4 c[3];
    uint32_t plane;
    uint32_t cb;   // shared-memory address of the codebook
    int part;      // first 16-column quarter of each K step owned
};

template <int P> struct RawMx4 { // four 64-column K steps: per step P of the row's weights (P / 32 MX blocks)
    uint4 c[4][P / 32];
    uint32_t sc[4][P / 32]; // their E8M0 bytes
};

// part: first 16-column quarter of the step owned (P = 64: 0, P = 32: 2 * half).
template <int P> __device__ __forceinline__ void read_raw(uint32_t slot, int r, int part, RawQ2<P> &x) {
#pragma unroll
    for (int i = 0; i < P / 16; i++)
        x.c[i] = lds128(slot + ((part + i) * 128 + r) * 16);
    if (P == 64) {
        const uint4 v = lds128(slot + 8192 + r * 16);
        x.sc[0] = v.x;
        x.sc[1] = v.y;
        x.sc[P / 16 - 2] = v.z;
        x.sc[P / 16 - 1] = v.w;
    } else if (P == 32) {
        const uint2 v = lds64(slot + 8192 + r * 16 + (part / 2) * 8);
        x.sc[0] = v.x;
        x.sc[P / 16 - 1] = v.y;
    } else {
        x.sc[0] = lds32(slot + 8192 + r * 16 + part * 4);
    }
    x.dm = lds32(slot + 10240 + r * 4);
}

// 8-bit raw block: the two steps' codes (8192 B each), then their scales (512 B each).
template <int P> __device__ __forceinline__ void read_raw(uint32_t slot, int r, int part, RawQ8<P> &x) {
#pragma unroll
    for (int s = 0; s < 2; s++) {
#pragma unroll
        for (int i = 0; i < P / 16; i++)
            x.c[s][i] = lds128(slot + s * 8192 + ((part + i) * 128 + r) * 16);
        const uint32_t d = lds32(slot + 2 * 8192 + s * 512 + r * 4);
        if (P > 32) {
            x.d[s][0] = d & 0xFFFFu;
            x.d[s][P > 32 ? 1 : 0] = d >> 16;
        } else {
            x.d[s][0] = (d >> (16 * (part / 2))) & 0xFFFFu;
        }
    }
}

template <int P> __device__ __forceinline__ void read_raw(uint32_t slot, int r, int part, RawBF<P> &x) {
#pragma unroll
    for (int i = 0; i < P / 8; i++)
        x.c[i] = lds128(slot + ((2 * part + i) * 128 + r) * 16);
}

template <int P> __device__ __forceinline__ void read_raw(uint32_t slot, int r, int part, RawMx4<P> &x) {
#pragma unroll
    for (int s = 0; s < 4; s++) {
        const uint32_t st = slot + s * kMx4TileRec;
        const uint32_t sw = lds32(st + 2 * 128 * 16 + (r & ~1) * 2) >> (16 * (r & 1)); // the row's two scale bytes
#pragma unroll
        for (int i = 0; i < P / 32; i++) {
            const int half = part / 2 + i;
            x.c[s][i] = lds128(st + (half * 128 + r) * 16);
            x.sc[s][i] = (sw >> (8 * half)) & 0xFFu;
        }
    }
}

template <int P> __device__ __forceinline__ void read_raw(uint32_t slot, int r, int part, RawVq<P> &x) {
#pragma unroll
    for (int c = 0; c < 3; c++)
        x.c[c] = lds128(slot + (c * 128 + r) * 16);
    x.plane = lds32(slot + 3 * 128 * 16 + r * 4);
    x.part = part;
}

// Expand one sub-block word (16 weights, pair p of codes at bits 2p and
// 16 + 2p) into 8 bf16 pairs.
__device__ __forceinline__ void expand_q2_word(uint32_t W, uint32_t S2, uint32_t N2, uint32_t *o) {
    constexpr uint32_t kMagic = 0x43004300u; // bf16 128 in both halves
    const uint32_t W6 = W >> 6, W12 = W >> 12;
    // 128 + q * 4^j  ->  q, exactly
    const uint32_t q0 = hfma2(lop3_or(W, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    const uint32_t q1 = hfma2(lop3_or(W, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    const uint32_t q2 = hfma2(lop3_or(W, 0x00300030u, kMagic), 0x3D803D80u, 0xC100C100u);
    const uint32_t q3 = hfma2(lop3_or(W6, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    const uint32_t q4 = hfma2(lop3_or(W6, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    const uint32_t q5 = hfma2(lop3_or(W6, 0x00300030u, kMagic), 0x3D803D80u, 0xC100C100u);
    const uint32_t q6 = hfma2(lop3_or(W12, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    const uint32_t q7 = hfma2(lop3_or(W12, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    o[0] = hfma2(q0, S2, N2);
    o[1] = hfma2(q1, S2, N2);
    o[2] = hfma2(q2, S2, N2);
    o[3] = hfma2(q3, S2, N2);
    o[4] = hfma2(q4, S2, N2);
    o[5] = hfma2(q5, S2, N2);
    o[6] = hfma2(q6, S2, N2);
    o[7] = hfma2(q7, S2, N2);
}

__device__ __forceinline__ float nib_to_f(uint32_t n) { return __uint_as_float(0x4B000000u | n) - 8388608.0f; }

// K step s (0..3) of the block -> P/2 bf16 pairs.
template <int P> __device__ __forceinline__ void expand_step(const RawQ2<P> &r, int s, uint32_t (&o)[P / 2]) {
    const float d = f16_to_f32(r.dm), dmin = f16_to_f32(r.dm >> 16);
#pragma unroll
    for (int v = 0; v < P / 16; v++) {
        const uint32_t words[4] = {r.c[v].x, r.c[v].y, r.c[v].z, r.c[v].w};
        const uint32_t b = (r.sc[v] >> (8 * s)) & 0xFFu;
        const float S = d * nib_to_f(b & 15u), C = dmin * nib_to_f(b >> 4);
        expand_q2_word(words[s], pack_bf16x2(S, S), pack_bf16x2(-C, -C), o + 8 * v);
    }
}

// Two int8 codes -> the binary16 pair d * q, rounded once. u is the code word
// with every byte's top bit flipped (code + 128); sel picks its bytes j, j + 1
// under the byte 0x64, giving the exact binary16 pair 1152 + q; minus 1152 is
// the exact q, and one packed multiply by the block's binary16 scale d2 (both
// halves) rounds d * q.
__device__ __forceinline__ uint32_t q8_pair_f16(uint32_t u, uint32_t sel, uint32_t d2) {
    uint32_t p, q, r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(u), "r"(0x64646464u), "r"(sel));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(p), "r"(0x64806480u)); // 1152 in both halves
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(q), "r"(d2));
    return r;
}

template <int P> __device__ __forceinline__ void expand_step(const RawQ8<P> &r, int s, uint32_t (&o)[P / 2]) {
#pragma unroll
    for (int v = 0; v < P / 16; v++) {
        const uint32_t d = r.d[s][P > 32 ? v >> 1 : 0] & 0xFFFFu;
        const uint32_t d2 = d | (d << 16);
        const uint32_t w[4] = {r.c[s][v].x, r.c[s][v].y, r.c[s][v].z, r.c[s][v].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t u = w[i] ^ 0x80808080u;
            o[8 * v + 2 * i] = q8_pair_f16(u, 0x4140u, d2);     // bytes 0, 1
            o[8 * v + 2 * i + 1] = q8_pair_f16(u, 0x4342u, d2); // bytes 2, 3
        }
    }
}

template <int P> __device__ __forceinline__ void expand_step(const RawBF<P> &r, int /*s*/, uint32_t (&o)[P / 2]) {
#pragma unroll
    for (int i = 0; i < P / 8; i++) {
        o[4 * i] = r.c[i].x;
        o[4 * i + 1] = r.c[i].y;
        o[4 * i + 2] = r.c[i].z;
        o[4 * i + 3] = r.c[i].w;
    }
}

// MXFP4 block -> binary16 pairs X * e2m1: the hardware E2M1-pair conversion
// (byte j = weights 2j, 2j+1, the even one in the low nibble and the low half)
// and one packed multiply by X (exact while X * 6 and X / 2 are normal or
// subnormal binary16 values: scale bytes 104..141).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{ .reg .b8 t;\n\t"
        "cvt.u8.u32 t, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t; }"
        : "=r"(r)
        : "r"(byte));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <int P> __device__ __forceinline__ void expand_step(const RawMx4<P> &r, int s, uint32_t (&o)[P / 2]) {
#pragma unroll
    for (int i = 0; i < P / 32; i++) {
        const float X = r.sc[s][i] == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(r.sc[s][i] << 23);
        const uint32_t xh = __half_as_ushort(__float2half_rn(X));
        const uint32_t X2 = xh | xh << 16;
        const uint32_t w[4] = {r.c[s][i].x, r.c[s][i].y, r.c[s][i].z, r.c[s][i].w};
#pragma unroll
        for (int j = 0; j < 16; j++)
            o[16 * i + j] = hmul2_f16(e2m1x2_to_f16x2(w[j >> 2] >> (8 * (j & 3))), X2);
    }
}

// Index i (0..31) of a 48-byte index string (12 bits, least significant bit first).
__device__ __forceinline__ uint32_t vq_index12(const uint32_t (&w)[12], int i) {
    const int b = 12 * i, wd = b >> 5, sh = b & 31;
    uint32_t v = w[wd] >> sh;
    if (sh > 20)
        v |= w[wd + 1] << (32 - sh);
    return v & 0xFFFu;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    asm("{ .reg .b16 t;\n\t"
        "cvt.u16.u32 t, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, t; }"
        : "=r"(r)
        : "r"(two));
    return r;
}

// VQ: K step s of the block -> the codewords of the owned indices as binary16
// pairs (E4M3 is exact in binary16). P = 64: the step's 8 indices; P = 32: the
// 4 of the owned half.
template <int N> __device__ __forceinline__ void vq_expand(const uint32_t (&w)[12], uint32_t plane, uint32_t cb,
                                                          int i0, uint32_t *o) {
#pragma unroll
    for (int q = 0; q < N; q++) {
        const int i = i0 + q;
        const uint32_t idx = vq_index12(w, i) | ((plane >> i) & 1u) << 12; // plane bits are 0 in 12-bit layers
        const uint2 cw = lds64(cb + idx * 8);
        o[4 * q] = e4m3x2_to_f16x2(cw.x);
        o[4 * q + 1] = e4m3x2_to_f16x2(cw.x >> 16);
        o[4 * q + 2] = e4m3x2_to_f16x2(cw.y);
        o[4 * q + 3] = e4m3x2_to_f16x2(cw.y >> 16);
    }
}

template <int P> __device__ __forceinline__ void expand_step(const RawVq<P> &r, int s, uint32_t (&o)[P / 2]) {
    const uint32_t w[12] = {r.c[0].x, r.c[0].y, r.c[0].z, r.c[0].w, r.c[1].x, r.c[1].y,
                            r.c[1].z, r.c[1].w, r.c[2].x, r.c[2].y, r.c[2].z, r.c[2].w};
    // the index positions stay compile-time constants (the string is in registers)
    if (P == 64 || r.part == 0)
        vq_expand<P / 8>(w, r.plane, r.cb, 8 * s, o);
    else // part 2: columns 32..63 of the step
        vq_expand<P / 8>(w, r.plane, r.cb, 8 * s + 4, o);
}

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<kFmtQ2> {
    template <int P> using Raw = RawQ2<P>;
};
template <> struct FmtTraits<kFmtQ8> {
    template <int P> using Raw = RawQ8<P>;
};
template <> struct FmtTraits<kFmtBF16> {
    template <int P> using Raw = RawBF<P>;
};
template <> struct FmtTraits<kFmtMx4> {
    template <int P> using Raw = RawMx4<P>;
};
template <> struct FmtTraits<kFmtVq> {
    template <int P> using Raw = RawVq<P>;
};

// The loader's bulk copies of raw block kb of 128-row tile rt of matrix m
// into `dst` (kRawMat bytes); returns the bytes.
__device__ __forceinline__ unsigned copy_raw(const Q2Mat &m, int64_t rt, int kb, uint32_t dst, uint64_t *bar) {
    const int64_t tb = rt * m.nb + kb;
    bulk_g2s(dst, m.qs + tb * 512, 8192, bar);
    bulk_g2s(dst + 8192, m.sc + tb * 128, 2048, bar);
    bulk_g2s(dst + 10240, m.dm + tb * 128, 512, bar);
    return 8192 + 2048 + 512;
}

// 8-bit: raw block kb is K steps 2 kb and 2 kb + 1 (consecutive in both streams).
__device__ __forceinline__ unsigned copy_raw(const Q8Mat &m, int64_t rt, int kb, uint32_t dst, uint64_t *bar) {
    const int64_t ts = rt * m.nks + 2 * kb;
    bulk_g2s(dst, m.qs + ts * 512, 2 * 8192, bar);
    bulk_g2s(dst + 2 * 8192, m.d + ts * 128, 2 * 512, bar);
    return 2 * (8192 + 512);
}

// MXFP4: raw block kb is K steps 4 kb .. 4 kb + 3, four consecutive records.
__device__ __forceinline__ unsigned copy_raw(const Mx4Tile &m, int64_t rt, int kb, uint32_t dst, uint64_t *bar) {
    bulk_g2s(dst, m.rec + (rt * m.nks + 4 * kb) * kMx4TileRec, 4 * kMx4TileRec, bar);
    return 4 * kMx4TileRec;
}

// VQ: raw block kb is the 256-column block kb of tile rt: one record.
__device__ __forceinline__ unsigned copy_raw(const VqTile &m, int64_t rt, int kb, uint32_t dst, uint64_t *bar) {
    bulk_g2s(dst, m.rec + (rt * m.nkb + kb) * kVqTileRec, kVqTileRec, bar);
    return kVqTileRec;
}

__device__ __forceinline__ unsigned copy_raw(const BfMat &m, int64_t rt, int ks, uint32_t dst, uint64_t *bar) {
    bulk_g2s(dst, m.p + (rt * m.nks + ks) * 1024, 16384, bar);
    return 16384;
}

template <int FMT> struct MatOf;
template <> struct MatOf<kFmtQ2> {
    __device__ static const Q2Mat &get(const Args &a, int i) { return a.q2[i]; }
};
template <> struct MatOf<kFmtQ8> {
    __device__ static const Q8Mat &get(const Args &a, int i) { return a.q8[i]; }
};
template <> struct MatOf<kFmtBF16> {
    __device__ static const BfMat &get(const Args &a, int i) { return a.bf[0]; }
};
template <> struct MatOf<kFmtMx4> {
    __device__ static const Mx4Tile &get(const Args &a, int i) { return a.mx4[i]; }
};
template <> struct MatOf<kFmtVq> {
    __device__ static const VqTile &get(const Args &a, int i) { return a.vq[i]; }
};

// ---- tiles ------------------------------------------------------------------------

__device__ __forceinline__ int num_groups(const Args &a, int nmax) {
    return a.dense_n > 0 ? (a.dense_n + nmax - 1) / nmax : *a.ngroups;
}

__device__ __forceinline__ int4 group_at(const Args &a, int g, int nmax) {
    if (a.dense_n > 0)
        return make_int4(0, g * nmax, min(nmax, a.dense_n - g * nmax), 0);
    return a.groups[g];
}

// Accumulator placement of a tile with n_mma columns: a narrow tile
// (n_mma <= 64) takes one 128-column slot (the next one in turn) for its two
// accumulators, a wide tile both slots.
struct AccPlace {
    uint32_t col;    // first accumulator
    uint32_t stride; // columns to the second accumulator
    int slot;        // first slot
    bool wide;
};

__device__ __forceinline__ AccPlace acc_place(int n_mma, int next1) {
    AccPlace p;
    p.wide = n_mma > 64;
    p.slot = p.wide ? 0 : next1;
    p.col = p.wide ? 0u : (uint32_t)(next1 * 128);
    p.stride = p.wide ? 128u : 64u;
    return p;
}

// ---- the kernel -------------------------------------------------------------------

template <int FMT, int NA, int EPI>
__global__ void __launch_bounds__(Cfg<FMT, NA>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ BMaps bm, const Args a) {
    using C = Cfg<FMT, NA>;
    constexpr int kPart = C::kPart;
    using Raw = typename FmtTraits<FMT>::template Raw<kPart>;
    constexpr int kNMax = C::kNMax;
    constexpr int kSPB = C::kSPB;
    constexpr int kStages = C::kStages;
    constexpr int kRaw = C::kRaw;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + kStages;
    uint64_t *rfull = empty + kStages;
    uint64_t *rempty = rfull + kRaw;
    uint64_t *accf = rempty + kRaw;
    uint64_t *acce = accf + 2;
    uint64_t *fin = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile unsigned *abort = reinterpret_cast<volatile unsigned *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(full + s, C::kProdWarps + 1); // one arrival per producer warp + the loader's expect_tx
            mbar_init(empty + s, NA == 2 ? 2 : 1);
        }
        for (int s = 0; s < kRaw; s++) {
            mbar_init(rfull + s, 1);
            mbar_init(rempty + s, C::kProdWarps);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(accf + b, 2);
            mbar_init(acce + b, 4);
        }
        mbar_init(fin, 2);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::kMmaWarp)
        umma::tmem_alloc(tmem_slot, kTmemCols);
    if constexpr (FMT == kFmtVq) { // the codebook, once per CTA
        const int n16 = (8 << a.vq_bits) / 16;
        for (int i = tid; i < n16; i += C::kThreads)
            reinterpret_cast<uint4 *>(smem + C::kCbOffset)[i] = __ldg(reinterpret_cast<const uint4 *>(a.codebook) + i);
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int MT = (a.M + kTileM - 1) / kTileM; // a partial last m-tile only for plain bf16 rows
    const int ksplit = a.ksplit > 1 ? a.ksplit : 1;
    const int nk = a.Kd / kTileK / ksplit; // K steps of one (partial) tile
    const int nblk = nk / kSPB;
    const int ntiles = num_groups(a, kNMax) * MT * ksplit; // tile t: (group, m-tile) t / ksplit, K part t % ksplit
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nsteps = my_tiles * nk;
    const uint32_t smem_base = umma::smem_addr(smem);
    const uint32_t raw_base = smem_base + C::kRawOffset;

    if (warp < C::kProdWarps) {
        // ---------------- producers ----------------
        // Step j (the CTA's tiles' K steps in order) uses ring slot j % kStages;
        // raw block rb (kSPB steps) arrives in raw slot rb % kRaw.
        const int q = warp & 3, u = warp >> 2;
        const int row = 32 * q + lane;
        const int mat = u / C::kPartsPerMat;
        const int part = (u % C::kPartsPerMat) * (kPart / 16); // first quarter of the step owned
        const uint32_t a_lane = tmem + ((uint32_t)(32 * q) << 16) + 256 + mat * (kTileK / 2) + part * 8;
        const int nblocks = nsteps / kSPB;
        for (int rb = 0; rb < nblocks; rb++) {
            const int rs = rb % kRaw;
            if (!mbar_wait(rfull + rs, (rb / kRaw) & 1, abort, a.status))
                break;
            Raw cur;
            read_raw(raw_base + (rs * NA + mat) * C::kRawMat, row, part, cur);
            if constexpr (FMT == kFmtVq)
                cur.cb = smem_base + C::kCbOffset;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(rempty + rs);
            bool ok = true;
#pragma unroll
            for (int s = 0; s < kSPB; s++) {
                const int j = rb * kSPB + s;
                const int slot = j % kStages;
                if (!mbar_wait(empty + slot, ((j / kStages) & 1) ^ 1, abort, a.status)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                uint32_t o[kPart / 2];
                expand_step(cur, s, o);
                const uint32_t ta = a_lane + slot * C::kACols;
                if (kPart == 64) {
                    tmem_st16(ta, *reinterpret_cast<uint32_t(*)[16]>(o));
                    tmem_st16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
                } else if (kPart == 32) {
                    tmem_st16(ta, *reinterpret_cast<uint32_t(*)[16]>(o));
                } else {
                    tmem_st8(ta, *reinterpret_cast<uint32_t(*)[8]>(o));
                }
                tmem_st_wait();
                umma::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(full + slot);
            }
            if (!ok)
                break;
        }
    } else if (warp == C::kLoadWarp) {
        // ---------------- loader ----------------
        // Two cursors over the CTA's tiles: raw blocks run a full raw ring
        // ahead of the B copies, which advance with the MMA's stage releases.
        if (lane == 0) {
            const int nblocks = my_tiles * nblk;
            // raw cursor: global block rb = (tile ordinal r_tl, block r_kb)
            int r_tl = 0, r_kb = 0, r_kb0 = 0;
            int64_t r_rt = 0;
            auto raw_tile = [&]() {
                const int t = (int)blockIdx.x + r_tl * (int)gridDim.x;
                const int tg = t / ksplit;
                const int4 g = group_at(a, tg / MT, kNMax);
                r_rt = (int64_t)g.x * (a.M / kTileM) + tg % MT;
                r_kb0 = (t % ksplit) * nblk;
            };
            auto issue_raw = [&](int rb) -> bool {
                const int rs = rb % kRaw;
                if (!mbar_wait(rempty + rs, ((rb / kRaw) & 1) ^ 1, abort, a.status))
                    return false;
                mbar_arrive_tx(rfull + rs, NA * C::kRawMat);
#pragma unroll
                for (int m = 0; m < NA; m++)
                    copy_raw(MatOf<FMT>::get(a, m), r_rt, r_kb0 + r_kb, raw_base + (rs * NA + m) * C::kRawMat,
                             rfull + rs);
                if (++r_kb == nblk) {
                    r_kb = 0;
                    if (++r_tl < my_tiles)
                        raw_tile();
                }
                return true;
            };
            bool ok = true;
            int rb_next = 0;
            if (nblocks > 0)
                raw_tile();
            for (; rb_next < nblocks && rb_next < kRaw && ok; rb_next++)
                ok = issue_raw(rb_next);
            int j = 0, gb = 0;
            for (int tl = 0; tl < my_tiles && ok; tl++) {
                const int t = (int)blockIdx.x + tl * (int)gridDim.x;
                const int4 g = group_at(a, t / ksplit / MT, kNMax);
                const int n_mma = max(16, (g.z + 15) & ~15);
                const int box = n_mma <= 16 ? 0 : (n_mma <= 32 ? 1 : (n_mma <= 64 ? 2 : 3));
                const unsigned bbytes = (16u << box) * kTileK * 2;
                int col = (t % ksplit) * nk * kTileK;
                if (a.b_kwrap > 0)
                    col %= a.b_kwrap;
                for (int kb = 0; kb < nblk && ok; kb++, gb++) {
                    for (int s = 0; s < kSPB; s++, j++) {
                        const int slot = j % kStages;
                        if (!mbar_wait(empty + slot, ((j / kStages) & 1) ^ 1, abort, a.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_tx(full + slot, bbytes);
                        tma_2d(smem_base + slot * C::kBBytes, &bm.m[box], col, g.y, full + slot);
                        col += kTileK;
                        if (col == a.b_kwrap)
                            col = 0;
                    }
                    // the producers have started block gb: its raw slot is free for gb + kRaw
                    if (ok && rb_next < nblocks) {
                        ok = issue_raw(rb_next);
                        rb_next++;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == C::kMmaWarp || warp == C::kMmaWarp + 1) {
        // ---------------- MMA issuers ----------------
        const int iss = warp - C::kMmaWarp;
        if (lane == 0) {
            int stage = 0;
            unsigned fph = 0;
            unsigned use = 0u; // bit b: parity of the next use of accumulator slot b
            int next1 = 0;     // slot of the next narrow tile
            bool ok = true;
            const uint64_t bdesc0 = umma::desc_sw128(smem_base);
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int4 g = group_at(a, t / ksplit / MT, kNMax);
                const int n_mma = max(16, (g.z + 15) & ~15);
                const AccPlace pl = acc_place(n_mma, next1);
                const bool wide = pl.wide;
                const int s0 = pl.slot;
                if (!mbar_wait(acce + s0, ((use >> s0) & 1u) ^ 1u, abort, a.status))
                    break;
                if (wide && !mbar_wait(acce + 1, ((use >> 1) & 1u) ^ 1u, abort, a.status))
                    break;
                umma::fence_after_sync();
                // MXFP4, VQ and 8-bit: both operands binary16 (the expanded weights and the activations)
                const uint32_t idesc = FMT == kFmtMx4 || FMT == kFmtVq || FMT == kFmtQ8
                                           ? umma::idesc_f16_f32(kTileM, n_mma)
                                           : umma::idesc_bf16_f32(kTileM, n_mma);
                const uint32_t dacc = tmem + pl.col + iss * pl.stride;
                const uint32_t a_off = NA == 2 ? iss * (kTileK / 2) : 0;
                for (int ks = 0; ks < nk; ks++) {
                    if (NA == 2 || (ks & 1) == iss) {
                        if (!mbar_wait(full + stage, fph, abort, a.status)) {
                            ok = false;
                            break;
                        }
                        umma::fence_after_sync();
                        const uint64_t bdesc = bdesc0 + (uint64_t)(stage * (C::kBBytes >> 4));
                        const uint32_t acol = tmem + 256 + stage * C::kACols + a_off;
                        const bool acc = NA == 2 ? ks > 0 : ks > 1;
#pragma unroll
                        for (int kk = 0; kk < kTileK / 16; kk++)
                            mma_ts(dacc, acol + kk * 8, bdesc + 2 * kk, idesc, acc || kk > 0);
                        umma::commit(empty + stage);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        fph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma::commit(accf + s0);
                use ^= 1u << s0;
                if (wide) {
                    umma::commit(accf + 1);
                    use ^= 2u;
                } else {
                    next1 ^= 1;
                }
            }
            // all issued MMAs have completed before TMEM is released
            umma::commit(fin);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(fin, 0)) {
                if (globaltimer() - t0 > kWaitNs) {
                    atomicOr(a.status, kErrTimeout);
                    *abort = 1u;
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        unsigned use = 0u;
        int next1 = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int4 g = group_at(a, t / ksplit / MT, kNMax);
            const int n_mma = max(16, (g.z + 15) & ~15);
            const AccPlace pl = acc_place(n_mma, next1);
            const bool wide = pl.wide;
            const int s0 = pl.slot;
            if (!mbar_wait(accf + s0, (use >> s0) & 1u, abort, a.status))
                break;
            if (wide && !mbar_wait(accf + 1, (use >> 1) & 1u, abort, a.status))
                break;
            umma::fence_after_sync();
            const int mrow = (t / ksplit % MT) * kTileM + 32 * q + lane;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + pl.col;
            for (int c0 = 0; c0 < g.z; c0 += 8) {
                // NA == 2: v[0] gate, v[1] up; NA == 1: the two partial sums, added
                float v[2][8];
#pragma unroll
                for (int m = 0; m < 2; m++) {
                    uint32_t r[8];
                    umma::tmem_ld8(tbase + m * pl.stride + c0, r);
                    umma::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 8; jj++)
                        v[m][jj] = __uint_as_float(r[jj]);
                }
                if (NA == 1) {
#pragma unroll
                    for (int jj = 0; jj < 8; jj++)
                        v[0][jj] += v[1][jj];
                }
                if constexpr (FMT == kFmtVq) { // the rows' gains (expert g.x, row mrow)
#pragma unroll
                    for (int m = 0; m < NA; m++) {
                        const float gr = f16_to_f32(__ldg(a.rgain[m] + (int64_t)g.x * a.M + mrow));
#pragma unroll
                        for (int jj = 0; jj < 8; jj++)
                            v[m][jj] *= gr;
                    }
                }
                if (EPI == kEpiSwiGLUFp4) {
                    // one MX block per token column: this warp's 32 rows (M is a multiple of 128)
                    uint16_t *out = static_cast<uint16_t *>(a.out);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        const float h = silu(v[0][jj]) * v[1][jj];
                        const float amax =
                            __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h))));
                        const uint16_t q = fp4_grid_f16(h, amax);
                        if (c0 + jj < g.z)
                            out[(int64_t)(g.y + c0 + jj) * a.ldo + mrow] = q;
                    }
                } else if (mrow >= a.M) {
                    // rows past a partial last m-tile
                } else if (EPI == kEpiSwiGLUF16) {
                    uint16_t *out = static_cast<uint16_t *>(a.out);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++)
                        if (c0 + jj < g.z)
                            out[(int64_t)(g.y + c0 + jj) * a.ldo + mrow] = f32_to_f16_sat(silu(v[0][jj]) * v[1][jj]);
                } else if (EPI == kEpiSwiGLU) {
                    uint16_t *out = static_cast<uint16_t *>(a.out);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        if (c0 + jj < g.z) {
                            const float h = silu(v[0][jj]) * v[1][jj];
                            out[(int64_t)(g.y + c0 + jj) * a.ldo + mrow] = (uint16_t)(pack_bf16x2(h, 0.f) & 0xFFFFu);
                        }
                    }
                } else {
                    float *out = static_cast<float *>(a.out) + (int64_t)(t % ksplit) * a.out_kstride;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++)
                        if (c0 + jj < g.z)
                            out[(int64_t)(g.y + c0 + jj) * a.ldo + mrow] = v[0][jj];
                }
            }
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce + s0);
            use ^= 1u << s0;
            if (wide) {
                if (lane == 0)
                    mbar_arrive(acce + 1);
                use ^= 2u;
            } else {
                next1 ^= 1;
            }
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

// B rows of the routed gate/up in expert-grouped order: xp[pos] = x[perm[pos] / K];
// one CTA per row.
__global__ void gather_rows_kernel(const uint16_t *x, const int32_t *perm, int K, int H,
                                   uint16_t *xp) {
    pdl_launch_next();
    pdl_wait();
    const int pos = blockIdx.x;
    const int t = perm[pos] / K;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H);
    uint4 *dst = reinterpret_cast<uint4 *>(xp + (int64_t)pos * H);
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x)
        dst[c] = src[c];
}

// ---- routed tile groups -------------------------------------------------------------

// One block of 1024 threads (distinct experts <= 1024). For each distinct
// expert u with rows [uoff[u], uoff[u+1]) emit ceil(rows / nmax) groups of at
// most nmax rows, for two group sizes at once.
__global__ void plan_groups_kernel(const int32_t *uexp, const int32_t *uoff,
                                   const int32_t *nuniq, int nmax_a, int4 *ga,
                                   int32_t *na, int nmax_b, int4 *gb,
                                   int32_t *nb) {
    pdl_launch_next();
    pdl_wait();
    __shared__ int32_t sa[1024], sb[1024];
    const int u = threadIdx.x;
    const int U = *nuniq;
    int e = 0, p0 = 0, cnt = 0;
    if (u < U) {
        e = uexp[u];
        p0 = uoff[u];
        cnt = uoff[u + 1] - p0;
    }
    const int ca = (cnt + nmax_a - 1) / nmax_a, cb = (cnt + nmax_b - 1) / nmax_b;
    sa[u] = ca;
    sb[u] = cb;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive scans
        const int x = u >= o ? sa[u - o] : 0;
        const int y = u >= o ? sb[u - o] : 0;
        __syncthreads();
        sa[u] += x;
        sb[u] += y;
        __syncthreads();
    }
    for (int i = 0; i < ca; i++)
        ga[sa[u] - ca + i] = make_int4(e, p0 + i * nmax_a, min(nmax_a, cnt - i * nmax_a), 0);
    for (int i = 0; i < cb; i++)
        gb[sb[u] - cb + i] = make_int4(e, p0 + i * nmax_b, min(nmax_b, cnt - i * nmax_b), 0);
    if (u == 1023) {
        *na = sa[1023];
        *nb = sb[1023];
    }
}

} // namespace pf

} // namespace ds4
