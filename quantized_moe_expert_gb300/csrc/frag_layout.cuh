// Fragment-major weight layouts for the tensor-core GEMV of the decode path.
//
// A warp multiplies a tile of 16 weight rows by the activations with
// mma.sync.m16n8k16 (A = weights, 16 rows x 16 k per MMA; B = activations,
// 16 k x 8 token columns). The layouts below store each (16-row tile, column
// range) so that lane l = 4*g + tig fetches exactly the bits its A fragment
// needs with 16-byte loads, and a warp's loads cover contiguous 512-byte spans.
//
// 2-bit blocks: one 1344-byte record per (16-row tile, 256-column block) (the
// 84 bytes of each of its 16 rows' blocks). Inside a block the MMA's k index
// is the 16-weight sub-block j and MMA number c (0..15) takes column 16 j + c
// of every sub-block, so lane (g, tig) meets the same sub-blocks
// {2tig, 2tig+1} (fragment registers a0, a1) and {2tig+8, 2tig+9} (a2, a3) of
// rows g and g+8 in all 16 MMAs of a block: their scales are turned into
// multipliers once per block.
//   codes   [0, 1024): lane l's 32 bytes are words W0..W7 (W0..W3 at 16 l,
//           W4..W7 at 512 + 16 l). Words W(2i), W(2i+1) hold MMAs c = 4i..4i+3:
//           each A register (row g + 8 rho, sub-block pair kappa) is two codes
//           at bits s + 2p of the low and high halves of one word (the low half
//           the even sub-block), placed by q2_slot below; one LOP3 with 0x4300
//           makes the bf16 pair 128 + q 4^p exactly (p <= 2). Within an MMA
//           the two rows of a sub-block pair share p, so p(c, kappa) can be
//           undone on the activation side.
//   scales  [1024, 1280): lane l, uint2 {row g, row g+8}; each word holds
//           sc(2tig), sc(2tig+8), m(2tig), m(2tig+8) in nibbles 0..3 and
//           sc(2tig+1), sc(2tig+9), m(2tig+1), m(2tig+9) in nibbles 4..7,
//           so one LOP3 (after a shift of 0, 4, 8 or 12) gives the bf16 pair
//           128 + v for the two sub-blocks of a register.
//   d/dmin  [1280, 1344): entry g (uint2) = the d | dmin << 16 words of rows g
//           and g + 8.
// With the sub-block scale folded in, A = (128 + q 4^p) sc - 128 sc = sc q 4^p
// (one packed bf16 FMA, exact), the activations are x 4^-p (exact), so every
// product is sc q x exactly; the min term sum_j m_j (sum of x over j) is two
// more MMAs per block (m as exact bf16, the sums as a bf16 hi + lo pair).
//
// 8-bit codes, per (tile, bq), bq = 32-column block: lane l holds a uint4
//   { V(g, 0), V(g+8, 0), V(g, 1), V(g+8, 1) }
// where V(row, c) = bytes of `row` at columns 32bq + 16c + 2tig + {0, 1, 8, 9}
// in that order, each XOR 0x80 (the code plus 128). One PRMT with 0x64 bytes
// turns two of them into the binary16 pair 1024 + (q + 128), and subtracting
// 1152 gives q exactly. Scales per (tile, bq): 8 x uint32; entry g holds the
// binary16 d of row g (low half) and row g+8 (high half). Codes and scales of
// a (tile, bq) sit together in one 544-byte record (512 B of codes, 32 B of
// scales), a tile's column range being one contiguous run of records.
#pragma once

#include "common.cuh"

namespace ds4 {

constexpr int kQ2Rec = 1344; // bytes per (16-row tile, 256-column block) record
constexpr int kQ2RecScales = 1024, kQ2RecDm = 1280; // offsets of the scale and d/dmin entries

// Where the two codes of A register (rho, kappa) of MMA c = 4 i + cl live:
// word W(2i + w) shifted right by s, at bit 2p of each half, for row g (rho 0)
// and row g + 8 (rho 1). Every (word, s, p) slot of a word pair is used once.
struct Q2Slot {
    int w0, s0, w1, s1, p;
};
__host__ __device__ constexpr Q2Slot q2_slot(int cl, int kappa) {
    return cl == 0 ? (kappa == 0 ? Q2Slot{0, 0, 0, 6, 0} : Q2Slot{0, 0, 0, 6, 1})
         : cl == 1 ? (kappa == 0 ? Q2Slot{0, 0, 0, 6, 2} : Q2Slot{0, 12, 1, 0, 0})
         : cl == 2 ? (kappa == 0 ? Q2Slot{0, 12, 1, 0, 1} : Q2Slot{1, 0, 1, 6, 2})
                   : (kappa == 0 ? Q2Slot{1, 6, 1, 12, 0} : Q2Slot{1, 6, 1, 12, 1});
}

// Exponent p of the activations of MMA c, sub-block pair kappa (the B side
// carries the factor 4^-p).
__host__ __device__ constexpr int q2_p(int c, int kappa) { return q2_slot(c & 3, kappa).p; }

// Position of column k (0..K) in the permuted activation layout of the decode
// kernel: per 256-column block, per MMA c, per tig: the bf16 pairs of the
// sub-blocks (2tig, 2tig+1) then (2tig+8, 2tig+9). Returns the element index.
__host__ __device__ constexpr int64_t q2_act_index(int64_t k) {
    const int64_t b = k >> 8;
    const int j = (int)((k >> 4) & 15), c = (int)(k & 15);
    const int kappa = j >> 3, tig = (j & 7) >> 1, half = j & 1;
    return (((b * 16 + c) * 4 + tig) * 2 + kappa) * 2 + half;
}

// Position of the sum of sub-block j of block b in the permuted sum layout:
// per block, hi parts then lo parts, each per tig the pairs (2tig, 2tig+1),
// (2tig+8, 2tig+9). part: 0 hi, 1 lo.
__host__ __device__ constexpr int64_t q2_sum_index(int64_t b, int j, int part) {
    const int kappa = j >> 3, tig = (j & 7) >> 1, half = j & 1;
    return ((b * 2 + part) * 4 + tig) * 4 + kappa * 2 + half;
}

constexpr int kQ8Rec = 544;  // bytes per (16-row tile, 32-column block) record
constexpr int kQ8RecD = 512; // offset of the scale entries

struct Q2Frag {
    const uint8_t *rec; // [rows/16][nkc/2] records of kQ2Rec bytes
    int64_t rows;
    int32_t nkc;        // K / 128
};

struct Q8Frag {
    const uint8_t *rec; // [rows/16][nbq] records of kQ8Rec bytes
    int64_t rows;
    int32_t nbq;        // K / 32
};

// Canonical 2-bit block field readers (84-byte blocks, see include/ds4moe.h).
__device__ __forceinline__ const uint8_t *canon_block(const uint8_t *src, int64_t row, int nb, int blk) {
    return src + (row * nb + blk) * kQ2Bytes;
}

__device__ __forceinline__ uint32_t canon_code(const uint8_t *blk, int i) { return (blk[16 + (i >> 2)] >> (2 * (i & 3))) & 3u; }

// One thread per (tile, 256-column block, lane): the lane's code words, its
// scale words and (tig == 0) the d/dmin entry of its row pair.
__global__ void repack_q2_frag_kernel(const uint8_t *__restrict__ src, int64_t rows, int nb, uint8_t *__restrict__ rec) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (rows / 16) * nb * 32;
    if (i >= total)
        return;
    const int lane = (int)(i & 31);
    const int blk = (int)((i >> 5) % nb);
    const int64_t tile = (i >> 5) / nb;
    const int g = lane >> 2, tig = lane & 3;
    const uint8_t *rb[2] = {canon_block(src, tile * 16 + g, nb, blk), canon_block(src, tile * 16 + g + 8, nb, blk)};
    uint8_t *const out = rec + (tile * nb + blk) * kQ2Rec;
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int c = 0; c < 16; c++) {
        const int pair = c >> 2, cl = c & 3;
        for (int kappa = 0; kappa < 2; kappa++) {
            const Q2Slot sl = q2_slot(cl, kappa);
            for (int rho = 0; rho < 2; rho++) {
                const int word = 2 * pair + (rho ? sl.w1 : sl.w0);
                const int bit = (rho ? sl.s1 : sl.s0) + 2 * sl.p;
                for (int half = 0; half < 2; half++) {
                    const int j = 2 * tig + 8 * kappa + half; // sub-block
                    w[word] |= canon_code(rb[rho], 16 * j + c) << (16 * half + bit);
                }
            }
        }
    }
    reinterpret_cast<uint4 *>(out)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(out + 512)[lane] = make_uint4(w[4], w[5], w[6], w[7]);
    uint32_t s[2];
    for (int rho = 0; rho < 2; rho++) {
        const uint8_t *sc = rb[rho]; // scales[16]: low nibble sc, high nibble m
        const uint32_t j0 = sc[2 * tig], j1 = sc[2 * tig + 1], j2 = sc[2 * tig + 8], j3 = sc[2 * tig + 9];
        s[rho] = (j0 & 15u) | (j2 & 15u) << 4 | (j0 >> 4) << 8 | (j2 >> 4) << 12 | (j1 & 15u) << 16 |
                 (j3 & 15u) << 20 | (j1 >> 4) << 24 | (j3 >> 4) << 28;
    }
    reinterpret_cast<uint2 *>(out + kQ2RecScales)[lane] = make_uint2(s[0], s[1]);
    if (tig == 0) {
        const uint8_t *da = rb[0] + 80, *db = rb[1] + 80;
        const uint32_t wa = da[0] | (da[1] << 8) | (da[2] << 16) | ((uint32_t)da[3] << 24);
        const uint32_t wb = db[0] | (db[1] << 8) | (db[2] << 16) | ((uint32_t)db[3] << 24);
        reinterpret_cast<uint2 *>(out + kQ2RecDm)[g] = make_uint2(wa, wb);
    }
}

// One thread per (tile, bq, lane).
__global__ void repack_q8_frag_kernel(const uint8_t *__restrict__ src, int64_t rows, int nbq, uint8_t *__restrict__ rec) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (rows / 16) * nbq * 32;
    if (i >= total)
        return;
    const int lane = (int)(i & 31);
    const int bq = (int)((i >> 5) % nbq);
    const int64_t tile = (i >> 5) / nbq;
    const int g = lane >> 2, tig = lane & 3;
    uint32_t v[4];
#pragma unroll
    for (int h = 0; h < 4; h++) {
        const int64_t row = tile * 16 + g + 8 * (h & 1);
        const int c = h >> 1;
        const uint8_t *q = src + (row * nbq + bq) * kQ8Bytes + 2 + 16 * c + 2 * tig;
        v[h] = ((uint32_t)(q[0] ^ 0x80)) | ((uint32_t)(q[1] ^ 0x80) << 8) | ((uint32_t)(q[8] ^ 0x80) << 16) |
               ((uint32_t)(q[9] ^ 0x80) << 24);
    }
    uint8_t *const rec_blk = rec + (tile * nbq + bq) * kQ8Rec; // this block's record
    reinterpret_cast<uint4 *>(rec_blk)[lane] = make_uint4(v[0], v[1], v[2], v[3]);
    if (lane < 8) {
        const int64_t ra = tile * 16 + lane, rb = ra + 8;
        const uint8_t *da = src + (ra * nbq + bq) * kQ8Bytes;
        const uint8_t *db = src + (rb * nbq + bq) * kQ8Bytes;
        reinterpret_cast<uint32_t *>(rec_blk + kQ8RecD)[lane] =
            (uint32_t)(da[0] | (da[1] << 8)) | ((uint32_t)(db[0] | (db[1] << 8)) << 16);
    }
}

} // namespace ds4
