// Fragment-major weight layouts for the tensor-core GEMV of the decode path.
//
// A warp multiplies a tile of 16 weight rows by the activations with
// mma.sync.m16n8k16 (A = weights, row-major 16x16 per chunk of 16 columns).
// The layouts below store each (16-row tile, column range) so that lane
// l = 4*g + tig fetches exactly the bits its A fragment needs with one 16-byte
// load, and a warp's 32 loads cover one contiguous 512-byte span.
//
// 2-bit codes, per (tile, kc), kc = 128-column chunk: lane l holds a uint4
//   { W(g, G0), W(g+8, G0), W(g, G1), W(g+8, G1) },  G0 = 2kc, G1 = 2kc+1
// where W(row, G) packs the 16 codes of `row` at columns 64G + 16c + 2tig + o
// (+0 and +1), c = 0..3, o in {0, 8}. Register r = 2c + o/8 of the fragment
// takes the code of column k at bit s_r + p_r and of column k+1 at bit
// 16 + s_r + p_r, with (s_r, p_r) = (0,0) (0,2) (0,4) (6,0) (6,2) (6,4) (12,0)
// (12,2). After shifting the word right by s_r, one LOP3
//   (v & (3 << p | 3 << (16 + p))) | 0x3F803F80
// yields the bf16 pair (1 + q_k 2^(p-7), 1 + q_(k+1) 2^(p-7)) exactly.
// The activations are pre-scaled by 2^(7-p) per column, so each product is
// x_k 2^(7-p) + q_k x_k and the per-sub-block offset sum_k x_k 2^(7-p) is
// subtracted in the epilogue.
//
// Scale/min bytes, per (tile, kc): 8 x uint4; entry g holds the 8 scale bytes
// (one per 16-column sub-block of the chunk) of row g (bytes 0-7) and row g+8
// (bytes 8-15). d/dmin, per (tile, 256-column block): 8 x uint2; entry g holds
// the d|dmin word of row g and of row g+8.
// All three sit together, one 1344-byte record per (tile, 256-column block)
// (the 84 bytes of each of its 16 rows' blocks): codes of the block's two
// chunks (2 x 512 B), their scale entries (2 x 128 B), the d/dmin entries
// (64 B). A tile's column range is one contiguous run of records, so a stage
// of one matrix tile is a single bulk copy.
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

__host__ __device__ constexpr int frag_shift(int r) { return r < 3 ? 0 : (r < 6 ? 6 : 12); }
__host__ __device__ constexpr int frag_pos(int r) { return r < 3 ? 2 * r : (r < 6 ? 2 * (r - 3) : 2 * (r - 6)); }

// Pre-scale exponent of column k for the 2-bit fragment: 7 - p of the register
// holding it (depends on k mod 64 only).
__host__ __device__ inline int frag_exp(int k) {
    const int c = (k & 63) >> 4, o = (k & 15) >= 8 ? 1 : 0;
    return 7 - frag_pos(2 * c + o);
}

// Canonical 2-bit block field readers (84-byte blocks, see include/ds4moe.h).
__device__ __forceinline__ int canon_code(const uint8_t *src, int64_t row, int nb, int k) {
    const uint8_t *blk = src + (row * nb + (k >> 8)) * kQ2Bytes;
    const int i = k & 255;
    return (blk[16 + (i >> 2)] >> (2 * (i & 3))) & 3;
}

__device__ __forceinline__ uint32_t canon_word2(const uint8_t *src, int64_t row, int nb, int G, int tig) {
    uint32_t w = 0;
#pragma unroll
    for (int r = 0; r < 8; r++) {
        const int k = 64 * G + 16 * (r >> 1) + 2 * tig + 8 * (r & 1);
        const int b = frag_shift(r) + frag_pos(r);
        w |= (uint32_t)canon_code(src, row, nb, k) << b;
        w |= (uint32_t)canon_code(src, row, nb, k + 1) << (16 + b);
    }
    return w;
}

// One thread per (tile, kc, lane): codes; lanes < 8 also write the scale entry
// of (tile, kc, g = lane); even kc also writes the d/dmin entry of the block.
__global__ void repack_q2_frag_kernel(const uint8_t *__restrict__ src, int64_t rows, int nb, uint8_t *__restrict__ rec) {
    const int nkc = nb * 2;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (rows / 16) * nkc * 32;
    if (i >= total)
        return;
    const int lane = (int)(i & 31);
    const int kc = (int)((i >> 5) % nkc);
    const int64_t tile = (i >> 5) / nkc;
    const int g = lane >> 2, tig = lane & 3;
    const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
    uint8_t *const rec_blk = rec + (tile * nb + (kc >> 1)) * kQ2Rec; // this block's record
    reinterpret_cast<uint4 *>(rec_blk + (kc & 1) * 512)[lane] =
        make_uint4(canon_word2(src, r0, nb, 2 * kc, tig), canon_word2(src, r1, nb, 2 * kc, tig),
                   canon_word2(src, r0, nb, 2 * kc + 1, tig), canon_word2(src, r1, nb, 2 * kc + 1, tig));
    if (lane < 8) {
        const int64_t ra = tile * 16 + lane, rb = ra + 8;
        const int blk = kc >> 1, j0 = (kc & 1) * 8; // 8 sub-blocks of this chunk within the block
        const uint8_t *sa = src + (ra * nb + blk) * kQ2Bytes + j0;
        const uint8_t *sb = src + (rb * nb + blk) * kQ2Bytes + j0;
        uint32_t v[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            v[0] |= (uint32_t)sa[j] << (8 * j);
            v[1] |= (uint32_t)sa[4 + j] << (8 * j);
            v[2] |= (uint32_t)sb[j] << (8 * j);
            v[3] |= (uint32_t)sb[4 + j] << (8 * j);
        }
        reinterpret_cast<uint4 *>(rec_blk + kQ2RecScales + (kc & 1) * 128)[lane] = make_uint4(v[0], v[1], v[2], v[3]);
        if ((kc & 1) == 0) {
            const uint8_t *da = src + (ra * nb + blk) * kQ2Bytes + 80;
            const uint8_t *db = src + (rb * nb + blk) * kQ2Bytes + 80;
            const uint32_t wa = da[0] | (da[1] << 8) | (da[2] << 16) | ((uint32_t)da[3] << 24);
            const uint32_t wb = db[0] | (db[1] << 8) | (db[2] << 16) | ((uint32_t)db[3] << 24);
            reinterpret_cast<uint2 *>(rec_blk + kQ2RecDm)[lane] = make_uint2(wa, wb);
        }
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
