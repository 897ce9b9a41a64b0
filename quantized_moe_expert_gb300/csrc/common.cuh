// Shared device-side definitions of the ds4moe library: the repacked weight
// layout, the handle's scratch, error bits and small helpers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds4moe.h"

namespace ds4 {

constexpr int kQ2Block = 256;      // weights per 2-bit super-block
constexpr int kQ2Sub = 16;         // weights per sub-block (one scale/min nibble pair)
constexpr int kQ2Bytes = 84;       // canonical bytes per 2-bit block
constexpr int kQ8Block = 32;       // weights per 8-bit block
constexpr int kQ8Bytes = 34;       // canonical bytes per 8-bit block
constexpr int kMaxTopK = 8;

// Sticky device error bits (OR-ed into the handle's status word).
constexpr unsigned kErrIndex = 1u << 0;    // a routed index was out of range and was clamped
constexpr unsigned kErrTimeout = 1u << 1;  // a bounded wait gave up
constexpr unsigned kErrInternal = 1u << 2; // an internal consistency check failed

// 2-bit matrix in the prefill kernels' layout: three separately aligned
// streams over (128-row tile rt, 256-weight block b, row r of the tile), so
// that 32 consecutive rows' pieces of one block are adjacent in memory and a
// warp (one lane per row) reads them with 512-byte coalesced loads.
//   codes  16-byte quarter i of (rt, b, r): ((rt * nb + b) * 4 + i) * 128 + r
//   scales 16 bytes of (rt, b, r):           (rt * nb + b) * 128 + r
//   dm     one word of (rt, b, r):           (rt * nb + b) * 128 + r,
//          binary16 d in the low half, dmin in the high half
// Rows are a multiple of 128. Sub-block sb = 4 s + v of a block (s: its
// 64-column step, v: the step's 16-column quarter) is the word s of quarter
// v and scale byte 4 v + s (low nibble scale, high nibble min). Inside the
// word, weight pair p (weights 2p, 2p+1 of the sub-block) sits at bits 2p and
// 16 + 2p, so a mask picks both codes of a pair into the two halves.
struct Q2Mat {
    const uint4 *qs;
    const uint4 *sc;
    const uint32_t *dm;
    int64_t rows;
    int32_t nb; // blocks per row = K / 256
};

// 8-bit matrix in the prefill kernels' layout, per 128-row tile rt and
// 64-column step ks (two 32-weight blocks), consecutive rows adjacent:
//   codes  16-byte quarter i of (rt, ks, r): ((rt * nks + ks) * 4 + i) * 128 + r
//   d      one word of (rt, ks, r):          (rt * nks + ks) * 128 + r,
//          binary16 scale of the first block low, of the second block high
struct Q8Mat {
    const uint4 *qs;
    const uint32_t *d;
    int64_t rows;
    int32_t nks; // K / 64
};

// bf16 matrix in the prefill kernels' layout, per 128-row tile rt and 64-column
// step ks: 16-byte chunk c (columns 8c .. 8c+7) of row r at
// ((rt * nks + ks) * 8 + c) * 128 + r. Rows are padded with zeros to a
// multiple of 128.
struct BfMat {
    const uint4 *p;
    int64_t rows;
    int32_t nks;
};

__device__ __forceinline__ float f16_to_f32(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

// fp32 -> binary16 bits, round to nearest, magnitudes beyond the largest
// finite binary16 saturating to it.
__device__ __forceinline__ uint16_t f32_to_f16_sat(float v) {
    uint16_t h;
    asm("cvt.rn.satfinite.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits) {
    return __uint_as_float((bits & 0xFFFFu) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Programmatic dependent launch. A kernel launched with the programmatic
// stream-serialization attribute may be scheduled while its predecessor in
// the stream still runs: pdl_wait() blocks until that grid has completed and
// its writes are visible (a no-op after an ordinary launch), so it comes before
// the kernel's first global access; pdl_launch_next() lets the next such
// kernel be scheduled early. Only the launch and the prologue overlap.
// Because such a kernel can be resident while every earlier grid of the chain
// still runs, it reaches the data those grids write through pointers without
// __restrict__ (a noalias pointer lets the compiler move a load or a store
// across the wait) and with ordinary loads: the non-coherent path (__ldg, or
// what the compiler makes of a const __restrict__ pointer) is only for data no
// grid writes while the kernel is resident, such as the layer's weights.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float sigmoid(float z) { return 1.0f / (1.0f + expf(-z)); }

// Order-preserving unsigned key of a float (larger float, larger key; -0 and
// +0 share one key; NaN maps to 0, below every number) and its inverse for
// non-NaN keys.
__device__ __forceinline__ unsigned order_key(float v) {
    const unsigned u = v == 0.f ? 0u : __float_as_uint(v);
    if (v != v)
        return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_key_value(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Selection key of a selection score: order_key with NaN moved from 0 to 1,
// so that 0 can mark a taken expert. The selection policy of every kernel:
// larger score first, equal scores (and NaNs among themselves) by lower
// expert index, a NaN score below every number including -inf. Keys of
// numbers are >= order_key(-inf) > 1.
__device__ __forceinline__ unsigned sel_key(float v) { return v == v ? order_key(v) : 1u; }

// The score a selection key stands for (NaN for the NaN key).
__device__ __forceinline__ float sel_key_value(unsigned k) {
    return k > 1u ? order_key_value(k) : __uint_as_float(0x7FC00000u);
}

// Down-gain blocks ("YoungAi - DeepSeek V4.1 Flash on one DGX Spark", sections
// 3 and 4.2): per expert and 32 output channels, 16 bytes of FP4 E2M1 codes
// (channel i at byte i/2, even channel in the low nibble) and one E8M0 scale
// byte; gain i = 1 + 2^(scale - 127) * e2m1(code_i).
constexpr int kGainBlockBytes = 17;

// Twice the E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, one per nibble.
constexpr unsigned kE2M1Twice = 0xC8643210u;

// Gain of channel c (0..31) of the block at blk. Scale byte 0 gives 2^-127,
// which leaves 1 + X * v at 1 in fp32 either way; 0xFF is NaN.
__device__ __forceinline__ float down_gain(const uint8_t *blk, int c) {
    const unsigned code = ((unsigned)__ldg(blk + (c >> 1)) >> ((c & 1) * 4)) & 15u;
    const unsigned sb = __ldg(blk + 16);
    const float X = __uint_as_float(sb == 255u ? 0x7FC00000u : sb << 23);
    const float v = 0.5f * (float)((kE2M1Twice >> (4 * (code & 7u))) & 15u);
    return fmaf(X, (code & 8u) ? -v : v, 1.0f);
}

// Scratch owned by a handle, sized for max_tokens at create time.
// Pair index p = t * K + k names the k-th routed choice of token t.
struct Scratch {
    float *logits;     // [Tmax][E]
    int32_t *idx;      // [Tmax][K] routed experts
    float *w;          // [Tmax][K] mixing weights
    float *gap;        // [Tmax]
    int32_t *counts;   // [E] pairs per expert
    int32_t *offsets;  // [E+1] exclusive scan of counts
    int32_t *uexp;     // [min(E, Tmax*K)] distinct experts in ascending order
    int32_t *uoff;     // [min(E, Tmax*K) + 1] first pair position of each distinct expert
    int32_t *nuniq;    // [1] number of distinct experts
    int32_t *perm;     // [Tmax*K] pair index at each expert-grouped position
    int32_t *inv;      // [Tmax*K] expert-grouped position of each pair
    uint16_t *h;       // [Tmax*K][I] bf16 routed SwiGLU activations, expert-grouped order
    float *ye;         // [Tmax*K][H] routed expert outputs, expert-grouped order
    uint16_t *hsh;     // [Tmax][I_sh] binary16 shared-expert SwiGLU activations
    uint16_t *xp;      // [Tmax*K][H] bf16 token rows in expert-grouped order (routed gate/up B)
    int4 *grp_gu;      // routed tile groups of at most 128 rows (gate/up)
    int4 *grp_dn;      // routed tile groups of at most 256 rows (down)
    int32_t *ngrp;     // [2] number of groups in grp_gu, grp_dn
    float *ysh;        // [Tmax][H]
    uint16_t *xstage;  // [Tmax][H] bf16 staging for host-memory calls
    float *ystage;     // [Tmax][H]
    float *ax;         // VQ layers: [Tmax][H] x in fp32
    uint16_t *x4;      // [Tmax][H] binary16 token rows: on the FP4 grid (MXFP4 routed GEMMs) or x itself (VQ routed
                       // GEMMs, then the shared expert's GEMMs of every layer)
    int8_t *xq;        // MXFP4 layers: [Tmax][H] Q8 codes of the token rows
    float *xd;         // MXFP4 layers: [Tmax][H/32] their block scales
    float *hf;         // MXFP4 and VQ layers: [Tmax*K][I] fp32 SwiGLU rows, expert-grouped order
    int8_t *hq;        // MXFP4 layers: [Tmax*K][I] Q8 codes of the SwiGLU rows
    float *hd;         // MXFP4 layers: [Tmax*K][I/32] their block scales
};

// MXFP4 weights: per row and 32-weight block the 16 E2M1 code bytes as one
// uint4 and the E8M0 scale byte.
struct Mx4Mat {
    const uint4 *codes;   // [rows][nb]
    const uint8_t *scale; // [rows][nb]
    int64_t rows;
    int32_t nb; // 32-weight blocks per row
};

// MXFP4 weights in the prefill GEMM's tile order: one kMx4TileRec-byte record
// per (128-row tile, 64-column step): the 16 code bytes of each row's two
// 32-weight blocks ([block][row][16 B]), then the rows' two E8M0 bytes
// ([row][block]). A loader moves one step of a tile with one bulk copy.
constexpr int kMx4TileRec = 2 * 128 * 16 + 128 * 2;
struct Mx4Tile {
    const uint8_t *rec; // [rows / 128][nks] records
    int64_t rows;
    int32_t nks; // K / 64
};

// VQ weights of one matrix: per expert the index stream, the bit plane
// (13-bit layers) and the binary16 row gains.
struct VqMat {
    const uint32_t *stream; // [E][rows * k * 3 / 64] words
    const uint8_t *plane;   // [E][rows * k / 64] or nullptr
    const uint16_t *gain;   // [E][rows]
    int64_t rows;           // rows per expert
    int32_t k;              // weights per row
};

// VQ indices in the prefill GEMM's tile order: one kVqTileRec-byte record per
// (128-row tile, 256-column block): each row's 32 indices (48 bytes: the index
// stream's bytes for those columns, 12 bits per index, least significant bit
// first) as three 16-byte chunks [chunk][row][16 B], then each row's 32 bit-plane
// bits (13-bit layers) [row][4 B]. Rows run over all experts (expert e's rows at
// e * rows_per_expert).
constexpr int kVqTileRec = 3 * 128 * 16 + 128 * 4;
struct VqTile {
    const uint8_t *rec; // [E * rows / 128][k / 256] records
    int64_t rows;       // rows of all experts
    int32_t nkb;        // k / 256
};

struct LayerDev {
    int H, I, E, K, Ish, Tmax;
    const float *router_w;
    BfMat router_w3; // [E][3H] bf16 (tile layout): hi, mid and lo parts of router_w, which sum to it exactly
    const float *router_bias;
    Q2Mat gate, up, down; // rows: gate/up E*I (K = H), down E*H (K = I)
    Q8Mat sh_gate, sh_up, sh_down;
    const float *gain; // [E][H] per-expert down gains s1 * s2 expanded from the tables, or nullptr
    bool mx4;          // routed experts in MXFP4 (mgate, mup, mdown) instead of 2-bit
    Mx4Mat mgate, mup, mdown;
    Mx4Tile tgate, tup, tdown; // the same weights in the prefill GEMM's tile order
    int vq;            // 12 or 13: routed experts vector-quantised (vgate, vup, vdown, codebook); 0: not
    VqMat vgate, vup, vdown;
    VqTile tvgate, tvup, tvdown; // the same indices in the prefill GEMM's tile order
    const uint8_t *codebook; // [2^vq][8] E4M3
};

} // namespace ds4
