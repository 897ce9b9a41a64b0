// Tile GEMVs of the decode-sized paths (the fused decode kernel and the batch
// kernels): mma.sync.m16n8k16 over the fragment-major records of
// frag_layout.cuh. 2-bit blocks with the sub-block scales folded into the A
// operand; 8-bit blocks as exact binary16 integers with one scale per
// 32-column block.
#pragma once

#include "common.cuh"
#include "frag_layout.cuh"

namespace ds4 {

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t hsub2_1152(uint32_t v) {
    uint32_t r;
    const uint32_t c = 0x64806480u; // binary16 1152 in both halves
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(c));
    return r;
}

// bf16 pair (as u32) -> binary16 pair, round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// fp32 -> bf16 bits, round to nearest even
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float v) {
    uint32_t u = __float_as_uint(v);
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

constexpr uint32_t kBf2Mag = 0x43004300u;   // bf16 pair (128, 128)
constexpr uint32_t kBf2One = 0x3F803F80u;   // (1, 1)
constexpr uint32_t kBf2M128 = 0xC300C300u;  // (-128, -128)
constexpr uint32_t kBf2P16384 = 0x46804680u; // (16384, 16384)

// (v & mask) | (128, 128) as a bf16 pair: 128 + the masked bits
__device__ __forceinline__ uint32_t lop_mag(uint32_t v, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(kBf2Mag));
    return r;
}

__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Multipliers of one block for one matrix: C = (sc, sc') and O = -128 C for
// the four registers (rho, kappa), and the min-term A fragment M.
struct Q2Mult {
    uint32_t C[4], O[4], M[4]; // index 2 kappa + rho: the MMA's a0, a1, a2, a3
};

__device__ __forceinline__ void q2_mult(const uint2 sw, Q2Mult &q) {
#pragma unroll
    for (int rho = 0; rho < 2; rho++) {
        const uint32_t w = rho ? sw.y : sw.x;
#pragma unroll
        for (int kappa = 0; kappa < 2; kappa++) {
            const uint32_t cr = lop_mag(w >> (4 * kappa), 0x000F000Fu);    // 128 + sc
            const uint32_t mr = lop_mag(w >> (8 + 4 * kappa), 0x000F000Fu); // 128 + m
            q.C[2 * kappa + rho] = bf2_fma(cr, kBf2One, kBf2M128);        // sc
            q.O[2 * kappa + rho] = bf2_fma(cr, kBf2M128, kBf2P16384);     // -128 sc
            q.M[2 * kappa + rho] = bf2_fma(mr, kBf2One, kBf2M128);        // m
        }
    }
}

// A register of MMA c (c & 3 == cl) from the lane's word pair (wa, wb) and
// its shifts: the two codes at q2_slot(cl, kappa), row rho.
template <int CL, int KAPPA, int RHO>
__device__ __forceinline__ uint32_t q2_areg(const uint32_t (&sh)[2][3], const Q2Mult &q) {
    constexpr Q2Slot s = q2_slot(CL, KAPPA);
    constexpr int w = RHO ? s.w1 : s.w0;
    constexpr int si = (RHO ? s.s1 : s.s0) / 6;
    const uint32_t raw = lop_mag(sh[w][si], 0x00030003u << (2 * s.p));
    return bf2_fma(raw, q.C[2 * KAPPA + RHO], q.O[2 * KAPPA + RHO]);
}

template <int CL, int NMAT>
__device__ __forceinline__ void q2_mma4(float (&D)[NMAT][4], const uint32_t (&sh)[NMAT][2][3], const Q2Mult (&q)[NMAT],
                                        uint2 b) {
#pragma unroll
    for (int m = 0; m < NMAT; m++)
        mma_bf16(D[m], q2_areg<CL, 0, 0>(sh[m], q[m]), q2_areg<CL, 0, 1>(sh[m], q[m]), q2_areg<CL, 1, 0>(sh[m], q[m]),
                 q2_areg<CL, 1, 1>(sh[m], q[m]), b.x, b.y);
}

// The 2-bit tile GEMV over 256-column blocks [b0, b1) of NMAT 16-row tiles
// that share the activations: rec[m] is matrix m's record of block 0 (records
// of consecutive blocks back to back), xrow / lrow the bf16 activation row of
// this lane's MMA column at block 0 in the permuted layout (hi, and lo when
// SPLIT), srow its sub-block sums at block 0. Per block and matrix the scales
// and mins of the lane's two rows and four sub-blocks become bf16 multipliers
// once; each of the 16 MMAs then builds its A registers with one LOP3 and one
// packed FMA (sc q 4^p, exact); the min term is two MMAs on the hi + lo sums.
// out[m][rho][col] (row g + 8 rho, MMA column 2 tig + col) gains d D - dmin Dm
// per block.
template <int NMAT, bool SPLIT>
__device__ __forceinline__ void q2_gemv(const uint8_t *const (&rec)[NMAT], const uint8_t *xrow, const uint8_t *lrow,
                                        const uint8_t *srow, int b0, int b1, int lane, float (&out)[2][2][2]) {
    const int g = lane >> 2, tig = lane & 3;
    const uint8_t *xa = xrow + 8 * tig;
    const uint8_t *xl = lrow + 8 * tig;
    const uint8_t *xs = srow + 8 * tig;
    for (int b = b0; b < b1; b++) {
        const uint8_t *rb[NMAT];
        Q2Mult q[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; m++) {
            rb[m] = rec[m] + b * kQ2Rec;
            q2_mult(reinterpret_cast<const uint2 *>(rb[m] + kQ2RecScales)[lane], q[m]);
        }
        float D[NMAT][4], Dm[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int i = 0; i < 4; i++)
                D[m][i] = Dm[m][i] = 0.f;
        // min term: m x (sum of the activations over each sub-block), hi and lo parts
        {
            const uint2 shi = *reinterpret_cast<const uint2 *>(xs + 64 * b);
            const uint2 slo = *reinterpret_cast<const uint2 *>(xs + 64 * b + 32);
#pragma unroll
            for (int m = 0; m < NMAT; m++) {
                mma_bf16(Dm[m], q[m].M[0], q[m].M[1], q[m].M[2], q[m].M[3], shi.x, shi.y);
                mma_bf16(Dm[m], q[m].M[0], q[m].M[1], q[m].M[2], q[m].M[3], slo.x, slo.y);
            }
        }
#pragma unroll
        for (int half = 0; half < 2; half++) {
            uint4 qw[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; m++)
                qw[m] = reinterpret_cast<const uint4 *>(rb[m] + 512 * half)[lane];
#pragma unroll
            for (int pr = 0; pr < 2; pr++) {
                uint32_t sh[NMAT][2][3];
#pragma unroll
                for (int m = 0; m < NMAT; m++) {
                    const uint32_t wa = pr ? qw[m].z : qw[m].x, wb = pr ? qw[m].w : qw[m].y;
                    sh[m][0][0] = wa;
                    sh[m][0][1] = wa >> 6;
                    sh[m][0][2] = wa >> 12;
                    sh[m][1][0] = wb;
                    sh[m][1][1] = wb >> 6;
                    sh[m][1][2] = wb >> 12;
                }
                const int c0 = 8 * half + 4 * pr;
                const uint8_t *xb = xa + 32 * (16 * b + c0);
                const uint8_t *lb = xl + 32 * (16 * b + c0);
                q2_mma4<0, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(xb));
                if (SPLIT)
                    q2_mma4<0, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(lb));
                q2_mma4<1, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(xb + 32));
                if (SPLIT)
                    q2_mma4<1, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(lb + 32));
                q2_mma4<2, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(xb + 64));
                if (SPLIT)
                    q2_mma4<2, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(lb + 64));
                q2_mma4<3, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(xb + 96));
                if (SPLIT)
                    q2_mma4<3, NMAT>(D, sh, q, *reinterpret_cast<const uint2 *>(lb + 96));
            }
        }
        // the block's d and dmin
#pragma unroll
        for (int m = 0; m < NMAT; m++) {
            const uint2 dw = reinterpret_cast<const uint2 *>(rb[m] + kQ2RecDm)[g];
            const float dg = f16_to_f32(dw.x), mg = f16_to_f32(dw.x >> 16);
            const float dg8 = f16_to_f32(dw.y), mg8 = f16_to_f32(dw.y >> 16);
            out[m][0][0] += dg * D[m][0] - mg * Dm[m][0];
            out[m][0][1] += dg * D[m][1] - mg * Dm[m][1];
            out[m][1][0] += dg8 * D[m][2] - mg8 * Dm[m][2];
            out[m][1][1] += dg8 * D[m][3] - mg8 * Dm[m][3];
        }
    }
}

// The 8-bit tile GEMV over 32-column blocks [b0, b1) of NMAT 16-row tiles that
// share the activations, eight columns (tokens) per MMA: rec[m] is matrix m's
// record of block 0 (records of consecutive blocks back to back), xrow the
// activation row of this lane's MMA column at block 0 (bf16 when FROM_BF16,
// converted to binary16 here; else binary16), lrow its low part when SPLIT.
// A = the codes as exact binary16 integers (one PRMT, one subtraction); per
// block the two MMAs' sum is scaled by the row's d. out[m][rho][col] (row
// g + 8 rho, MMA column 2 tig + col) gains d D per block.
template <int NMAT, bool SPLIT, bool FROM_BF16>
__device__ __forceinline__ void q8_gemv(const uint8_t *const (&rec)[NMAT], const uint8_t *xrow, const uint8_t *lrow,
                                        int b0, int b1, int lane, float (&out)[2][2][2]) {
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t *act = reinterpret_cast<const uint32_t *>(xrow) + tig;
    const uint32_t *act_lo = reinterpret_cast<const uint32_t *>(lrow) + tig;
    for (int b = b0; b < b1; b++) {
        float D[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int i = 0; i < 4; i++)
                D[m][i] = 0.f;
        uint4 q[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
            q[m] = reinterpret_cast<const uint4 *>(rec[m] + b * kQ8Rec)[lane];
#pragma unroll
        for (int c = 0; c < 2; c++) {
            // columns 32 b + 16 c + 2 tig + {0, 1} and + {8, 9}: words (16 b + 8 c) + tig and + 4
            uint32_t bx0 = act[16 * b + 8 * c], bx1 = act[16 * b + 8 * c + 4];
            if (FROM_BF16) {
                bx0 = bf16x2_to_f16x2(bx0);
                bx1 = bf16x2_to_f16x2(bx1);
            }
            uint32_t lx0 = 0u, lx1 = 0u;
            if (SPLIT) {
                lx0 = act_lo[16 * b + 8 * c];
                lx1 = act_lo[16 * b + 8 * c + 4];
            }
#pragma unroll
            for (int m = 0; m < NMAT; m++) {
                const uint32_t vg = c ? q[m].z : q[m].x, vg8 = c ? q[m].w : q[m].y;
                const uint32_t a0 = hsub2_1152(prmt(vg, 0x64646464u, 0x4140u));
                const uint32_t a1 = hsub2_1152(prmt(vg8, 0x64646464u, 0x4140u));
                const uint32_t a2 = hsub2_1152(prmt(vg, 0x64646464u, 0x4342u));
                const uint32_t a3 = hsub2_1152(prmt(vg8, 0x64646464u, 0x4342u));
                mma_f16(D[m], a0, a1, a2, a3, bx0, bx1);
                if (SPLIT)
                    mma_f16(D[m], a0, a1, a2, a3, lx0, lx1);
            }
        }
#pragma unroll
        for (int m = 0; m < NMAT; m++) {
            const uint32_t dw = reinterpret_cast<const uint32_t *>(rec[m] + b * kQ8Rec + kQ8RecD)[g];
            const float dg = f16_to_f32(dw), dg8 = f16_to_f32(dw >> 16);
            out[m][0][0] = fmaf(dg, D[m][0], out[m][0][0]);
            out[m][0][1] = fmaf(dg, D[m][1], out[m][0][1]);
            out[m][1][0] = fmaf(dg8, D[m][2], out[m][1][0]);
            out[m][1][1] = fmaf(dg8, D[m][3], out[m][1][1]);
        }
    }
}

} // namespace ds4
