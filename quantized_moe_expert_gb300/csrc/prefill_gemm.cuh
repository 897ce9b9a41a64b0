// Prefill expert stage: grouped GEMMs on the 5th-generation tensor cores with
// the quantised weights expanded to bf16 in shared memory on the fly.
//
// For a batch of many tokens the routed layer is a dense contraction per
// expert ("a grouped GEMM that dequantizes tiles into shared memory as bf16",
// the prefill design of the routed-MoE layer): expert e's gate/up rows times
// the activations of the tokens routed to e, SwiGLU, then the down rows times
// those SwiGLU rows. One kernel template serves the four GEMMs of the layer:
//
//   routed gate/up   A = 2-bit gate and up rows of e,  B = x rows of e's tokens,
//                    out = bf16 silu(g) * u in expert-grouped order
//   routed down      A = 2-bit down rows of e,         B = those bf16 rows,
//                    out = fp32 expert outputs in expert-grouped order
//   shared gate/up   A = 8-bit shared gate and up,     B = every x row
//   shared down      A = 8-bit shared down,            B = the shared SwiGLU rows
//
// A tile is (group, 128-row m-tile): D[128 x n] = A[128 x K] * B[n x K]^T with
// n <= 128 tokens (two accumulators, gate and up) or n <= 256 (one). The
// kernel is persistent (one CTA per SM, tiles dealt round robin) and warp
// specialised:
//   warps 0-7   producers: load the quantised rows of the tile (one 256-weight
//               block ahead in registers), expand 128 x 64 bf16 A tiles into
//               a 4-stage ring in the 128-byte-swizzled K-major layout, and
//               copy the B rows of the stage with cp.async;
//   warp 8      allocates TMEM (512 columns = two accumulator sets) and one
//               lane issues tcgen05.mma (M=128, N=n rounded up to 16, K=16)
//               and commits stage releases and finished accumulators to
//               mbarriers;
//   warps 9-12  epilogue: tcgen05.ld the finished accumulator (warp w reads
//               TMEM lanes 32 (w % 4) ..), apply SwiGLU or nothing, store.
// With two accumulator sets the epilogue of one tile overlaps the MMAs of
// the next. Every mbarrier wait is bounded; a wait that runs out sets the
// timeout bit of the status word and every role of the CTA stops.
//
// 2-bit expansion. For a 16-weight sub-block with scale sc, min m and the
// block's d, dmin: w = (d sc) q - (dmin m). S = d sc and C = dmin m are exact
// in fp32 and rounded once to bf16; each pair of codes becomes an exact bf16
// pair q through a magic-number OR and one packed fma, and a second packed
// fma gives round_bf16(q S - C). 8-bit expansion: w = round_bf16(d q), d q
// exact in fp32.
#pragma once

#include "common.cuh"
#include "umma.cuh"

namespace ds4 {
namespace pf {

constexpr int kStages = 4;
constexpr int kProdWarps = 8;
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kMmaWarp = kProdWarps;
constexpr int kEpiWarp0 = kProdWarps + 1;
constexpr int kThreads = 32 * (kProdWarps + 1 + 4);
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull; // 1 s: far beyond any legitimate wait

enum { kFmtQ2 = 0, kFmtQ8 = 1 };
enum { kEpiSwiGLU = 0, kEpiF32 = 1 };

// Routed tile groups: {expert, first expert-grouped position, rows, 0}.
struct Args {
    Q2Mat q2[2];
    Q8Mat q8[2];
    int M;                 // rows of one expert's matrix (output features)
    int Kd;                // reduction length
    const int4 *groups;    // routed groups (ignored when dense_n > 0)
    const int32_t *ngroups;
    int dense_n;           // > 0: one dense group of dense_n rows, in n-tiles
    const uint16_t *b;     // bf16 B rows [..][ldb]
    int ldb;
    const int32_t *bmap;   // nullable: B row of position p is bmap[p] / bmap_div
    int bmap_div;
    void *out;             // bf16 (SwiGLU) or fp32 rows [position][ldo]
    int ldo;
    unsigned *status;
};

template <int NA> struct Cfg {
    static constexpr int kNMax = NA == 2 ? 128 : 256;
    static constexpr int kABytes = kTileM * kTileK * 2;
    static constexpr int kBBytes = kNMax * kTileK * 2;
    static constexpr int kStageBytes = NA * kABytes + kBBytes;
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOffset + 256 + 1024; // + barriers + alignment slack
    static constexpr int kAccStride = 256;                     // TMEM columns per accumulator set
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
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

// {lo, hi} rounded to bf16, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- quantised row data of one producer thread ----------------------------------
//
// Producer thread tid owns row (tid >> 1) of the m-tile and half (tid & 1) of
// every 64-column K step, in each of the NA matrices.

struct RawQ2 { // one 256-weight block, this thread's half: 8 sub-blocks
    uint4 c0, c1;
    uint2 sc;
    uint32_t dm;
};

struct RawQ8 { // one 64-column K step, this thread's half: one 32-weight block
    uint4 c0, c1;
    uint32_t d;
};

__device__ __forceinline__ void load_raw(const Q2Mat &m, int64_t row, int kb, int half, RawQ2 &r) {
    const int64_t blk = row * m.nb + kb;
    const uint4 *q = reinterpret_cast<const uint4 *>(m.qs + blk * 64 + half * 32);
    r.c0 = __ldg(q);
    r.c1 = __ldg(q + 1);
    r.sc = __ldg(reinterpret_cast<const uint2 *>(m.sc + blk * 16 + half * 8));
    r.dm = __ldg(m.dm + blk);
}

__device__ __forceinline__ void load_raw(const Q8Mat &m, int64_t row, int ks, int half, RawQ8 &r) {
    const int blk = 2 * ks + half;
    const uint4 *q = reinterpret_cast<const uint4 *>(m.qs + row * m.k + blk * 32);
    r.c0 = __ldg(q);
    r.c1 = __ldg(q + 1);
    r.d = __ldg(m.d + row * (m.k / 32) + blk);
}

// Expand one sub-block word (16 weights, pair p of codes at bits 2p and
// 16 + 2p) into 8 bf16 pairs.
__device__ __forceinline__ void expand_q2_word(uint32_t W, uint32_t S2, uint32_t N2, uint32_t (&o)[8]) {
    constexpr uint32_t kMagic = 0x43004300u; // bf16 128 in both halves
    const uint32_t W6 = W >> 6, W12 = W >> 12;
    // 128 + q * 4^j  ->  q, exactly
    uint32_t q0 = hfma2(lop3_or(W, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    uint32_t q1 = hfma2(lop3_or(W, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    uint32_t q2 = hfma2(lop3_or(W, 0x00300030u, kMagic), 0x3D803D80u, 0xC100C100u);
    uint32_t q3 = hfma2(lop3_or(W6, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    uint32_t q4 = hfma2(lop3_or(W6, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    uint32_t q5 = hfma2(lop3_or(W6, 0x00300030u, kMagic), 0x3D803D80u, 0xC100C100u);
    uint32_t q6 = hfma2(lop3_or(W12, 0x00030003u, kMagic), 0x3F803F80u, 0xC300C300u);
    uint32_t q7 = hfma2(lop3_or(W12, 0x000C000Cu, kMagic), 0x3E803E80u, 0xC200C200u);
    o[0] = hfma2(q0, S2, N2);
    o[1] = hfma2(q1, S2, N2);
    o[2] = hfma2(q2, S2, N2);
    o[3] = hfma2(q3, S2, N2);
    o[4] = hfma2(q4, S2, N2);
    o[5] = hfma2(q5, S2, N2);
    o[6] = hfma2(q6, S2, N2);
    o[7] = hfma2(q7, S2, N2);
}

// K step s (0..3) of the block in r -> chunks 4 half .. 4 half + 3 of row `row`.
__device__ __forceinline__ void expand_step(const RawQ2 &r, int s, int row, int half, uint32_t a_tile) {
    const float d = f16_to_f32(r.dm), dmin = f16_to_f32(r.dm >> 16);
    const uint32_t words[8] = {r.c0.x, r.c0.y, r.c0.z, r.c0.w, r.c1.x, r.c1.y, r.c1.z, r.c1.w};
    const uint32_t scw = s < 2 ? r.sc.x : r.sc.y;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t b = (scw >> (16 * (s & 1) + 8 * j)) & 0xFFu;
        const float S = d * (float)(b & 15u), C = dmin * (float)(b >> 4);
        const uint32_t S2 = pack_bf16x2(S, S), N2 = pack_bf16x2(-C, -C);
        uint32_t o[8];
        expand_q2_word(words[2 * s + j], S2, N2, o);
        const int c = 4 * half + 2 * j;
        sts128(a_tile + umma::sw128_offset(row, c), o[0], o[1], o[2], o[3]);
        sts128(a_tile + umma::sw128_offset(row, c + 1), o[4], o[5], o[6], o[7]);
    }
}

__device__ __forceinline__ float s8_to_f(uint32_t byte) {
    // (byte ^ 0x80) is the code + 128; 2^23 + that, minus 2^23 + 128, is exact.
    return __uint_as_float(0x4B000000u | ((byte ^ 0x80u) & 0xFFu)) - 8388736.0f;
}

__device__ __forceinline__ uint32_t q8_pair(uint32_t w, int j, float d) {
    return pack_bf16x2(d * s8_to_f(w >> (16 * j)), d * s8_to_f(w >> (16 * j + 8)));
}

__device__ __forceinline__ void expand_step(const RawQ8 &r, int /*s*/, int row, int half, uint32_t a_tile) {
    const float d = f16_to_f32(r.d);
    const uint32_t w[8] = {r.c0.x, r.c0.y, r.c0.z, r.c0.w, r.c1.x, r.c1.y, r.c1.z, r.c1.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t a = w[2 * i], b = w[2 * i + 1];
        sts128(a_tile + umma::sw128_offset(row, 4 * half + i), q8_pair(a, 0, d), q8_pair(a, 1, d), q8_pair(b, 0, d),
               q8_pair(b, 1, d));
    }
}

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<kFmtQ2> {
    using Raw = RawQ2;
    static constexpr int kStepsPerBlk = 4;
    __device__ static const Q2Mat &mat(const Args &a, int i) { return a.q2[i]; }
};
template <> struct FmtTraits<kFmtQ8> {
    using Raw = RawQ8;
    static constexpr int kStepsPerBlk = 1;
    __device__ static const Q8Mat &mat(const Args &a, int i) { return a.q8[i]; }
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

// ---- the kernel -------------------------------------------------------------------

template <int FMT, int NA, int EPI>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const Args a) {
    using C = Cfg<NA>;
    using Tr = FmtTraits<FMT>;
    using Raw = typename Tr::Raw;
    constexpr int kNMax = C::kNMax;
    constexpr int kSPB = Tr::kStepsPerBlk;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + kStages;
    uint64_t *accf = empty + kStages;
    uint64_t *acce = accf + 2;
    uint64_t *fin = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile unsigned *abort = reinterpret_cast<volatile unsigned *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(full + s, kProdThreads);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, 128);
        }
        mbar_init(fin, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp)
        umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int MT = a.M / kTileM;
    const int nk = a.Kd / kTileK;
    const int nblk = nk / kSPB;
    const int ntiles = num_groups(a, kNMax) * MT;
    const uint32_t smem_base = umma::smem_addr(smem);

    if (warp < kProdWarps) {
        // ---------------- producers ----------------
        const int row = tid >> 1, half = tid & 1;
        const int bc = tid & 7;                 // B chunk column of this thread
        constexpr int kBRows = kNMax / 32;      // B rows per thread per stage
        int stage = 0;
        unsigned eph = 1;
        int t = blockIdx.x, kb = 0;
        int4 gcur = make_int4(0, 0, 0, 0);
        Raw nxt[NA];
        if (t < ntiles) {
            gcur = group_at(a, t / MT, kNMax);
            const int64_t grow = (int64_t)gcur.x * a.M + (t % MT) * kTileM + row;
#pragma unroll
            for (int m = 0; m < NA; m++)
                load_raw(Tr::mat(a, m), grow, 0, half, nxt[m]);
        }
        int brow[kBRows];
        bool ok = true;
        while (t < ntiles && ok) {
            Raw cur[NA];
#pragma unroll
            for (int m = 0; m < NA; m++)
                cur[m] = nxt[m];
            const int4 g = gcur;
            if (kb == 0) { // B row sources of this tile
#pragma unroll
                for (int i = 0; i < kBRows; i++) {
                    const int n = (tid >> 3) + 32 * i;
                    int r = -1;
                    if (n < g.z) {
                        const int p = g.y + n;
                        r = a.bmap ? __ldg(a.bmap + p) / a.bmap_div : p;
                    }
                    brow[i] = r;
                }
            }
            // prefetch the next block (possibly of the next tile)
            int t2 = t, kb2 = kb + 1;
            if (kb2 == nblk) {
                kb2 = 0;
                t2 += gridDim.x;
                if (t2 < ntiles)
                    gcur = group_at(a, t2 / MT, kNMax);
            }
            if (t2 < ntiles) {
                const int64_t grow = (int64_t)gcur.x * a.M + (t2 % MT) * kTileM + row;
#pragma unroll
                for (int m = 0; m < NA; m++)
                    load_raw(Tr::mat(a, m), grow, kb2, half, nxt[m]);
            }
#pragma unroll
            for (int s = 0; s < kSPB; s++) {
                const int ks = kb * kSPB + s;
                if (!mbar_wait(empty + stage, eph, abort, a.status)) {
                    ok = false;
                    break;
                }
                const uint32_t st_base = smem_base + stage * C::kStageBytes;
                const uint32_t b_tile = st_base + NA * C::kABytes;
#pragma unroll
                for (int i = 0; i < kBRows; i++)
                    if (brow[i] >= 0)
                        cp_async16(b_tile + umma::sw128_offset((tid >> 3) + 32 * i, bc),
                                   a.b + (int64_t)brow[i] * a.ldb + ks * kTileK + bc * 8);
#pragma unroll
                for (int m = 0; m < NA; m++)
                    expand_step(cur[m], s, row, half, st_base + m * C::kABytes);
                cp_async_wait_all();
                umma::fence_smem_to_async();
                mbar_arrive(full + stage);
                if (++stage == kStages) {
                    stage = 0;
                    eph ^= 1u;
                }
            }
            t = t2;
            kb = kb2;
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int stage = 0;
            unsigned fph = 0;
            unsigned use = 0u; // bit b: parity of the next use of accumulator set b
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, it++) {
                const int b = it & 1;
                if (!mbar_wait(acce + b, ((use >> b) & 1u) ^ 1u, abort, a.status))
                    break;
                umma::fence_after_sync();
                const int4 g = group_at(a, t / MT, kNMax);
                const int n_mma = max(16, (g.z + 15) & ~15);
                const uint32_t idesc = umma::idesc_bf16_f32(kTileM, n_mma);
                for (int ks = 0; ks < nk; ks++) {
                    if (!mbar_wait(full + stage, fph, abort, a.status)) {
                        ok = false;
                        break;
                    }
                    umma::fence_after_sync();
                    const uint32_t st_base = smem_base + stage * C::kStageBytes;
                    const uint64_t bdesc = umma::desc_sw128(st_base + NA * C::kABytes);
#pragma unroll
                    for (int m = 0; m < NA; m++) {
                        const uint64_t adesc = umma::desc_sw128(st_base + m * C::kABytes);
                        const uint32_t d_tmem = tmem + b * C::kAccStride + m * 128;
#pragma unroll
                        for (int kk = 0; kk < kTileK / 16; kk++)
                            umma::mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, ks > 0 || kk > 0);
                    }
                    umma::commit(empty + stage);
                    if (++stage == kStages) {
                        stage = 0;
                        fph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma::commit(accf + b);
                use ^= 1u << b;
            }
            // all issued MMAs have completed before TMEM is released
            umma::commit(fin);
            uint64_t t0 = globaltimer();
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
        int it = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, it++) {
            const int b = it & 1;
            if (!mbar_wait(accf + b, (use >> b) & 1u, abort, a.status))
                break;
            use ^= 1u << b;
            umma::fence_after_sync();
            const int4 g = group_at(a, t / MT, kNMax);
            const int mrow = (t % MT) * kTileM + 32 * q + lane;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + b * C::kAccStride;
            for (int c0 = 0; c0 < g.z; c0 += 16) {
                uint32_t r0[16];
                umma::tmem_ld16(tbase + c0, r0);
                if (EPI == kEpiSwiGLU) {
                    uint32_t r1[16];
                    umma::tmem_ld16(tbase + 128 + c0, r1);
                    umma::tmem_ld_wait();
                    uint16_t *out = static_cast<uint16_t *>(a.out);
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        if (c0 + j < g.z) {
                            const float h = silu(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                            out[(int64_t)(g.y + c0 + j) * a.ldo + mrow] =
                                (uint16_t)(pack_bf16x2(h, 0.f) & 0xFFFFu);
                        }
                    }
                } else {
                    umma::tmem_ld_wait();
                    float *out = static_cast<float *>(a.out);
#pragma unroll
                    for (int j = 0; j < 16; j++)
                        if (c0 + j < g.z)
                            out[(int64_t)(g.y + c0 + j) * a.ldo + mrow] = __uint_as_float(r0[j]);
                }
            }
            umma::fence_before_sync();
            mbar_arrive(acce + b);
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- routed tile groups -------------------------------------------------------------

// One block of 1024 threads (distinct experts <= 1024). For each distinct
// expert u with rows [uoff[u], uoff[u+1]) emit ceil(rows / nmax) groups of at
// most nmax rows, for two group sizes at once.
__global__ void plan_groups_kernel(const int32_t *__restrict__ uexp, const int32_t *__restrict__ uoff,
                                   const int32_t *__restrict__ nuniq, int nmax_a, int4 *__restrict__ ga,
                                   int32_t *__restrict__ na, int nmax_b, int4 *__restrict__ gb,
                                   int32_t *__restrict__ nb) {
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

// y[t][j] = sum_k w[t][k] * ye[inv[t*K+k]][j] + ysh[t][j], summed in k order
// and then the shared term, so the result does not depend on the schedule.
__global__ void combine_kernel(const float *__restrict__ ye, const float *__restrict__ ysh,
                               const float *__restrict__ w, const int32_t *__restrict__ inv, int T, int H, int K,
                               float *__restrict__ y) {
    const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = (int64_t)T * H / 4;
    if (i4 >= n4)
        return;
    const int t = (int)((i4 * 4) / H);
    const int j = (int)((i4 * 4) % H);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; k++) {
        const float wk = w[(int64_t)t * K + k];
        const float4 v = *reinterpret_cast<const float4 *>(ye + (int64_t)inv[(int64_t)t * K + k] * H + j);
        acc.x = fmaf(wk, v.x, acc.x);
        acc.y = fmaf(wk, v.y, acc.y);
        acc.z = fmaf(wk, v.z, acc.z);
        acc.w = fmaf(wk, v.w, acc.w);
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
