// ds4moe C ABI: handle lifetime, argument checks, weight repacking and the
// launch sequence of the layer. Kernels live in the headers included below.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/ds4moe.h"
#include "common.cuh"
#include "decode_fused.cuh"
#include "batch_experts.cuh"
#include "frag_layout.cuh"
#include "dispatch.cuh"
#include "mx4_experts.cuh"
#include "vq_experts.cuh"
#include "prefill_gemm.cuh"
#include "router.cuh"

using namespace ds4;

// Per-kernel CUDA-event timing (ds4moe_profile).
struct Profiler {
    bool on = false;
    struct Rec {
        int name;
        cudaEvent_t a, b;
    };
    std::vector<std::string> names;
    std::vector<int32_t> launches;
    std::vector<double> total_ms;
    std::vector<Rec> pending;
    std::vector<cudaEvent_t> pool;

    cudaEvent_t take() {
        if (pool.empty()) {
            cudaEvent_t e;
            cudaEventCreate(&e);
            return e;
        }
        cudaEvent_t e = pool.back();
        pool.pop_back();
        return e;
    }
    int name_id(const char *n) {
        for (size_t i = 0; i < names.size(); i++)
            if (names[i] == n)
                return (int)i;
        names.emplace_back(n);
        launches.push_back(0);
        total_ms.push_back(0.0);
        return (int)names.size() - 1;
    }
    void drain() { // caller has synchronised the stream
        for (const Rec &r : pending) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, r.a, r.b);
            launches[r.name] += 1;
            total_ms[r.name] += ms;
            pool.push_back(r.a);
            pool.push_back(r.b);
        }
        pending.clear();
    }
    void clear() {
        drain();
        names.clear();
        launches.clear();
        total_ms.clear();
    }
    ~Profiler() {
        for (const Rec &r : pending) {
            cudaEventDestroy(r.a);
            cudaEventDestroy(r.b);
        }
        for (cudaEvent_t e : pool)
            cudaEventDestroy(e);
    }
};

// Buffers and state of the fused decode kernel (sized for 8 tokens).
struct DecodeState {
    Q2Frag gate, up, down;
    Q8Frag sh_gate, sh_up, sh_down;
    unsigned long long *lgt = nullptr, *srec = nullptr; // epoch-tagged logits and routing records
    float *gap = nullptr;
    int32_t *counts = nullptr, *nuniq = nullptr, *inv = nullptr;
    uint16_t *xq = nullptr, *xsums = nullptr;
    uint16_t *hq_hi = nullptr, *hq_lo = nullptr, *hsums = nullptr;
    uint16_t *hs_hi = nullptr, *hs_lo = nullptr;
    float *ye = nullptr, *ysh = nullptr;
    unsigned *ctl = nullptr;
    int ctl_words = 0;
    int grid = 0;
    unsigned epoch = 0;
};

static_assert(kBatchMaxT == DS4MOE_BATCH_MAX_T, "batch path token limit");

// Buffers and launch shape of the batch path (2-bit layers, up to kBatchMaxT
// tokens per call) and of its shared-expert items, which every layer's
// shared expert takes for calls of up to sh_tmax tokens.
struct BatchState {
    uint16_t *xq = nullptr, *xsums = nullptr;                      // [Tb][H], [Tb][H/8]
    uint16_t *hq_hi = nullptr, *hq_lo = nullptr, *hsums = nullptr; // [Pb][I], [Pb][I], [Pb][I/8]
    uint16_t *hs_hi = nullptr, *hs_lo = nullptr;                   // [Tb][Ish] binary16
    int4 *vslot = nullptr;                                         // [Pb] virtual slots
    int32_t *nvslot = nullptr;
    int tmax = 0;                 // tokens per call; 0: the path is unavailable for this layer
    int sh_tmax = 0;              // tokens per call of the shared expert on the 8-bit tile GEMV; 0: never
    int nstage[2] = {0, 0}; // ring depth of the gate/up and the down product kernel
    int smem[2] = {0, 0};   // their dynamic shared memory
    int chunk[2] = {0, 0};  // columns per stage of their shared-expert (8-bit) items
    int grid = 0;
};

struct ds4moe {
    Profiler prof;
    pf::BMaps map_xp, map_h, map_hsh, map_x4; // B tensor maps over scratch (fixed addresses)
    pf::BMaps map_x;                  // over the caller's x of the last call
    const void *map_x_ptr = nullptr;
    int map_x_rows = -1;
    LayerDev L;
    Scratch S;
    DecodeState D;
    BatchState B;
    int device = 0;
    cudaStream_t stream = nullptr;
    unsigned *status = nullptr; // device word of kErr* bits
    void *weight_mem = nullptr;
    uint64_t weight_bytes = 0;
    void *scratch_mem = nullptr;
    uint64_t scratch_bytes = 0;
    ds4moe_stats stats{};
    bool has_gain[2] = {false, false};
    int skip_signal = 0; // test hook: batch product launches still to skip one stage's signal
};

namespace {

// ---- argument checks -------------------------------------------------------

bool is_device_ptr(const void *p) {
    if (!p)
        return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_desc(const ds4moe_layer_desc *d) {
    if (!d || d->magic != DS4MOE_MAGIC || d->version != DS4MOE_VERSION ||
        (d->flags != 0 && d->flags != DS4MOE_FLAG_MXFP4 && d->flags != DS4MOE_FLAG_VQ12 &&
         d->flags != DS4MOE_FLAG_VQ13))
        return DS4MOE_EINVAL;
    if (d->hidden <= 0 || d->hidden % 256 || d->inter <= 0 || d->inter % 256)
        return DS4MOE_EINVAL;
    if (d->n_experts < 1 || d->n_experts > 1024 || d->top_k < 1 || d->top_k > kMaxTopK ||
        d->top_k > d->n_experts)
        return DS4MOE_EINVAL;
    if (d->shared_inter < 0 || d->shared_inter % 256)
        return DS4MOE_EINVAL;
    if (d->max_tokens < 1 || d->max_tokens > 65536)
        return DS4MOE_EINVAL;
    if ((int64_t)d->hidden * d->inter > (int64_t)1 << 30)
        return DS4MOE_EINVAL;
    return DS4MOE_OK;
}

// ---- repacking: canonical 84/34-byte blocks -> per-field streams -----------

__global__ void repack_q2_kernel(const uint32_t *__restrict__ src, int64_t nblocks, int nb, uint4 *__restrict__ qs,
                                 uint4 *__restrict__ sc, uint32_t *__restrict__ dm) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; // canonical block: row * nb + b
    if (idx >= nblocks)
        return;
    const int64_t row = idx / nb;
    const int b = (int)(idx - row * nb);
    const int64_t tb = (row >> 7) * nb + b; // (tile, block)
    const int r = (int)(row & 127);
    const uint32_t *s = src + idx * (kQ2Bytes / 4);
    uint32_t w[21];
#pragma unroll
    for (int i = 0; i < 21; i++)
        w[i] = s[i];
    // canonical: scales[16] (words 0-3), codes[64] (words 4-19, code i at byte i/4,
    // bits 2 (i % 4)), d and dmin (word 20)
    uint32_t osc[4] = {0u, 0u, 0u, 0u}, oqs[16];
#pragma unroll
    for (int sb = 0; sb < 16; sb++) {
        const int slot = 4 * (sb & 3) + (sb >> 2); // quarter major, step minor
        const uint32_t byte = (w[sb >> 2] >> (8 * (sb & 3))) & 0xFFu;
        osc[slot >> 2] |= byte << (8 * (slot & 3));
        uint32_t word = 0u;
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const int i = 16 * sb + k;
            const uint32_t q = (w[4 + (i >> 4)] >> (2 * (i & 15))) & 3u;
            word |= q << ((k & 1) ? 16 + (k - 1) : k);
        }
        oqs[slot] = word;
    }
    sc[tb * 128 + r] = make_uint4(osc[0], osc[1], osc[2], osc[3]);
#pragma unroll
    for (int i = 0; i < 4; i++)
        qs[(tb * 4 + i) * 128 + r] = make_uint4(oqs[4 * i], oqs[4 * i + 1], oqs[4 * i + 2], oqs[4 * i + 3]);
    dm[tb * 128 + r] = w[20]; // d in the low half, dmin in the high half
}

__global__ void repack_q8_kernel(const uint16_t *__restrict__ src, int64_t nblocks, int nblk32, uint4 *__restrict__ qs,
                                 uint16_t *__restrict__ d) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; // canonical block: row * nblk32 + blk
    if (idx >= nblocks)
        return;
    const int64_t row = idx / nblk32;
    const int blk = (int)(idx - row * nblk32);
    const int nks = nblk32 / 2, ks = blk >> 1, hb = blk & 1;
    const int64_t ts = (row >> 7) * nks + ks;
    const int r = (int)(row & 127);
    const uint16_t *s = src + idx * (kQ8Bytes / 2);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        w[i] = (uint32_t)s[1 + 2 * i] | ((uint32_t)s[2 + 2 * i] << 16);
    qs[(ts * 4 + 2 * hb) * 128 + r] = make_uint4(w[0], w[1], w[2], w[3]);
    qs[(ts * 4 + 2 * hb + 1) * 128 + r] = make_uint4(w[4], w[5], w[6], w[7]);
    d[(ts * 128 + r) * 2 + hb] = s[0];
}

// Down-gain tables ([E][H/32] 17-byte blocks each, either may be null) -> one
// fp32 gain per expert and output channel, the product s1 * s2.
__global__ void expand_gain_kernel(const uint8_t *__restrict__ g1, const uint8_t *__restrict__ g2, int E, int H,
                                   float *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)E * H)
        return;
    const int64_t blk = (i / 32) * kGainBlockBytes; // channel blocks of 32 run over [E][H/32]
    const int c = (int)(i % 32);
    float g = 1.f;
    if (g1)
        g = down_gain(g1 + blk, c);
    if (g2)
        g *= down_gain(g2 + blk, c);
    out[i] = g;
}

// fp32 router rows -> three bf16 parts (round to nearest each), stored side by
// side per row: w = hi + mid + lo exactly, since each remainder is exact in fp32
// and three 8-bit significands cover fp32's 24.
__global__ void split_router_kernel(const float *__restrict__ w, int E, int H, uint16_t *__restrict__ w3) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)E * H)
        return;
    const int64_t e = i / H;
    const int h = (int)(i - e * H);
    const int nks = 3 * H / 64;
    float v = w[i];
#pragma unroll
    for (int part = 0; part < 3; part++) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        const int k = part * H + h; // column of the [E][3H] matrix
        const int64_t chunk = (((e >> 7) * nks + k / 64) * 8 + (k % 64) / 8) * 128 + (e & 127);
        w3[chunk * 8 + k % 8] = __bfloat16_as_ushort(b);
        v -= __bfloat162float(b);
    }
}

// Bump allocator over one device allocation, 256-byte aligned pieces.
struct Carver {
    char *base;
    uint64_t used = 0;
    template <class T> T *take(uint64_t count) {
        T *p = reinterpret_cast<T *>(base ? base + used : nullptr);
        used += (count * sizeof(T) + 255) & ~uint64_t(255);
        return p;
    }
};

void layout_weights(ds4moe *h, Carver &c) {
    LayerDev &L = h->L;
    auto q2 = [&](Q2Mat &m, int64_t rows, int k) {
        m.rows = rows;
        m.nb = k / 256;
        const uint64_t nblk = (uint64_t)rows * m.nb;
        m.qs = c.take<uint4>(nblk * 4);
        m.sc = c.take<uint4>(nblk);
        m.dm = c.take<uint32_t>(nblk);
    };
    auto q8 = [&](Q8Mat &m, int64_t rows, int k) {
        m.rows = rows;
        m.nks = k / 64;
        m.qs = c.take<uint4>((uint64_t)rows * k / 16);
        m.d = c.take<uint32_t>((uint64_t)rows * (k / 64));
    };
    L.router_w = c.take<float>((uint64_t)L.E * L.H);
    L.router_w3.rows = L.E;
    L.router_w3.nks = 3 * L.H / 64;
    L.router_w3.p = c.take<uint4>((uint64_t)((L.E + 127) / 128) * 128 * 3 * L.H / 8);
    L.router_bias = c.take<float>(L.E);
    auto m4 = [&](Mx4Mat &m, int64_t rows, int k) {
        m.rows = rows;
        m.nb = k / 32;
        m.codes = c.take<uint4>((uint64_t)rows * m.nb);
        m.scale = c.take<uint8_t>((uint64_t)rows * m.nb);
    };
    auto vqm = [&](VqMat &m, int64_t rows, int k) {
        m.rows = rows;
        m.k = k;
        const uint64_t n = (uint64_t)L.E * rows * (k / 8); // indices of all experts
        m.stream = c.take<uint32_t>(n * 12 / 32);
        m.plane = L.vq == 13 ? c.take<uint8_t>(n / 8) : nullptr;
        m.gain = c.take<uint16_t>((uint64_t)L.E * rows);
    };
    if (L.vq) {
        vqm(L.vgate, L.I, L.H);
        vqm(L.vup, L.I, L.H);
        vqm(L.vdown, L.H, L.I);
        L.codebook = c.take<uint8_t>((uint64_t)8 << L.vq);
        auto tv = [&](VqTile &m, int64_t rows, int k) {
            m.rows = rows;
            m.nkb = k / 256;
            m.rec = c.take<uint8_t>((uint64_t)(rows / 128) * m.nkb * kVqTileRec);
        };
        tv(L.tvgate, (int64_t)L.E * L.I, L.H);
        tv(L.tvup, (int64_t)L.E * L.I, L.H);
        tv(L.tvdown, (int64_t)L.E * L.H, L.I);
    } else if (L.mx4) {
        m4(L.mgate, (int64_t)L.E * L.I, L.H);
        m4(L.mup, (int64_t)L.E * L.I, L.H);
        m4(L.mdown, (int64_t)L.E * L.H, L.I);
        auto t4 = [&](Mx4Tile &m, int64_t rows, int k) {
            m.rows = rows;
            m.nks = k / 64;
            m.rec = c.take<uint8_t>((uint64_t)(rows / 128) * m.nks * kMx4TileRec);
        };
        t4(L.tgate, (int64_t)L.E * L.I, L.H);
        t4(L.tup, (int64_t)L.E * L.I, L.H);
        t4(L.tdown, (int64_t)L.E * L.H, L.I);
    } else {
        q2(L.gate, (int64_t)L.E * L.I, L.H);
        q2(L.up, (int64_t)L.E * L.I, L.H);
        q2(L.down, (int64_t)L.E * L.H, L.I);
    }
    if (L.Ish > 0) {
        q8(L.sh_gate, L.Ish, L.H);
        q8(L.sh_up, L.Ish, L.H);
        q8(L.sh_down, L.H, L.Ish);
    }
    L.gain = h->has_gain[0] || h->has_gain[1] ? c.take<float>((uint64_t)L.E * L.H) : nullptr;
    DecodeState &D = h->D;
    auto f2 = [&](Q2Frag &m, int64_t rows, int k) {
        m.rows = rows;
        m.nkc = k / 128;
        m.rec = c.take<uint8_t>((uint64_t)(rows / 16) * (m.nkc / 2) * kQ2Rec);
    };
    auto f8 = [&](Q8Frag &m, int64_t rows, int k) {
        m.rows = rows;
        m.nbq = k / 32;
        m.rec = c.take<uint8_t>((uint64_t)(rows / 16) * m.nbq * kQ8Rec);
    };
    // the shared expert's 8-bit tile GEMV layout serves every layer (the batch kernel's shared
    // items); the 2-bit one only 2-bit layers (MXFP4 and VQ layers do not use the fused decode kernel)
    if (L.Ish > 0) {
        f8(D.sh_gate, L.Ish, L.H);
        f8(D.sh_up, L.Ish, L.H);
        f8(D.sh_down, L.H, L.Ish);
    }
    if (L.mx4 || L.vq)
        return;
    f2(D.gate, (int64_t)L.E * L.I, L.H);
    f2(D.up, (int64_t)L.E * L.I, L.H);
    f2(D.down, (int64_t)L.E * L.H, L.I);
}

// Logits rows reserved for the router GEMM's K-split partials: tiles * split <=
// grid <= 256 CTAs of 128 rows.
constexpr int64_t kLogitRowsSplit = 256 * 128;

void layout_scratch(ds4moe *h, Carver &c) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    const int64_t T = L.Tmax, P = (int64_t)L.Tmax * L.K;
    const int64_t U = P < L.E ? P : L.E;
    // the router GEMM may write up to (SM count * 128 / m-tiles) rows of K-split partial logits
    S.logits = c.take<float>((T > kLogitRowsSplit ? T : kLogitRowsSplit) * L.E);
    S.idx = c.take<int32_t>(P);
    S.w = c.take<float>(P);
    S.gap = c.take<float>(T);
    S.counts = c.take<int32_t>(L.E);
    S.offsets = c.take<int32_t>(L.E + 1);
    S.uexp = c.take<int32_t>(U);
    S.uoff = c.take<int32_t>(U + 1);
    S.nuniq = c.take<int32_t>(1);
    S.perm = c.take<int32_t>(P);
    S.inv = c.take<int32_t>(P);
    S.h = c.take<uint16_t>(P * L.I);
    S.ye = c.take<float>(P * L.H);
    S.hsh = c.take<uint16_t>(T * (L.Ish > 0 ? L.Ish : 2));
    S.xp = c.take<uint16_t>(P * L.H);
    S.grp_gu = c.take<int4>(U + P / 128 + 1);
    S.grp_dn = c.take<int4>(U + P / 128 + 1);
    S.ngrp = c.take<int32_t>(2);
    S.ysh = c.take<float>(T * L.H);
    S.xstage = c.take<uint16_t>(T * L.H);
    S.ystage = c.take<float>(T * L.H);
    S.ax = L.vq ? c.take<float>(T * L.H) : nullptr;
    S.xq = L.mx4 ? c.take<int8_t>(T * L.H) : nullptr;
    S.x4 = c.take<uint16_t>(T * L.H); // binary16 x: MXFP4 and VQ forms, the shared expert's GEMMs
    S.xd = L.mx4 ? c.take<float>(T * (L.H / 32)) : nullptr;
    S.hf = L.mx4 || L.vq ? c.take<float>(P * L.I) : nullptr;
    S.hq = L.mx4 ? c.take<int8_t>(P * L.I) : nullptr;
    S.hd = L.mx4 ? c.take<float>(P * (L.I / 32)) : nullptr;
    DecodeState &D = h->D;
    const int64_t Td = kDecodeT, Pd = (int64_t)kDecodeT * L.K;
    D.lgt = c.take<unsigned long long>(Td * L.E);
    D.srec = c.take<unsigned long long>(2 * kMaxSlots);
    D.gap = c.take<float>(Td);
    D.counts = c.take<int32_t>(L.E);
    D.nuniq = c.take<int32_t>(1);
    D.inv = c.take<int32_t>(Pd);
    D.xq = c.take<uint16_t>(Td * L.H);
    D.xsums = c.take<uint16_t>(Td * (L.H / 8));
    D.hq_hi = c.take<uint16_t>(Pd * L.I);
    D.hq_lo = c.take<uint16_t>(Pd * L.I);
    D.hsums = c.take<uint16_t>(Pd * (L.I / 8));
    D.hs_hi = c.take<uint16_t>(Td * (L.Ish > 0 ? L.Ish : 2));
    D.hs_lo = c.take<uint16_t>(Td * (L.Ish > 0 ? L.Ish : 2));
    D.ye = c.take<float>(Pd * L.H);
    D.ysh = c.take<float>(Td * L.H);
    D.ctl_words = kCtlTileCnt + L.H / 32;
    D.ctl = c.take<unsigned>(D.ctl_words);
    BatchState &B = h->B;
    const int64_t Tb = T < kBatchMaxT ? T : kBatchMaxT, Pb = Tb * L.K;
    B.hs_hi = c.take<uint16_t>(Tb * (L.Ish > 0 ? L.Ish : 2));
    B.hs_lo = c.take<uint16_t>(Tb * (L.Ish > 0 ? L.Ish : 2));
    B.vslot = c.take<int4>(Pb); // the one-launch grouping writes them for every layer
    B.nvslot = c.take<int32_t>(1);
    if (!L.mx4 && !L.vq) {
        B.xq = c.take<uint16_t>(Tb * L.H);
        B.xsums = c.take<uint16_t>(Tb * (L.H / 8));
        B.hq_hi = c.take<uint16_t>(Pb * L.I);
        B.hq_lo = c.take<uint16_t>(Pb * L.I);
        B.hsums = c.take<uint16_t>(Pb * (L.I / 8));
    }
}

int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess)
        return DS4MOE_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? DS4MOE_ENOMEM : DS4MOE_ECUDA;
}

int launch_rc() { return cuda_rc(cudaGetLastError()); }

unsigned blocks_for(int64_t n, int per) { return (unsigned)((n + per - 1) / per); }

// A launch with programmatic stream serialization: the kernel (which calls
// pdl_wait() before its first global access) may be scheduled while its
// predecessor in the stream finishes.
template <typename... KArgs, typename... Args>
void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch `body` (a kernel launch on h->stream), bracketed by timing events when
// profiling is on, and count it.
template <class F> void launch(ds4moe *h, const char *name, F &&body) {
    if (h->prof.on) {
        Profiler::Rec r{h->prof.name_id(name), h->prof.take(), h->prof.take()};
        cudaEventRecord(r.a, h->stream);
        body();
        cudaEventRecord(r.b, h->stream);
        h->prof.pending.push_back(r);
    } else {
        body();
    }
    h->stats.kernel_count += 1;
}

// Grid size and dynamic shared memory of the prefill GEMM kernels.
int g_pf_grid = 0;

template <int FMT, int NA, int EPI> int setup_gemm() {
    return cuda_rc(cudaFuncSetAttribute(pf::grouped_gemm_kernel<FMT, NA, EPI>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, pf::Cfg<FMT, NA>::kSmemBytes));
}

template <int FMT, int NA, int EPI>
void launch_gemm(ds4moe *h, const char *name, const pf::BMaps &bm, const pf::Args &a) {
    launch(h, name, [&] {
        pf::grouped_gemm_kernel<FMT, NA, EPI>
            <<<g_pf_grid, pf::Cfg<FMT, NA>::kThreads, pf::Cfg<FMT, NA>::kSmemBytes, h->stream>>>(bm, a);
    });
}

// Tensor maps of a bf16 matrix [rows][cols] for the GEMM's B operand: 64-column
// boxes of 16, 32, 64 and 128 rows, 128-byte swizzle, zero fill past the end.
int make_bmaps(const void *base, int64_t rows, int cols, pf::BMaps *out) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void **>(&encode), 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !encode) {
            cudaGetLastError();
            encode = nullptr;
            return DS4MOE_ECUDA;
        }
    }
    for (int i = 0; i < pf::kBoxes; i++) {
        const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
        const cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
        const cuuint32_t box[2] = {64u, 16u << i};
        const cuuint32_t estride[2] = {1u, 1u};
        if (encode(&out->m[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim, gstride, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DS4MOE_ECUDA;
    }
    return DS4MOE_OK;
}

// Tensor maps over the caller's x [T][H] (re-encoded when x or T changes).
int x_maps(ds4moe *h, const void *x, int T) {
    if (x == h->map_x_ptr && T == h->map_x_rows)
        return DS4MOE_OK;
    const int rc = make_bmaps(x, T, h->L.H, &h->map_x);
    h->map_x_ptr = rc ? nullptr : x;
    h->map_x_rows = rc ? -1 : T;
    return rc;
}

// ---- the launch sequence ----------------------------------------------------

// Router logits. Up to kRtMaxT tokens: fp32 dot products on CUDA cores in
// 256-column slices (router_tile_kernel; with xq/xsums given it also writes x
// in the 2-bit GEMV's activation layout for the batch path). More tokens: a
// tensor-core GEMM over the three bf16 parts of the router rows (K = 3 H, x
// repeated per part) whose near-boundary scores the selection recomputes.
int run_router(ds4moe *h, const void *x, int T, float *sel_out, uint16_t *xq = nullptr, uint16_t *xsums = nullptr) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int nsplit = 1;
    const bool tiled = T <= kRtMaxT;
    if (!tiled) {
        int rc = x_maps(h, x, T);
        if (rc)
            return rc;
        pf::Args a{};
        a.status = h->status;
        a.bf[0] = L.router_w3;
        a.M = L.E;
        a.Kd = 3 * L.H;
        a.dense_n = T;
        a.b_kwrap = L.H;
        a.out = S.logits;
        a.ldo = L.E;
        // split K so that the partial tiles fill the GPU: the divisor of the K steps
        // with the fewest K steps on the busiest CTA (rounds of partial tiles times
        // K steps per partial tile; the smaller split on a tie), at least 4 K steps
        // per partial tile, within the partial-logit rows
        const int64_t tiles = ((L.E + 127) / 128) * ((T + 127) / 128);
        const int nk = 3 * L.H / 64;
        int split = 1;
        int64_t best = -1;
        for (int d = 1; d <= nk; d++) {
            if (nk % d != 0 || nk / d < 4 || (int64_t)d * T > (T > kLogitRowsSplit ? T : kLogitRowsSplit))
                continue;
            const int64_t steps = (tiles * d + g_pf_grid - 1) / g_pf_grid * (nk / d);
            if (best < 0 || steps < best) {
                best = steps;
                split = d;
            }
        }
        a.ksplit = split;
        a.out_kstride = (int64_t)T * L.E;
        nsplit = split;
        launch_gemm<pf::kFmtBF16, 1, pf::kEpiF32>(h, "router_logits_tc", h->map_x, a);
    } else {
        nsplit = L.H / kRtSlice;
        launch(h, "router_logits", [&] {
            const dim3 grid((L.E + kRtExperts - 1) / kRtExperts, nsplit);
            const uint16_t *xb = static_cast<const uint16_t *>(x);
            if (T <= 16)
                launch_pdl(router_tile_kernel<16>, grid, dim3(kRtThreads), router_tile_smem(16), st, xb, T, L.H,
                           L.router_w, L.E, S.logits, xq, xsums, h->status);
            else
                launch_pdl(router_tile_kernel<64>, grid, dim3(kRtThreads), router_tile_smem(64), st, xb, T, L.H,
                           L.router_w, L.E, S.logits, xq, xsums, h->status);
        });
    }
    launch(h, "router_select", [&] {
        const size_t smem = (size_t)kSelectSmemPerExpert * L.E;
        // one thread per expert (at least kSelectThreads, at most 1024)
        const int threads = L.E < kSelectThreads ? kSelectThreads : L.E > 1024 ? 1024 : (L.E + 31) / 32 * 32;
        launch_pdl(router_select_kernel, dim3(T), dim3(threads), smem, st, S.logits, L.router_bias, T, L.E, L.K,
                   S.idx, S.w, S.gap, sel_out, tiled ? nullptr : static_cast<const uint16_t *>(x), L.router_w, L.H,
                   nsplit, (int64_t)T * L.E);
    });
    return launch_rc();
}

// Dynamic shared memory of the one-block grouping: the histograms (128 E bytes,
// at most 128 KB) and, where they fit beside them, the staged indices.
constexpr size_t kGroupSmemMax = 200 * 1024;

// Expert grouping for the routing in S.idx, one launch: for up to kBatchMaxT
// tokens the batch path's grouping (which also writes its virtual slots),
// else the one-block grouping over per-warp histograms.
int run_group(ds4moe *h, int T) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    if (T > kBatchMaxT) {
        const int P = T * L.K;
        const size_t hist = (size_t)128 * L.E, staged = hist + (size_t)4 * P;
        const bool stage = staged <= kGroupSmemMax;
        launch(h, "group", [&] {
            launch_pdl(group_kernel, dim3(1), dim3(1024), stage ? staged : hist, h->stream, S.idx, P, L.E, stage,
                       S.counts, S.offsets, S.uexp, S.uoff, S.nuniq, S.perm, S.inv, h->status);
        });
        return launch_rc();
    }
    launch(h, "batch_group", [&] {
        launch_pdl(batch_group_kernel, dim3(1), dim3(1024), 0, h->stream, S.idx, T * L.K, L.E, S.counts, S.offsets,
                   S.uexp, S.uoff, S.nuniq, S.perm, S.inv, h->B.vslot, h->B.nvslot, h->status);
    });
    return launch_rc();
}

// The shared expert on tensor cores (dense over the T token rows of x, in
// binary16 like the expanded 8-bit weights): SwiGLU rows (binary16) into
// S.hsh, then the down product into S.ysh.
int run_shared_gemms(ds4moe *h, const void *x, int T) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    launch(h, "shared_x_f16", [&] {
        launch_pdl(bf16_to_f16_kernel, dim3(blocks_for((int64_t)T * L.H / 8, 256)), dim3(256), 0, h->stream,
                   static_cast<const uint16_t *>(x), (int64_t)T * L.H, S.x4);
    });
    pf::Args s{};
    s.status = h->status;
    s.q8[0] = L.sh_gate;
    s.q8[1] = L.sh_up;
    s.M = L.Ish;
    s.Kd = L.H;
    s.dense_n = T;
    s.out = S.hsh;
    s.ldo = L.Ish;
    launch_gemm<pf::kFmtQ8, 2, pf::kEpiSwiGLUF16>(h, "prefill_gateup_q8", h->map_x4, s);
    s.q8[0] = L.sh_down;
    s.M = L.H;
    s.Kd = L.Ish;
    s.out = S.ysh;
    s.ldo = L.H;
    launch_gemm<pf::kFmtQ8, 1, pf::kEpiF32>(h, "prefill_down_q8", h->map_hsh, s);
    return launch_rc();
}

// The shared expert on the batch kernel's 8-bit items (token groups of up to
// 8 columns over the exact tile GEMV; SwiGLU rows as a binary16 hi + lo pair):
// gate/up, then down into S.ysh.
int run_shared_batch(ds4moe *h, const void *x, int T) {
    const LayerDev &L = h->L;
    BatchState &B = h->B;
    DecodeState &D = h->D;
    BatchArgs a{};
    a.H = L.H;
    a.I = L.I;
    a.K = L.K;
    a.Ish = L.Ish;
    a.T = T;
    a.sh_gate = D.sh_gate;
    a.sh_up = D.sh_up;
    a.sh_down = D.sh_down;
    a.x = static_cast<const uint16_t *>(x);
    a.hs_hi = B.hs_hi;
    a.hs_lo = B.hs_lo;
    a.ysh = h->S.ysh;
    a.status = h->status;
    for (int down = 0; down < 2; down++) {
        a.nstage = B.nstage[down];
        a.chunk = B.chunk[down];
        auto fn = down ? batch_product_kernel<true, kBatchShared> : batch_product_kernel<false, kBatchShared>;
        launch(h, down ? "batch_down_shared" : "batch_gateup_shared", [&] {
            launch_pdl(fn, dim3(B.grid), dim3(kBatchThreads), B.smem[down], h->stream, a);
        });
    }
    return launch_rc();
}

// The shared expert of a call: the tile GEMV for up to B.sh_tmax tokens (a
// tensor-core tile of 128 rows would leave most SMs idle there), else the
// tensor-core GEMMs.
int run_shared(ds4moe *h, const void *x, int T) {
    return T <= h->B.sh_tmax ? run_shared_batch(h, x, T) : run_shared_gemms(h, x, T);
}

// Experts and combine for the routing already in S.idx / S.w: grouped
// tensor-core GEMMs over the expert-grouped rows.
int run_experts_prefill(ds4moe *h, const void *x, int T, float *y) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int rc = run_group(h, T);
    if (rc)
        return rc;
    launch(h, "plan_groups", [&] {
        launch_pdl(pf::plan_groups_kernel, dim3(1), dim3(1024), 0, st, S.uexp, S.uoff, S.nuniq,
                   pf::Cfg<pf::kFmtQ2, 2>::kNMax, S.grp_gu, S.ngrp, pf::Cfg<pf::kFmtQ2, 1>::kNMax, S.grp_dn,
                   S.ngrp + 1);
    });
    launch(h, "gather_rows", [&] {
        launch_pdl(pf::gather_rows_kernel, dim3(T * L.K), dim3(256), 0, st, static_cast<const uint16_t *>(x), S.perm,
                   L.K, L.H, S.xp);
    });
    pf::Args a{};
    a.status = h->status;
    // routed gate/up: B rows are the gathered token rows, in expert-grouped order
    a.q2[0] = L.gate;
    a.q2[1] = L.up;
    a.M = L.I;
    a.Kd = L.H;
    a.groups = S.grp_gu;
    a.ngroups = S.ngrp;
    a.dense_n = 0;
    a.out = S.h;
    a.ldo = L.I;
    launch_gemm<pf::kFmtQ2, 2, pf::kEpiSwiGLU>(h, "prefill_gateup_q2", h->map_xp, a);
    // routed down
    a.q2[0] = L.down;
    a.M = L.H;
    a.Kd = L.I;
    a.groups = S.grp_dn;
    a.ngroups = S.ngrp + 1;
    a.out = S.ye;
    a.ldo = L.H;
    launch_gemm<pf::kFmtQ2, 1, pf::kEpiF32>(h, "prefill_down_q2", h->map_h, a);
    if (L.Ish > 0) {
        rc = run_shared(h, x, T);
        if (rc)
            return rc;
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// Experts and combine for the routing already in S.idx / S.w, T <= B.tmax:
// x in the 2-bit tile GEMV's layout (unless the router wrote it), the grouping
// with the virtual slots, the two persistent products (gate/up, then down;
// each over the routed experts' 2-bit items and the shared expert's 8-bit
// items), the combine.
int run_experts_batch(ds4moe *h, const void *x, int T, float *y, bool x_prepared) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    BatchState &B = h->B;
    DecodeState &D = h->D;
    cudaStream_t st = h->stream;
    if (!x_prepared)
        launch(h, "batch_prep_x", [&] {
            launch_pdl(batch_prep_x_kernel, dim3(blocks_for((int64_t)T * L.H / 16, 256)), dim3(256), 0, st,
                       static_cast<const uint16_t *>(x), T, L.H, B.xq, B.xsums);
        });
    int rc = run_group(h, T);
    if (rc)
        return rc;
    BatchArgs a;
    a.H = L.H;
    a.I = L.I;
    a.K = L.K;
    a.Ish = L.Ish;
    a.T = T;
    a.gate = D.gate;
    a.up = D.up;
    a.down = D.down;
    a.sh_gate = D.sh_gate;
    a.sh_up = D.sh_up;
    a.sh_down = D.sh_down;
    a.x = static_cast<const uint16_t *>(x);
    a.xq = B.xq;
    a.xsums = B.xsums;
    a.hq_hi = B.hq_hi;
    a.hq_lo = B.hq_lo;
    a.hsums = B.hsums;
    a.ye = S.ye;
    a.hs_hi = B.hs_hi;
    a.hs_lo = B.hs_lo;
    a.ysh = S.ysh;
    a.vslot = B.vslot;
    a.nvslot = B.nvslot;
    a.perm = S.perm;
    a.status = h->status;
    auto product = [&](int mode, const char *name, void (*fn)(BatchArgs)) {
        a.nstage = B.nstage[mode];
        a.chunk = B.chunk[mode];
        a.skip_signal = h->skip_signal > 0;
        if (h->skip_signal > 0)
            h->skip_signal--;
        launch(h, name, [&] { launch_pdl(fn, dim3(B.grid), dim3(kBatchThreads), B.smem[mode], st, a); });
    };
    // few tokens: one launch per product over both kinds of items (the shared expert fills the
    // routed items' tail); more: separate launches, each split evenly over the SMs
    if (T <= kBatchMergeMaxT || L.Ish == 0) {
        product(0, "batch_gateup", batch_product_kernel<false, kBatchBoth>);
        product(1, "batch_down", batch_product_kernel<true, kBatchBoth>);
    } else {
        product(0, "batch_gateup", batch_product_kernel<false, kBatchRouted>);
        product(0, "batch_gateup_shared", batch_product_kernel<false, kBatchShared>);
        product(1, "batch_down", batch_product_kernel<true, kBatchRouted>);
        product(1, "batch_down_shared", batch_product_kernel<true, kBatchShared>);
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// MXFP4 routed experts for the routing already in S.idx / S.w, every T: Q8
// token rows, the gate/up product with SwiGLU, Q8 SwiGLU rows, the down
// product, the shared expert, the combine.
int run_experts_mx4(ds4moe *h, const void *x, int T, float *y) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int rc = run_group(h, T);
    if (rc)
        return rc;
    const int P = T * L.K;
    const int U = P < L.E ? P : L.E; // bound on the distinct experts
    launch(h, "mx4_act_x", [&] {
        launch_pdl(act_q8_kernel, dim3(blocks_for((int64_t)T * L.H, 256)), dim3(256), 0, st, x, 1, (int64_t)T * L.H,
                   S.xq, S.xd);
    });
    // an expert holds at most T rows when a token's experts are distinct; more come in chunks
    const int nt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    launch(h, "mx4_gateup", [&] {
        const dim3 grid((L.I + 7) / 8, U);
        auto k = nt == 1   ? mx4_product_kernel<true, 1>
                 : nt == 2 ? mx4_product_kernel<true, 2>
                 : nt == 4 ? mx4_product_kernel<true, 4>
                           : mx4_product_kernel<true, 8>;
        launch_pdl(k, grid, dim3(256), 0, st, L.mgate, L.mup, S.xq, S.xd, S.uexp, S.uoff, S.nuniq, S.perm, L.K, L.I,
                   L.H, S.hf);
    });
    launch(h, "mx4_act_h", [&] {
        launch_pdl(act_q8_kernel, dim3(blocks_for((int64_t)P * L.I, 256)), dim3(256), 0, st, S.hf, 0,
                   (int64_t)P * L.I, S.hq, S.hd);
    });
    launch(h, "mx4_down", [&] {
        const dim3 grid((L.H + 7) / 8, U);
        auto k = nt == 1   ? mx4_product_kernel<false, 1>
                 : nt == 2 ? mx4_product_kernel<false, 2>
                 : nt == 4 ? mx4_product_kernel<false, 4>
                           : mx4_product_kernel<false, 8>;
        launch_pdl(k, grid, dim3(256), 0, st, L.mdown, L.mdown, S.hq, S.hd, S.uexp, S.uoff, S.nuniq, S.perm, L.K, L.H,
                   L.I, S.ye);
    });
    if (L.Ish > 0) {
        rc = run_shared(h, x, T);
        if (rc)
            return rc;
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// MXFP4 routed experts on the tensor cores (the prefill form) for the routing
// already in S.idx / S.w: the grouping and the tile groups, x on the FP4 grid
// (binary16) gathered into expert-grouped order, the grouped GEMMs on the MXFP4
// tile records (weights expanded exactly to binary16 in TMEM; the gate/up
// epilogue puts the SwiGLU rows on the FP4 grid), the shared expert, the combine.
int run_experts_mx4_tc(ds4moe *h, const void *x, int T, float *y) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int rc = run_group(h, T);
    if (rc)
        return rc;
    launch(h, "plan_groups", [&] {
        launch_pdl(pf::plan_groups_kernel, dim3(1), dim3(1024), 0, st, S.uexp, S.uoff, S.nuniq,
                   pf::Cfg<pf::kFmtMx4, 2>::kNMax, S.grp_gu, S.ngrp, pf::Cfg<pf::kFmtMx4, 1>::kNMax, S.grp_dn,
                   S.ngrp + 1);
    });
    launch(h, "mx4_act_fp4", [&] {
        launch_pdl(act_fp4_kernel, dim3(blocks_for((int64_t)T * L.H / 8, 256)), dim3(256), 0, st,
                   static_cast<const uint16_t *>(x), (int64_t)T * L.H, S.x4);
    });
    launch(h, "gather_rows", [&] {
        launch_pdl(pf::gather_rows_kernel, dim3(T * L.K), dim3(256), 0, st, S.x4, S.perm, L.K, L.H, S.xp);
    });
    pf::Args a{};
    a.status = h->status;
    a.mx4[0] = L.tgate;
    a.mx4[1] = L.tup;
    a.M = L.I;
    a.Kd = L.H;
    a.groups = S.grp_gu;
    a.ngroups = S.ngrp;
    a.dense_n = 0;
    a.out = S.h;
    a.ldo = L.I;
    launch_gemm<pf::kFmtMx4, 2, pf::kEpiSwiGLUFp4>(h, "prefill_gateup_mx4", h->map_xp, a);
    a.mx4[0] = L.tdown;
    a.M = L.H;
    a.Kd = L.I;
    a.groups = S.grp_dn;
    a.ngroups = S.ngrp + 1;
    a.out = S.ye;
    a.ldo = L.H;
    launch_gemm<pf::kFmtMx4, 1, pf::kEpiF32>(h, "prefill_down_mx4", h->map_h, a);
    if (L.Ish > 0) {
        rc = run_shared(h, x, T);
        if (rc)
            return rc;
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// VQ routed experts on the tensor cores (the prefill form) for the routing
// already in S.idx / S.w: the grouping and the tile groups, x as binary16
// gathered into expert-grouped order, the grouped GEMMs on the VQ tile records
// (codewords from the codebook in shared memory, exact in binary16; row gains
// in the epilogues; the SwiGLU rows as binary16), the shared expert, the combine.
int run_experts_vq_tc(ds4moe *h, const void *x, int T, float *y) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int rc = run_group(h, T);
    if (rc)
        return rc;
    launch(h, "plan_groups", [&] {
        launch_pdl(pf::plan_groups_kernel, dim3(1), dim3(1024), 0, st, S.uexp, S.uoff, S.nuniq,
                   pf::Cfg<pf::kFmtVq, 2>::kNMax, S.grp_gu, S.ngrp, pf::Cfg<pf::kFmtVq, 1>::kNMax, S.grp_dn,
                   S.ngrp + 1);
    });
    launch(h, "gather_rows_f16", [&] {
        launch_pdl(gather_rows_f16_kernel, dim3(T * L.K), dim3(256), 0, st, static_cast<const uint16_t *>(x), S.perm,
                   L.K, L.H, S.xp);
    });
    pf::Args a{};
    a.status = h->status;
    a.vq[0] = L.tvgate;
    a.vq[1] = L.tvup;
    a.rgain[0] = L.vgate.gain;
    a.rgain[1] = L.vup.gain;
    a.codebook = L.codebook;
    a.vq_bits = L.vq;
    a.M = L.I;
    a.Kd = L.H;
    a.groups = S.grp_gu;
    a.ngroups = S.ngrp;
    a.dense_n = 0;
    a.out = S.h;
    a.ldo = L.I;
    launch_gemm<pf::kFmtVq, 2, pf::kEpiSwiGLUF16>(h, "prefill_gateup_vq", h->map_xp, a);
    a.vq[0] = L.tvdown;
    a.rgain[0] = L.vdown.gain;
    a.M = L.H;
    a.Kd = L.I;
    a.groups = S.grp_dn;
    a.ngroups = S.ngrp + 1;
    a.out = S.ye;
    a.ldo = L.H;
    launch_gemm<pf::kFmtVq, 1, pf::kEpiF32>(h, "prefill_down_vq", h->map_h, a);
    if (L.Ish > 0) {
        rc = run_shared(h, x, T);
        if (rc)
            return rc;
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// VQ routed experts for the routing already in S.idx / S.w, every T: x in fp32,
// the gate/up product with SwiGLU, the down product, the shared expert, the
// combine. The product kernels are persistent (two CTAs per SM) and load the
// codebook into shared memory once per CTA.
int run_experts_vq(ds4moe *h, const void *x, int T, float *y) {
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    int rc = run_group(h, T);
    if (rc)
        return rc;
    const int P = T * L.K;
    const int U = P < L.E ? P : L.E; // bound on the distinct experts
    const int nt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    const int entries = 1 << L.vq;
    const size_t smem = (size_t)8 << L.vq;
    launch(h, "vq_widen_x", [&] {
        launch_pdl(widen_bf16_kernel, dim3(blocks_for((int64_t)T * L.H / 8, 256)), dim3(256), 0, st,
                   static_cast<const uint16_t *>(x), (int64_t)T * L.H, S.ax);
    });
    launch(h, "vq_gateup", [&] {
        const int work = U * ((L.I + 7) / 8);
        const int grid = work < 2 * g_pf_grid ? work : 2 * g_pf_grid;
        auto k = nt == 1   ? vq_product_kernel<true, 1>
                 : nt == 2 ? vq_product_kernel<true, 2>
                 : nt == 4 ? vq_product_kernel<true, 4>
                           : vq_product_kernel<true, 8>;
        launch_pdl(k, dim3(grid), dim3(256), smem, st, L.vgate, L.vup, L.codebook, entries, S.ax, S.uexp, S.uoff,
                   S.nuniq, S.perm, L.K,
                                   L.I, L.H, U, S.hf);
    });
    launch(h, "vq_down", [&] {
        const int work = U * ((L.H + 7) / 8);
        const int grid = work < 2 * g_pf_grid ? work : 2 * g_pf_grid;
        auto k = nt == 1   ? vq_product_kernel<false, 1>
                 : nt == 2 ? vq_product_kernel<false, 2>
                 : nt == 4 ? vq_product_kernel<false, 4>
                           : vq_product_kernel<false, 8>;
        launch_pdl(k, dim3(grid), dim3(256), smem, st, L.vdown, L.vdown, L.codebook, entries, S.hf, S.uexp, S.uoff,
                   S.nuniq, S.perm, L.K,
                                   L.H, L.I, U, S.ye);
    });
    if (L.Ish > 0) {
        rc = run_shared(h, x, T);
        if (rc)
            return rc;
    }
    launch(h, "combine", [&] {
        launch_pdl(combine_kernel, dim3(blocks_for((int64_t)T * L.H / 4, 256)), dim3(256), 0, st, S.ye,
                   L.Ish > 0 ? S.ysh : nullptr, S.w, S.inv, S.idx, L.gain, T, L.H, L.K, y);
    });
    return launch_rc();
}

// The fused decode kernel over tokens [0, T) in launches of up to 8 tokens.
// forced_idx/forced_w: caller routing (nullptr = route here). idx_out/w_out
// receive the routing of every token ([T][K]).
int run_decode(ds4moe *h, const void *x, int T, float *y, const int32_t *forced_idx, const float *forced_w) {
    const LayerDev &L = h->L;
    DecodeState &D = h->D;
    Scratch &S = h->S;
    for (int t0 = 0; t0 < T; t0 += kDecodeT) {
        const int Tc = T - t0 < kDecodeT ? T - t0 : kDecodeT;
        DecodeArgs a;
        a.H = L.H;
        a.I = L.I;
        a.E = L.E;
        a.K = L.K;
        a.Ish = L.Ish;
        a.router_w = L.router_w;
        a.router_bias = L.router_bias;
        a.gate = D.gate;
        a.up = D.up;
        a.down = D.down;
        a.sh_gate = D.sh_gate;
        a.sh_up = D.sh_up;
        a.sh_down = D.sh_down;
        a.x = static_cast<const uint16_t *>(x) + (int64_t)t0 * L.H;
        a.T = Tc;
        a.y = y + (int64_t)t0 * L.H;
        a.forced_idx = forced_idx ? forced_idx + (int64_t)t0 * L.K : nullptr;
        a.forced_w = forced_w ? forced_w + (int64_t)t0 * L.K : nullptr;
        a.epoch = ++D.epoch;
        if (a.epoch == 0)
            a.epoch = ++D.epoch;
        a.lgt = D.lgt;
        a.srec = D.srec;
        a.idx = S.idx + (int64_t)t0 * L.K;
        a.w = S.w + (int64_t)t0 * L.K;
        a.gap = S.gap + t0;
        a.counts = D.counts;
        a.nuniq = D.nuniq;
        a.inv = D.inv;
        a.xq = D.xq;
        a.xsums = D.xsums;
        a.hq_hi = D.hq_hi;
        a.hq_lo = D.hq_lo;
        a.hsums = D.hsums;
        a.hs_hi = D.hs_hi;
        a.hs_lo = D.hs_lo;
        a.ye = D.ye;
        a.ysh = D.ysh;
        a.ctl = D.ctl;
        a.status = h->status;
        a.io = SelIO{a.lgt, a.epoch, a.idx, a.w, a.gap, a.inv, a.counts, a.nuniq, a.srec};
        a.gain = L.gain;
        void *args[] = {&a};
        launch(h, "decode_fused", [&] {
            // with down gains: the kernels built for them (one token; up to 8)
            const void *fn = L.gain    ? (Tc <= 1 ? (const void *)decode_fused_kernel<1, true>
                                                  : (const void *)decode_fused_kernel<8, true>)
                             : Tc <= 1 ? (const void *)decode_fused_kernel<1>
                             : Tc <= 2 ? (const void *)decode_fused_kernel<2>
                             : Tc <= 4 ? (const void *)decode_fused_kernel<4>
                                       : (const void *)decode_fused_kernel<8>;
            cudaLaunchCooperativeKernel(fn, dim3(D.grid), dim3(kDecodeThreads), args, sizeof(DecodeSmem), h->stream);
        });
        int rc = launch_rc();
        if (rc)
            return rc;
    }
    return DS4MOE_OK;
}

int check_call(ds4moe *h, const void *x, int T) {
    if (!h)
        return DS4MOE_EINVAL;
    if (T < 0 || T > h->L.Tmax)
        return DS4MOE_EINVAL;
    if (T > 0 && !is_device_ptr(x))
        return DS4MOE_EINVAL;
    if (T > 0 && !aligned(x, 16))
        return DS4MOE_EINVAL;
    return DS4MOE_OK;
}

// The path a call takes: DS4MOE_PATH_AUTO resolved by T; -1 if an explicit
// batch path cannot take the call (more than B.tmax tokens, or no batch path
// for this layer). MXFP4 and VQ layers run one pipeline whatever the path.
int resolve_path(const ds4moe *h, int T, int path) {
    if (h->L.mx4) { // two forms: decode (Q8 activations, CUDA cores), prefill (FP4 activations, tensor cores)
        if (path == DS4MOE_PATH_AUTO)
            return T >= DS4MOE_AUTO_MX4_PREFILL_MIN_T ? DS4MOE_PATH_PREFILL : DS4MOE_PATH_DECODE;
        return path == DS4MOE_PATH_PREFILL ? DS4MOE_PATH_PREFILL : DS4MOE_PATH_DECODE;
    }
    if (h->L.vq) { // CUDA-core products for decode sizes, tensor cores for prefill sizes
        if (path == DS4MOE_PATH_AUTO)
            return T >= DS4MOE_AUTO_VQ_PREFILL_MIN_T ? DS4MOE_PATH_PREFILL : DS4MOE_PATH_DECODE;
        return path == DS4MOE_PATH_PREFILL ? DS4MOE_PATH_PREFILL : DS4MOE_PATH_DECODE;
    }
    if (path == DS4MOE_PATH_AUTO) {
        if (T <= DS4MOE_AUTO_DECODE_MAX_T)
            return DS4MOE_PATH_DECODE;
        return T <= DS4MOE_AUTO_BATCH_MAX_T && T <= h->B.tmax ? DS4MOE_PATH_BATCH : DS4MOE_PATH_PREFILL;
    }
    if (path == DS4MOE_PATH_BATCH && !h->L.mx4 && !h->L.vq && T > h->B.tmax)
        return -1;
    return path;
}

int forward_impl(ds4moe *h, const void *x, int T, int path, float *y) {
    h->stats = ds4moe_stats{};
    h->stats.tokens = T;
    h->stats.path = path;
    if (h->L.mx4 || h->L.vq) {
        int rc = run_router(h, x, T, nullptr);
        if (rc)
            return rc;
        if (h->L.vq)
            return path == DS4MOE_PATH_PREFILL ? run_experts_vq_tc(h, x, T, y) : run_experts_vq(h, x, T, y);
        return path == DS4MOE_PATH_PREFILL ? run_experts_mx4_tc(h, x, T, y) : run_experts_mx4(h, x, T, y);
    }
    if (path == DS4MOE_PATH_DECODE)
        return run_decode(h, x, T, y, nullptr, nullptr);
    if (path == DS4MOE_PATH_BATCH) {
        int rc = run_router(h, x, T, nullptr, h->B.xq, h->B.xsums);
        return rc ? rc : run_experts_batch(h, x, T, y, true);
    }
    int rc = run_router(h, x, T, nullptr);
    if (rc)
        return rc;
    return run_experts_prefill(h, x, T, y);
}

} // namespace

extern "C" {

const char *ds4moe_strerror(int code) {
    switch (code) {
    case DS4MOE_OK: return "ok";
    case DS4MOE_EINVAL: return "invalid argument";
    case DS4MOE_ENOMEM: return "device allocation failed";
    case DS4MOE_ECUDA: return "CUDA call or launch failed";
    case DS4MOE_EUNSUPPORTED: return "device is not a GB300 (compute capability 10.3)";
    case DS4MOE_ETIMEOUT: return "a bounded device-side wait timed out";
    case DS4MOE_EDEVICE: return "a kernel reported an inconsistency (e.g. an out-of-range expert index)";
    case DS4MOE_ESCRATCH:
        return "request needs more than the fixed DS4MOE_NOALLOC_SCRATCH bytes of ds4moe_route_noalloc";
    default: return "unknown ds4moe error";
    }
}

int ds4moe_create(const ds4moe_layer_desc *desc, const ds4moe_weights *w, ds4moe_t **out) {
    if (!out)
        return DS4MOE_EINVAL;
    *out = nullptr;
    int rc = check_desc(desc);
    if (rc)
        return rc;
    if (!w || !is_device_ptr(w->router_w) || !is_device_ptr(w->gate) || !is_device_ptr(w->up) ||
        !is_device_ptr(w->down))
        return DS4MOE_EINVAL;
    if (w->router_bias && !is_device_ptr(w->router_bias))
        return DS4MOE_EINVAL;
    if ((w->down_gain && !is_device_ptr(w->down_gain)) || (w->down_gain2 && !is_device_ptr(w->down_gain2)))
        return DS4MOE_EINVAL;
    {
        const int vq = desc->flags == DS4MOE_FLAG_VQ12 ? 12 : desc->flags == DS4MOE_FLAG_VQ13 ? 13 : 0;
        const void *rowgains[3] = {w->gate_rowgain, w->up_rowgain, w->down_rowgain};
        const void *planes[3] = {w->gate_plane, w->up_plane, w->down_plane};
        if ((vq != 0) != (w->vq_codebook != nullptr) || (vq && !is_device_ptr(w->vq_codebook)))
            return DS4MOE_EINVAL;
        for (int m = 0; m < 3; m++) {
            if ((vq != 0) != (rowgains[m] != nullptr) || (vq && !is_device_ptr(rowgains[m])))
                return DS4MOE_EINVAL;
            if ((vq == 13) != (planes[m] != nullptr) || (vq == 13 && !is_device_ptr(planes[m])))
                return DS4MOE_EINVAL;
        }
    }
    const bool has_shared = desc->shared_inter > 0;
    if (has_shared != (w->sh_gate != nullptr) || has_shared != (w->sh_up != nullptr) ||
        has_shared != (w->sh_down != nullptr))
        return DS4MOE_EINVAL;
    if (has_shared && (!is_device_ptr(w->sh_gate) || !is_device_ptr(w->sh_up) || !is_device_ptr(w->sh_down)))
        return DS4MOE_EINVAL;
    if (!aligned(w->router_w, 16) || !aligned(w->gate, 4) || !aligned(w->up, 4) || !aligned(w->down, 4) ||
        (has_shared && (!aligned(w->sh_gate, 2) || !aligned(w->sh_up, 2) || !aligned(w->sh_down, 2))) ||
        (w->router_bias && !aligned(w->router_bias, 4)))
        return DS4MOE_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DS4MOE_ECUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return DS4MOE_ECUDA;
    if (prop.major != 10 || prop.minor != 3)
        return DS4MOE_EUNSUPPORTED;

    ds4moe *h = new (std::nothrow) ds4moe();
    if (!h)
        return DS4MOE_ENOMEM;
    h->device = dev;
    LayerDev &L = h->L;
    L.H = desc->hidden;
    L.I = desc->inter;
    L.E = desc->n_experts;
    L.K = desc->top_k;
    L.Ish = desc->shared_inter;
    L.Tmax = desc->max_tokens;
    L.mx4 = (desc->flags & DS4MOE_FLAG_MXFP4) != 0;
    L.vq = desc->flags == DS4MOE_FLAG_VQ12 ? 12 : desc->flags == DS4MOE_FLAG_VQ13 ? 13 : 0;
    h->has_gain[0] = w->down_gain != nullptr;
    h->has_gain[1] = w->down_gain2 != nullptr;

    Carver probe{nullptr};
    layout_weights(h, probe);
    h->weight_bytes = probe.used;
    Carver sprobe{nullptr};
    layout_scratch(h, sprobe);
    h->scratch_bytes = sprobe.used;

    rc = cuda_rc(cudaMalloc(&h->weight_mem, h->weight_bytes));
    if (!rc)
        rc = cuda_rc(cudaMalloc(&h->scratch_mem, h->scratch_bytes));
    if (!rc)
        rc = cuda_rc(cudaMalloc(reinterpret_cast<void **>(&h->status), sizeof(unsigned)));
    if (rc) {
        ds4moe_destroy(h);
        return rc;
    }
    Carver wc{static_cast<char *>(h->weight_mem)};
    layout_weights(h, wc);
    Carver sc{static_cast<char *>(h->scratch_mem)};
    layout_scratch(h, sc);
    {
        const int64_t P = (int64_t)L.Tmax * L.K;
        rc = make_bmaps(h->S.xp, P, L.H, &h->map_xp);
        if (!rc)
            rc = make_bmaps(h->S.h, P, L.I, &h->map_h);
        if (!rc && L.Ish > 0)
            rc = make_bmaps(h->S.hsh, L.Tmax, L.Ish, &h->map_hsh);
        if (!rc && L.Ish > 0)
            rc = make_bmaps(h->S.x4, L.Tmax, L.H, &h->map_x4);
        if (rc) {
            ds4moe_destroy(h);
            return rc;
        }
    }

    cudaStream_t st = nullptr; // create-time work runs on the legacy stream and is waited for
    cudaMemsetAsync(h->status, 0, sizeof(unsigned), st);
    cudaMemcpyAsync(const_cast<float *>(L.router_w), w->router_w, sizeof(float) * L.E * L.H,
                    cudaMemcpyDeviceToDevice, st);
    cudaMemsetAsync(const_cast<uint4 *>(L.router_w3.p), 0,
                    (size_t)((L.E + 127) / 128) * 128 * 3 * L.H * sizeof(uint16_t), st);
    split_router_kernel<<<blocks_for((int64_t)L.E * L.H, 256), 256, 0, st>>>(
        L.router_w, L.E, L.H, reinterpret_cast<uint16_t *>(const_cast<uint4 *>(L.router_w3.p)));
    if (w->router_bias)
        cudaMemcpyAsync(const_cast<float *>(L.router_bias), w->router_bias, sizeof(float) * L.E,
                        cudaMemcpyDeviceToDevice, st);
    else
        L.router_bias = nullptr;
    auto rq2 = [&](const void *src, Q2Mat &m) {
        const int64_t nblk = m.rows * m.nb;
        repack_q2_kernel<<<blocks_for(nblk, 256), 256, 0, st>>>(
            static_cast<const uint32_t *>(src), nblk, m.nb, const_cast<uint4 *>(m.qs), const_cast<uint4 *>(m.sc),
            const_cast<uint32_t *>(m.dm));
    };
    auto rq8 = [&](const void *src, Q8Mat &m) {
        const int64_t nblk = m.rows * (m.nks * 2);
        repack_q8_kernel<<<blocks_for(nblk, 256), 256, 0, st>>>(
            static_cast<const uint16_t *>(src), nblk, m.nks * 2, const_cast<uint4 *>(m.qs),
            reinterpret_cast<uint16_t *>(const_cast<uint32_t *>(m.d)));
    };
    auto rm4 = [&](const void *src, Mx4Mat &m) {
        const int64_t nblk = m.rows * m.nb;
        repack_mx4_kernel<<<blocks_for(nblk, 256), 256, 0, st>>>(static_cast<const uint8_t *>(src), nblk,
                                                                 const_cast<uint4 *>(m.codes),
                                                                 const_cast<uint8_t *>(m.scale));
    };
    auto cvq = [&](const void *stream, const void *plane, const void *rowgain, VqMat &m) {
        const uint64_t n = (uint64_t)L.E * m.rows * (m.k / 8);
        cudaMemcpyAsync(const_cast<uint32_t *>(m.stream), stream, n * 12 / 8, cudaMemcpyDeviceToDevice, st);
        if (m.plane)
            cudaMemcpyAsync(const_cast<uint8_t *>(m.plane), plane, n / 8, cudaMemcpyDeviceToDevice, st);
        cudaMemcpyAsync(const_cast<uint16_t *>(m.gain), rowgain, (uint64_t)L.E * m.rows * 2, cudaMemcpyDeviceToDevice,
                        st);
    };
    auto rm4t = [&](const void *src, Mx4Tile &m) {
        const int nb = m.nks * 2;
        repack_mx4_tile_kernel<<<blocks_for(m.rows * nb, 256), 256, 0, st>>>(static_cast<const uint8_t *>(src),
                                                                           m.rows, nb, const_cast<uint8_t *>(m.rec));
    };
    if (L.vq) {
        cvq(w->gate, w->gate_plane, w->gate_rowgain, L.vgate);
        cvq(w->up, w->up_plane, w->up_rowgain, L.vup);
        cvq(w->down, w->down_plane, w->down_rowgain, L.vdown);
        auto rvt = [&](const VqMat &m, VqTile &t) {
            repack_vq_tile_kernel<<<blocks_for(t.rows * t.nkb, 256), 256, 0, st>>>(m.stream, m.plane, t.rows, m.k,
                                                                                 const_cast<uint8_t *>(t.rec));
        };
        rvt(L.vgate, L.tvgate);
        rvt(L.vup, L.tvup);
        rvt(L.vdown, L.tvdown);
        cudaMemcpyAsync(const_cast<uint8_t *>(L.codebook), w->vq_codebook, (size_t)8 << L.vq, cudaMemcpyDeviceToDevice,
                        st);
    } else if (L.mx4) {
        rm4(w->gate, L.mgate);
        rm4(w->up, L.mup);
        rm4(w->down, L.mdown);
        rm4t(w->gate, L.tgate);
        rm4t(w->up, L.tup);
        rm4t(w->down, L.tdown);
    } else {
        rq2(w->gate, L.gate);
        rq2(w->up, L.up);
        rq2(w->down, L.down);
    }
    if (has_shared) {
        rq8(w->sh_gate, L.sh_gate);
        rq8(w->sh_up, L.sh_up);
        rq8(w->sh_down, L.sh_down);
    }
    if (L.gain)
        expand_gain_kernel<<<blocks_for((int64_t)L.E * L.H, 256), 256, 0, st>>>(
            static_cast<const uint8_t *>(w->down_gain), static_cast<const uint8_t *>(w->down_gain2), L.E, L.H,
            const_cast<float *>(L.gain));
    DecodeState &D = h->D;
    auto rf2 = [&](const void *src, Q2Frag &m) {
        const int64_t n = (m.rows / 16) * (m.nkc / 2) * 32; // one thread per (tile, block, lane)
        repack_q2_frag_kernel<<<blocks_for(n, 256), 256, 0, st>>>(static_cast<const uint8_t *>(src), m.rows, m.nkc / 2,
                                                                   const_cast<uint8_t *>(m.rec));
    };
    auto rf8 = [&](const void *src, Q8Frag &m) {
        const int64_t n = (m.rows / 16) * m.nbq * 32;
        repack_q8_frag_kernel<<<blocks_for(n, 256), 256, 0, st>>>(static_cast<const uint8_t *>(src), m.rows, m.nbq,
                                                                   const_cast<uint8_t *>(m.rec));
    };
    if (!L.mx4 && !L.vq) {
        rf2(w->gate, D.gate);
        rf2(w->up, D.up);
        rf2(w->down, D.down);
    }
    if (has_shared) {
        rf8(w->sh_gate, D.sh_gate);
        rf8(w->sh_up, D.sh_up);
        rf8(w->sh_down, D.sh_down);
    }
    cudaMemsetAsync(D.ctl, 0, sizeof(unsigned) * D.ctl_words, st);
    // no stale word may carry a future launch's epoch (epochs start at 1)
    cudaMemsetAsync(D.lgt, 0, sizeof(unsigned long long) * kDecodeT * L.E, st);
    cudaMemsetAsync(D.srec, 0, sizeof(unsigned long long) * 2 * kMaxSlots, st);
    // the rehearsal's logits: 0.0 with epoch 0, present from the start
    int per_sm = 0, nsm = 0;
    for (const void *fn : {(const void *)decode_fused_kernel<1>, (const void *)decode_fused_kernel<2>,
                           (const void *)decode_fused_kernel<4>, (const void *)decode_fused_kernel<8>,
                           (const void *)decode_fused_kernel<1, true>, (const void *)decode_fused_kernel<8, true>})
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(DecodeSmem));
    for (const void *fn : {(const void *)vq_product_kernel<true, 1>, (const void *)vq_product_kernel<true, 2>,
                           (const void *)vq_product_kernel<true, 4>, (const void *)vq_product_kernel<true, 8>,
                           (const void *)vq_product_kernel<false, 1>, (const void *)vq_product_kernel<false, 2>,
                           (const void *)vq_product_kernel<false, 4>, (const void *)vq_product_kernel<false, 8>})
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 << 13);
    // every variant has the same threads and shared memory and the same launch bound of two CTAs per SM
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel<8>, kDecodeThreads, sizeof(DecodeSmem));
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    D.grid = per_sm * nsm;
    g_pf_grid = nsm;
    {
        // the batch path where its shared memory fits: three stages per ring, else two (the
        // attribute belongs to the kernel, not to the layer: it allows the device maximum).
        // An 8-bit stage holds the widest column range that divides K within kBatchStageCap.
        // Its routed items serve 2-bit layers only, its shared items every layer.
        BatchState &B = h->B;
        const int optin = (int)prop.sharedMemPerBlockOptin;
        bool fits = true;
        for (int down = 0; down < 2; down++) {
            int chunk = 32;
            if (L.Ish > 0) {
                const int K = down ? L.Ish : L.H, tiles = down ? 4 : 2;
                for (int c = K; c >= 32; c -= 32)
                    if (K % c == 0 && tiles * (c / 32) * kQ8Rec <= kBatchStageCap) {
                        chunk = c;
                        break;
                    }
            }
            int ns = 3;
            while (ns >= 2 && BatchPlan(down, L.H, L.I, L.Ish, chunk, ns).total > optin)
                ns--;
            fits = fits && ns >= 2;
            B.nstage[down] = ns;
            B.chunk[down] = chunk;
            B.smem[down] = BatchPlan(down, L.H, L.I, L.Ish, chunk, ns).total;
        }
        if (fits) {
            const int tb = L.Tmax < kBatchMaxT ? L.Tmax : kBatchMaxT;
            B.tmax = L.mx4 || L.vq ? 0 : tb;
            B.sh_tmax = L.Ish > 0 ? tb : 0;
            B.grid = nsm;
            for (const void *fn :
                 {(const void *)batch_product_kernel<false, kBatchBoth>,
                  (const void *)batch_product_kernel<true, kBatchBoth>,
                  (const void *)batch_product_kernel<false, kBatchRouted>,
                  (const void *)batch_product_kernel<true, kBatchRouted>,
                  (const void *)batch_product_kernel<false, kBatchShared>,
                  (const void *)batch_product_kernel<true, kBatchShared>})
                cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        }
    }
    cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGroupSmemMax);
    cudaFuncSetAttribute(router_tile_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, router_tile_smem(16));
    cudaFuncSetAttribute(router_tile_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, router_tile_smem(64));
    rc = setup_gemm<pf::kFmtQ2, 2, pf::kEpiSwiGLU>();
    if (!rc)
        rc = setup_gemm<pf::kFmtQ2, 1, pf::kEpiF32>();
    if (!rc)
        rc = setup_gemm<pf::kFmtQ8, 2, pf::kEpiSwiGLUF16>();
    if (!rc)
        rc = setup_gemm<pf::kFmtQ8, 1, pf::kEpiF32>();
    if (!rc)
        rc = setup_gemm<pf::kFmtBF16, 1, pf::kEpiF32>();
    if (!rc)
        rc = setup_gemm<pf::kFmtMx4, 2, pf::kEpiSwiGLUFp4>();
    if (!rc)
        rc = setup_gemm<pf::kFmtMx4, 1, pf::kEpiF32>();
    if (!rc)
        rc = setup_gemm<pf::kFmtVq, 2, pf::kEpiSwiGLUF16>();
    if (!rc)
        rc = setup_gemm<pf::kFmtVq, 1, pf::kEpiF32>();
    if (rc || D.grid <= 0) {
        ds4moe_destroy(h);
        return DS4MOE_ECUDA;
    }
    rc = launch_rc();
    if (!rc)
        rc = cuda_rc(cudaStreamSynchronize(st));
    if (rc) {
        ds4moe_destroy(h);
        return rc;
    }
    *out = h;
    return DS4MOE_OK;
}

int ds4moe_destroy(ds4moe_t *h) {
    if (!h)
        return DS4MOE_OK;
    if (h->stream)
        cudaStreamSynchronize(h->stream);
    else
        cudaDeviceSynchronize();
    cudaFree(h->weight_mem);
    cudaFree(h->scratch_mem);
    cudaFree(h->status);
    delete h;
    return DS4MOE_OK;
}

int ds4moe_set_stream(ds4moe_t *h, void *stream) {
    if (!h)
        return DS4MOE_EINVAL;
    h->stream = static_cast<cudaStream_t>(stream);
    return DS4MOE_OK;
}

int ds4moe_route_detail(ds4moe_t *h, const void *x, int32_t T, int32_t *idx_out, float *w_out, float *gap_out,
                        float *sel_out) {
    int rc = check_call(h, x, T);
    if (rc)
        return rc;
    if (T == 0)
        return DS4MOE_OK;
    if (!is_device_ptr(idx_out) || !is_device_ptr(w_out) || (gap_out && !is_device_ptr(gap_out)) ||
        (sel_out && !is_device_ptr(sel_out)))
        return DS4MOE_EINVAL;
    h->stats = ds4moe_stats{};
    rc = run_router(h, x, T, sel_out);
    if (rc)
        return rc;
    const LayerDev &L = h->L;
    cudaStream_t st = h->stream;
    cudaMemcpyAsync(idx_out, h->S.idx, sizeof(int32_t) * T * L.K, cudaMemcpyDeviceToDevice, st);
    cudaMemcpyAsync(w_out, h->S.w, sizeof(float) * T * L.K, cudaMemcpyDeviceToDevice, st);
    if (gap_out)
        cudaMemcpyAsync(gap_out, h->S.gap, sizeof(float) * T, cudaMemcpyDeviceToDevice, st);
    return launch_rc();
}

int ds4moe_route(ds4moe_t *h, const void *x, int32_t T, int32_t *idx_out, float *w_out) {
    return ds4moe_route_detail(h, x, T, idx_out, w_out, nullptr, nullptr);
}

int ds4moe_forward_path(ds4moe_t *h, const void *x, int32_t T, int32_t path, float *y) {
    int rc = check_call(h, x, T);
    if (rc)
        return rc;
    if (path < DS4MOE_PATH_AUTO || path > DS4MOE_PATH_BATCH)
        return DS4MOE_EINVAL;
    if (T == 0)
        return DS4MOE_OK;
    if (!is_device_ptr(y) || !aligned(y, 16))
        return DS4MOE_EINVAL;
    path = resolve_path(h, T, path);
    if (path < 0)
        return DS4MOE_EINVAL;
    return forward_impl(h, x, T, path, y);
}

int ds4moe_forward(ds4moe_t *h, const void *x, int32_t T, float *y) {
    return ds4moe_forward_path(h, x, T, DS4MOE_PATH_AUTO, y);
}

int ds4moe_forward_routed(ds4moe_t *h, const void *x, int32_t T, const int32_t *idx, const float *w,
                          int32_t path, float *y) {
    int rc = check_call(h, x, T);
    if (rc)
        return rc;
    if (path < DS4MOE_PATH_AUTO || path > DS4MOE_PATH_BATCH)
        return DS4MOE_EINVAL;
    if (T == 0)
        return DS4MOE_OK;
    if (!is_device_ptr(idx) || !is_device_ptr(w) || !is_device_ptr(y) || !aligned(y, 16))
        return DS4MOE_EINVAL;
    path = resolve_path(h, T, path);
    if (path < 0)
        return DS4MOE_EINVAL;
    const LayerDev &L = h->L;
    Scratch &S = h->S;
    cudaStream_t st = h->stream;
    h->stats = ds4moe_stats{};
    h->stats.tokens = T;
    h->stats.path = path;
    if (path == DS4MOE_PATH_DECODE && !L.mx4 && !L.vq)
        return run_decode(h, x, T, y, idx, w);
    cudaMemcpyAsync(S.idx, idx, sizeof(int32_t) * T * L.K, cudaMemcpyDeviceToDevice, st);
    cudaMemcpyAsync(S.w, w, sizeof(float) * T * L.K, cudaMemcpyDeviceToDevice, st);
    rc = launch_rc();
    if (rc)
        return rc;
    if (L.vq)
        return path == DS4MOE_PATH_PREFILL ? run_experts_vq_tc(h, x, T, y) : run_experts_vq(h, x, T, y);
    if (L.mx4)
        return path == DS4MOE_PATH_PREFILL ? run_experts_mx4_tc(h, x, T, y) : run_experts_mx4(h, x, T, y);
    return path == DS4MOE_PATH_BATCH ? run_experts_batch(h, x, T, y, false) : run_experts_prefill(h, x, T, y);
}

int ds4moe_forward_host(ds4moe_t *h, const void *x_host, int32_t T, float *y_host) {
    if (!h || T < 0 || T > h->L.Tmax)
        return DS4MOE_EINVAL;
    if (T == 0)
        return DS4MOE_OK;
    if (!x_host || !y_host)
        return DS4MOE_EINVAL;
    const LayerDev &L = h->L;
    cudaStream_t st = h->stream;
    int rc = cuda_rc(cudaMemcpyAsync(h->S.xstage, x_host, sizeof(uint16_t) * T * L.H, cudaMemcpyHostToDevice, st));
    if (rc)
        return rc;
    rc = forward_impl(h, h->S.xstage, T, resolve_path(h, T, DS4MOE_PATH_AUTO), h->S.ystage);
    if (rc)
        return rc;
    rc = cuda_rc(cudaMemcpyAsync(y_host, h->S.ystage, sizeof(float) * T * L.H, cudaMemcpyDeviceToHost, st));
    if (rc)
        return rc;
    return cuda_rc(cudaStreamSynchronize(st));
}

int ds4moe_debug_skip_signal(ds4moe_t *h, int32_t launches) {
    if (!h || launches < 0)
        return DS4MOE_EINVAL;
    h->skip_signal = launches;
    return DS4MOE_OK;
}

int ds4moe_status(ds4moe_t *h) {
    if (!h)
        return DS4MOE_EINVAL;
    int rc = cuda_rc(cudaStreamSynchronize(h->stream));
    if (rc)
        return rc;
    unsigned bits = 0;
    rc = cuda_rc(cudaMemcpy(&bits, h->status, sizeof(unsigned), cudaMemcpyDeviceToHost));
    if (rc)
        return rc;
    if (bits)
        cudaMemset(h->status, 0, sizeof(unsigned));
    if (bits & kErrTimeout) {
        cudaMemset(h->D.ctl, 0, sizeof(unsigned) * h->D.ctl_words); // an aborted launch leaves them dirty
        return DS4MOE_ETIMEOUT;
    }
    if (bits)
        return DS4MOE_EDEVICE;
    return DS4MOE_OK;
}

int ds4moe_get_stats(ds4moe_t *h, ds4moe_stats *out) {
    if (!h || !out)
        return DS4MOE_EINVAL;
    int rc = cuda_rc(cudaStreamSynchronize(h->stream));
    if (rc)
        return rc;
    *out = h->stats;
    if (h->stats.tokens > 0) {
        // the fused decode kernel keeps its own grouping; every other path (and every
        // MXFP4 layer) the dispatch kernels'
        const bool dec = h->stats.path == DS4MOE_PATH_DECODE && !h->L.mx4 && !h->L.vq;
        int32_t n = 0;
        cudaMemcpy(&n, dec ? h->D.nuniq : h->S.nuniq, sizeof(int32_t), cudaMemcpyDeviceToHost);
        out->n_unique = n;
        int32_t *counts = static_cast<int32_t *>(malloc(sizeof(int32_t) * h->L.E));
        if (counts && cudaMemcpy(counts, dec ? h->D.counts : h->S.counts, sizeof(int32_t) * h->L.E,
                                 cudaMemcpyDeviceToHost) ==
                          cudaSuccess) {
            int mx = 0;
            for (int e = 0; e < h->L.E; e++)
                mx = counts[e] > mx ? counts[e] : mx;
            out->max_load = mx;
        }
        free(counts);
    }
    return cuda_rc(cudaGetLastError());
}

int ds4moe_inspect(ds4moe_t *h, int32_t T, int32_t *idx, float *w, float *gap, int32_t *counts, int32_t *inv,
                   int32_t *uexp, int32_t *ustart, int32_t *n_unique) {
    if (!h || T < 0 || T != h->stats.tokens)
        return DS4MOE_EINVAL;
    int rc = cuda_rc(cudaStreamSynchronize(h->stream));
    if (rc || T == 0)
        return rc;
    const LayerDev &L = h->L;
    const Scratch &S = h->S;
    const int64_t P = (int64_t)T * L.K;
    auto get = [&](void *dst, const void *src, size_t bytes) {
        if (dst && rc == DS4MOE_OK)
            rc = cuda_rc(cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
    };
    get(idx, S.idx, sizeof(int32_t) * P);
    get(w, S.w, sizeof(float) * P);
    get(gap, S.gap, sizeof(float) * T);
    if (rc || !(counts || inv || uexp || ustart || n_unique))
        return rc;
    const bool dec = h->stats.path == DS4MOE_PATH_DECODE && !L.mx4 && !L.vq;
    if (dec && T > kDecodeT)
        return DS4MOE_EINVAL; // the fused kernel keeps the grouping of its last launch only
    int32_t nu = 0;
    get(&nu, dec ? h->D.nuniq : S.nuniq, sizeof(int32_t));
    if (rc)
        return rc;
    if (nu < 0 || nu > P || nu > L.E)
        return DS4MOE_EDEVICE;
    if (n_unique)
        *n_unique = nu;
    get(counts, dec ? h->D.counts : S.counts, sizeof(int32_t) * L.E);
    get(inv, dec ? h->D.inv : S.inv, sizeof(int32_t) * P);
    if (!dec) {
        get(uexp, S.uexp, sizeof(int32_t) * nu);
        get(ustart, S.uoff, sizeof(int32_t) * (nu + 1));
        return rc;
    }
    // the decode kernel's slot records: expert in bits 0-10, first position in bits 11-17
    std::vector<unsigned long long> rec(2 * (size_t)nu);
    get(rec.data(), h->D.srec, sizeof(unsigned long long) * rec.size());
    if (rc)
        return rc;
    for (int s = 0; s < nu; s++) {
        const unsigned w0 = (unsigned)rec[2 * s];
        if (uexp)
            uexp[s] = (int32_t)(w0 & 0x7FFu);
        if (ustart)
            ustart[s] = (int32_t)((w0 >> 11) & 0x7Fu);
    }
    if (ustart)
        ustart[nu] = (int32_t)P;
    return rc;
}

int ds4moe_profile(ds4moe_t *h, int32_t enable) {
    if (!h)
        return DS4MOE_EINVAL;
    int rc = cuda_rc(cudaStreamSynchronize(h->stream));
    if (rc)
        return rc;
    if (enable)
        h->prof.clear();
    else
        h->prof.drain();
    h->prof.on = enable != 0;
    return DS4MOE_OK;
}

int ds4moe_profile_read(ds4moe_t *h, ds4moe_kernel_time *out, int32_t max, int32_t *n_out) {
    if (!h || !n_out || max < 0 || (max > 0 && !out))
        return DS4MOE_EINVAL;
    int rc = cuda_rc(cudaStreamSynchronize(h->stream));
    if (rc)
        return rc;
    h->prof.drain();
    const int n = (int)h->prof.names.size();
    for (int i = 0; i < n && i < max; i++) {
        memset(out[i].name, 0, sizeof(out[i].name));
        strncpy(out[i].name, h->prof.names[i].c_str(), sizeof(out[i].name) - 1);
        out[i].launches = h->prof.launches[i];
        out[i].total_ms = h->prof.total_ms[i];
    }
    *n_out = n;
    return DS4MOE_OK;
}

int ds4moe_memory(ds4moe_t *h, uint64_t *weight_bytes, uint64_t *scratch_bytes) {
    if (!h)
        return DS4MOE_EINVAL;
    if (weight_bytes)
        *weight_bytes = h->weight_bytes;
    if (scratch_bytes)
        *scratch_bytes = h->scratch_bytes;
    return DS4MOE_OK;
}

} // extern "C"

// ---- routing without allocation ------------------------------------------------
//
// The scratch of ds4moe_route_noalloc lives in this file-scope device array.
// Host code may not use the symbol as a pointer: its device address is looked
// up with cudaGetSymbolAddress for the current device and context on every
// call (a lookup, no allocation), so a context that was reset or replaced
// never receives a stale address.

static __device__ __align__(256) unsigned char g_noalloc_scratch[DS4MOE_NOALLOC_SCRATCH];

namespace {

// Device address of the scratch array on the current device; *dev gets that device.
int noalloc_scratch(void **out, int *dev) {
    int rc = cuda_rc(cudaGetDevice(dev));
    if (rc)
        return rc;
    int major = 0, minor = 0;
    rc = cuda_rc(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev));
    if (!rc)
        rc = cuda_rc(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev));
    if (rc)
        return rc;
    if (major != 10 || minor != 3)
        return DS4MOE_EUNSUPPORTED;
    void *p = nullptr;
    rc = cuda_rc(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    if (rc)
        return rc;
    *out = p;
    return DS4MOE_OK;
}

// A device (or managed) pointer of device `dev`.
bool on_device(const void *p, int dev) {
    if (!p)
        return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
}

uint64_t round256(uint64_t n) { return (n + 255) & ~uint64_t(255); }

} // namespace

extern "C" int ds4moe_route_noalloc(const float *router_w, const float *router_bias, const void *x_bf16,
                                    int32_t T, int32_t H, int32_t E, int32_t K, int32_t *idx_out, float *w_out,
                                    void *stream) {
    if (T < 0 || H <= 0 || H % 256 || E < 1 || E > 1024 || K < 1 || K > kMaxTopK || K > E)
        return DS4MOE_EINVAL;
    if (T == 0)
        return DS4MOE_OK;
    const uint64_t x32_bytes = round256(4ull * T * H);
    const uint64_t xsum_bytes = round256(4ull * T * (H / 16));
    const uint64_t logit_bytes = round256(4ull * T * E);
    if (x32_bytes + xsum_bytes + logit_bytes > DS4MOE_NOALLOC_SCRATCH)
        return DS4MOE_ESCRATCH;
    void *base = nullptr;
    int dev = 0;
    int rc = noalloc_scratch(&base, &dev);
    if (rc)
        return rc;
    // every buffer and the stream on the current device (the scratch's)
    if (!on_device(router_w, dev) || !aligned(router_w, 16) || !on_device(x_bf16, dev) || !aligned(x_bf16, 16) ||
        !on_device(idx_out, dev) || !on_device(w_out, dev) || (router_bias && !on_device(router_bias, dev)))
        return DS4MOE_EINVAL;
    if (stream) {
        int sdev = -1;
        if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
            cudaGetLastError();
            return DS4MOE_EINVAL;
        }
        if (sdev != dev)
            return DS4MOE_EINVAL;
    }
    float *x32 = static_cast<float *>(base);
    float *xsum = reinterpret_cast<float *>(static_cast<char *>(base) + x32_bytes);
    float *logits = reinterpret_cast<float *>(static_cast<char *>(base) + x32_bytes + xsum_bytes);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prep_x_kernel<<<blocks_for((int64_t)T * (H / 16), 256), 256, 0, st>>>(static_cast<const uint16_t *>(x_bf16), T,
                                                                         H, x32, xsum);
    router_logits_kernel<<<dim3(blocks_for(E, 8), blocks_for(T, kRouterTok)), 256, 0, st>>>(x32, T, H, router_w, E,
                                                                                          logits);
    const size_t smem = (size_t)kSelectSmemPerExpert * E;
    router_select_kernel<<<T, kSelectThreads, smem, st>>>(
        logits, router_bias, T, E, K, idx_out, w_out, nullptr, nullptr, nullptr, nullptr, 0, 1, 0);
    return launch_rc();
}
