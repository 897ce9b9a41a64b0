/*
 * ds4moe: the routed mixture-of-experts FFN layer of a DeepSeek-V4-Flash-shaped
 * model on one NVIDIA GB300 (sm_103a), as a C ABI.
 *
 * What one call computes, for T tokens x[T][H] (bf16):
 *
 *   L[t,e]   = sum_h x[t,h] Wr[e,h]                         router logits (fp32)
 *   s[t,e]   = sigmoid(L[t,e]);  sel = s + b_e              selection score (b optional)
 *   idx[t,:] = the K experts of largest sel, in descending order, equal scores
 *              resolved towards the lower expert index
 *   w[t,k]   = s[t,idx[t,k]] / sum_j s[t,idx[t,j]]          mixing weights (bias-free)
 *   ye       = Wd[e] (silu(Wg[e] x_t) * (Wu[e] x_t))        SwiGLU expert, 2-bit weights
 *   ysh      = same with the 8-bit shared expert
 *   y[t]     = sum_k w[t,k] (g_{idx[t,k]} * ye_{idx[t,k]}(x_t)) + ysh(x_t)
 *              with g_e[j] = s1_e[j] * s2_e[j] the optional per-expert down
 *              gains (elementwise over the H output channels; 1 when absent)
 *
 * The block sum with an unweighted shared expert is the engine's MoE sum of
 * "YoungAi - DeepSeek V4.1 Flash on one DGX Spark", section 4.2 ("The
 * objective"). Its per-expert, per-output-channel gains s_e are the sidecar and
 * post-training files of the same page (section 3: g_eff = g_base * s_sidecar *
 * s_posttrain, one factor per down-projection row of an expert; section 4.2:
 * FP4 E2M1 values of s - 1 with one scale per 32 in 17-byte blocks): the two
 * optional gain tables s1, s2 below. The router bias is added to the
 * selection score only, mixing weights untouched (same page, section 3 and
 * section 4.2, "The router bias"). 384 experts, 6 per token: same page,
 * section 2.2. Only the routed experts are 2-bit; the shared expert stays
 * 8-bit ("Running DeepSeek V4 Flash on an RTX 5080 ...": routed up/gate and
 * down are 2-bit, shared experts are left untouched; the ds4 teardown on
 * txtmix.com, section 3, names the shared-expert recipe SExpQ8).
 *
 * Storage formats the caller hands to ds4moe_create (little-endian, rows of
 * consecutive weights along the reduction dimension K):
 *   2-bit block, 84 bytes per 256 weights:
 *     [0,16)  scales[j], j = 0..15: low nibble sc_j, high nibble m_j of the
 *             sub-block of weights 16j..16j+15
 *     [16,80) qs: code q_i of weight i at byte 16 + i/4, bits 2*(i%4)..+1
 *     [80,82) d (binary16)   [82,84) dmin (binary16)
 *     weight i = d * sc_{i/16} * q_i - dmin * m_{i/16}
 *   8-bit block, 34 bytes per 32 weights: [0,2) d (binary16), [2,34) int8 q_i;
 *     weight i = d * q_i
 *   router_w   fp32 [E][H];  router_bias fp32 [E] or NULL
 *   gate, up   2-bit [E][I][H/256] blocks;  down 2-bit [E][H][I/256] blocks
 *   sh_gate, sh_up 8-bit [I_sh][H/32];  sh_down 8-bit [H][I_sh/32]
 *   down-gain block, 17 bytes per 32 consecutive output channels of one expert:
 *     [0,16)  FP4 E2M1 code c_i of channel i at byte i/2, low nibble for even i
 *             (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa;
 *             magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6)
 *     [16]    E8M0 scale X = 2^(byte - 127) (0xFF is NaN and propagates)
 *     gain i = 1 + X * e2m1(c_i)
 *   down_gain, down_gain2   [E][H/32] gain blocks each, or NULL (all gains 1)
 *
 * Conventions of every entry point:
 *   - Return 0 (DS4MOE_OK) or a negative DS4MOE_E* code; nothing is launched
 *     when an argument is rejected. ds4moe_strerror names each code.
 *   - "device" pointers must be CUDA device (or managed) memory of the handle's
 *     device; host pointers are rejected with DS4MOE_EINVAL.
 *   - Compute calls are asynchronous on the handle's stream (ds4moe_set_stream;
 *     default: the legacy default stream). Caller buffers must stay valid until
 *     the stream reaches the call. A handle may not be used by two host threads
 *     at once; calls on one handle are serialised by its stream.
 *   - Errors found by kernels (a wait that timed out, a routed index that had
 *     to be clamped or replaced) are sticky in the handle and reported by
 *     ds4moe_status.
 *   - NaN or Inf inputs are not checked and propagate.
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4MOE_MAGIC 0x454D3444u /* "D4ME" */
#define DS4MOE_VERSION 3u /* 2: ds4moe_weights gained down_gain, down_gain2; 3: the VQ fields */

enum {
    DS4MOE_OK = 0,
    DS4MOE_EINVAL = -1,       /* bad argument: pointer, shape, token count, magic/version */
    DS4MOE_ENOMEM = -2,       /* device allocation failed */
    DS4MOE_ECUDA = -3,        /* a CUDA call or launch failed */
    DS4MOE_EUNSUPPORTED = -4, /* device is not compute capability 10.3 (GB300) */
    DS4MOE_ETIMEOUT = -5,     /* a bounded device-side wait gave up */
    DS4MOE_EDEVICE = -6,      /* a kernel reported an internal inconsistency */
    DS4MOE_ESCRATCH = -7      /* request needs more than the fixed scratch of ds4moe_route_noalloc */
};

/*
 * Layer flag: the routed gate/up/down weights are MXFP4 instead of 2-bit
 * ("Running DeepSeek V4 Flash on an RTX 5080 ...", model list: the MXFP4 GGUF
 * keeps DeepSeek's released MXFP4 routed experts; decode runs them on Q8
 * activations). OCP microscaling element and scale types:
 *   MXFP4 block, 17 bytes per 32 consecutive weights of one row: 16 bytes of
 *     E2M1 codes (weight i at byte i/2, low nibble for even i), then the E8M0
 *     scale X = 2^(byte - 127);   w_i = X * e2m1(c_i).
 *   gate, up [E][I][H/32] blocks; down [E][H][I/32] blocks (router, shared
 *   expert and down gains unchanged).
 * Each routed-expert product quantises its input per 32 values first (x, and
 * the SwiGLU rows, rounded to binary32, before the down product). Decode form:
 * d = amax / 127, q = x / d rounded to the nearest integer (ties to even), both
 * in binary32; the product uses d * q. Prefill form (the model page's note on
 * Blackwell: batched expert work runs on FP4 matrix instructions with FP4
 * activations): the OCP MX conversion, X = 2^(floor(log2 amax) - 2) and the E2M1 value nearest
 * to x / X (ties to even, saturating at 6); the product uses X * e2m1. The
 * prefill form runs on the tensor cores with both operands in binary16, exact
 * for weight scale bytes 104..141 and activation blocks with amax in
 * [2^-21, 2^16). The path argument picks the form (see
 * DS4MOE_AUTO_MX4_PREFILL_MIN_T); DS4MOE_AUTO_DECODE_MAX_T does not apply.
 */
#define DS4MOE_FLAG_MXFP4 1u

/*
 * Layer flags: the routed experts are vector-quantised ("YoungAi - DeepSeek
 * V4.1 Flash on one DGX Spark", section 4.1): every 8 consecutive weights of a
 * row are one codeword of a per-layer codebook (2^bits entries of 8 OCP FP8
 * E4M3 values, shared by all experts and the three matrices) times one
 * binary16 gain per row, w[r, 8j .. 8j+7] = g_r * C[idx[r, j]].
 *   gate, up, down: per expert the index stream of the matrix, its rows back
 *     to back (row r, group j = index r * K/8 + j), 12 bits per index, least
 *     significant bit first (index k at bits 12k .. 12k+11): I*H*3/16 bytes
 *     per expert for gate and up, H*I*3/16 for down;
 *   *_plane: 13-bit layers, bit k (least significant first) = bit 12 of index k;
 *   *_rowgain: binary16 g_r per row; vq_codebook: entry n at bytes 8n .. 8n+7.
 * Activations are not quantised (the tensor-core form rounds x and the SwiGLU
 * rows to binary16, see DS4MOE_AUTO_VQ_PREFILL_MIN_T).
 */
#define DS4MOE_FLAG_VQ12 2u
#define DS4MOE_FLAG_VQ13 4u

/*
 * DS4MOE_PATH_AUTO takes the decode path for T <= DS4MOE_AUTO_DECODE_MAX_T,
 * the batch path for T <= DS4MOE_AUTO_BATCH_MAX_T (where the layer has one)
 * and the prefill path above: the measured crossovers on a GB300 at H=4096,
 * I=2048, E=384, top-6.
 */
#define DS4MOE_AUTO_DECODE_MAX_T 1
#define DS4MOE_AUTO_BATCH_MAX_T 64

/*
 * Layers with MXFP4 routed experts (DS4MOE_FLAG_MXFP4) have two forms: decode
 * (Q8 activations, CUDA-core integer products; DS4MOE_PATH_DECODE and _BATCH)
 * and prefill (FP4 activations, grouped GEMMs on the tensor cores;
 * DS4MOE_PATH_PREFILL). DS4MOE_PATH_AUTO takes the prefill form from this many
 * tokens on: the measured crossover on a GB300 at H=4096, I=2048, E=384, top-6
 * (the pages pair Q8 activations with decode and FP4 activations with batched
 * expert work; the boundary between the two sits where the tensor-core form
 * becomes the faster one).
 */
#define DS4MOE_AUTO_MX4_PREFILL_MIN_T 3

/*
 * Layers with VQ routed experts (DS4MOE_FLAG_VQ12, _VQ13) have two forms of
 * the same arithmetic: CUDA-core products (DS4MOE_PATH_DECODE and _BATCH) and
 * grouped GEMMs on the tensor cores (DS4MOE_PATH_PREFILL: codewords exact in
 * binary16, x and the SwiGLU rows rounded to binary16). DS4MOE_PATH_AUTO takes
 * the tensor-core form from this many tokens on: measured on a GB300 at H=4096,
 * I=2048, E=384, top-6, it is the faster form at every T (174 vs 226 us at T=1).
 */
#define DS4MOE_AUTO_VQ_PREFILL_MIN_T 1

/*
 * Most tokens one call of the batch path takes. The shared expert takes the
 * batch path's 8-bit tile GEMV (exact products, fp32 sums) in every path and
 * format up to this many tokens (and max_tokens); the fused decode kernel
 * holds its own, and larger calls take the tensor-core GEMMs.
 */
#define DS4MOE_BATCH_MAX_T 64

/* Execution paths for ds4moe_forward_path. */
enum {
    DS4MOE_PATH_AUTO = 0,    /* by T, see DS4MOE_AUTO_DECODE_MAX_T */
    DS4MOE_PATH_DECODE = 1,  /* fused dequant-GEMV kernel, launches of up to 8 tokens */
    DS4MOE_PATH_PREFILL = 2, /* grouped GEMM on tcgen05 tensor cores */
    DS4MOE_PATH_BATCH = 3    /* 2-bit layers, T <= min(max_tokens, DS4MOE_BATCH_MAX_T): routing and
                                grouping, then two persistent tile-GEMV kernels that read each
                                chosen expert once for up to 8 of its (token, k) pairs */
};

typedef struct ds4moe ds4moe_t; /* opaque handle */

/* Layer description. All sizes are element counts. */
typedef struct {
    uint32_t magic;       /* DS4MOE_MAGIC */
    uint32_t version;     /* DS4MOE_VERSION */
    int32_t hidden;       /* H, multiple of 256 */
    int32_t inter;        /* I (routed intermediate), multiple of 256 */
    int32_t n_experts;    /* E, 1..1024 */
    int32_t top_k;        /* K, 1..min(E, 8) */
    int32_t shared_inter; /* I_sh, multiple of 256, or 0 for no shared expert */
    int32_t max_tokens;   /* largest T any call will pass, 1..65536 */
    uint32_t flags;       /* 0 or one of DS4MOE_FLAG_MXFP4, DS4MOE_FLAG_VQ12, DS4MOE_FLAG_VQ13 */
} ds4moe_layer_desc;

/* Device pointers to the weights in the storage formats above. */
typedef struct {
    const float *router_w;    /* [E][H] */
    const float *router_bias; /* [E] or NULL */
    const void *gate;         /* 2-bit [E][I][H/256] (MXFP4: [E][I][H/32] blocks; VQ: index streams) */
    const void *up;           /* 2-bit [E][I][H/256] (MXFP4: [E][I][H/32]; VQ: index streams) */
    const void *down;         /* 2-bit [E][H][I/256] (MXFP4: [E][H][I/32]; VQ: index streams) */
    const void *sh_gate;      /* 8-bit [I_sh][H/32], NULL iff I_sh == 0 */
    const void *sh_up;        /* 8-bit [I_sh][H/32], NULL iff I_sh == 0 */
    const void *sh_down;      /* 8-bit [H][I_sh/32], NULL iff I_sh == 0 */
    const void *down_gain;    /* gain blocks [E][H/32] (sidecar), or NULL */
    const void *down_gain2;   /* gain blocks [E][H/32] (post-training), or NULL */
    /* VQ layers only (DS4MOE_FLAG_VQ12 / DS4MOE_FLAG_VQ13), else NULL: */
    const void *vq_codebook;  /* 2^bits x 8 E4M3 bytes */
    const void *gate_plane;   /* bit planes [E][I*H/64] bytes (13-bit only, else NULL) */
    const void *up_plane;     /* [E][I*H/64] */
    const void *down_plane;   /* [E][H*I/64] */
    const void *gate_rowgain; /* binary16 [E][I] */
    const void *up_rowgain;   /* binary16 [E][I] */
    const void *down_rowgain; /* binary16 [E][H] */
} ds4moe_weights;

/*
 * Validate the description, copy every weight into library-owned device
 * memory in the kernels' layout, size the scratch for max_tokens, and
 * synchronise. The caller's weight buffers may be freed once this returns.
 * Down-gain tables, when given, are decoded here into one fp32 gain per expert
 * and output channel (the product of the two tables; 4*E*H bytes); a handle
 * created with gains runs the decode kernel built for them.
 * Runs on the current device, which must be a GB300 (sm_103).
 * Errors: EINVAL (desc, NULL or host pointer), EUNSUPPORTED, ENOMEM, ECUDA.
 */
int ds4moe_create(const ds4moe_layer_desc *desc, const ds4moe_weights *weights, ds4moe_t **out);

/* Free everything the handle owns (synchronises its stream first). NULL is OK. */
int ds4moe_destroy(ds4moe_t *h);

/* Issue later calls on this cudaStream_t (NULL = legacy default stream). */
int ds4moe_set_stream(ds4moe_t *h, void *cuda_stream);

/*
 * Routing only. x_bf16: device [T][H] bf16. Writes idx_out device int32 [T][K]
 * and w_out device fp32 [T][K]. 0 <= T <= max_tokens; T == 0 does nothing.
 */
int ds4moe_route(ds4moe_t *h, const void *x_bf16, int32_t T, int32_t *idx_out, float *w_out);

/*
 * The layer. x_bf16: device [T][H] bf16; y: device fp32 [T][H].
 * 0 <= T <= max_tokens; T == 0 does nothing. Picks the path by T
 * (DS4MOE_PATH_AUTO, see DS4MOE_AUTO_DECODE_MAX_T).
 */
int ds4moe_forward(ds4moe_t *h, const void *x_bf16, int32_t T, float *y);

/*
 * The layer from and to HOST memory: copies x_host (bf16 [T][H]) to the device,
 * runs ds4moe_forward, copies y back to y_host (fp32 [T][H]) and waits for the
 * copy. Pinned host buffers give the fastest copies; pageable ones work.
 */
int ds4moe_forward_host(ds4moe_t *h, const void *x_host, int32_t T, float *y_host);

/*
 * ds4moe_forward with an explicit path (DS4MOE_PATH_*). The decode and prefill
 * paths accept any T; the batch path T <= min(max_tokens, DS4MOE_BATCH_MAX_T)
 * (DS4MOE_EINVAL above that, or when the layer's shared memory plan does not
 * fit the device). MXFP4 and VQ layers run their one pipeline for every path.
 */
int ds4moe_forward_path(ds4moe_t *h, const void *x_bf16, int32_t T, int32_t path, float *y);

/*
 * The layer for a caller-given routing (no router): idx device int32 [T][K]
 * with 0 <= idx < E, w device fp32 [T][K]. Used to compare the expert and
 * combine stages on tokens whose routing is a near-tie. Indices out of range
 * are clamped by the kernels and reported as DS4MOE_EDEVICE by ds4moe_status.
 * A token's K indices should be distinct: the decode path (T <= 8 per launch)
 * replaces a repeated index by the smallest index the token's row does not
 * hold and reports DS4MOE_EDEVICE; the prefill and batch paths apply the expert once per
 * occurrence.
 */
int ds4moe_forward_routed(ds4moe_t *h, const void *x_bf16, int32_t T, const int32_t *idx,
                          const float *w, int32_t path, float *y);

/*
 * Routing with diagnostics: like ds4moe_route, and also gap_out device fp32 [T]
 * = the K-th minus the (K+1)-th largest fp32 selection score (+inf when K == E),
 * and, if sel_out is not NULL, the fp32 selection scores [T][E].
 */
int ds4moe_route_detail(ds4moe_t *h, const void *x_bf16, int32_t T, int32_t *idx_out, float *w_out,
                        float *gap_out, float *sel_out);

/* Synchronise the handle's stream; return and clear the sticky device error. */
int ds4moe_status(ds4moe_t *h);

/*
 * Test hook for the failure detection of the persistent kernels: in each of
 * the next `launches` product launches of the batch path (DS4MOE_PATH_BATCH),
 * CTA 0 issues nothing for its first ring stage, so the bounded waits on that
 * stage run out (about a second), the CTA's roles stop and drain their own
 * copies, and ds4moe_status then returns DS4MOE_ETIMEOUT; the device and the
 * handle stay usable, the outputs of those calls are undefined. 0 turns it off.
 * Errors: EINVAL (NULL handle, launches < 0).
 */
int ds4moe_debug_skip_signal(ds4moe_t *h, int32_t launches);

/* Statistics of the last forward call (read after ds4moe_status). */
typedef struct {
    int32_t tokens;        /* T of the last call */
    int32_t path;          /* DS4MOE_PATH_DECODE, DS4MOE_PATH_PREFILL or DS4MOE_PATH_BATCH */
    int32_t n_unique;      /* distinct routed experts touched */
    int32_t max_load;      /* most (token, k) pairs on one expert */
    int32_t kernel_count;  /* kernels the call launched */
} ds4moe_stats;

int ds4moe_get_stats(ds4moe_t *h, ds4moe_stats *out);

/*
 * Test entry point: the routing and the token-to-expert grouping of the last
 * forward call, copied to HOST buffers (synchronises the stream). T must be
 * that call's token count. Any output may be NULL.
 *   idx [T][K], w [T][K], gap [T]   the routing the call used (for the router
 *                                   paths: the experts, weights and K-th minus
 *                                   (K+1)-th selection score of each token)
 *   counts [E]                      (token, k) pairs per expert
 *   inv [T][K]                      position of pair p = t*K + k in the
 *                                   expert-grouped order: experts ascending,
 *                                   pairs of one expert in ascending p
 *   uexp [n_unique], ustart [n_unique + 1]
 *                                   the distinct experts in that order and the
 *                                   first position of each (ustart[n] = T*K)
 *   n_unique                        number of distinct experts
 * The decode path keeps the grouping of its last launch of up to 8 tokens only:
 * after a decode call with T > 8 the grouping outputs must be NULL.
 * Errors: EINVAL (NULL handle, T not the last call's, grouping after a long
 * decode call), ECUDA, EDEVICE (a grouping the kernels left inconsistent).
 */
int ds4moe_inspect(ds4moe_t *h, int32_t T, int32_t *idx, float *w, float *gap, int32_t *counts, int32_t *inv,
                   int32_t *uexp, int32_t *ustart, int32_t *n_unique);

/*
 * Device bytes the handle owns: repacked weights and scratch. The weights
 * count every resident layout: the routed experts twice (the tensor-core
 * tile layout and the layout of the CUDA-core products: 2 x 3.17 GB for a
 * 2-bit layer at H=4096, I=2048, E=384) and the 8-bit shared expert twice
 * (tile layout and the tile GEMV's fragment layout), besides the router.
 */
int ds4moe_memory(ds4moe_t *h, uint64_t *weight_bytes, uint64_t *scratch_bytes);

/*
 * Per-kernel timing with CUDA events recorded on the handle's stream around
 * every kernel the library launches. ds4moe_profile(h, 1) clears the records
 * and starts recording; ds4moe_profile(h, 0) stops. ds4moe_profile_read
 * synchronises the stream and writes up to max entries (one per kernel name,
 * in first-launch order) with the number of launches and their summed device
 * time; *n_out gets the number of entries. Recording adds one event pair per
 * launch; leave it off when timing whole calls.
 */
typedef struct {
    char name[48];
    int32_t launches;
    double total_ms;
} ds4moe_kernel_time;

int ds4moe_profile(ds4moe_t *h, int32_t enable);
int ds4moe_profile_read(ds4moe_t *h, ds4moe_kernel_time *out, int32_t max, int32_t *n_out);

/*
 * Routing that allocates nothing. The pages have no counterpart; this entry
 * point exists for callers that cannot allocate device memory at call time:
 * an engine that reserves all of HBM for its own pools at start-up, or a
 * latency-critical caller for whom cudaMalloc's implicit device-wide
 * synchronisation is not acceptable. It also routes without building a handle
 * (ds4moe_create copies the whole layer).
 *
 * Computes what ds4moe_route computes, from the caller's router weights:
 *   router_w    device fp32 [E][H], 16-byte aligned
 *   router_bias device fp32 [E] or NULL (added to the selection score only)
 *   x_bf16      device bf16 [T][H], 16-byte aligned
 *   idx_out     device int32 [T][K];  w_out device fp32 [T][K]
 *   stream      cudaStream_t the kernels run on (NULL = legacy default stream)
 * with H a multiple of 256, 1 <= E <= 1024, 1 <= K <= min(E, 8), T >= 0.
 *
 * The scratch (activations widened to fp32, their 16-element sums and the
 * logits) is one statically allocated device array of DS4MOE_NOALLOC_SCRATCH
 * bytes, which every GPU that loads the library keeps until the process
 * exits. A call needs 4*T*(H + H/16 + E) bytes plus up to 768 bytes of
 * alignment; larger requests return DS4MOE_ESCRATCH and launch nothing (with
 * H=4096 and E=384 that is T <= 221). The call never calls cudaMalloc or
 * cudaFree and launches three kernels on `stream`.
 *
 * Every call runs on the current device: all buffers must be memory of that
 * device and `stream` a stream of it (else EINVAL). Each call looks the
 * array's device address up for the current device and context
 * (cudaGetSymbolAddress: a lookup that allocates nothing), so the entry point
 * stays valid after cudaDeviceReset or under another context. The first call
 * on a device may load the library's device code: make it before any stream
 * capture. All calls share the one array, which keeps the last call's
 * contents (nothing in it needs to start at zero): calls whose kernels can
 * overlap on the GPU, such as calls on different streams that are not
 * ordered, race on it and must be serialised by the caller.
 * Errors: EINVAL, ESCRATCH (checked first), EUNSUPPORTED (device not sm_103),
 * ECUDA.
 */
#define DS4MOE_NOALLOC_SCRATCH (4u << 20)

int ds4moe_route_noalloc(const float *router_w, const float *router_bias, const void *x_bf16, int32_t T,
                         int32_t H, int32_t E, int32_t K, int32_t *idx_out, float *w_out, void *stream);

/* Static string for a return code. */
const char *ds4moe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* DS4MOE_H */
