/*
 * Seeded synthetic inputs for the routed-MoE layer: weights in their canonical
 * storage layout, router matrices, router biases and bf16 activations.
 *
 * This file holds no arithmetic of the layer itself. It only draws random
 * numbers and encodes them into the storage formats (IEEE binary16, bfloat16,
 * the 84-byte 2-bit block and the 34-byte 8-bit block). Both the CPU oracle
 * tests and the GPU path consume what it writes.
 *
 * Random numbers come from a counter-based SplitMix64 (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; the finaliser
 * constants are those of Vigna's public-domain splitmix64.c). Output i of a
 * stream with key k is mix(k + (i + 1) * gamma), so every element can be drawn
 * independently and the fill loops parallelise without changing any value.
 * Normals use the Box-Muller transform.
 *
 * Canonical layouts written here (little-endian):
 *   2-bit block, 84 bytes per 256 consecutive weights of one row:
 *     [0,16)  scales[j] : low nibble = scale of sub-block j, high nibble = min
 *     [16,80) qs        : code of weight i at byte 16 + i/4, bits 2*(i%4)..+1
 *     [80,82) d    binary16
 *     [82,84) dmin binary16
 *   8-bit block, 34 bytes per 32 consecutive weights of one row:
 *     [0,2) d binary16, [2,34) int8 codes
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of stream `stream` under seed `seed`. */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return sm64_mix(seed ^ sm64_mix(stream * GAMMA + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i)
{
    return sm64_mix(key + (i + 1) * GAMMA);
}

/* Uniform in (0, 1] and [0, 1) from the top 53 bits. */
static inline double unit_open0(uint64_t r) { return ((double)(r >> 11) + 1.0) * 0x1.0p-53; }
static inline double unit_closed0(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }

/* Two standard normals from two draws (Box-Muller). */
static inline void normal_pair(uint64_t r1, uint64_t r2, double *z0, double *z1)
{
    const double two_pi = 6.283185307179586476925286766559;
    double rad = sqrt(-2.0 * log(unit_open0(r1)));
    double th = two_pi * unit_closed0(r2);
    *z0 = rad * cos(th);
    *z1 = rad * sin(th);
}

static inline uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* float -> bfloat16, round to nearest even (inputs here are finite). */
static inline uint16_t to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* float -> IEEE binary16, round to nearest even, with subnormals and overflow
 * to infinity (inputs here are finite). */
static inline uint16_t to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag >= 0x477FF000u) /* rounds to >= 65520: infinity */
        return (uint16_t)(sign | 0x7C00u);
    int e = (int)(mag >> 23) - 127;
    uint32_t m = (mag & 0x7FFFFFu) | 0x800000u; /* 24-bit significand */
    if (mag == 0)
        return (uint16_t)sign;
    if (e >= -14) {
        /* normal half: keep 11 bits of the 24-bit significand */
        uint32_t shift = 13;
        uint32_t keep = m >> shift, rem = m & ((1u << shift) - 1), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (keep & 1u)))
            keep++;
        uint32_t he = (uint32_t)(e + 15);
        if (keep == 0x800u) { keep = 0x400u; he++; }
        if (he >= 31)
            return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (he << 10) | (keep & 0x3FFu));
    }
    /* subnormal half: value = m * 2^(e-23); unit is 2^-24 */
    int shift = -e - 14 + 13; /* bits to drop from m */
    if (shift > 24)
        return (uint16_t)sign;
    uint32_t keep = m >> shift, rem = m & ((1u << shift) - 1), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (keep & 1u)))
        keep++;
    return (uint16_t)(sign | keep); /* keep == 0x400 becomes the smallest normal */
}

/* Exposed for the generator's own tests. */
uint16_t synth_to_f16(float f) { return to_f16(f); }
uint16_t synth_to_bf16(float f) { return to_bf16(f); }

/*
 * 2-bit blocks: codes and the 4-bit scales/mins uniform, d and dmin |N(0, sigma)|.
 * Block b uses draws 12*b .. 12*b+11 of the stream.
 */
void synth_fill_q2(uint8_t *out, int64_t nblocks, uint64_t seed, uint64_t stream, double sigma)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint8_t *blk = out + b * 84;
        uint64_t base = (uint64_t)b * 12;
        for (int w = 0; w < 10; w++) { /* 80 random bytes: scales then codes */
            uint64_t r = draw(key, base + w);
            memcpy(blk + 8 * w, &r, 8);
        }
        double z0, z1;
        normal_pair(draw(key, base + 10), draw(key, base + 11), &z0, &z1);
        uint16_t d = to_f16((float)(fabs(z0) * sigma));
        uint16_t dmin = to_f16((float)(fabs(z1) * sigma));
        blk[80] = (uint8_t)(d & 0xFF);
        blk[81] = (uint8_t)(d >> 8);
        blk[82] = (uint8_t)(dmin & 0xFF);
        blk[83] = (uint8_t)(dmin >> 8);
    }
}

/*
 * Down-gain blocks (17 bytes per 32 channels): 16 bytes of uniform random FP4
 * codes, then the E8M0 scale byte `scale_byte` (the same for every block).
 * Block b uses draws 2*b, 2*b+1 of the stream.
 */
void synth_fill_gain(uint8_t *out, int64_t nblocks, uint64_t seed, uint64_t stream, uint8_t scale_byte)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint8_t *blk = out + b * 17;
        for (int w = 0; w < 2; w++) {
            uint64_t r = draw(key, (uint64_t)b * 2 + w);
            memcpy(blk + 8 * w, &r, 8);
        }
        blk[16] = scale_byte;
    }
}

/*
 * MXFP4 blocks (17 bytes per 32 weights): 16 bytes of uniform random E2M1
 * codes, then the E8M0 scale byte base_byte - (r mod 3) (three scales a
 * factor of 2 apart). Block b uses draws 3*b .. 3*b+2 of the stream.
 */
void synth_fill_mx4(uint8_t *out, int64_t nblocks, uint64_t seed, uint64_t stream, uint8_t base_byte)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint8_t *blk = out + b * 17;
        for (int w = 0; w < 2; w++) {
            uint64_t r = draw(key, (uint64_t)b * 3 + w);
            memcpy(blk + 8 * w, &r, 8);
        }
        blk[16] = (uint8_t)(base_byte - (uint8_t)(draw(key, (uint64_t)b * 3 + 2) % 3));
    }
}

/* Uniform random bytes: byte i is byte i % 8 of draw i / 8 of the stream. */
void synth_fill_bytes(uint8_t *out, int64_t n, uint64_t seed, uint64_t stream)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < (n + 7) / 8; w++) {
        uint64_t r = draw(key, (uint64_t)w);
        for (int b = 0; b < 8 && 8 * w + b < n; b++)
            out[8 * w + b] = (uint8_t)(r >> (8 * b));
    }
}

/*
 * VQ codebook entries as FP8 E4M3 bytes: random sign and mantissa, exponent
 * field uniform in 5..9 (magnitudes 2^-2 .. 2^2 * 1.875), never NaN.
 * Byte i uses draw i of the stream.
 */
void synth_fill_e4m3_codebook(uint8_t *out, int64_t n, uint64_t seed, uint64_t stream)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        uint64_t r = draw(key, (uint64_t)i);
        const unsigned sign = (unsigned)(r & 1), man = (unsigned)((r >> 1) & 7);
        const unsigned ex = 5u + (unsigned)(((r >> 32) * 5u) >> 32);
        out[i] = (uint8_t)(sign << 7 | ex << 3 | man);
    }
}

/* Row gains: binary16 of |N(0, sigma)|; row i uses draws 2i and 2i+1 of the stream. */
void synth_fill_f16_abs_normal(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream, double sigma)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        double z0, z1;
        normal_pair(draw(key, 2 * (uint64_t)i), draw(key, 2 * (uint64_t)i + 1), &z0, &z1);
        out[i] = to_f16((float)(fabs(z0) * sigma));
    }
}

/*
 * 8-bit blocks: codes uniform in [-127, 127], d = |N(0, sigma)|.
 * Block b uses draws 18*b .. 18*b+17.
 */
void synth_fill_q8(uint8_t *out, int64_t nblocks, uint64_t seed, uint64_t stream, double sigma)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint8_t *blk = out + b * 34;
        uint64_t base = (uint64_t)b * 18;
        for (int w = 0; w < 16; w++) {
            uint64_t r = draw(key, base + w);
            for (int h = 0; h < 2; h++) {
                uint32_t v = (uint32_t)(r >> (32 * h));
                int q = (int)(((uint64_t)v * 255u) >> 32) - 127; /* 0..254 -> -127..127 */
                blk[2 + 2 * w + h] = (uint8_t)(int8_t)q;
            }
        }
        double z0, z1;
        normal_pair(draw(key, base + 16), draw(key, base + 17), &z0, &z1);
        uint16_t d = to_f16((float)(fabs(z0) * sigma));
        blk[0] = (uint8_t)(d & 0xFF);
        blk[1] = (uint8_t)(d >> 8);
    }
}

/* n fp32 values ~ N(0, sigma^2). Pair p uses draws 2p, 2p+1. */
void synth_fill_normal_f32(float *out, int64_t n, uint64_t seed, uint64_t stream, double sigma)
{
    uint64_t key = stream_key(seed, stream);
    int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; p++) {
        double z0, z1;
        normal_pair(draw(key, 2 * (uint64_t)p), draw(key, 2 * (uint64_t)p + 1), &z0, &z1);
        out[2 * p] = (float)(z0 * sigma);
        if (2 * p + 1 < n)
            out[2 * p + 1] = (float)(z1 * sigma);
    }
}

/* n bfloat16 values ~ N(0, sigma^2), as raw bits. */
void synth_fill_normal_bf16(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream, double sigma)
{
    uint64_t key = stream_key(seed, stream);
    int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; p++) {
        double z0, z1;
        normal_pair(draw(key, 2 * (uint64_t)p), draw(key, 2 * (uint64_t)p + 1), &z0, &z1);
        out[2 * p] = to_bf16((float)(z0 * sigma));
        if (2 * p + 1 < n)
            out[2 * p + 1] = to_bf16((float)(z1 * sigma));
    }
}

/*
 * A seeded permutation of the ranks 1..n (Fisher-Yates, draw i picks the swap
 * partner for position n-1-i). rank_out[e] is the rank of expert e.
 */
void synth_rank_permutation(int32_t *rank_out, int32_t n, uint64_t seed, uint64_t stream)
{
    uint64_t key = stream_key(seed, stream);
    for (int32_t e = 0; e < n; e++)
        rank_out[e] = e + 1;
    for (int32_t i = n - 1; i > 0; i--) {
        uint64_t r = draw(key, (uint64_t)(n - 1 - i));
        int32_t j = (int32_t)(((r >> 32) * (uint64_t)(i + 1)) >> 32);
        int32_t t = rank_out[i];
        rank_out[i] = rank_out[j];
        rank_out[j] = t;
    }
}
