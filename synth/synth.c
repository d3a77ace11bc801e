/*
 * synth.c -- seeded synthetic inputs for the routed sparse-MoE layer.
 *
 * This module only draws inputs: Gaussian weights and activations, the
 * MLX-style affine group quantisation that turns a drawn weight matrix into
 * (q, scale, bias) arrays, bf16 router weights, a Zipf expert-popularity bias
 * and its drift.  It computes nothing of the layer itself (no router, no
 * dequantisation, no expert FFN, no blob packing).  Both the CUDA path and the
 * CPU oracle receive what it produces as plain arrays.
 *
 * Random numbers: Philox4x32-10, implemented from its published definition
 * (J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random Numbers: As Easy
 * as 1, 2, 3", SC'11): a 4x32-bit counter and a 2x32-bit key, ten rounds of
 * two 32x32->64 multiplies, with the key bumped by the Weyl constants between
 * rounds.  Gaussians come from the Box-Muller transform (Box & Muller 1958).
 *
 * Stream addressing: key = the 64-bit seed; counter = (block, row, kind<<20 |
 * expert, layer).  Every (layer, kind, expert, row) therefore owns an
 * independent stream, and any expert can be regenerated on its own.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_PHILOX_M0 0xD2511F53u
#define SYN_PHILOX_M1 0xCD9E8D57u
#define SYN_PHILOX_W0 0x9E3779B9u
#define SYN_PHILOX_W1 0xBB67AE85u

static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)SYN_PHILOX_M0 * c[0];
    uint64_t p1 = (uint64_t)SYN_PHILOX_M1 * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

/* Philox4x32 with 10 rounds; exported so a test can check the published
 * known-answer vectors. */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += SYN_PHILOX_W0;
            k[1] += SYN_PHILOX_W1;
        }
        philox_round(c, k);
    }
    out[0] = c[0];
    out[1] = c[1];
    out[2] = c[2];
    out[3] = c[3];
}

/* uniform on the open interval (0, 1) from the top 24 bits */
static inline float u01(uint32_t v) { return ((float)(v >> 8) + 0.5f) * (1.0f / 16777216.0f); }

static inline void box_muller(uint32_t a, uint32_t b, float* z0, float* z1) {
    float r = sqrtf(-2.0f * logf(u01(a)));
    float t = 6.28318530717958647692f * u01(b);
    float st, ct;
    sincosf(t, &st, &ct);
    *z0 = r * ct;
    *z1 = r * st;
}

/* n Gaussian N(0, sigma^2) values of stream (layer, kind, expert, row). */
void synth_normal_row(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t expert, uint32_t row,
                      uint32_t n, float sigma, float* out) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t tag = (kind << 20) | (expert & 0xFFFFFu);
    for (uint32_t blk = 0; blk * 4 < n; ++blk) {
        uint32_t ctr[4] = {blk, row, tag, layer};
        uint32_t r[4];
        float z[4];
        synth_philox4x32_10(ctr, key, r);
        box_muller(r[0], r[1], &z[0], &z[1]);
        box_muller(r[2], r[3], &z[2], &z[3]);
        for (uint32_t j = 0; j < 4 && blk * 4 + j < n; ++j) out[blk * 4 + j] = sigma * z[j];
    }
}

/* rows x cols Gaussian matrix, row r drawn from stream row (row0 + r). */
void synth_normal_matrix(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t expert, uint32_t row0,
                         uint32_t rows, uint32_t cols, float sigma, float* out) {
    for (uint32_t r = 0; r < rows; ++r)
        synth_normal_row(seed, layer, kind, expert, row0 + r, cols, sigma, out + (size_t)r * cols);
}

/* ---- IEEE half / bfloat16 rounding (round to nearest, ties to even) ---- */

uint16_t synth_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ex = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (ex == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
    int e = (int)ex - 127 + 15;
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e <= 0) {
        /* half subnormal: value / 2^-24 = (1.man) * 2^(e-14) */
        if (ex == 0) return (uint16_t)sign; /* f32 subnormals are far below half's range */
        int shift = 14 - e;
        if (shift > 24) return (uint16_t)sign;
        uint32_t full = man | 0x800000u;
        uint32_t res = full >> shift;
        uint32_t rem = full & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (res & 1u))) res += 1u;
        return (uint16_t)(sign | res);
    }
    uint32_t res = ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (res & 1u))) res += 1u; /* may carry into the exponent */
    return (uint16_t)(sign | res);
}

float synth_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t ex = (h >> 10) & 0x1Fu;
    uint32_t man = h & 0x3FFu;
    float v;
    if (ex == 0) {
        v = ldexpf((float)man, -24);
    } else if (ex == 31) {
        uint32_t bits = 0x7F800000u | (man << 13);
        memcpy(&v, &bits, 4);
    } else {
        v = ldexpf((float)(man | 0x400u), (int)ex - 25);
    }
    uint32_t bits;
    memcpy(&bits, &v, 4);
    bits |= sign;
    memcpy(&v, &bits, 4);
    return v;
}

uint16_t synth_f32_to_bf16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu)) return (uint16_t)((x >> 16) | 0x40u);
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7FFFu + lsb;
    return (uint16_t)(x >> 16);
}

/*
 * MLX-style affine group quantisation of one matrix (rows x cols, cols a
 * multiple of `group`).  Per group of `group` consecutive columns of a row:
 *   scale = fp16((max - min) / (2^bits - 1)),  bias = fp16(min),
 *   q     = clamp(rint((w - bias) / scale), 0, 2^bits - 1)   (fp32, ties to even)
 * with q = 0 when the rounded scale is 0.  q is written one value per byte;
 * sb holds (scale, bias) as fp16 bit patterns, interleaved, per group.
 * The dequantised weight is scale*q + bias.
 */
void synth_quantize_affine(const float* w, uint32_t rows, uint32_t cols, uint32_t group, int bits,
                           uint8_t* q, uint16_t* sb) {
    const float qmax = (float)((1u << bits) - 1u);
    const uint32_t ng = cols / group;
    for (uint32_t r = 0; r < rows; ++r) {
        for (uint32_t g = 0; g < ng; ++g) {
            const float* wg = w + (size_t)r * cols + (size_t)g * group;
            uint8_t* qg = q + (size_t)r * cols + (size_t)g * group;
            float mn = wg[0], mx = wg[0];
            for (uint32_t c = 1; c < group; ++c) {
                if (wg[c] < mn) mn = wg[c];
                if (wg[c] > mx) mx = wg[c];
            }
            uint16_t sh = synth_f32_to_f16((mx - mn) / qmax);
            uint16_t bh = synth_f32_to_f16(mn);
            float s = synth_f16_to_f32(sh), b = synth_f16_to_f32(bh);
            for (uint32_t c = 0; c < group; ++c) {
                float v = 0.0f;
                if (s != 0.0f) {
                    v = rintf((wg[c] - b) / s);
                    if (v < 0.0f) v = 0.0f;
                    if (v > qmax) v = qmax;
                }
                qg[c] = (uint8_t)v;
            }
            sb[((size_t)r * ng + g) * 2 + 0] = sh;
            sb[((size_t)r * ng + g) * 2 + 1] = bh;
        }
    }
}

/* Stream kinds (the `kind` field of the counter). */
enum {
    SYN_GATE = 1,
    SYN_UP = 2,
    SYN_DOWN = 3,
    SYN_ROUTER = 4,
    SYN_SHARED_GATE = 5,
    SYN_TOKENS = 6,
    SYN_RANK = 7,
    SYN_DRIFT = 8
};

/*
 * One expert: gate and up are inter x hidden, down is hidden x inter, each
 * drawn N(0, sigma^2) and quantised with group 64.  `scratch` must hold
 * inter*hidden floats.  expert = 0xFFFFF addresses the shared expert.
 */
int synth_expert(uint64_t seed, uint32_t layer, uint32_t expert, uint32_t hidden, uint32_t inter, int bits,
                 float sigma, uint8_t* qg, uint16_t* sbg, uint8_t* qu, uint16_t* sbu, uint8_t* qd, uint16_t* sbd,
                 float* scratch) {
    if ((hidden % 64) || (inter % 64) || (bits != 4 && bits != 8)) return -1;
    synth_normal_matrix(seed, layer, SYN_GATE, expert, 0, inter, hidden, sigma, scratch);
    synth_quantize_affine(scratch, inter, hidden, 64, bits, qg, sbg);
    synth_normal_matrix(seed, layer, SYN_UP, expert, 0, inter, hidden, sigma, scratch);
    synth_quantize_affine(scratch, inter, hidden, 64, bits, qu, sbu);
    synth_normal_matrix(seed, layer, SYN_DOWN, expert, 0, hidden, inter, sigma, scratch);
    synth_quantize_affine(scratch, hidden, inter, 64, bits, qd, sbd);
    return 0;
}

/* bf16 matrix rows x cols ~ N(0, sigma^2) of stream (layer, kind, expert=0). */
void synth_bf16_matrix(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t rows, uint32_t cols, float sigma,
                       uint16_t* out, float* scratch_row) {
    for (uint32_t r = 0; r < rows; ++r) {
        synth_normal_row(seed, layer, kind, 0, r, cols, sigma, scratch_row);
        for (uint32_t c = 0; c < cols; ++c) out[(size_t)r * cols + c] = synth_f32_to_bf16(scratch_row[c]);
    }
}

void synth_router_weights(uint64_t seed, uint32_t layer, uint32_t n_experts, uint32_t hidden, float sigma,
                          uint16_t* out, float* scratch_row) {
    synth_bf16_matrix(seed, layer, SYN_ROUTER, n_experts, hidden, sigma, out, scratch_row);
}

void synth_shared_gate_weights(uint64_t seed, uint32_t layer, uint32_t hidden, float sigma, uint16_t* out,
                               float* scratch_row) {
    synth_bf16_matrix(seed, layer, SYN_SHARED_GATE, 1, hidden, sigma, out, scratch_row);
}

/* B tokens x hidden fp32 activations ~ N(0,1) for decode step `step`. */
void synth_tokens(uint64_t seed, uint32_t step, uint32_t n_tokens, uint32_t hidden, float* x) {
    for (uint32_t t = 0; t < n_tokens; ++t) synth_normal_row(seed, step, SYN_TOKENS, 0, t, hidden, 1.0f, x + (size_t)t * hidden);
}

static uint32_t draw_u32(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t a, uint32_t b) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {a, b, kind << 20, layer};
    uint32_t r[4];
    synth_philox4x32_10(ctr, key, r);
    return r[0];
}

/* uniform integer in [0, n) by the multiply-shift map of a 32-bit draw */
static inline uint32_t below(uint32_t v, uint32_t n) { return (uint32_t)(((uint64_t)v * n) >> 32); }

/*
 * Per-layer expert-popularity permutation: expert_at[r] is the expert with
 * popularity rank r+1 (Fisher-Yates shuffle of 0..E-1).
 */
void synth_rank_permutation(uint64_t seed, uint32_t layer, uint32_t n_experts, int32_t* expert_at) {
    for (uint32_t i = 0; i < n_experts; ++i) expert_at[i] = (int32_t)i;
    for (uint32_t i = n_experts - 1; i > 0; --i) {
        uint32_t j = below(draw_u32(seed, layer, SYN_RANK, i, 0), i + 1);
        int32_t t = expert_at[i];
        expert_at[i] = expert_at[j];
        expert_at[j] = t;
    }
}

/*
 * Zipf(s) popularity bias: p(r) = r^-s / sum_{j=1..E} j^-s for rank r, and
 * beta[e] = ln p(rank of e).  Added to the router logits.
 */
void synth_zipf_bias(uint32_t n_experts, double s, const int32_t* expert_at, float* beta) {
    double z = 0.0;
    for (uint32_t r = 1; r <= n_experts; ++r) z += pow((double)r, -s);
    for (uint32_t r = 1; r <= n_experts; ++r) beta[expert_at[r - 1]] = (float)(log(pow((double)r, -s) / z));
}

/*
 * Temporally correlated popularity drift: at decode step `step`, swap the
 * experts holding `n_swaps` randomly chosen pairs of adjacent ranks.
 */
void synth_drift_step(uint64_t seed, uint32_t layer, uint32_t step, uint32_t n_experts, uint32_t n_swaps,
                      int32_t* expert_at) {
    for (uint32_t i = 0; i < n_swaps; ++i) {
        uint32_t p = below(draw_u32(seed, layer, SYN_DRIFT, step, i), n_experts - 1);
        int32_t t = expert_at[p];
        expert_at[p] = expert_at[p + 1];
        expert_at[p + 1] = t;
    }
}
