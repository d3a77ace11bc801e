// gemv.cuh -- the arithmetic of the decode path, written once and shared by
// the per-layer kernels and the persistent stack kernel, so both produce the
// same bits.  Every reduction order is fixed here.
//
// Dequantised GEMV, MLX affine int4/int8 group 64 [Swiftlet README,
// "Relation to TurboFieldfare": MLX affine int4/int8 group quantisation
// computed on the GPU; cooperative SIMD-group GEMV fast path]:
//   row . v = sum_g ( s_g * sum_{c in g} q_c v_c  +  b_g * sum_{c in g} v_c )
//
// The activation vector v (a token's x, or one expert's SwiGLU output h) is
// held as 24-bit block fixed point: V_c = rint(v_c * 2^e) with one exponent e
// per vector chosen so that |V_c| <= 2^22, split into three signed base-256
// digits V = D2*2^16 + D1*2^8 + D0 (D0, D1 in [-128, 127], D2 in [-64, 64]).
// The representation error is at most 2^-22 of max|v| per element, the same
// order as fp32 rounding of v.  Products with the 4- or 8-bit codes are then
// exact integer dot products (DP4A: four byte products per instruction):
//   int4: a 32-bit word holds codes c0..c7; (w & 0x0f0f0f0f) holds the even
//         codes, (w & 0xf0f0f0f0) sixteen times the odd ones, each byte
//         paired with the matching digit bytes of the even/odd columns.
//   int8: a word holds four codes, paired with four digit bytes.
// Integer sums are exact, so their order does not matter; the float steps
// (digit recombination, scale/bias, the warp butterfly) are fixed below.
//
// A warp owns a row; lane L owns the 16-byte code chunks L, L+32, ... of it
// (32 int4 or 16 int8 columns each, always inside one 64-column group).
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

template <int BITS>
struct Codes;

template <>
struct Codes<4> {
    static constexpr int kCols = 32;   // columns per 16-byte chunk
    static constexpr int kDigitWords = 24;  // digit words per chunk (4 code words x 3 digits x even/odd)
};

template <>
struct Codes<8> {
    static constexpr int kCols = 16;
    static constexpr int kDigitWords = 12;  // 4 code words x 3 digits
};

__device__ __forceinline__ float bf16_lo(uint32_t t) { return __uint_as_float(t << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t t) { return __uint_as_float(t & 0xffff0000u); }

__device__ __forceinline__ int dp4a_us(uint32_t codes, uint32_t digits, int acc) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(codes), "r"(digits), "r"(acc));
    return d;
}

// ---------------------------------------------------------------------------
// block fixed point of one vector
// ---------------------------------------------------------------------------
// exponent for max|v| (0 when the vector is all zero): 21 - floor(log2 max|v|)
__device__ __forceinline__ int bfp_exponent(float maxabs) {
    if (!(maxabs > 0.0f)) return 0;
    const uint32_t b = __float_as_uint(maxabs);
    const int be = (int)((b >> 23) & 0xffu);
    const int lg = be ? be - 127 : (31 - __clz((int)(b & 0x7fffffu))) - 149;  // subnormals: from the mantissa
    return 21 - lg;
}

// v * 2^e, as one or two power-of-two multiplies (each factor a normal float)
__device__ __forceinline__ float pow2_scale(float v, int e) {
    if (e >= -126 && e <= 127) return __fmul_rn(v, __int_as_float((127 + e) << 23));
    const int a = e / 2, b = e - a;
    return __fmul_rn(__fmul_rn(v, __int_as_float((127 + a) << 23)), __int_as_float((127 + b) << 23));
}

__device__ __forceinline__ int bfp_int(float v, int e) { return __float2int_rn(pow2_scale(v, e)); }

// the three signed base-256 digits of V, as bytes
__device__ __forceinline__ void bfp_digits(int V, uint32_t& d0, uint32_t& d1, uint32_t& d2) {
    const int D0 = (int)(int8_t)(V & 0xff);
    const int V1 = (V - D0) >> 8;
    const int D1 = (int)(int8_t)(V1 & 0xff);
    const int D2 = (V1 - D1) >> 8;
    d0 = (uint32_t)D0 & 0xffu;
    d1 = (uint32_t)D1 & 0xffu;
    d2 = (uint32_t)D2 & 0xffu;
}

// Digit words and integer sum of one chunk from its columns' V values.
// int4 layout per code word i: [E0 O0 E1 O1 E2 O2] (E = columns 0,2,4,6 of
// the word, O = 1,3,5,7; digit j in byte order of the columns); int8 layout
// per code word i: [L0 L1 L2] for its four columns.
template <int BITS>
__device__ __forceinline__ void bfp_chunk(const int* V, uint32_t* dw, int& S) {
    S = 0;
    if (BITS == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t e[3] = {0, 0, 0}, o[3] = {0, 0, 0};
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t a0, a1, a2, c0, c1, c2;
                bfp_digits(V[8 * i + 2 * b], a0, a1, a2);
                bfp_digits(V[8 * i + 2 * b + 1], c0, c1, c2);
                e[0] |= a0 << (8 * b), e[1] |= a1 << (8 * b), e[2] |= a2 << (8 * b);
                o[0] |= c0 << (8 * b), o[1] |= c1 << (8 * b), o[2] |= c2 << (8 * b);
                S += V[8 * i + 2 * b] + V[8 * i + 2 * b + 1];
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                dw[6 * i + 2 * j] = e[j];
                dw[6 * i + 2 * j + 1] = o[j];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t l[3] = {0, 0, 0};
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t a0, a1, a2;
                bfp_digits(V[4 * i + b], a0, a1, a2);
                l[0] |= a0 << (8 * b), l[1] |= a1 << (8 * b), l[2] |= a2 << (8 * b);
                S += V[4 * i + b];
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) dw[3 * i + j] = l[j];
        }
    }
}

// Block-fixed-point digits of B tokens' x (xs [B][H], exponents xe[B]) by the
// warps w0 .. w0+nw-1 of the block:
// a warp covers 32 consecutive columns of one token (one int4 chunk, two int8
// chunks); the digit words are assembled with shuffles in the layout of
// bfp_chunk and stored whole.
template <int BITS>
__device__ __forceinline__ void make_digits(int B, int H, const float* xs, uint32_t* xdw, int32_t* xS, const int* xe,
                                            int w0, int nw) {
    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nc = H / CC, ng = H / 32;
#pragma unroll 1
    for (int g = warp - w0; g < B * ng; g += nw) {
        const int t = g / ng, col = (g - t * ng) * 32 + lane;
        const int V = bfp_int(xs[t * H + col], xe[t]);
        uint32_t d0, d1, d2;
        bfp_digits(V, d0, d1, d2);
        const uint32_t dig = d0 | (d1 << 8) | (d2 << 16);
        if (BITS == 4) {
            // word L = 6 cw + 2 j + odd: digit j of columns 8 cw + 2 b + odd, b = 0..3
            const int Lw = lane < 24 ? lane : 0;
            const int cw = Lw / 6, r = Lw - 6 * cw, j = r >> 1, odd = r & 1;
            const uint32_t g0 = __shfl_sync(kFullMask, dig, 8 * cw + 0 + odd);
            const uint32_t g1 = __shfl_sync(kFullMask, dig, 8 * cw + 2 + odd);
            const uint32_t g2 = __shfl_sync(kFullMask, dig, 8 * cw + 4 + odd);
            const uint32_t g3 = __shfl_sync(kFullMask, dig, 8 * cw + 6 + odd);
            const uint32_t sel = (uint32_t)j | ((uint32_t)(j + 4) << 4);
            const uint32_t word = __byte_perm(__byte_perm(g0, g1, sel), __byte_perm(g2, g3, sel), 0x5410);
            const int ch = col / CC;
            if (lane < 24) xdw[(size_t)(t * nc + ch) * DW + lane] = word;
            const int S = __reduce_add_sync(kFullMask, V);
            if (lane == 0) xS[t * nc + ch] = S;
        } else {
            // per half-warp chunk: word 3 cw + j = digit j of columns 4 cw + b, b = 0..3
            const int hb = lane & 16, L = lane & 15;
            const int Lw = L < 12 ? L : 0;
            const int cw = Lw / 3, j = Lw - 3 * cw;
            const uint32_t g0 = __shfl_sync(kFullMask, dig, hb + 4 * cw + 0);
            const uint32_t g1 = __shfl_sync(kFullMask, dig, hb + 4 * cw + 1);
            const uint32_t g2 = __shfl_sync(kFullMask, dig, hb + 4 * cw + 2);
            const uint32_t g3 = __shfl_sync(kFullMask, dig, hb + 4 * cw + 3);
            const uint32_t sel = (uint32_t)j | ((uint32_t)(j + 4) << 4);
            const uint32_t word = __byte_perm(__byte_perm(g0, g1, sel), __byte_perm(g2, g3, sel), 0x5410);
            const int ch = col / CC;
            if (L < 12) xdw[(size_t)(t * nc + ch) * DW + L] = word;
            const int S = lane < 16 ? __reduce_add_sync(0x0000ffffu, V) : __reduce_add_sync(0xffff0000u, V);
            if (L == 0) xS[t * nc + ch] = S;
        }
    }
}

// sum over the chunk of q_c * V_c, as a float (digits recombined in a fixed order)
__device__ __forceinline__ float chunk_dot(uint4 v, const uint32_t* dw, Codes<4>) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    int ae[3] = {0, 0, 0}, ao[3] = {0, 0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = wd[i] & 0x0f0f0f0fu, hi = wd[i] & 0xf0f0f0f0u;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            ae[j] = dp4a_us(lo, dw[6 * i + 2 * j], ae[j]);
            ao[j] = dp4a_us(hi, dw[6 * i + 2 * j + 1], ao[j]);
        }
    }
    const int A0 = ae[0] + (ao[0] >> 4), A1 = ae[1] + (ao[1] >> 4), A2 = ae[2] + (ao[2] >> 4);
    return __fmaf_rn((float)A2, 65536.0f, __fmaf_rn((float)A1, 256.0f, (float)A0));
}

__device__ __forceinline__ float chunk_dot(uint4 v, const uint32_t* dw, Codes<8>) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    int a[3] = {0, 0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 3; ++j) a[j] = dp4a_us(wd[i], dw[3 * i + j], a[j]);
    }
    return __fmaf_rn((float)a[2], 65536.0f, __fmaf_rn((float)a[1], 256.0f, (float)a[0]));
}

// part += s*A + b*S for the chunk's (scale, bias) word
__device__ __forceinline__ float chunk_term(float part, float A, int S, uint32_t sbw) {
    const float2 sb = __half22float2(*reinterpret_cast<const __half2*>(&sbw));
    part = __fmaf_rn(sb.x, A, part);
    return __fmaf_rn(sb.y, (float)S, part);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}

// two independent butterflies interleaved (each result equals warp_sum of it)
__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float oa = __shfl_xor_sync(kFullMask, a, off), ob = __shfl_xor_sync(kFullMask, b, off);
        a = __fadd_rn(a, oa);
        b = __fadd_rn(b, ob);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}

// SiLU(g) * u.  The element-wise transcendental math of the decode path
// (SiLU, the sigmoid gate, softmax weights, 1/sqrt of the renormalisation)
// uses the hardware approximations (ex2, rcp, rsqrt: a few ulp); both decode
// paths share these functions, so they agree bit for bit, and the error is
// far inside the layer tolerance.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

// ---------------------------------------------------------------------------
// router logit (fp32, fixed order): element h accumulates into lane (h/8)%32
// in ascending h, butterfly 16..1, + bias.  w_row bf16 [H], x fp32 [H].
// ---------------------------------------------------------------------------
__device__ __forceinline__ float router_logit(const uint16_t* w_row, const float* x, int H, float bias, int lane) {
    const uint4* w4 = reinterpret_cast<const uint4*>(w_row);
    float a = 0.0f;
#pragma unroll 4
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 v = w4[c];
        const float4 xa = *reinterpret_cast<const float4*>(x + 8 * c);
        const float4 xb = *reinterpret_cast<const float4*>(x + 8 * c + 4);
        a = __fmaf_rn(bf16_lo(v.x), xa.x, a);
        a = __fmaf_rn(bf16_hi(v.x), xa.y, a);
        a = __fmaf_rn(bf16_lo(v.y), xa.z, a);
        a = __fmaf_rn(bf16_hi(v.y), xa.w, a);
        a = __fmaf_rn(bf16_lo(v.z), xb.x, a);
        a = __fmaf_rn(bf16_hi(v.z), xb.y, a);
        a = __fmaf_rn(bf16_lo(v.w), xb.z, a);
        a = __fmaf_rn(bf16_hi(v.w), xb.w, a);
    }
    return __fadd_rn(warp_sum(a), bias);
}

// sigmoid(w_sg . x), the dot product in the router's fixed order
__device__ __forceinline__ float shared_gate(const uint16_t* w_sg, const float* x, int H, int lane) {
    const float g = router_logit(w_sg, x, H, 0.0f, lane);
    return __fdividef(1.0f, __fadd_rn(1.0f, __expf(-g)));
}

// Renormalisation statistics of one token over kRenormThreads threads:
// thread i accumulates y_j^2 (fma) over the column pairs j = 2i + 2 m
// kRenormThreads and j + 1, m ascending; each warp's partials are summed by a
// butterfly and the warp sums in warp order.  Also max |y|.  The pairing
// matches the persistent kernel's exchange reads (one 16-byte word pair per
// thread and step), so there each thread sums the values it fetched itself.
constexpr int kRenormThreads = 512;

// this thread's partial sum of squares and max |y| of one token (thread i of kRenormThreads)
__device__ __forceinline__ void renorm_partial(const float* y, int H, int i, float& s, float& m) {
    s = 0.0f;
    m = 0.0f;
#pragma unroll 1
    for (int j = 2 * i; j < H; j += 2 * kRenormThreads) {
        s = __fmaf_rn(y[j], y[j], s);
        s = __fmaf_rn(y[j + 1], y[j + 1], s);
        m = fmaxf(m, fmaxf(fabsf(y[j]), fabsf(y[j + 1])));
    }
}

// r = 1/sqrt(mean + eps) from the kRenormThreads/32 warp sums, added in warp order
__device__ __forceinline__ float renorm_scale(const float* warp_sums, int H, float eps) {
    float tot = warp_sums[0];
#pragma unroll 1
    for (int w = 1; w < kRenormThreads / 32; ++w) tot = __fadd_rn(tot, warp_sums[w]);
    return rsqrtf(__fadd_rn(__fmul_rn(tot, 1.0f / (float)H), eps));
}

// The statistics above computed by a whole block of kRenormThreads threads.
// Returns r to every thread and max |y| via *maxabs.  red: kRenormThreads/32 * 2
// floats of shared memory.
__device__ __forceinline__ float renorm_block(const float* y, int H, float eps, float* red, float* maxabs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kRenormThreads / 32;
    float s, m;
    renorm_partial(y, H, tid, s, m);
    s = warp_sum(s);
    m = warp_max(m);
    if (lane == 0) {
        red[warp] = s;
        red[NW + warp] = m;
    }
    __syncthreads();
    float mx = red[NW];
    for (int w = 1; w < NW; ++w) mx = fmaxf(mx, red[NW + w]);
    const float r = renorm_scale(red, H, eps);
    __syncthreads();
    *maxabs = mx;
    return r;
}

// ---------------------------------------------------------------------------
// top-k of one token by one warp (descending logit, ties -> lower index) and
// the routing weights.  lg fp32 [E] (E <= 1024, shared or global memory);
// idx/val/w: k entries in shared memory.
// Logits compare as order-preserving 32-bit keys (+0 and -0 equal); each
// round takes the warp maximum key and, among equal keys, the lowest index
// (two warp reductions); the winning lane rescans its own 32-strided slice.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// routing weights of the k chosen logits val[] (one warp): lane i < k takes
// exp(val[i] - val[0]); the denominator is their warp butterfly sum (or, for
// the full softmax, of every logit's exponential, lane-strided then the
// butterfly)
__device__ __forceinline__ void topk_weights(const float* lg, int E, int k, int norm_topk, int lane, const float* val,
                                             float* w) {
    const float m = val[0];
    const float ei = lane < k ? __expf(__fsub_rn(val[lane], m)) : 0.0f;
    float den;
    if (norm_topk) {
        den = warp_sum(ei);
    } else {
        float d = 0.0f;
#pragma unroll 1
        for (int e = lane; e < E; e += 32) d = __fadd_rn(d, __expf(__fsub_rn(lg[e], m)));
        den = warp_sum(d);
    }
    if (lane < k) w[lane] = __fdividef(ei, den);
    __syncwarp();
}

// k best (key desc, index asc) of n candidates cand_key/cand_idx (n <= 32*MAXM)
// by one warp; writes idx[] and the chosen keys.
template <int MAXM>
__device__ __forceinline__ void warp_select(const uint32_t* cand_key, const int32_t* cand_idx, int n, int k, int lane,
                                            int32_t* idx, uint32_t* keys) {
    uint32_t key[MAXM];
    int32_t id[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int i = lane + 32 * m;
        key[m] = i < n ? cand_key[i] : 0u;
        id[m] = i < n ? cand_idx[i] : 0x7fffffff;
    }
    uint32_t taken = 0;
    auto local_best = [&](uint32_t& bk, int32_t& bi, int& bm) {
        bk = 0u;
        bi = 0x7fffffff;
        bm = -1;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const bool live = lane + 32 * m < n && !(taken & (1u << m));
            if (live && (bm < 0 || key[m] > bk || (key[m] == bk && id[m] < bi))) {
                bk = key[m];
                bi = id[m];
                bm = m;
            }
        }
    };
    uint32_t bk;
    int32_t bi;
    int bm;
    local_best(bk, bi, bm);
    for (int i = 0; i < k; ++i) {
        const uint32_t K = __reduce_max_sync(kFullMask, bm >= 0 ? bk : 0u);
        const uint32_t cand = (bm >= 0 && bk == K) ? (uint32_t)bi : 0xffffffffu;
        const uint32_t win = __reduce_min_sync(kFullMask, cand);
        if (bm >= 0 && (uint32_t)bi == win && bk == K) {
            taken |= 1u << bm;
            local_best(bk, bi, bm);
        }
        if (lane == 0) {
            idx[i] = (int32_t)win;
            keys[i] = K;
        }
    }
    __syncwarp();
}

__device__ __forceinline__ void warp_topk(const float* lg, int E, int k, int norm_topk, int lane, int32_t* idx,
                                          float* val, float* w) {
    uint32_t key[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) key[m] = (lane + 32 * m < E) ? order_key(lg[lane + 32 * m]) : 0u;
    uint32_t taken = 0;
    auto local_best = [&](uint32_t& bk, int& bm) {
        bk = 0u;
        bm = -1;
#pragma unroll
        for (int m = 0; m < 32; ++m) {
            const bool live = lane + 32 * m < E && !(taken & (1u << m));
            if (live && (bm < 0 || key[m] > bk)) {
                bk = key[m];
                bm = m;
            }
        }
    };
    uint32_t bk;
    int bm;
    local_best(bk, bm);
    for (int i = 0; i < k; ++i) {
        const uint32_t K = __reduce_max_sync(kFullMask, bm >= 0 ? bk : 0u);
        const uint32_t cand = (bm >= 0 && bk == K) ? (uint32_t)(lane + 32 * bm) : 0xffffffffu;
        const uint32_t win = __reduce_min_sync(kFullMask, cand);
        if ((int)(win & 31u) == lane) {
            taken |= 1u << (win >> 5);
            local_best(bk, bm);
        }
        if (lane == 0) {
            idx[i] = (int32_t)win;
            val[i] = lg[win];
        }
    }
    __syncwarp();
    topk_weights(lg, E, k, norm_topk, lane, val, w);
}

// ---------------------------------------------------------------------------
// down rows: h in fp32 registers, codes expanded to fp32 (FFMA)
// ---------------------------------------------------------------------------
// A down row meets each (token, expert) h only for this block's few output
// rows, so converting h to digits would cost more than it saves; the down
// projection multiplies fp32 h directly:
//   int4: a LOP3 turns two nibbles into the bf16 pair (128 + q_lo, 128 + q_hi)
//         whose halves are fp32 values; sum (128 + q) h - 128 * sum h is
//         folded into the bias term (OFF = 128).
//   int8: a byte permute puts q in the mantissa of 2^23, one subtract gives q.
template <int BITS>
struct HF {
    float v[Codes<BITS>::kCols];  // this lane's chunk of h
    float s;                      // their sum (sequential)
};

__device__ __forceinline__ float bf16_pair_lo(uint32_t t) { return __uint_as_float(t << 16); }
__device__ __forceinline__ float bf16_pair_hi(uint32_t t) { return __uint_as_float(t & 0xffff0000u); }
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int shift) {
    return ((w >> shift) & 0x000f000fu) | 0x43004300u;
}

// 128 + (byte b of x) as a float, for a byte below 16: byte b goes to bits 16..23
// under the exponent byte of 128.0 (the bits of bf16_pair_lo(nib_pair(...)))
__device__ __forceinline__ float q128(uint32_t x, int b) {
    return __uint_as_float(__byte_perm(x, 0x43000000u, 0x7044u | ((unsigned)b << 8)));
}

// sum over the chunk of (128 + q_c) * h_c
__device__ __forceinline__ float chunk_dot_f(uint4 v, const float* h, Codes<4>) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* hw = h + 8 * i;
        // even codes (columns 0, 2, 4, 6 of the word) and odd codes, one per byte;
        // one byte permute then places a code in the mantissa of 128.0 (128 + q)
        const uint32_t ev = wd[i] & 0x0f0f0f0fu, od = (wd[i] >> 4) & 0x0f0f0f0fu;
        float s = __fmul_rn(q128(ev, 0), hw[0]);
        s = __fmaf_rn(q128(ev, 2), hw[4], s);
        s = __fmaf_rn(q128(od, 0), hw[1], s);
        s = __fmaf_rn(q128(od, 2), hw[5], s);
        s = __fmaf_rn(q128(ev, 1), hw[2], s);
        s = __fmaf_rn(q128(ev, 3), hw[6], s);
        s = __fmaf_rn(q128(od, 1), hw[3], s);
        s = __fmaf_rn(q128(od, 3), hw[7], s);
        a[i] = s;
    }
    return __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
}

__device__ __forceinline__ float byte_q(uint32_t w, int i) {
    return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4b000000u, 0x7440u | (unsigned)i)), 8388608.0f);
}

// sum over the chunk of q_c * h_c
__device__ __forceinline__ float chunk_dot_f(uint4 v, const float* h, Codes<8>) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* hw = h + 4 * i;
        float s = __fmul_rn(byte_q(wd[i], 0), hw[0]);
        s = __fmaf_rn(byte_q(wd[i], 1), hw[1], s);
        s = __fmaf_rn(byte_q(wd[i], 2), hw[2], s);
        s = __fmaf_rn(byte_q(wd[i], 3), hw[3], s);
        a[i] = s;
    }
    return __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
}

template <int BITS>
__device__ __forceinline__ void hf_sum(HF<BITS>& h) {
    float s = h.v[0];
#pragma unroll
    for (int i = 1; i < Codes<BITS>::kCols; ++i) s = __fadd_rn(s, h.v[i]);
    h.s = s;
}

// s * A + (b - OFF * s) * S for one chunk
template <int BITS>
__device__ __forceinline__ float chunk_term_f(float A, float S, uint32_t sbw) {
    const float2 sb = __half22float2(*reinterpret_cast<const __half2*>(&sbw));
    const float off = BITS == 4 ? 128.0f : 0.0f;
    const float d = __fmaf_rn(-off, sb.x, sb.y);
    return __fmaf_rn(d, S, __fmul_rn(sb.x, A));
}

// one down row (cols / CC <= 32 chunks, one per lane) . h
template <int BITS>
__device__ __forceinline__ float row_dot_h(const uint8_t* q_row, const uint32_t* sb_row, const HF<BITS>& h, int cols,
                                           int lane) {
    constexpr int CC = Codes<BITS>::kCols, CPG = 64 / CC;
    float part = 0.0f;
    if (lane < cols / CC) {
        const float A = chunk_dot_f(reinterpret_cast<const uint4*>(q_row)[lane], h.v, Codes<BITS>{});
        part = chunk_term_f<BITS>(A, h.s, sb_row[lane / CPG]);
    }
    return warp_sum(part);
}

// a token's digits for gate/up rows: lane L holds chunks L, L+32, ... (NPER of them)
template <int BITS, int NPER>
struct XDigits {
    uint32_t dw[NPER][Codes<BITS>::kDigitWords];
    int S[NPER];
};

template <int BITS, int NPER>
__device__ __forceinline__ void load_xdigits(XDigits<BITS, NPER>& xd, const uint32_t* words, const int32_t* sums,
                                             int nchunk, int lane) {
    constexpr int DW = Codes<BITS>::kDigitWords;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int c = lane + 32 * i;
        if (c < nchunk) {
#pragma unroll
            for (int j = 0; j < DW; j += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(words + (size_t)c * DW + j);
                xd.dw[i][j] = v.x, xd.dw[i][j + 1] = v.y, xd.dw[i][j + 2] = v.z, xd.dw[i][j + 3] = v.w;
            }
            xd.S[i] = sums[c];
        }
    }
}

// one gate/up row . x, same order as a chunk loop c = lane, lane+32, ...
template <int BITS, int NPER>
__device__ __forceinline__ float row_dot_x(const uint8_t* q_row, const uint32_t* sb_row, const XDigits<BITS, NPER>& xd,
                                           int e, int nchunk, int lane) {
    constexpr int CPG = 64 / Codes<BITS>::kCols;
    const uint4* q = reinterpret_cast<const uint4*>(q_row);
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int c = lane + 32 * i;
        if (c < nchunk) {
            const float A = chunk_dot(q[c], xd.dw[i], Codes<BITS>{});
            part = chunk_term(part, A, xd.S[i], sb_row[c / CPG]);
        }
    }
    return pow2_scale(warp_sum(part), -e);
}

// gate and up rows against the same x, butterflies interleaved; each result
// equals row_dot_x of that row
template <int BITS, int NPER>
__device__ __forceinline__ void row_dot_x2(const uint8_t* q0, const uint32_t* sb0, const uint8_t* q1, const uint32_t* sb1,
                                           const XDigits<BITS, NPER>& xd, int e, int nchunk, int lane, float& r0,
                                           float& r1) {
    constexpr int CPG = 64 / Codes<BITS>::kCols;
    float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int c = lane + 32 * i;
        if (c < nchunk) {
            const float A0 = chunk_dot(reinterpret_cast<const uint4*>(q0)[c], xd.dw[i], Codes<BITS>{});
            const float A1 = chunk_dot(reinterpret_cast<const uint4*>(q1)[c], xd.dw[i], Codes<BITS>{});
            p0 = chunk_term(p0, A0, xd.S[i], sb0[c / CPG]);
            p1 = chunk_term(p1, A1, xd.S[i], sb1[c / CPG]);
        }
    }
    warp_sum2(p0, p1);
    r0 = pow2_scale(p0, -e);
    r1 = pow2_scale(p1, -e);
}

// row_dot_x2 with the token's digit words read from shared memory chunk by
// chunk (chunk c's words at xdw[c * DW], its integer sum at xS[c]) in a rolled
// loop: the same chunks in the same order, the same butterfly, so each result
// equals row_dot_x2's bit for bit, with a fraction of the code.
template <int BITS>
__device__ __forceinline__ void row_dot_x2_sm(const uint8_t* q0, const uint32_t* sb0, const uint8_t* q1,
                                              const uint32_t* sb1, const uint32_t* xdw, const int32_t* xS, int e,
                                              int nchunk, int lane, float& r0, float& r1) {
    constexpr int DW = Codes<BITS>::kDigitWords, CPG = 64 / Codes<BITS>::kCols;
    float p0 = 0.0f, p1 = 0.0f;
#pragma unroll 1
    for (int c = lane; c < nchunk; c += 32) {
        uint32_t dw[DW];
#pragma unroll
        for (int j = 0; j < DW; j += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(xdw + (size_t)c * DW + j);
            dw[j] = v.x, dw[j + 1] = v.y, dw[j + 2] = v.z, dw[j + 3] = v.w;
        }
        const int S = xS[c];
        const float A0 = chunk_dot(reinterpret_cast<const uint4*>(q0)[c], dw, Codes<BITS>{});
        const float A1 = chunk_dot(reinterpret_cast<const uint4*>(q1)[c], dw, Codes<BITS>{});
        p0 = chunk_term(p0, A0, S, sb0[c / CPG]);
        p1 = chunk_term(p1, A1, S, sb1[c / CPG]);
    }
    warp_sum2(p0, p1);
    r0 = pow2_scale(p0, -e);
    r1 = pow2_scale(p1, -e);
}

// two down rows against the same h, butterflies interleaved (each result equals row_dot_h)
template <int BITS>
__device__ __forceinline__ void row_dot_h2(const uint8_t* q0, const uint32_t* sb0, const uint8_t* q1, const uint32_t* sb1,
                                           const HF<BITS>& h, int cols, int lane, float& r0, float& r1) {
    constexpr int CC = Codes<BITS>::kCols, CPG = 64 / CC;
    float p0 = 0.0f, p1 = 0.0f;
    if (lane < cols / CC) {
        const float A0 = chunk_dot_f(reinterpret_cast<const uint4*>(q0)[lane], h.v, Codes<BITS>{});
        const float A1 = chunk_dot_f(reinterpret_cast<const uint4*>(q1)[lane], h.v, Codes<BITS>{});
        p0 = chunk_term_f<BITS>(A0, h.s, sb0[lane / CPG]);
        p1 = chunk_term_f<BITS>(A1, h.s, sb1[lane / CPG]);
    }
    warp_sum2(p0, p1);
    r0 = p0;
    r1 = p1;
}

// Two down rows at once when a row has exactly 16 chunks (int4, 512 columns):
// lanes 0-15 take row q0, lanes 16-31 row q1, lane L holding chunk L & 15 of
// h.  Each half reduces with the butterfly offsets 8, 4, 2, 1, the same pairs
// as row_dot_h's 32-lane butterfly (whose offset-16 step adds the zeros of the
// idle lanes), so each result equals row_dot_h of that row.  Returns the row
// of this lane's half (r0 on lanes 0-15, r1 on lanes 16-31); lanes 0 and 16
// hold the finished values.
template <int BITS>
__device__ __forceinline__ float row_dot_h_halves(const uint8_t* q0, const uint32_t* sb0, const uint8_t* q1,
                                                  const uint32_t* sb1, const HF<BITS>& h, int lane) {
    constexpr int CPG = 64 / Codes<BITS>::kCols;
    const int c = lane & 15;
    const uint8_t* q = lane < 16 ? q0 : q1;
    const uint32_t* sb = lane < 16 ? sb0 : sb1;
    const float A = chunk_dot_f(reinterpret_cast<const uint4*>(q)[c], h.v, Codes<BITS>{});
    float v = chunk_term_f<BITS>(A, h.s, sb[c / CPG]);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}

// NP row pairs of row_dot_h_halves at once (rows q[2i] on lanes 0-15 and
// q[2i+1] on lanes 16-31), their butterflies interleaved; v[i] equals
// row_dot_h_halves of pair i.
template <int BITS, int NP>
__device__ __forceinline__ void row_dot_h_halves_n(const uint8_t* const (&q)[2 * NP], const uint32_t* const (&sb)[2 * NP],
                                                   const HF<BITS>& h, int lane, float (&v)[NP]) {
    constexpr int CPG = 64 / Codes<BITS>::kCols;
    const int c = lane & 15, hi = lane >> 4;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const uint8_t* qi = hi ? q[2 * i + 1] : q[2 * i];  // static indices: the arrays stay in registers
        const uint32_t* si = hi ? sb[2 * i + 1] : sb[2 * i];
        const float A = chunk_dot_f(reinterpret_cast<const uint4*>(qi)[c], h.v, Codes<BITS>{});
        v[i] = chunk_term_f<BITS>(A, h.s, si[c / CPG]);
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < NP; ++i) v[i] = __fadd_rn(v[i], __shfl_xor_sync(kFullMask, v[i], off));
}

}  // namespace moe