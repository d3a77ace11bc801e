/*
 * moe_oracle.c -- CPU oracle for the routed sparse-MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code with the CUDA library.
 *
 * It is the plain definition of the layer the Swiftlet pages describe, written
 * out slowly in fp64 (the pages give no formulas; each reading is marked):
 *
 *  - Routed MoE with one shared expert: every layer routes each token to k of E
 *    experts (8 of 256 for the 35B model, 10 of 512 for the 80B model) and also
 *    runs one always-resident shared expert.  [Swiftlet article (linlog.top),
 *    section "Why MoE architectures can be streamed"; README translation
 *    (news.paixiangai.cn), section "How it works"]
 *  - Expert weights are MLX affine int4/int8 group-quantised and dequantised in
 *    the matvec: w = scale * q + bias per group.  [README translation, section
 *    "Relation to TurboFieldfare"; kerneldigest explainer, technology table row
 *    "data-processing"]  [reading: group 64, fp16 scale and bias, the MLX
 *    affine form; the pages give no formula]
 *  - Experts live as fixed-stride blobs, one read fetches one expert.  [Swiftlet
 *    article, section 2 "Fixed-stride pread reads"]  [reading: the blob byte
 *    layout below]
 *  - A bounded slot pool with LFU plus recency eviction caches experts.
 *    [Swiftlet article, section 3 "Expert cache pool and LFU+LRU eviction";
 *    README translation, section "How it works"]  [reading: the exact victim
 *    rule below]
 *
 * Readings where the pages are silent:
 *  - Router: logits l = W_r x (+ optional per-expert bias), experts chosen by
 *    descending logit (ties -> lower index), weights = softmax over the k
 *    chosen logits (softmax-then-top-k with renormalisation, the Qwen3-Next
 *    convention); norm_topk = 0 keeps the full-softmax denominator.
 *  - Because the chosen indices are an integer decision taken from floating
 *    point, the logits are computed in the precision of the GPU kernel (fp32)
 *    in one fixed order: 32 partial sums, element h going to partial
 *    (h / 8) mod 32 in ascending h with fused multiply-add, then a butterfly
 *    reduction with offsets 16, 8, 4, 2, 1, then + bias.
 *  - Expert FFN: SwiGLU, h = silu(G x) * (U x), silu(z) = z / (1 + e^-z),
 *    out = D h.  Shared expert gated by sigmoid(w_sg . x).
 *  - Prefill mode emulates the bf16 tensor-core operands of a grouped GEMM:
 *    weights rounded to bf16 after an fp32 fma(scale, q, bias) and the token
 *    activations rounded to bf16, products accumulated exactly (here in fp64).
 *    The SwiGLU output h is not rounded: rounding it to one bf16 would make
 *    the layer output jump by 2^-8 of an h element whenever the accumulation
 *    order moves h across a bf16 rounding boundary, far outside the layer
 *    tolerance, so the GPU path carries h as a pair of bf16 (hi + lo, h to
 *    about 2^-17) and this definition keeps h exact.
 *
 * Build: gcc -O2 -ffp-contract=off (every fused multiply-add is an explicit
 * fmaf; nothing else is contracted).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_EMISSING -2
#define ORC_EPOOL -3

/* ------------------------------------------------------------------------ */
/* number formats                                                             */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bits -> double (exact). */
double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man + 1024), ex - 25);
    return sign ? -v : v;
}

/* bfloat16 bits -> float (exact: the top half of an fp32). */
float orc_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet). */
uint16_t orc_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t keep = u >> 16, drop = u & 0xFFFFu;
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

static float bf16_round(float f) { return orc_bf16_to_float(orc_float_to_bf16(f)); }

/* ------------------------------------------------------------------------ */
/* dequantisation                                                             */
/* ------------------------------------------------------------------------ */

/*
 * Dequantise rows x cols: w[r][c] = scale[r][c/64] * q[r][c] + bias[r][c/64],
 * in fp64.  q holds one code per byte; sb holds fp16 (scale, bias) pairs per
 * 64-column group.
 */
void orc_dequant(const uint8_t* q, const uint16_t* sb, int rows, int cols, double* w) {
    int ng = cols / 64;
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < cols; ++c) {
            const uint16_t* p = sb + ((size_t)r * ng + c / 64) * 2;
            double s = orc_half_to_double(p[0]), b = orc_half_to_double(p[1]);
            w[(size_t)r * cols + c] = s * (double)q[(size_t)r * cols + c] + b;
        }
    }
}

/* Prefill operand: bf16(fp32 fma(scale, q, bias)). */
static void dequant_bf16(const uint8_t* q, const uint16_t* sb, int rows, int cols, double* w) {
    int ng = cols / 64;
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < cols; ++c) {
            const uint16_t* p = sb + ((size_t)r * ng + c / 64) * 2;
            float s = (float)orc_half_to_double(p[0]), b = (float)orc_half_to_double(p[1]);
            w[(size_t)r * cols + c] = (double)bf16_round(fmaf(s, (float)q[(size_t)r * cols + c], b));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* router                                                                     */
/* ------------------------------------------------------------------------ */

/* One router logit in the fixed fp32 order described in the header. */
float orc_router_logit(const uint16_t* w_row, const float* x, int hidden, float bias) {
    float p[32];
    for (int j = 0; j < 32; ++j) p[j] = 0.0f;
    for (int h = 0; h < hidden; ++h) {
        int lane = (h / 8) % 32;
        p[lane] = fmaf(orc_bf16_to_float(w_row[h]), x[h], p[lane]);
    }
    for (int off = 16; off >= 1; off /= 2) {
        float t[32];
        for (int j = 0; j < 32; ++j) t[j] = p[j] + p[j ^ off];
        for (int j = 0; j < 32; ++j) p[j] = t[j];
    }
    return p[0] + bias;
}

void orc_router_logits(const uint16_t* w, const float* bias, const float* x, int hidden, int n_experts,
                       float* logits) {
    for (int e = 0; e < n_experts; ++e)
        logits[e] = orc_router_logit(w + (size_t)e * hidden, x, hidden, bias ? bias[e] : 0.0f);
}

/* k indices by descending logit, ties to the lower index; output in that order. */
void orc_topk(const float* logits, int n_experts, int k, int32_t* idx) {
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < n_experts; ++e) {
            int taken = 0;
            for (int j = 0; j < i; ++j) taken |= (idx[j] == e);
            if (taken) continue;
            if (best < 0 || logits[e] > logits[best]) best = e;
        }
        idx[i] = best;
    }
}

/*
 * Routing weights of the chosen experts: softmax of the chosen logits
 * (norm_topk = 1) or their full-softmax probabilities (norm_topk = 0).
 */
void orc_topk_weights(const float* logits, int n_experts, int k, const int32_t* idx, int norm_topk,
                      double* w) {
    double m = logits[idx[0]];
    double den = 0.0;
    if (norm_topk) {
        for (int i = 0; i < k; ++i) den += exp((double)logits[idx[i]] - m);
    } else {
        for (int e = 0; e < n_experts; ++e) den += exp((double)logits[e] - m);
    }
    for (int i = 0; i < k; ++i) w[i] = exp((double)logits[idx[i]] - m) / den;
}

/* sigmoid(w_sg . x), dot product in fp64 */
double orc_shared_gate(const uint16_t* w_sg, const float* x, int hidden) {
    double d = 0.0;
    for (int h = 0; h < hidden; ++h) d += (double)orc_bf16_to_float(w_sg[h]) * (double)x[h];
    return 1.0 / (1.0 + exp(-d));
}

/* ------------------------------------------------------------------------ */
/* experts                                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* q_gate; /* inter x hidden codes, one per byte */
    const uint16_t* sb_gate; /* inter x hidden/64 x (scale, bias) fp16 */
    const uint8_t* q_up;
    const uint16_t* sb_up;
    const uint8_t* q_down; /* hidden x inter */
    const uint16_t* sb_down; /* hidden x inter/64 x 2 */
} orc_expert;

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * out = D (silu(G x) * (U x)), all in fp64 (decode mode), or with bf16
 * weights and x and fp64 accumulation (prefill mode).
 */
static int expert_ffn(const orc_expert* e, int hidden, int inter, const float* x, int prefill, double* out) {
    double* wg = malloc(sizeof(double) * (size_t)inter * hidden);
    double* wu = malloc(sizeof(double) * (size_t)inter * hidden);
    double* wd = malloc(sizeof(double) * (size_t)hidden * inter);
    double* xv = malloc(sizeof(double) * (size_t)hidden);
    double* hv = malloc(sizeof(double) * (size_t)inter);
    if (!wg || !wu || !wd || !xv || !hv) {
        free(wg); free(wu); free(wd); free(xv); free(hv);
        return ORC_EINVAL;
    }
    if (prefill) {
        dequant_bf16(e->q_gate, e->sb_gate, inter, hidden, wg);
        dequant_bf16(e->q_up, e->sb_up, inter, hidden, wu);
        dequant_bf16(e->q_down, e->sb_down, hidden, inter, wd);
        for (int c = 0; c < hidden; ++c) xv[c] = (double)bf16_round(x[c]);
    } else {
        orc_dequant(e->q_gate, e->sb_gate, inter, hidden, wg);
        orc_dequant(e->q_up, e->sb_up, inter, hidden, wu);
        orc_dequant(e->q_down, e->sb_down, hidden, inter, wd);
        for (int c = 0; c < hidden; ++c) xv[c] = (double)x[c];
    }
    for (int r = 0; r < inter; ++r) {
        double a = 0.0, u = 0.0;
        for (int c = 0; c < hidden; ++c) {
            a += wg[(size_t)r * hidden + c] * xv[c];
            u += wu[(size_t)r * hidden + c] * xv[c];
        }
        double h = silu(a) * u;
        hv[r] = h;
    }
    for (int j = 0; j < hidden; ++j) {
        double acc = 0.0;
        for (int r = 0; r < inter; ++r) acc += wd[(size_t)j * inter + r] * hv[r];
        out[j] = acc;
    }
    free(wg); free(wu); free(wd); free(xv); free(hv);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* one layer                                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t hidden, n_experts, top_k, inter, shared_inter, norm_topk;
    const uint16_t* router_w;      /* bf16 [n_experts x hidden] */
    const float* router_bias;      /* fp32 [n_experts] or NULL */
    const uint16_t* shared_gate_w; /* bf16 [hidden] */
    const orc_expert* experts;     /* [n_experts]; q_gate == NULL marks one not supplied */
    const orc_expert* shared;
} orc_layer;

static int check_layer(const orc_layer* L) {
    if (!L || L->hidden <= 0 || L->hidden % 64 || L->inter <= 0 || L->inter % 64 || L->shared_inter < 0 ||
        L->shared_inter % 64 || L->top_k < 1 || L->top_k > L->n_experts)
        return ORC_EINVAL;
    return ORC_OK;
}

/* Router half of the layer: logits, chosen experts, their weights, shared gate. */
int orc_route_token(const orc_layer* L, const float* x, float* logits, int32_t* idx, double* w, double* sigma) {
    if (check_layer(L)) return ORC_EINVAL;
    orc_router_logits(L->router_w, L->router_bias, x, L->hidden, L->n_experts, logits);
    orc_topk(logits, L->n_experts, L->top_k, idx);
    orc_topk_weights(logits, L->n_experts, L->top_k, idx, L->norm_topk, w);
    *sigma = (L->shared && L->shared_inter > 0) ? orc_shared_gate(L->shared_gate_w, x, L->hidden) : 0.0;
    return ORC_OK;
}

/* Expert half: y = sum_i w_i E_{idx_i}(x) + sigma * S(x). */
int orc_combine_token(const orc_layer* L, const float* x, const int32_t* idx, const double* w, double sigma,
                      int prefill, double* y) {
    if (check_layer(L)) return ORC_EINVAL;
    int H = L->hidden;
    double* o = malloc(sizeof(double) * (size_t)H);
    if (!o) return ORC_EINVAL;
    for (int j = 0; j < H; ++j) y[j] = 0.0;
    for (int i = 0; i < L->top_k; ++i) {
        const orc_expert* e = &L->experts[idx[i]];
        if (!e->q_gate) {
            free(o);
            return ORC_EMISSING;
        }
        int rc = expert_ffn(e, H, L->inter, x, prefill, o);
        if (rc) {
            free(o);
            return rc;
        }
        for (int j = 0; j < H; ++j) y[j] += w[i] * o[j];
    }
    if (L->shared && L->shared_inter > 0) {
        int rc = expert_ffn(L->shared, H, L->shared_inter, x, prefill, o);
        if (rc) {
            free(o);
            return rc;
        }
        for (int j = 0; j < H; ++j) y[j] += sigma * o[j];
    }
    free(o);
    return ORC_OK;
}

/*
 * The whole layer for one token.  prefill = 0: decode definition (fp64);
 * prefill = 1: bf16-operand emulation.  Routing is identical in both.
 * y is returned rounded to fp32; w and sigma in fp64.
 */
int orc_layer_token(const orc_layer* L, const float* x, int prefill, float* y, int32_t* idx, double* w,
                    double* sigma, float* logits) {
    if (check_layer(L)) return ORC_EINVAL;
    int rc = orc_route_token(L, x, logits, idx, w, sigma);
    if (rc) return rc;
    double* yd = malloc(sizeof(double) * (size_t)L->hidden);
    if (!yd) return ORC_EINVAL;
    rc = orc_combine_token(L, x, idx, w, *sigma, prefill, yd);
    for (int j = 0; j < L->hidden && rc == ORC_OK; ++j) y[j] = (float)yd[j];
    free(yd);
    return rc;
}

/* Stand-in for the omitted attention/norm layers between MoE layers:
 * x = y / sqrt(mean(y^2) + eps), fp64, rounded to fp32. */
void orc_renorm(const float* y, int hidden, double eps, float* x) {
    double ss = 0.0;
    for (int j = 0; j < hidden; ++j) ss += (double)y[j] * (double)y[j];
    double r = 1.0 / sqrt(ss / hidden + eps);
    for (int j = 0; j < hidden; ++j) x[j] = (float)((double)y[j] * r);
}

/* ------------------------------------------------------------------------ */
/* fixed-stride blob (the oracle's own packer and unpacker)                   */
/* ------------------------------------------------------------------------ */
/*
 * Layout v1 [reading: the pages fix only "one fixed-stride blob per expert,
 * one read fetches it"]: little-endian sections in the order
 *   gate.q, up.q, down.q, gate.sb, up.sb, down.sb, zero padding to the stride.
 * X.q: rows x (cols*bits/32) 32-bit words; element c of a row sits in word
 *      c / (32/bits) at bit offset (c mod (32/bits)) * bits (low bits first).
 * X.sb: rows x (cols/64) 32-bit words, low half = fp16 scale, high half =
 *      fp16 bias.
 * Stride = blob bytes rounded up to 4096.
 */

size_t orc_blob_bytes(int hidden, int inter, int bits) {
    size_t q = (size_t)3 * hidden * inter * bits / 8;
    size_t sb = (size_t)3 * (hidden * inter / 64) * 4;
    return q + sb;
}

size_t orc_blob_stride(int hidden, int inter, int bits) {
    return (orc_blob_bytes(hidden, inter, bits) + 4095) / 4096 * 4096;
}

static void put_u32(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

static uint32_t get_u32(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static uint8_t* pack_codes(uint8_t* p, const uint8_t* q, int rows, int cols, int bits) {
    int per = 32 / bits;
    for (int r = 0; r < rows; ++r) {
        for (int wd = 0; wd < cols / per; ++wd) {
            uint32_t v = 0;
            for (int i = 0; i < per; ++i) v |= (uint32_t)q[(size_t)r * cols + wd * per + i] << (i * bits);
            put_u32(p, v);
            p += 4;
        }
    }
    return p;
}

static uint8_t* pack_sb(uint8_t* p, const uint16_t* sb, int rows, int cols) {
    for (size_t g = 0; g < (size_t)rows * (cols / 64); ++g) {
        put_u32(p, (uint32_t)sb[2 * g] | ((uint32_t)sb[2 * g + 1] << 16));
        p += 4;
    }
    return p;
}

int orc_pack_blob(int hidden, int inter, int bits, const orc_expert* e, uint8_t* blob, size_t cap) {
    if ((bits != 4 && bits != 8) || hidden % 64 || inter % 64) return ORC_EINVAL;
    size_t stride = orc_blob_stride(hidden, inter, bits);
    if (cap < stride) return ORC_EINVAL;
    for (int i = 0; i < 3; ++i) {
        const uint8_t* q = i == 0 ? e->q_gate : i == 1 ? e->q_up : e->q_down;
        size_t n = (size_t)hidden * inter;
        for (size_t j = 0; j < n; ++j)
            if (q[j] >> bits) return ORC_EINVAL; /* code out of range for the bit width */
    }
    memset(blob, 0, stride);
    uint8_t* p = blob;
    p = pack_codes(p, e->q_gate, inter, hidden, bits);
    p = pack_codes(p, e->q_up, inter, hidden, bits);
    p = pack_codes(p, e->q_down, hidden, inter, bits);
    p = pack_sb(p, e->sb_gate, inter, hidden);
    p = pack_sb(p, e->sb_up, inter, hidden);
    p = pack_sb(p, e->sb_down, hidden, inter);
    return ORC_OK;
}

static const uint8_t* unpack_codes(const uint8_t* p, uint8_t* q, int rows, int cols, int bits) {
    int per = 32 / bits;
    uint32_t mask = (1u << bits) - 1u;
    for (int r = 0; r < rows; ++r) {
        for (int wd = 0; wd < cols / per; ++wd) {
            uint32_t v = get_u32(p);
            p += 4;
            for (int i = 0; i < per; ++i) q[(size_t)r * cols + wd * per + i] = (uint8_t)((v >> (i * bits)) & mask);
        }
    }
    return p;
}

static const uint8_t* unpack_sb(const uint8_t* p, uint16_t* sb, int rows, int cols) {
    for (size_t g = 0; g < (size_t)rows * (cols / 64); ++g) {
        uint32_t v = get_u32(p);
        p += 4;
        sb[2 * g] = (uint16_t)v;
        sb[2 * g + 1] = (uint16_t)(v >> 16);
    }
    return p;
}

int orc_unpack_blob(int hidden, int inter, int bits, const uint8_t* blob, uint8_t* q_gate, uint16_t* sb_gate,
                    uint8_t* q_up, uint16_t* sb_up, uint8_t* q_down, uint16_t* sb_down) {
    if ((bits != 4 && bits != 8) || hidden % 64 || inter % 64) return ORC_EINVAL;
    const uint8_t* p = blob;
    p = unpack_codes(p, q_gate, inter, hidden, bits);
    p = unpack_codes(p, q_up, inter, hidden, bits);
    p = unpack_codes(p, q_down, hidden, inter, bits);
    p = unpack_sb(p, sb_gate, inter, hidden);
    p = unpack_sb(p, sb_up, inter, hidden);
    unpack_sb(p, sb_down, hidden, inter);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* slot pool simulator                                                        */
/* ------------------------------------------------------------------------ */
/*
 * [reading of "LFU + LRU" / "LFU plus recency": use count first, recency as
 * the tie-break]  Per layer: `slots` slots, slot_expert[s] (-1 = free),
 * slot_freq[s], slot_last[s]; expert_slot[e] (-1 = not resident).  One call
 * requests the set R (ascending, distinct expert ids) at clock t:
 *  - e resident: HIT, freq += 1, last = t.
 *  - e not resident: MISS into the lowest free slot; with no free slot the
 *    victim is the slot, among those whose expert is not in R, with the
 *    smallest (freq, last, slot index) (policy 0, LFU + recency) or the
 *    smallest (last, slot index) (policy 1, LRU).  The loaded expert starts
 *    with freq = 1, last = t.  Counts live only while resident.
 *  - |R| > slots is an error.
 * Two variants of the count, not on the pages, for comparison with the
 * pages' policy (the article's section 3 reports hit rates of 43-70% with
 * speed nearly flat in cache size; the pages say "LFU" without fixing whether
 * a count outlives an eviction, so both lifetimes are given a definition):
 *  - policy 2, persistent LFU: expert_count[e] counts every call that ever
 *    requested e (incremented for all of R when the call starts, kept across
 *    evictions); the victim minimises (expert_count of its expert, last,
 *    slot index).
 *  - policy 3, aged LFU: policy 0, except that a call whose clock t is a
 *    positive multiple of aging_period first halves (rounding down) the
 *    count of every occupied slot.
 * Events (expert, kind 0 = HIT / 1 = MISS, slot, evicted expert or -1) are
 * written in ascending expert order; returns their count.
 */
int orc_pool_request(int slots, int n_experts, int policy, int aging_period, int32_t* slot_expert,
                     int64_t* slot_freq, int64_t* slot_last, int32_t* expert_slot, int64_t* expert_count,
                     int64_t t, const int32_t* req, int n_req, int32_t* events) {
    if (policy < 0 || policy > 3 || (policy == 3 && aging_period < 1)) return ORC_EINVAL;
    if (n_req > slots) return ORC_EPOOL;
    for (int i = 0; i < n_req; ++i) {
        if (req[i] < 0 || req[i] >= n_experts || (i > 0 && req[i] <= req[i - 1])) return ORC_EINVAL;
    }
    if (policy == 3 && t > 0 && t % aging_period == 0) {
        for (int k = 0; k < slots; ++k)
            if (slot_expert[k] >= 0) slot_freq[k] /= 2;
    }
    if (policy == 2) {
        for (int i = 0; i < n_req; ++i) expert_count[req[i]] += 1;
    }
    for (int i = 0; i < n_req; ++i) {
        int e = req[i];
        int32_t* ev = events + 4 * i;
        int s = expert_slot[e];
        if (s >= 0) {
            slot_freq[s] += 1;
            slot_last[s] = t;
            ev[0] = e; ev[1] = 0; ev[2] = s; ev[3] = -1;
            continue;
        }
        int victim = -1;
        for (int k = 0; k < slots; ++k) {
            if (slot_expert[k] < 0) {
                victim = k;
                break;
            }
        }
        int evicted = -1;
        if (victim < 0) {
            for (int k = 0; k < slots; ++k) {
                int in_req = 0;
                for (int j = 0; j < n_req; ++j) in_req |= (req[j] == slot_expert[k]);
                if (in_req) continue;
                if (victim < 0) {
                    victim = k;
                    continue;
                }
                int better;
                if (policy == 1) {
                    better = slot_last[k] < slot_last[victim];
                } else {
                    int64_t fk = slot_freq[k], fv = slot_freq[victim];
                    if (policy == 2) {
                        fk = expert_count[slot_expert[k]];
                        fv = expert_count[slot_expert[victim]];
                    }
                    better = fk < fv || (fk == fv && slot_last[k] < slot_last[victim]);
                }
                if (better) victim = k;
            }
            if (victim < 0) return ORC_EPOOL;
            evicted = slot_expert[victim];
            expert_slot[evicted] = -1;
        }
        slot_expert[victim] = e;
        slot_freq[victim] = 1;
        slot_last[victim] = t;
        expert_slot[e] = victim;
        ev[0] = e; ev[1] = 1; ev[2] = victim; ev[3] = evicted;
    }
    return n_req;
}
