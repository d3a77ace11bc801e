// decode_kernels.cu -- per-layer decode kernels for sm_103a: router logits,
// top-k + dispatch (+ the tokens' block-fixed-point digits), batched dequant
// gate/up + SwiGLU and down (a CTA per active expert and row block, so each
// expert's weights are read once for all of its tokens), the per-token
// weighted combine, and the between-layer renormalisation.  They serve streaming contexts (which read the routing
// back between kernels), batches above the persistent kernel's limit and
// single-layer calls; the arithmetic is the one in gemv.cuh, shared with the
// persistent stack kernel, so both paths give the same bits.
#include "gemv.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxE = 1024, kMaxK = 16, kMaxB = 64;
constexpr int kThreads = 256, kNWarps = kThreads / 32;
constexpr int kWorkPairs = 8;  // pairs per work item of the batched kernels

// ---------------------------------------------------------------------------
// router logits: one warp per expert, all tokens
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) router_kernel(const uint16_t* __restrict__ w_r,
                                                          const float* __restrict__ bias,
                                                          const float* __restrict__ x, int B, int H, int E,
                                                          float* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kNWarps + warp;
    if (e >= E) return;
    const float be = bias ? bias[e] : 0.0f;
    for (int t = 0; t < B; ++t) {
        const float v = router_logit(w_r + (size_t)e * H, x + (size_t)t * H, H, be, lane);
        if (lane == 0) logits[(size_t)t * E + e] = v;
    }
}

// ---------------------------------------------------------------------------
// top-k, routing weights, shared gate, token digits, and the dispatch lists
// ---------------------------------------------------------------------------
__device__ int block_scan_incl(int v, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFullMask, s, off);
            if (lane >= off) s += o;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    return v;
}

template <int BITS>
__device__ void token_digits(const float* x, int H, int lane, uint32_t* words, int32_t* sums, int32_t* expo) {
    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    float mx = 0.0f;
    for (int j = lane; j < H; j += 32) mx = fmaxf(mx, fabsf(x[j]));
    const int e = bfp_exponent(warp_max(mx));
    for (int c = lane; c < H / CC; c += 32) {
        int V[CC];
#pragma unroll
        for (int i = 0; i < CC; ++i) V[i] = bfp_int(x[c * CC + i], e);
        uint32_t dw[DW];
        int S;
        bfp_chunk<BITS>(V, dw, S);
#pragma unroll
        for (int i = 0; i < DW; ++i) words[(size_t)c * DW + i] = dw[i];
        sums[c] = S;
    }
    if (lane == 0) *expo = e;
}

// Routing of one token per CTA of kRtThreads threads: top-k of its logits
// (each warp the k best of its 32-expert slices, one warp merging the sorted
// lists by k rounds over their heads: logit descending, ties to the lower
// id, the order of warp_topk), the routing weights, the shared gate and
// (unless mode & 4) the block-fixed-point digits of its x.  Published to the
// host when pub.ready is set (one token only: several tokens publish with
// publish_kernel afterwards).
constexpr int kRtThreads = 512, kRtWarps = kRtThreads / 32;

template <int BITS>
__global__ void __launch_bounds__(kRtThreads) route_token_kernel(
    Shapes s, int mode, const float* __restrict__ logits, const float* __restrict__ x,
    const uint16_t* __restrict__ wsg, int32_t* idx, float* w, float* sigma, int32_t* uidx, float* uw, TokenDigits xd,
    HostGate pub, int pub_layer) {
    const int E = s.n_experts, k = s.top_k, H = s.hidden;
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ __align__(16) float rt_x[];  // [H] this token's x
    __shared__ float s_lg[kMaxE];
    __shared__ uint32_t s_ck[kRtWarps][kMaxK];
    __shared__ int32_t s_ci[kRtWarps][kMaxK];
    __shared__ float s_val[kMaxK], s_w[kMaxK];
    __shared__ float s_red[kRtWarps];
    __shared__ int s_xe;
    const float* lg = logits + (size_t)t * E;
    const int M = (E + kRtThreads - 1) / kRtThreads;  // keys per lane (<= 2)
    const int nlist = (E + 32 * M - 1) / (32 * M);
    // level 1: the k best of this warp's experts w*32*M + 32 m + lane
    uint32_t key0 = 0u, key1 = 0u;
    for (int m = 0; m < M; ++m) {
        const int j = warp * 32 * M + 32 * m + lane;
        if (j < E) {
            const float v = lg[j];
            s_lg[j] = v;
            if (m == 0)
                key0 = order_key(v);
            else
                key1 = order_key(v);
        }
    }
    if (warp < nlist) {
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            const int bm = key1 > key0 ? 1 : 0;
            const uint32_t best = bm ? key1 : key0;
            const uint32_t mx = __reduce_max_sync(kFullMask, best);
            const uint32_t win = __reduce_min_sync(
                kFullMask, (best == mx && mx != 0u) ? (uint32_t)(warp * 32 * M + 32 * bm + lane) : 0xffffffffu);
            if (lane == 0) {
                s_ck[warp][r] = mx;
                s_ci[warp][r] = (int)win;
            }
            if (win == 0xffffffffu) break;
            if (lane == (int)(win & 31u)) {
                if (((win - (uint32_t)(warp * 32 * M)) >> 5) == 0u)
                    key0 = 0u;
                else
                    key1 = 0u;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        // level 2: merge the lists' heads; lane i < nlist holds list i's head and next entry
        uint32_t hk = 0u, hi = 0xffffffffu, nk = 0u, ni = 0xffffffffu;
        if (lane < nlist) {
            if (s_ci[lane][0] >= 0) hk = s_ck[lane][0], hi = (uint32_t)s_ci[lane][0];
            if (k > 1 && hi != 0xffffffffu && s_ci[lane][1] >= 0) nk = s_ck[lane][1], ni = (uint32_t)s_ci[lane][1];
        }
        int pos = 1;
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            const uint32_t mx = __reduce_max_sync(kFullMask, hk);
            const uint32_t win = __reduce_min_sync(kFullMask, hk == mx ? hi : 0xffffffffu);
            if (lane == 0) {
                idx[t * k + r] = (int)win;
                if (uidx) uidx[t * k + r] = (int)win;
                s_val[r] = s_lg[win];
            }
            if (hi == win) {
                hk = nk, hi = ni;
                ++pos;
                nk = 0u, ni = 0xffffffffu;
                if (hi != 0xffffffffu && pos < k && s_ci[lane][pos] >= 0) nk = s_ck[lane][pos], ni = (uint32_t)s_ci[lane][pos];
            }
        }
        __syncwarp();
        topk_weights(s_lg, E, k, s.norm_topk, lane, s_val, s_w);
        if (lane < k) {
            w[t * k + lane] = s_w[lane];
            if (uw) uw[t * k + lane] = s_w[lane];
        }
    } else if (warp == 1) {
        const float sg = wsg ? shared_gate(wsg, x + (size_t)t * H, H, lane) : 0.0f;
        if (lane == 0) sigma[t] = sg;
    }
    if (!(mode & 4)) {
        // digits of x: max |x| over the block, then a warp per 32 columns
        float mx = 0.0f;
        for (int j = threadIdx.x; j < H; j += kRtThreads) {
            const float v = x[(size_t)t * H + j];
            rt_x[j] = v;
            mx = fmaxf(mx, fabsf(v));
        }
        mx = warp_max(mx);
        if (lane == 0) s_red[warp] = mx;
        __syncthreads();
        if (threadIdx.x == 0) {
            float m2 = s_red[0];
            for (int i = 1; i < kRtWarps; ++i) m2 = fmaxf(m2, s_red[i]);
            s_xe = bfp_exponent(m2);
            xd.exps[t] = s_xe;
        }
        __syncthreads();
        const int nc = H / Codes<BITS>::kCols;
        make_digits<BITS>(1, H, rt_x, xd.words + (size_t)t * nc * Codes<BITS>::kDigitWords, xd.sums + (size_t)t * nc,
                          &s_xe, 0, kRtWarps);
    }
    if (pub.ready) {
        // one token: publish the routing to the host
        __syncthreads();
        for (int i = threadIdx.x; i < k; i += kRtThreads) pub.idx[(size_t)pub_layer * pub.idx_stride + i] = idx[i];
        __threadfence_system();
        __syncthreads();
        if (threadIdx.x == 0) pub.ready[pub_layer] = *pub.epoch;
    }
}

__global__ void __launch_bounds__(1024) route_dispatch_kernel(
    Shapes s, int mode, const float* __restrict__ logits, const float* __restrict__ x,
    const uint16_t* __restrict__ wsg, int B, int32_t* idx, float* w, float* sigma, int32_t* uidx, float* uw,
    const uint8_t* const* dir, const uint8_t* shared_blob, Dispatch d, TokenDigits xd,
    unsigned long long* hit_counter, HostGate pub, int pub_layer) {
    const int E = s.n_experts, k = s.top_k, H = s.hidden;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __shared__ int32_t s_idx[kMaxB][kMaxK];
    __shared__ float s_val[kMaxB][kMaxK], s_w[kMaxB][kMaxK];
    __shared__ int s_cnt[kMaxE];
    __shared__ unsigned long long s_msk[kMaxE];
    __shared__ int s_scan[kMaxE];
    __shared__ int s_wsum[32];
    __shared__ int s_total;

    if (mode & 1) {
        for (int t = blockIdx.x * nw + warp; t < B; t += gridDim.x * nw) {
            warp_topk(logits + (size_t)t * E, E, k, s.norm_topk, lane, s_idx[t], s_val[t], s_w[t]);
            if (lane < k) {
                idx[t * k + lane] = s_idx[t][lane];
                w[t * k + lane] = s_w[t][lane];
                if (uidx) uidx[t * k + lane] = s_idx[t][lane];
                if (uw) uw[t * k + lane] = s_w[t][lane];
            }
            const float sg = wsg ? shared_gate(wsg, x + (size_t)t * H, H, lane) : 0.0f;
            if (lane == 0) sigma[t] = sg;
            if (mode & 4) continue;  // routing only: no token digits
            const int nc = H / (s.bits == 4 ? 32 : 16);
            const int dwn = s.bits == 4 ? 24 : 12;
            if (s.bits == 4)
                token_digits<4>(x + (size_t)t * H, H, lane, xd.words + (size_t)t * nc * dwn, xd.sums + (size_t)t * nc,
                                xd.exps + t);
            else
                token_digits<8>(x + (size_t)t * H, H, lane, xd.words + (size_t)t * nc * dwn, xd.sums + (size_t)t * nc,
                                xd.exps + t);
        }
    }
    if ((mode & 1) && pub.ready) {
        // streaming, single CTA: publish the routing to the host
        __syncthreads();
        for (int i = threadIdx.x; i < B * k; i += blockDim.x) pub.idx[(size_t)pub_layer * pub.idx_stride + i] = idx[i];
        __threadfence_system();
        __syncthreads();
        if (threadIdx.x == 0) pub.ready[pub_layer] = *pub.epoch;
    }
    if (!(mode & 2)) return;
    __syncthreads();  // (mode 2 runs as a single CTA)
    const int tid = threadIdx.x;
    for (int e = tid; e < kMaxE; e += blockDim.x) {
        s_cnt[e] = 0;
        s_msk[e] = 0ull;
    }
    __syncthreads();
    const int npair = B * k;
    for (int p = tid; p < npair; p += blockDim.x) {
        const int e = idx[p], t = p / k;
        atomicAdd(&s_cnt[e], 1);
        atomicOr(&s_msk[e], 1ull << t);
    }
    __syncthreads();
    // packed scan: high 16 bits = pair count, low 16 bits = active flag
    const int mine = (tid < E) ? ((s_cnt[tid] << 16) | (s_cnt[tid] > 0 ? 1 : 0)) : 0;
    const int incl = block_scan_incl(mine, s_wsum);
    const int excl = incl - mine;
    if (tid < E) s_scan[tid] = excl;
    if (tid == blockDim.x - 1) s_total = incl;
    __syncthreads();
    const int n_routed = s_total & 0xffff;
    if (tid < E && s_cnt[tid] > 0) {
        const int a = excl & 0xffff;
        const uint8_t* blob = dir[tid];
        if (!blob) atomicExch(d.status, 1);
        d.act_expert[a] = tid;
        d.act_blob[a] = blob;
        d.act_off[a] = excl >> 16;
    }
    // pair of (token t, expert e): tokens ascending within each expert's run
    for (int p = tid; p < npair; p += blockDim.x) {
        const int e = idx[p], t = p / k;
        const int rank = __popcll(s_msk[e] & ((1ull << t) - 1ull));
        const int q = (s_scan[e] >> 16) + rank;
        d.pair_token[q] = t;
        d.pair_w[q] = w[p];
    }
    if (tid == 0) {
        if (shared_blob) {
            d.act_expert[n_routed] = -1;
            d.act_blob[n_routed] = shared_blob;
            d.act_off[n_routed] = npair;
            d.act_off[n_routed + 1] = npair + B;
            *d.n_act = n_routed + 1;
        } else {
            d.act_off[n_routed] = npair;
            *d.n_act = n_routed;
        }
        if (hit_counter) atomicAdd(hit_counter, (unsigned long long)n_routed);
    }
    if (shared_blob) {
        for (int t = tid; t < B; t += blockDim.x) {
            d.pair_token[npair + t] = t;
            d.pair_w[npair + t] = sigma[t];
        }
    }
    // each token's pairs in ascending pair order (ascending expert, the shared one last)
    __syncthreads();
    const int npt = k + (shared_blob ? 1 : 0);
    for (int t = tid; t < B; t += blockDim.x) {
        int v[kMaxK + 1];
        for (int i = 0; i < k; ++i) {
            const int e = idx[t * k + i];
            v[i] = (s_scan[e] >> 16) + __popcll(s_msk[e] & ((1ull << t) - 1ull));
        }
        for (int i = 1; i < k; ++i) {  // insertion sort, k <= 16
            const int x = v[i];
            int j = i - 1;
            while (j >= 0 && v[j] > x) {
                v[j + 1] = v[j];
                --j;
            }
            v[j + 1] = x;
        }
        if (shared_blob) v[k] = npair + t;
        for (int i = 0; i < npt; ++i) d.tok_pairs[t * (kMaxK + 1) + i] = v[i];
    }
    // work items of the batched kernels: (active expert, first pair, <= kWorkPairs pairs),
    // so an expert chosen by many tokens is spread over many CTAs
    __syncthreads();
    const int n_all = n_routed + (shared_blob ? 1 : 0);
    const int P = tid < n_all ? d.act_off[tid + 1] - d.act_off[tid] : 0;
    const int grp = (P + kWorkPairs - 1) / kWorkPairs;
    const int gincl = block_scan_incl(grp, s_wsum);
    for (int g = 0; g < grp; ++g)
        d.work[gincl - grp + g] = make_int4(tid, d.act_off[tid] + g * kWorkPairs, min(kWorkPairs, P - g * kWorkPairs), 0);
    if (tid == blockDim.x - 1) *d.n_work = gincl;
}

// ---------------------------------------------------------------------------
// down rows multiply fp32 h (HF: one chunk per lane)
// ---------------------------------------------------------------------------
// this lane's chunk of an h vector of `cols` values (cols / CC <= 32), zeros past the end
template <int BITS>
__device__ __forceinline__ void load_hf(const float* h, int cols, int lane, HF<BITS>& hf) {
    constexpr int CC = Codes<BITS>::kCols;
    const bool mine = lane < cols / CC;
#pragma unroll
    for (int i = 0; i < CC; i += 4) {
        const float4 f = mine ? *reinterpret_cast<const float4*>(h + lane * CC + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        hf.v[i] = f.x, hf.v[i + 1] = f.y, hf.v[i + 2] = f.z, hf.v[i + 3] = f.w;
    }
    hf_sum(hf);
}

// ---------------------------------------------------------------------------
// batched gate/up: a CTA per (active expert, kGuRows rows); the digits of the
// expert's tokens staged in shared memory kGuTok at a time; each warp's rows
// against each token with row_dot_x2 (the persistent kernel's arithmetic)
// ---------------------------------------------------------------------------
constexpr int kGuRows = 32, kGuTok = 8;

template <int BITS, int NPER>
__global__ void __launch_bounds__(kThreads, 2) gateup_batched_kernel(Shapes s, Dispatch d, TokenDigits xd,
                                                                  float* __restrict__ h) {
    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    static_assert(kGuTok >= kWorkPairs, "a work item's tokens fit the staging area");
    extern __shared__ __align__(16) uint32_t g_sm[];
    if ((int)blockIdx.y >= *d.n_work) return;
    const int4 wi = d.work[blockIdx.y];
    const int a = wi.x, pg = wi.y, n = wi.z;
    const bool shared = d.act_expert[a] < 0;
    const int rows = shared ? s.shared_inter : s.inter;
    const int r0 = blockIdx.x * kGuRows;
    if (r0 >= rows) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden, nc = H / CC, ng = H / 64;
    uint32_t* sw = g_sm;                                                 // [kGuTok][nc * DW]
    int32_t* ss = reinterpret_cast<int32_t*>(g_sm + kGuTok * nc * DW);  // [kGuTok][nc]
    const uint8_t* blob = d.act_blob[a];
    const BlobLayout L = blob_layout(H, rows, BITS);
    const size_t row_bytes = (size_t)H * BITS / 8;
    for (int i = threadIdx.x; i < n * nc * DW / 4; i += kThreads) {
        const int j = i / (nc * DW / 4), o = i - j * (nc * DW / 4);
        const int t = d.pair_token[pg + j];
        reinterpret_cast<uint4*>(sw)[i] = reinterpret_cast<const uint4*>(xd.words + (size_t)t * nc * DW)[o];
    }
    for (int i = threadIdx.x; i < n * nc; i += kThreads) {
        const int j = i / nc;
        ss[i] = xd.sums[(size_t)d.pair_token[pg + j] * nc + (i - j * nc)];
    }
    __syncthreads();
    constexpr int CPG = 64 / CC;
    int ex[kGuTok];
#pragma unroll
    for (int j = 0; j < kGuTok; ++j) ex[j] = j < n ? xd.exps[d.pair_token[pg + j]] : 0;
    for (int r = r0 + warp; r < min(r0 + kGuRows, rows); r += kNWarps) {
        // the row's code chunks and scale/bias words, once for all tokens
        const uint4* gq = reinterpret_cast<const uint4*>(blob + L.gate_q + r * row_bytes);
        const uint4* uq = reinterpret_cast<const uint4*>(blob + L.up_q + r * row_bytes);
        const uint32_t* gsb = reinterpret_cast<const uint32_t*>(blob + L.gate_sb) + (size_t)r * ng;
        const uint32_t* usb = reinterpret_cast<const uint32_t*>(blob + L.up_sb) + (size_t)r * ng;
        uint4 wg[NPER], wu[NPER];
        uint32_t sg[NPER], su[NPER];
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int c = lane + 32 * i;
            if (c < nc) {
                wg[i] = __ldg(gq + c), wu[i] = __ldg(uq + c);
                sg[i] = __ldg(gsb + c / CPG), su[i] = __ldg(usb + c / CPG);
            }
        }
        // per token: this lane's partial sums, in row_dot_x2's chunk order
        float v[2 * kGuTok];
#pragma unroll
        for (int j = 0; j < kGuTok; ++j) {
            float p0 = 0.0f, p1 = 0.0f;
            if (j < n) {
                XDigits<BITS, NPER> xr;
                load_xdigits(xr, sw + (size_t)j * nc * DW, ss + j * nc, nc, lane);
#pragma unroll
                for (int i = 0; i < NPER; ++i) {
                    const int c = lane + 32 * i;
                    if (c < nc) {
                        p0 = chunk_term(p0, chunk_dot(wg[i], xr.dw[i], Codes<BITS>{}), xr.S[i], sg[i]);
                        p1 = chunk_term(p1, chunk_dot(wu[i], xr.dw[i], Codes<BITS>{}), xr.S[i], su[i]);
                    }
                }
            }
            v[2 * j] = p0;
            v[2 * j + 1] = p1;
        }
        // reduce-scatter of the 16 partials over the warp: the xor-16, 8, 4, 2, 1
        // pairs of warp_sum, each value followed by the lanes that keep it;
        // lanes 2m and 2m + 1 end with value m (bitwise warp_sum of it)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool hi = lane & 16;
            const float send = hi ? v[i] : v[8 + i], keep = hi ? v[8 + i] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(kFullMask, send, 16));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool hi = lane & 8;
            const float send = hi ? v[i] : v[4 + i], keep = hi ? v[4 + i] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(kFullMask, send, 8));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const bool hi = lane & 4;
            const float send = hi ? v[i] : v[2 + i], keep = hi ? v[2 + i] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(kFullMask, send, 4));
        }
        {
            const bool hi = lane & 2;
            const float send = hi ? v[0] : v[1], keep = hi ? v[1] : v[0];
            v[0] = __fadd_rn(keep, __shfl_xor_sync(kFullMask, send, 2));
        }
        v[0] = __fadd_rn(v[0], __shfl_xor_sync(kFullMask, v[0], 1));
        // value m = 2 j (gate) on lanes 4j, 4j+1, value 2 j + 1 (up) on lanes 4j+2, 4j+3
        const float up = __shfl_down_sync(kFullMask, v[0], 2);
        const int j = lane >> 2;
        int e = 0;
#pragma unroll
        for (int q = 0; q < kGuTok; ++q)
            if (q == j) e = ex[q];
        if ((lane & 3) == 0 && j < n)
            h[(size_t)(pg + j) * s.h_stride + r] = silu_mul(pow2_scale(v[0], -e), pow2_scale(up, -e));
    }
}

// ---------------------------------------------------------------------------
// batched down: a CTA per (work item, kDnRows output rows); for each of the
// item's pairs, weighted row dots into part[pair][row].  The item's h rows are
// staged once per CTA in a chunk-interleaved layout (float4 i/4 of chunk c at
// [(i/4) * nch + c], so the lanes that each read one chunk hit consecutive
// addresses), with each chunk's sum (hf_sum's order) formed once per CTA.
// int4 rows of 16 chunks: each warp keeps the codes of 8 rows (4 half-warp
// row pairs) in registers for all of the item's pairs and interleaves their
// butterflies; other shapes: one row at a time (row_dot_h).
// ---------------------------------------------------------------------------
constexpr int kDnRows = 64;

template <int BITS>
__global__ void __launch_bounds__(kThreads, 2) down_batched_kernel(Shapes s, Dispatch d, const float* __restrict__ h,
                                                                float* __restrict__ part) {
    constexpr int CC = Codes<BITS>::kCols, CPG = 64 / CC, RW = kDnRows / kNWarps, NP = RW / 2;
    static_assert(RW == 8, "eight rows per warp: four half-warp row pairs");
    __shared__ __align__(16) float hs[kWorkPairs][1024];  // the item's h rows (cols <= 1024), chunk-interleaved
    __shared__ float hsum[kWorkPairs][64];                // per-chunk sums of h (<= 64 chunks)
    if ((int)blockIdx.y >= *d.n_work) return;
    const int4 wi = d.work[blockIdx.y];
    const int a = wi.x, pg = wi.y, n = wi.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden;
    const bool shared = d.act_expert[a] < 0;
    const int cols = shared ? s.shared_inter : s.inter;
    const int nch = cols / CC;
    const BlobLayout L = blob_layout(H, cols, BITS);
    const uint8_t* blob = d.act_blob[a];
    const size_t row_bytes = (size_t)cols * BITS / 8;
    const int ng = cols / 64;
    const int jb = blockIdx.x * kDnRows + warp * RW;
    const bool pairs16 = BITS == 4 && nch == 16 && jb + RW <= H;
    // this warp's codes first (the longest latency), then the staging
    uint4 q[NP];
    uint32_t sb[NP];
    const int c16 = lane & 15, hi = lane >> 4;
    if (pairs16) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int j = jb + 2 * i + hi;
            q[i] = __ldg(reinterpret_cast<const uint4*>(blob + L.down_q + j * row_bytes) + c16);
            sb[i] = __ldg(reinterpret_cast<const uint32_t*>(blob + L.down_sb) + (size_t)j * ng + c16 / CPG);
        }
    }
    for (int i = threadIdx.x; i < n * cols / 4; i += kThreads) {
        const int j = i / (cols / 4), o = i - j * (cols / 4);  // float4 o of pair j: chunk o*4/CC, element (o*4)%CC
        const float4 v = reinterpret_cast<const float4*>(h + (size_t)(pg + j) * s.h_stride)[o];
        const int cc = (o * 4) / CC, e4 = ((o * 4) % CC) >> 2;
        reinterpret_cast<float4*>(hs[j])[e4 * nch + cc] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n * nch; i += kThreads) {
        const int j = i / nch, cc = i - j * nch;
        float sum = hs[j][cc * 4];
#pragma unroll 1
        for (int e = 1; e < CC; ++e) sum = __fadd_rn(sum, hs[j][((e >> 2) * nch + cc) * 4 + (e & 3)]);
        hsum[j][cc] = sum;
    }
    __syncthreads();
    if (jb >= H) return;
    const int je = min(H, jb + RW);
    if (pairs16) {
        for (int p = 0; p < n; ++p) {
            HF<BITS> hd;
#pragma unroll
            for (int i = 0; i < CC; i += 4) {
                const float4 f = reinterpret_cast<const float4*>(hs[p])[(i >> 2) * nch + c16];
                hd.v[i] = f.x, hd.v[i + 1] = f.y, hd.v[i + 2] = f.z, hd.v[i + 3] = f.w;
            }
            hd.s = hsum[p][c16];
            // row_dot_h_halves of the four row pairs, butterflies interleaved
            float v[NP];
#pragma unroll
            for (int i = 0; i < NP; ++i) v[i] = chunk_term_f<BITS>(chunk_dot_f(q[i], hd.v, Codes<BITS>{}), hd.s, sb[i]);
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
                for (int i = 0; i < NP; ++i) v[i] = __fadd_rn(v[i], __shfl_xor_sync(kFullMask, v[i], off));
            if (c16 == 0) {
                const float wp = d.pair_w[pg + p];
                float* out = part + (size_t)(pg + p) * H + jb + hi;
#pragma unroll
                for (int i = 0; i < NP; ++i) out[2 * i] = __fmul_rn(wp, v[i]);
            }
        }
    } else {
        for (int p = 0; p < n; ++p) {
            HF<BITS> hd;
            const bool mine = lane < nch;
#pragma unroll
            for (int i = 0; i < CC; i += 4) {
                const float4 f = mine ? reinterpret_cast<const float4*>(hs[p])[(i >> 2) * nch + lane]
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                hd.v[i] = f.x, hd.v[i + 1] = f.y, hd.v[i + 2] = f.z, hd.v[i + 3] = f.w;
            }
            hd.s = mine ? hsum[p][lane] : 0.0f;
            const float wp = d.pair_w[pg + p];
            float* out = part + (size_t)(pg + p) * H;
            for (int j = jb; j < je; ++j) {
                const float v = row_dot_h<BITS>(blob + L.down_q + j * row_bytes,
                                                reinterpret_cast<const uint32_t*>(blob + L.down_sb) + (size_t)j * ng,
                                                hd, cols, lane);
                if (lane == 0) out[j] = __fmul_rn(wp, v);
            }
        }
    }
}

// y[t][j] = sum of the token's weighted pair rows in ascending pair order
__global__ void __launch_bounds__(kThreads) combine_kernel(Dispatch d, const float* __restrict__ part,
                                                           float* __restrict__ y, int B, int H, int npt) {
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= B * H) return;
    const int t = i / H, j = i - t * H;
    float acc = 0.0f;
    for (int q = 0; q < npt; ++q) acc = __fadd_rn(acc, part[(size_t)d.tok_pairs[t * (kMaxK + 1) + q] * H + j]);
    y[i] = acc;
}

// x = y / sqrt(mean(y^2) + eps), one block of kRenormThreads per token
__global__ void __launch_bounds__(kRenormThreads) renorm_kernel(const float* __restrict__ y, float* __restrict__ xn,
                                                                int H, float eps) {
    __shared__ float red[2 * kRenormThreads / 32];
    const int t = blockIdx.x;
    const float* yt = y + (size_t)t * H;
    float mx;
    const float r = renorm_block(yt, H, eps, red, &mx);
    for (int j = threadIdx.x; j < H; j += kRenormThreads) xn[(size_t)t * H + j] = __fmul_rn(yt[j], r);
}

// streaming: the routing of a layer to mapped host memory, then the call's epoch
__global__ void publish_kernel(const int32_t* __restrict__ idx, int n, int32_t* out, volatile uint32_t* ready,
                               const volatile uint32_t* epoch) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = idx[i];
    __threadfence_system();
    __syncthreads();
    if (threadIdx.x == 0) *ready = *epoch;
}

}  // namespace

cudaError_t launch_router(const Shapes& s, const uint16_t* w_r, const float* bias, const float* x, int B,
                          float* logits, cudaStream_t st) {
    if (s.hidden <= 2048) return launch_logits(w_r, bias, x, B, s.hidden, s.n_experts, 8, logits, st);
    router_kernel<<<(s.n_experts + kNWarps - 1) / kNWarps, kThreads, 0, st>>>(w_r, bias, x, B, s.hidden,
                                                                            s.n_experts, logits);
    return cudaGetLastError();
}

cudaError_t launch_route_dispatch(const Shapes& s, int mode, const float* logits, const float* x,
                                  const uint16_t* shared_gate_w, int B, int32_t* idx, float* w, float* sigma,
                                  int32_t* user_idx, float* user_w, const uint8_t* const* dir_layer,
                                  const uint8_t* shared_blob, Dispatch d, TokenDigits xd,
                                  unsigned long long* hit_counter, cudaStream_t st, const HostGate* pub,
                                  int pub_layer) {
    // the per-token part (top-k, weights, shared gate, digits): one CTA per token,
    // publishing itself for one token, else a small kernel follows; the dispatch
    // lists in one CTA of 1024 threads
    const bool fused_pub = pub && (mode & 1) && B == 1;
    const HostGate none{};
    if (mode & 1) {
        const size_t xs_bytes = (mode & 4) ? 0 : (size_t)s.hidden * sizeof(float);
        if (s.n_experts > kMaxE || s.top_k > kMaxK) return cudaErrorInvalidValue;
        cudaError_t e = cudaSuccess;
        if (s.bits == 4) {
            e = smem_limit(reinterpret_cast<const void*>(route_token_kernel<4>), (int)xs_bytes);
            if (e == cudaSuccess)
                route_token_kernel<4><<<B, kRtThreads, xs_bytes, st>>>(s, mode, logits, x, shared_gate_w, idx, w,
                                                                        sigma, user_idx, user_w, xd,
                                                                        fused_pub ? *pub : none, pub_layer);
        } else {
            e = smem_limit(reinterpret_cast<const void*>(route_token_kernel<8>), (int)xs_bytes);
            if (e == cudaSuccess)
                route_token_kernel<8><<<B, kRtThreads, xs_bytes, st>>>(s, mode, logits, x, shared_gate_w, idx, w,
                                                                        sigma, user_idx, user_w, xd,
                                                                        fused_pub ? *pub : none, pub_layer);
        }
        if (e != cudaSuccess) return e;
        if (pub && !fused_pub) {
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            publish_kernel<<<1, 256, 0, st>>>(idx, B * s.top_k, pub->idx + (size_t)pub_layer * pub->idx_stride,
                                              pub->ready + pub_layer, pub->epoch);
        }
    }
    if (mode & 2) {
        route_dispatch_kernel<<<1, 1024, 0, st>>>(s, mode & ~1, logits, x, shared_gate_w, B, idx, w, sigma,
                                                  user_idx, user_w, dir_layer, shared_blob, d, xd, hit_counter,
                                                  none, 0);
    }
    return cudaGetLastError();
}

cudaError_t launch_gateup_batched(const Shapes& s, Dispatch d, TokenDigits xd, float* h, cudaStream_t st) {
    const int rows = s.inter > s.shared_inter ? s.inter : s.shared_inter;
    dim3 grid((rows + kGuRows - 1) / kGuRows, s.max_work);
    const int nc = s.hidden / (s.bits == 4 ? 32 : 16), DW = s.bits == 4 ? 24 : 12;
    const size_t smem = (size_t)kGuTok * nc * (DW + 1) * 4;
    const int nper = (nc + 31) / 32;
    cudaError_t e = cudaSuccess;
#define MOE_GU(B_, N_)                                                                                         \
    do {                                                                                                     \
        e = smem_limit(reinterpret_cast<const void*>(gateup_batched_kernel<B_, N_>), (int)smem);              \
        if (e == cudaSuccess) gateup_batched_kernel<B_, N_><<<grid, kThreads, smem, st>>>(s, d, xd, h);       \
    } while (0)
    if (s.bits == 4) {
        if (nper <= 1) MOE_GU(4, 1); else if (nper == 2) MOE_GU(4, 2); else return cudaErrorInvalidValue;
    } else {
        if (nper <= 1) MOE_GU(8, 1); else if (nper == 2) MOE_GU(8, 2); else if (nper <= 4) MOE_GU(8, 4);
        else return cudaErrorInvalidValue;
    }
#undef MOE_GU
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_down_batched(const Shapes& s, Dispatch d, const float* h, float* part, cudaStream_t st) {
    dim3 grid((s.hidden + kDnRows - 1) / kDnRows, s.max_work);
    if (s.bits == 4)
        down_batched_kernel<4><<<grid, kThreads, 0, st>>>(s, d, h, part);
    else
        down_batched_kernel<8><<<grid, kThreads, 0, st>>>(s, d, h, part);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Shapes& s, Dispatch d, const float* part, float* y, int B, bool has_shared,
                           cudaStream_t st) {
    const int n = B * s.hidden;
    combine_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, st>>>(d, part, y, B, s.hidden,
                                                                       s.top_k + (has_shared ? 1 : 0));
    return cudaGetLastError();
}

cudaError_t launch_renorm(const float* y, float* x_next, int B, int hidden, float eps, cudaStream_t st) {
    renorm_kernel<<<B, kRenormThreads, 0, st>>>(y, x_next, hidden, eps);
    return cudaGetLastError();
}

}  // namespace moe
