// decode_kernels.cu -- per-layer decode kernels for sm_103a: router logits,
// top-k + dispatch (+ the tokens' block-fixed-point digits), fused dequant
// gate/up + SwiGLU, dequant down + weighted combine, and the between-layer
// renormalisation.  They serve streaming contexts (which read the routing
// back between kernels), batches above the persistent kernel's limit and
// single-layer calls; the arithmetic is the one in gemv.cuh, shared with the
// persistent stack kernel, so both paths give the same bits.
#include "gemv.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxE = 1024, kMaxK = 16, kMaxB = 64;
constexpr int kThreads = 256, kNWarps = kThreads / 32;
constexpr int kGateupRowsPerCta = 16;
constexpr int kDownRowsPerWarp = 2;

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

__global__ void __launch_bounds__(1024) route_dispatch_kernel(
    Shapes s, int mode, const float* __restrict__ logits, const float* __restrict__ x,
    const uint16_t* __restrict__ wsg, int B, int32_t* idx, float* w, float* sigma, int32_t* uidx, float* uw,
    const uint8_t* const* __restrict__ dir, const uint8_t* shared_blob, Dispatch d, TokenDigits xd,
    unsigned long long* hit_counter) {
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
        for (int t = warp; t < B; t += nw) {
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
    if (!(mode & 2)) return;
    __syncthreads();
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
}

// ---------------------------------------------------------------------------
// gate/up: one warp per row, the token's digits read from memory
// ---------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ float row_dot_tok(const uint8_t* q_row, const uint32_t* sb_row, const uint32_t* words,
                                             const int32_t* sums, int e, int cols, int lane) {
    constexpr int CC = Codes<BITS>::kCols, CPG = 64 / CC, DW = Codes<BITS>::kDigitWords;
    const int nchunk = cols / CC;
    const uint4* q = reinterpret_cast<const uint4*>(q_row);
    float part = 0.0f;
    for (int c = lane; c < nchunk; c += 32) {
        uint32_t dw[DW];
#pragma unroll
        for (int i = 0; i < DW; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(words + (size_t)c * DW + i);
            dw[i] = v.x, dw[i + 1] = v.y, dw[i + 2] = v.z, dw[i + 3] = v.w;
        }
        const float A = chunk_dot(__ldg(q + c), dw, Codes<BITS>{});
        part = chunk_term(part, A, sums[c], __ldg(sb_row + c / CPG));
    }
    return pow2_scale(warp_sum(part), -e);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) gateup_kernel(Shapes s, Dispatch d, TokenDigits xd,
                                                          float* __restrict__ h) {
    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    const int a = blockIdx.y;
    if (a >= *d.n_act) return;
    const bool shared = d.act_expert[a] < 0;
    const int rows = shared ? s.shared_inter : s.inter;
    const int r0 = blockIdx.x * kGateupRowsPerCta;
    if (r0 >= rows) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden, nc = H / CC;
    const uint8_t* blob = d.act_blob[a];
    const BlobLayout L = blob_layout(H, rows, BITS);
    const size_t row_bytes = (size_t)H * BITS / 8;
    const int ng = H / 64;
    const int p0 = d.act_off[a], p1 = d.act_off[a + 1];
    const int r1 = min(r0 + kGateupRowsPerCta, rows);
    for (int r = r0 + warp; r < r1; r += kNWarps) {
        const uint8_t* gq = blob + L.gate_q + r * row_bytes;
        const uint8_t* uq = blob + L.up_q + r * row_bytes;
        const uint32_t* gsb = reinterpret_cast<const uint32_t*>(blob + L.gate_sb) + (size_t)r * ng;
        const uint32_t* usb = reinterpret_cast<const uint32_t*>(blob + L.up_sb) + (size_t)r * ng;
        for (int p = p0; p < p1; ++p) {
            const int t = d.pair_token[p];
            const uint32_t* words = xd.words + (size_t)t * nc * DW;
            const int32_t* sums = xd.sums + (size_t)t * nc;
            const int e = xd.exps[t];
            const float g = row_dot_tok<BITS>(gq, gsb, words, sums, e, H, lane);
            const float u = row_dot_tok<BITS>(uq, usb, words, sums, e, H, lane);
            if (lane == 0) h[(size_t)p * s.h_stride + r] = silu_mul(g, u);
        }
    }
}

// ---------------------------------------------------------------------------
// down: the pair's h as digits in registers (one chunk per lane), rows of the warp
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

// y[t][j] = sum over active experts a (ascending, shared last) of w * (D_a[j] . h)
template <int BITS>
__global__ void __launch_bounds__(kThreads) down_kernel(Shapes s, Dispatch d, const float* __restrict__ h,
                                                        float* __restrict__ y, int B) {
    __shared__ float yacc[kNWarps][kDownRowsPerWarp][kMaxB];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden;
    const int n_act = *d.n_act;
    const int j0 = (blockIdx.x * kNWarps + warp) * kDownRowsPerWarp;
    if (j0 >= H) return;
    const int nj = min(kDownRowsPerWarp, H - j0);
    for (int jj = 0; jj < nj; ++jj)
        for (int t = lane; t < B; t += 32) yacc[warp][jj][t] = 0.0f;
    __syncwarp();
    for (int a = 0; a < n_act; ++a) {
        const bool shared = d.act_expert[a] < 0;
        const int cols = shared ? s.shared_inter : s.inter;
        const BlobLayout L = blob_layout(H, cols, BITS);
        const uint8_t* blob = d.act_blob[a];
        const size_t row_bytes = (size_t)cols * BITS / 8;
        const int ng = cols / 64;
        for (int p = d.act_off[a]; p < d.act_off[a + 1]; ++p) {
            HF<BITS> hd;
            load_hf<BITS>(h + (size_t)p * s.h_stride, cols, lane, hd);
            const int t = d.pair_token[p];
            const float wp = d.pair_w[p];
            for (int jj = 0; jj < nj; ++jj) {
                const int j = j0 + jj;
                const float v = row_dot_h<BITS>(blob + L.down_q + j * row_bytes,
                                                reinterpret_cast<const uint32_t*>(blob + L.down_sb) + (size_t)j * ng, hd,
                                                cols, lane);
                if (lane == 0) yacc[warp][jj][t] = __fadd_rn(yacc[warp][jj][t], __fmul_rn(wp, v));
            }
            __syncwarp();
        }
    }
    for (int jj = 0; jj < nj; ++jj)
        for (int t = lane; t < B; t += 32) y[(size_t)t * H + j0 + jj] = yacc[warp][jj][t];
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

}  // namespace

cudaError_t launch_router(const Shapes& s, const uint16_t* w_r, const float* bias, const float* x, int B,
                          float* logits, cudaStream_t st) {
    router_kernel<<<(s.n_experts + kNWarps - 1) / kNWarps, kThreads, 0, st>>>(w_r, bias, x, B, s.hidden,
                                                                            s.n_experts, logits);
    return cudaGetLastError();
}

cudaError_t launch_route_dispatch(const Shapes& s, int mode, const float* logits, const float* x,
                                  const uint16_t* shared_gate_w, int B, int32_t* idx, float* w, float* sigma,
                                  int32_t* user_idx, float* user_w, const uint8_t* const* dir_layer,
                                  const uint8_t* shared_blob, Dispatch d, TokenDigits xd,
                                  unsigned long long* hit_counter, cudaStream_t st) {
    route_dispatch_kernel<<<1, 1024, 0, st>>>(s, mode, logits, x, shared_gate_w, B, idx, w, sigma, user_idx,
                                              user_w, dir_layer, shared_blob, d, xd, hit_counter);
    return cudaGetLastError();
}

cudaError_t launch_gateup(const Shapes& s, Dispatch d, TokenDigits xd, float* h, int B, cudaStream_t st) {
    (void)B;
    const int rows = s.inter > s.shared_inter ? s.inter : s.shared_inter;
    dim3 grid((rows + kGateupRowsPerCta - 1) / kGateupRowsPerCta, s.max_act);
    if (s.bits == 4)
        gateup_kernel<4><<<grid, kThreads, 0, st>>>(s, d, xd, h);
    else
        gateup_kernel<8><<<grid, kThreads, 0, st>>>(s, d, xd, h);
    return cudaGetLastError();
}

cudaError_t launch_down(const Shapes& s, Dispatch d, const float* h, float* y, int B, cudaStream_t st) {
    const int rows_per_cta = kNWarps * kDownRowsPerWarp;
    const int grid = (s.hidden + rows_per_cta - 1) / rows_per_cta;
    if (s.bits == 4)
        down_kernel<4><<<grid, kThreads, 0, st>>>(s, d, h, y, B);
    else
        down_kernel<8><<<grid, kThreads, 0, st>>>(s, d, h, y, B);
    return cudaGetLastError();
}

cudaError_t launch_renorm(const float* y, float* x_next, int B, int hidden, float eps, cudaStream_t st) {
    renorm_kernel<<<B, kRenormThreads, 0, st>>>(y, x_next, hidden, eps);
    return cudaGetLastError();
}

}  // namespace moe
