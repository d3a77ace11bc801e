// decode_kernels.cu -- per-layer decode kernels for sm_103a: router logits,
// top-k + dispatch, fused dequant gate/up + SwiGLU, dequant down + combine,
// and the between-layer renormalisation.
//
// The router is a warp per expert; the expert GEMVs stream packed codes with
// 128-bit loads and reduce with warp shuffles, the CUDA counterpart of the
// "cooperative SIMD-group GEMV fast path" and the MLX affine int4/int8 group
// quantisation the Swiftlet README lists under "Relation to TurboFieldfare".
#include <cuda_fp16.h>
#include <math.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float2 scale_bias(uint32_t sb) {
    __half2 h = *reinterpret_cast<__half2*>(&sb);
    return __half22float2(h);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ---------------------------------------------------------------------------
// router logits
// ---------------------------------------------------------------------------
// One warp per expert.  The fp32 order is fixed so that the chosen experts are
// reproducible bit for bit: element h accumulates (fma) into lane (h/8) % 32 in
// ascending h, then a butterfly over offsets 16, 8, 4, 2, 1, then + bias.
__global__ void router_kernel(const uint16_t* __restrict__ w_r, const float* __restrict__ bias,
                              const float* __restrict__ x, int B, int H, int E, float* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + warp;
    if (e >= E) return;
    const uint4* wrow = reinterpret_cast<const uint4*>(w_r + (size_t)e * H);
    const int nchunk = H / 8;
    const float be = bias ? bias[e] : 0.0f;
    for (int t0 = 0; t0 < B; t0 += 8) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int c = lane; c < nchunk; c += 32) {
            const uint4 wv = __ldg(wrow + c);
            float wf[8] = {bf16lo(wv.x), bf16hi(wv.x), bf16lo(wv.y), bf16hi(wv.y),
                           bf16lo(wv.z), bf16hi(wv.z), bf16lo(wv.w), bf16hi(wv.w)};
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                if (t0 + tt < B) {
                    const float4* xp = reinterpret_cast<const float4*>(x + (size_t)(t0 + tt) * H + c * 8);
                    const float4 xa = __ldg(xp), xb = __ldg(xp + 1);
                    float a = acc[tt];
                    a = __fmaf_rn(wf[0], xa.x, a);
                    a = __fmaf_rn(wf[1], xa.y, a);
                    a = __fmaf_rn(wf[2], xa.z, a);
                    a = __fmaf_rn(wf[3], xa.w, a);
                    a = __fmaf_rn(wf[4], xb.x, a);
                    a = __fmaf_rn(wf[5], xb.y, a);
                    a = __fmaf_rn(wf[6], xb.z, a);
                    a = __fmaf_rn(wf[7], xb.w, a);
                    acc[tt] = a;
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
            if (t0 + tt < B) {
                float v = acc[tt];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, off));
                if (lane == 0) logits[(size_t)(t0 + tt) * E + e] = __fadd_rn(v, be);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// top-k, routing weights, shared gate, and the dispatch lists
// ---------------------------------------------------------------------------
constexpr int kMaxE = 1024, kMaxK = 16, kMaxB = 64;

// inclusive block scan of one int per thread (blockDim.x == 1024)
__device__ int block_scan_incl(int v, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(FULL, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(FULL, s, off);
            if (lane >= off) s += o;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    return v;
}

__global__ void __launch_bounds__(1024) route_dispatch_kernel(
    Shapes s, int mode, const float* __restrict__ logits, const float* __restrict__ x,
    const uint16_t* __restrict__ wsg, int B, int32_t* idx, float* w, float* sigma, int32_t* uidx, float* uw,
    const uint8_t* const* __restrict__ dir, const uint8_t* shared_blob, Dispatch d,
    unsigned long long* hit_counter) {
    const int E = s.n_experts, k = s.top_k, H = s.hidden;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __shared__ float s_lv[kMaxB][kMaxK];
    __shared__ int s_cnt[kMaxE];
    __shared__ unsigned long long s_msk[kMaxE];
    __shared__ int s_scan[kMaxE];
    __shared__ int s_wsum[32];
    __shared__ int s_total;

    if (mode & 1) {
        for (int t = warp; t < B; t += nw) {
            const float* lg = logits + (size_t)t * E;
            unsigned taken = 0;
            for (int i = 0; i < k; ++i) {
                float bv = -INFINITY;
                int be = 0x7fffffff;
                for (int m = 0; lane + 32 * m < E; ++m) {
                    if (taken & (1u << m)) continue;
                    const int e = lane + 32 * m;
                    const float v = lg[e];
                    if (v > bv || (v == bv && e < be)) {
                        bv = v;
                        be = e;
                    }
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const float ov = __shfl_xor_sync(FULL, bv, off);
                    const int oe = __shfl_xor_sync(FULL, be, off);
                    if (ov > bv || (ov == bv && oe < be)) {
                        bv = ov;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                if (lane == 0) {
                    s_lv[t][i] = bv;
                    idx[t * k + i] = be;
                    if (uidx) uidx[t * k + i] = be;
                }
            }
            __syncwarp();
            const float m = s_lv[t][0];
            float den = 0.0f;
            if (s.norm_topk) {
                for (int i = 0; i < k; ++i) den += expf(s_lv[t][i] - m);
            } else {
                for (int e = lane; e < E; e += 32) den += expf(lg[e] - m);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(FULL, den, off);
            }
            if (lane < k) {
                const float wi = expf(s_lv[t][lane] - m) / den;
                w[t * k + lane] = wi;
                if (uw) uw[t * k + lane] = wi;
            }
            float g = 0.0f;
            if (wsg) {
                for (int h = lane; h < H; h += 32) g = fmaf(__uint_as_float((uint32_t)wsg[h] << 16), x[(size_t)t * H + h], g);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) g += __shfl_xor_sync(FULL, g, off);
            }
            if (lane == 0) sigma[t] = wsg ? 1.0f / (1.0f + expf(-g)) : 0.0f;
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
        const bool has_shared = shared_blob != nullptr;
        if (has_shared) {
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
// expert GEMVs (v1: plain fp32 dequant-FMA)
// ---------------------------------------------------------------------------
constexpr int kGateupRowsPerCta = 32, kThreads = 256, kNWarps = kThreads / 32;

template <int BITS>
__device__ __forceinline__ float dot_chunk(uint4 v, float2 sb, const float* __restrict__ xv) {
    constexpr int PER = 32 / BITS;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float q = (float)((wd[i] >> (e * BITS)) & MASK);
            acc = fmaf(fmaf(sb.x, q, sb.y), xv[i * PER + e], acc);
        }
    }
    return acc;
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) gateup_kernel(Shapes s, Dispatch d, const float* __restrict__ x,
                                                          float* __restrict__ h) {
    const int a = blockIdx.y;
    if (a >= *d.n_act) return;
    const bool shared = d.act_expert[a] < 0;
    const int rows = shared ? s.shared_inter : s.inter;
    const int r0 = blockIdx.x * kGateupRowsPerCta;
    if (r0 >= rows) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden;
    const uint8_t* blob = d.act_blob[a];
    const BlobLayout L = blob_layout(H, rows, BITS);
    const int row_bytes = H * BITS / 8, nchunk = row_bytes / 16, chunk_cols = 128 / BITS, ng = H / 64;
    const int p0 = d.act_off[a], p1 = d.act_off[a + 1];
    const int r1 = min(r0 + kGateupRowsPerCta, rows);
    for (int r = r0 + warp; r < r1; r += kNWarps) {
        const uint4* gq = reinterpret_cast<const uint4*>(blob + L.gate_q + (size_t)r * row_bytes);
        const uint4* uq = reinterpret_cast<const uint4*>(blob + L.up_q + (size_t)r * row_bytes);
        const uint32_t* gsb = reinterpret_cast<const uint32_t*>(blob + L.gate_sb) + (size_t)r * ng;
        const uint32_t* usb = reinterpret_cast<const uint32_t*>(blob + L.up_sb) + (size_t)r * ng;
        for (int p = p0; p < p1; ++p) {
            const float* xt = x + (size_t)d.pair_token[p] * H;
            float ag = 0.0f, au = 0.0f;
            for (int c = lane; c < nchunk; c += 32) {
                const int col0 = c * chunk_cols, g = col0 / 64;
                ag += dot_chunk<BITS>(__ldg(gq + c), scale_bias(__ldg(gsb + g)), xt + col0);
                au += dot_chunk<BITS>(__ldg(uq + c), scale_bias(__ldg(usb + g)), xt + col0);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                ag += __shfl_xor_sync(FULL, ag, off);
                au += __shfl_xor_sync(FULL, au, off);
            }
            if (lane == 0) h[(size_t)p * s.h_stride + r] = silu(ag) * au;
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) down_kernel(Shapes s, Dispatch d, const float* __restrict__ h,
                                                        float* __restrict__ y, int B) {
    __shared__ float yacc[kNWarps][kMaxB];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = s.hidden;
    const int n_act = *d.n_act;
    for (int j = blockIdx.x * kNWarps + warp; j < H; j += gridDim.x * kNWarps) {
        for (int t = lane; t < B; t += 32) yacc[warp][t] = 0.0f;
        __syncwarp();
        for (int a = 0; a < n_act; ++a) {
            const bool shared = d.act_expert[a] < 0;
            const int cols = shared ? s.shared_inter : s.inter;
            const BlobLayout L = blob_layout(H, cols, BITS);
            const uint8_t* blob = d.act_blob[a];
            const int row_bytes = cols * BITS / 8, nchunk = row_bytes / 16, chunk_cols = 128 / BITS, ng = cols / 64;
            const uint4* dq = reinterpret_cast<const uint4*>(blob + L.down_q + (size_t)j * row_bytes);
            const uint32_t* dsb = reinterpret_cast<const uint32_t*>(blob + L.down_sb) + (size_t)j * ng;
            for (int p = d.act_off[a]; p < d.act_off[a + 1]; ++p) {
                const float* hp = h + (size_t)p * s.h_stride;
                float acc = 0.0f;
                for (int c = lane; c < nchunk; c += 32) {
                    const int col0 = c * chunk_cols, g = col0 / 64;
                    acc += dot_chunk<BITS>(__ldg(dq + c), scale_bias(__ldg(dsb + g)), hp + col0);
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(FULL, acc, off);
                if (lane == 0) yacc[warp][d.pair_token[p]] += d.pair_w[p] * acc;
                __syncwarp();
            }
        }
        for (int t = lane; t < B; t += 32) y[(size_t)t * H + j] = yacc[warp][t];
        __syncwarp();
    }
}

__global__ void renorm_kernel(const float* __restrict__ y, float* __restrict__ xn, int H, float eps) {
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float* yt = y + (size_t)t * H;
    float ss = 0.0f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) ss = fmaf(yt[j], yt[j], ss);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(FULL, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(FULL, v, off);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / (float)H + eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x) xn[(size_t)t * H + j] = yt[j] * r;
}

}  // namespace

cudaError_t launch_router(const Shapes& s, const uint16_t* w_r, const float* bias, const float* x, int B,
                          float* logits, cudaStream_t st) {
    const int wpb = 8;
    router_kernel<<<(s.n_experts + wpb - 1) / wpb, wpb * 32, 0, st>>>(w_r, bias, x, B, s.hidden, s.n_experts,
                                                                    logits);
    return cudaGetLastError();
}

cudaError_t launch_route_dispatch(const Shapes& s, int mode, const float* logits, const float* x,
                                  const uint16_t* shared_gate_w, int B, int32_t* idx, float* w, float* sigma,
                                  int32_t* user_idx, float* user_w, const uint8_t* const* dir_layer,
                                  const uint8_t* shared_blob, Dispatch d, unsigned long long* hit_counter,
                                  cudaStream_t st) {
    route_dispatch_kernel<<<1, 1024, 0, st>>>(s, mode, logits, x, shared_gate_w, B, idx, w, sigma, user_idx,
                                              user_w, dir_layer, shared_blob, d, hit_counter);
    return cudaGetLastError();
}

cudaError_t launch_gateup(const Shapes& s, Dispatch d, const float* x, float* h, int B, cudaStream_t st) {
    (void)B;
    const int rows = s.inter > s.shared_inter ? s.inter : s.shared_inter;
    dim3 grid((rows + kGateupRowsPerCta - 1) / kGateupRowsPerCta, s.max_act);
    if (s.bits == 4)
        gateup_kernel<4><<<grid, kThreads, 0, st>>>(s, d, x, h);
    else
        gateup_kernel<8><<<grid, kThreads, 0, st>>>(s, d, x, h);
    return cudaGetLastError();
}

cudaError_t launch_down(const Shapes& s, Dispatch d, const float* h, float* y, int B, cudaStream_t st) {
    const int grid = (s.hidden + kNWarps - 1) / kNWarps;
    if (s.bits == 4)
        down_kernel<4><<<grid, kThreads, 0, st>>>(s, d, h, y, B);
    else
        down_kernel<8><<<grid, kThreads, 0, st>>>(s, d, h, y, B);
    return cudaGetLastError();
}

cudaError_t launch_renorm(const float* y, float* x_next, int B, int hidden, float eps, cudaStream_t st) {
    renorm_kernel<<<B, 256, 0, st>>>(y, x_next, hidden, eps);
    return cudaGetLastError();
}

}  // namespace moe
