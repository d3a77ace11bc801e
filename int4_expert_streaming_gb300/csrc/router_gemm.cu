// router_gemm.cu -- the prefill router in two stages, with results identical
// to the exact fixed-order fp32 router.
//
//   1. split_kernel     x = hi + mid + lo, three bf16 pieces per element (the
//                       remainder is below 2^-26 |x|), as one [T][3H] bf16 array
//                       whose first H columns are bf16(x) itself; ||x_t||_2,
//                       ||W_e||_2 (upper bounds); y := 0
//   2. router_gemm      A_te = sum_h W_eh (hi + mid + lo)_th on the tensor cores
//                       (tcgen05, bf16 operands, fp32 accumulators in tensor memory)
//   3. refine_kernel    per token: every expert's logit lies within
//                       delta_e = 2^-8 ||W_e|| ||x_t|| (+ rounding slack) of
//                       A_te + bias_e; experts whose upper bound is below the
//                       k-th largest lower bound cannot be chosen; the others
//                       get their exact logit (the fixed fp32 order) and the
//                       top-k, routing weights and shared gate are taken on
//                       those exact values.
// The bound: bf16 x bf16 products are exact in fp32; an fp32 accumulation of
// 3H terms has error below 3H * 2^-23 * sum|W x| (< 2^-10.4 sum|W x| for
// H <= 2048), the split remainder adds < 2^-26 and the fixed-order fp32 dot
// itself < 2^-17 of sum|W x|, and sum|W x| <= ||W_e|| ||x_t|| (Cauchy-Schwarz);
// delta uses 2^-8, twice that, so even an accumulation that truncates every
// addition stays inside it.  The refine step also checks, for every candidate,
// that its exact logit lies within delta of the approximation, and reports a
// violation through the status word.
#include <cuda_bf16.h>

#include "gemv.cuh"
#include "prefill.h"
#include "umma.cuh"

namespace moe {
namespace {

using namespace umma;

__device__ __forceinline__ uint16_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------------------
// 1. split and norms
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) split_kernel(const float* __restrict__ x, int T, int H,
                                                    uint16_t* __restrict__ x3, float* __restrict__ xnorm,
                                                    float* __restrict__ y) {
    __shared__ float red[8];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* xt = x + (size_t)t * H;
    uint16_t* o = x3 + (size_t)t * 3 * H;
    float ss = 0.0f;
    for (int h = tid; h < H; h += 256) {
        const float v = xt[h];
        const uint16_t a = bf16_bits(v);
        const float r1 = __fsub_rn(v, bf16_val(a));
        const uint16_t b = bf16_bits(r1);
        const float r2 = __fsub_rn(r1, bf16_val(b));
        o[h] = a;
        o[H + h] = b;
        o[2 * H + h] = bf16_bits(r2);
        ss = __fmaf_rn(v, v, ss);
        y[(size_t)t * H + h] = 0.0f;
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float s = 0.0f;
        for (int w = 0; w < 8; ++w) s = __fadd_rn(s, red[w]);
        xnorm[t] = __fmul_rn(sqrtf(s), 1.0001f);  // an upper bound of ||x_t||_2
    }
}

__global__ void __launch_bounds__(256) wnorm_kernel(const uint16_t* __restrict__ w_r, int E, int H,
                                                    float* __restrict__ wnorm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    float ss = 0.0f;
    for (int h = lane; h < H; h += 32) {
        const float v = bf16_val(w_r[(size_t)e * H + h]);
        ss = __fmaf_rn(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) wnorm[e] = __fmul_rn(sqrtf(ss), 1.0001f);
}

// ---------------------------------------------------------------------------
// 2. approximate logits: one CTA per (128 experts, 128 tokens), K = 3H in
// 64-wide k-blocks (the A rows repeat W_r for each of the three pieces), a ring
// of kRS stages filled by cp.async from all 128 threads, one thread issuing
// the MMAs; D[e][t] in tensor memory, read back lane = expert.
// ---------------------------------------------------------------------------
constexpr int kRT = 128, kRS = 4;
constexpr int kRTile = 128 * 64 * 2;  // bytes of one 128 x 64 bf16 operand tile

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kRT, 1) router_gemm_kernel(const uint16_t* __restrict__ w_r,
                                                             const uint16_t* __restrict__ x3, int T, int H, int E,
                                                             float* __restrict__ approx, int* status,
                                                             unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t mma_bar[kRS], drain_bar;
    __shared__ uint32_t tmem_s;
    __shared__ volatile int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int e0 = blockIdx.x * 128, t0 = blockIdx.y * 128;
    const int KB = 3 * H / 64, HB = H / 64;
    if (tid == 0) {
        for (int s = 0; s < kRS; ++s) bar_init(&mma_bar[s], 1);
        bar_init(&drain_bar, 1);
        abort_s = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_s, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_s;
    // each thread copies rows (tid) of A and B of a k-block: 8 chunks of 16 bytes each
    auto load = [&](int kb) {
        const uint32_t st = smem0 + (kb % kRS) * 2 * kRTile;
        const int e = min(e0 + tid, E - 1), t = min(t0 + tid, T - 1);
        const uint16_t* a = w_r + (size_t)e * H + (kb % HB) * 64;
        const uint16_t* b = x3 + (size_t)t * 3 * H + kb * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            cp_async16(st + swz_chunk(tid, c), a + 8 * c);
            cp_async16(st + kRTile + swz_chunk(tid, c), b + 8 * c);
        }
    };
    for (int kb = 0; kb < kRS - 1; ++kb) {
        if (kb < KB) load(kb);
        cp_async_commit();
    }
    const uint32_t idesc = idesc_bf16(128, 128);
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
        cp_async_wait<kRS - 2>();  // this thread's copies of k-block kb have landed
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
            const uint32_t st = smem0 + (kb % kRS) * 2 * kRTile;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem, sdesc(st + kk * 32), sdesc(st + kRTile + kk * 32), idesc, (kb | kk) ? 1u : 0u);
            mma_commit(&mma_bar[kb % kRS]);
        }
        // the stage refilled next was read by the MMAs of k-block kb - 1
        const int nk = kb + kRS - 1;
        if (nk < KB && kb >= 1) {
            if (!bar_wait(&mma_bar[(kb - 1) % kRS], ((kb - 1) / kRS) & 1u, timeout_ns, &abort_s)) {
                *(volatile int*)status = 4;
                abort_s = 1;
                ok = false;
            }
        }
        if (ok && nk < KB) load(nk);
        cp_async_commit();
        if (__syncthreads_or(!ok)) ok = false;
    }
    cp_async_wait<0>();
    if (tid == 0) mma_commit(&drain_bar);
    if (!bar_wait(&drain_bar, 0, timeout_ns, &abort_s)) {
        *(volatile int*)status = 4;
        ok = false;
    }
    fence_after_sync();
    if (__syncthreads_and(ok ? 1 : 0)) {
        // lane = expert e0 + 32 warp + lane, columns = tokens
        const int e = e0 + 32 * warp + lane;
        for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int t = t0 + c0 + j;
                if (t < T && e < E) approx[(size_t)t * E + e] = __uint_as_float(v[j]);
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// 3. per token (one warp): candidates from the bound, exact logits for them,
// top-k / weights / shared gate on the exact values
// ---------------------------------------------------------------------------
constexpr int kMaxM = 32;  // E <= 1024: up to 32 experts per lane

__global__ void __launch_bounds__(256) refine_kernel(const float* __restrict__ approx, const float* __restrict__ xnorm,
                                                     const float* __restrict__ wnorm, const uint16_t* __restrict__ w_r,
                                                     const float* __restrict__ bias, const float* __restrict__ x,
                                                     const uint16_t* __restrict__ w_sg, int T, int H, int E, int k,
                                                     int32_t* __restrict__ idx, float* __restrict__ w,
                                                     float* __restrict__ sigma, int32_t* __restrict__ user_idx,
                                                     float* __restrict__ user_w, int* status) {
    __shared__ float s_lg[8][1024];  // exact logits of the candidates (-inf elsewhere)
    __shared__ int32_t s_idx[8][16];
    __shared__ float s_val[8][16], s_w[8][16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    const float* at = approx + (size_t)t * E;
    const float* xt = x + (size_t)t * H;
    const float nx = xnorm[t];
    const int M = (E + 31) / 32;
    // lower bounds as order keys; the k-th largest by rounds of warp max
    uint32_t lk[kMaxM];
#pragma unroll
    for (int m = 0; m < kMaxM; ++m) {
        const int e = lane + 32 * m;
        lk[m] = 0u;
        if (m < M && e < E) {
            const float ap = __fadd_rn(at[e], bias ? bias[e] : 0.0f);
            const float d = __fmaf_rn(0.00390625f * wnorm[e], nx, 2.4e-7f * fabsf(ap));  // 2^-8 ||W|| ||x|| + slack
            lk[m] = order_key(__fsub_rn(ap, d));
        }
    }
    uint32_t kth = 0u;
    {
        uint32_t taken = 0u;
        for (int r = 0; r < k; ++r) {
            uint32_t best = 0u;
            int bm = -1;
#pragma unroll
            for (int m = 0; m < kMaxM; ++m)
                if (!(taken & (1u << m)) && lk[m] > best) best = lk[m], bm = m;
            const uint32_t mx = __reduce_max_sync(kFullMask, best);
            const uint32_t win = __reduce_min_sync(kFullMask, (best == mx && bm >= 0) ? (uint32_t)(lane + 32 * bm)
                                                                                     : 0xffffffffu);
            if ((int)(win & 31u) == lane && bm >= 0) taken |= 1u << bm;
            kth = mx;
        }
    }
    // candidates: upper bound >= the k-th largest lower bound; exact logit for each
    float* lg = s_lg[warp];
    for (int e = lane; e < E; e += 32) lg[e] = -INFINITY;
    __syncwarp();
#pragma unroll 1
    for (int m = 0; m < M; ++m) {
        const int e = lane + 32 * m;
        bool cand = false;
        float ap = 0.0f, d = 0.0f;
        if (e < E) {
            ap = __fadd_rn(at[e], bias ? bias[e] : 0.0f);
            d = __fmaf_rn(0.00390625f * wnorm[e], nx, 2.4e-7f * fabsf(ap));
            cand = order_key(__fadd_rn(ap, d)) >= kth;
        }
        unsigned ball = __ballot_sync(kFullMask, cand);
        while (ball) {
            const int src = __ffs(ball) - 1;
            ball &= ball - 1;
            const int ec = src + 32 * m;
            const float v = router_logit(w_r + (size_t)ec * H, xt, H, bias ? bias[ec] : 0.0f, lane);
            if (lane == src) {
                lg[ec] = v;
                if (!(fabsf(v - ap) <= d)) atomicOr(status, 8);  // the bound failed: report
            }
        }
    }
    __syncwarp();
    // the exact top-k among the candidates (non-candidates hold -inf: never chosen
    // ahead of a real logit, and at least k candidates exist)
    warp_topk(lg, E, k, 1, lane, s_idx[warp], s_val[warp], s_w[warp]);
    if (lane < k) {
        idx[(size_t)t * k + lane] = s_idx[warp][lane];
        w[(size_t)t * k + lane] = s_w[warp][lane];
        if (user_idx) user_idx[(size_t)t * k + lane] = s_idx[warp][lane];
        if (user_w) user_w[(size_t)t * k + lane] = s_w[warp][lane];
    }
    if (w_sg) {
        const float sg = shared_gate(w_sg, xt, H, lane);
        if (lane == 0) sigma[t] = sg;
    }
}

}  // namespace

bool router_two_stage_ok(const Shapes& s) { return s.norm_topk && s.n_experts % 128 == 0 && s.hidden <= 2048; }

size_t router_two_stage_scratch(int max_tokens, const Shapes& s) {
    // approx [T][E] fp32, x3 [T][3H] bf16, xnorm [T], wnorm [E]
    return (size_t)max_tokens * s.n_experts * 4 + (size_t)max_tokens * 3 * s.hidden * 2 + (size_t)max_tokens * 4 +
           (size_t)s.n_experts * 4 + 4 * 256;
}

cudaError_t launch_router_two_stage(const Shapes& s, const PrefillScratch& p, const PrefillArgs& a, cudaStream_t st,
                                    int* launches) {
    const int T = a.T, H = s.hidden, E = s.n_experts, k = s.top_k;
    split_kernel<<<T, 256, 0, st>>>(a.x, T, H, p.x3, p.xnorm, a.y);
    wnorm_kernel<<<(E + 7) / 8, 256, 0, st>>>(a.router_w, E, H, p.wnorm);
    const size_t smem = (size_t)kRS * 2 * kRTile + 1024;
    cudaError_t e = smem_limit(reinterpret_cast<const void*>(router_gemm_kernel), (int)smem);
    if (e != cudaSuccess) return e;
    router_gemm_kernel<<<dim3(E / 128, (T + 127) / 128), kRT, smem, st>>>(a.router_w, p.x3, T, H, E, p.logits,
                                                                         p.status_dev, a.timeout_ns);
    refine_kernel<<<(T + 7) / 8, 256, 0, st>>>(p.logits, p.xnorm, p.wnorm, a.router_w, a.router_bias, a.x,
                                               a.shared_blob ? a.shared_gate : nullptr, T, H, E, k, p.idx, p.w,
                                               p.sigma, a.user_idx, a.user_w, p.status_dev);
    *launches += 4;
    return cudaGetLastError();
}

}  // namespace moe
