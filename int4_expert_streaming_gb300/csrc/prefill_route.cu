// prefill_route.cu -- routing and dispatch of a prefill call, and the host
// side of the prefill path.
//
//   1. logits_kernel   router logits of every (token, expert) in the fixed fp32
//                      order of the decode path (bit-identical logits)
//   2. select_kernel   per token: top-k, routing weights, the sigmoid shared
//                      gate, bf16 copy of x for the tensor cores, y := 0
//   3. hist_kernel     pairs (token, slot) counted per (expert, block of 1024
//                      pairs) and ranked inside their block (warp match)
//   4. scan_kernel     block counts -> first sorted position of every
//                      (expert, block); expert offsets; the chunk lists that
//                      drive the two grouped GEMMs
//   5. scatter_kernel  pair id, token and routing weight of every sorted
//                      position (stable: pairs of one expert keep ascending
//                      pair order)
//   6. gather_kernel   bf16 token rows in sorted pair order
//   7. grouped GEMM gate/up, 8. grouped GEMM down (prefill_gemm.cu)
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>

#include "gemv.cuh"
#include "prefill.h"

namespace moe {

cudaError_t launch_prefill_gemm(int mode, const Shapes& s, const PrefillScratch& p, const PrefillArgs& a,
                                cudaStream_t st);

namespace {

constexpr int kLgThreads = 256;   // 8 warps
constexpr int kLgExpertsPerWarp = 2;
constexpr int kLgExperts = 8 * kLgExpertsPerWarp;  // experts per CTA
constexpr int kLgTokens = 64;     // tokens per CTA
constexpr int kLgStageTok = 2;    // tokens per shared-memory stage
constexpr int kLgStages = 4;
constexpr int kMaxNC = 8;         // hidden / 256 <= 8
constexpr int kHistThreads = 1024;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// 1. logits.  Lane j of a warp owns the columns h with (h / 8) % 32 == j (the
// decode router's lane assignment), holds its slice of 4 router rows in
// registers, and accumulates every token against them in ascending h; the
// warp butterfly then sums the 32 partials.  Tokens are staged in shared
// memory in "lane-major" order: float4 (c, half, j) holds x[256c + 8j + 4half
// .. +4), so each lane's loads are contiguous across the warp.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLgThreads, 1) logits_kernel(const uint16_t* __restrict__ w_r,
                                                               const float* __restrict__ bias,
                                                               const float* __restrict__ x, int T, int H, int E,
                                                               int tok_tile, float* __restrict__ logits) {
    extern __shared__ __align__(16) float4 xs[];  // [kLgStages][kLgStageTok][H / 4]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nc = H / 256, q4 = H / 4;
    const int e0 = blockIdx.x * kLgExperts + warp * kLgExpertsPerWarp;
    const int t0 = blockIdx.y * tok_tile, tn = min(tok_tile, T - t0);
    const int nstage = (tn + kLgStageTok - 1) / kLgStageTok;

    auto load_stage = [&](int st) {
        if (st < nstage) {
            float4* dst = xs + (size_t)(st % kLgStages) * kLgStageTok * q4;
            for (int u = threadIdx.x; u < kLgStageTok * q4; u += kLgThreads) {
                const int tt = u / q4, v = u % q4;  // v: 16-byte unit of the row
                const int t = t0 + st * kLgStageTok + tt;
                if (t < T) {
                    const int c = v / 64, j = (v / 2) % 32, half = v % 2;
                    cp_async16((uint32_t)__cvta_generic_to_shared(dst + (size_t)tt * q4 + (c * 2 + half) * 32 + j),
                               x + (size_t)t * H + 4 * v);
                }
            }
        }
        cp_async_commit();
    };
    for (int st = 0; st < kLgStages - 1; ++st) load_stage(st);

    uint4 wr[kLgExpertsPerWarp][kMaxNC];
    float be[kLgExpertsPerWarp];
#pragma unroll
    for (int i = 0; i < kLgExpertsPerWarp; ++i) {
        const int e = min(e0 + i, E - 1);
        be[i] = bias ? bias[e] : 0.0f;
#pragma unroll
        for (int c = 0; c < kMaxNC; ++c)
            if (c < nc) wr[i][c] = *reinterpret_cast<const uint4*>(w_r + (size_t)e * H + 256 * c + 8 * lane);
    }

    for (int st = 0; st < nstage; ++st) {
        load_stage(st + kLgStages - 1);
        cp_async_wait<kLgStages - 1>();
        __syncthreads();
        const float4* xb = xs + (size_t)(st % kLgStages) * kLgStageTok * q4;
        float acc[kLgStageTok][kLgExpertsPerWarp];
#pragma unroll
        for (int tt = 0; tt < kLgStageTok; ++tt)
#pragma unroll
            for (int i = 0; i < kLgExpertsPerWarp; ++i) acc[tt][i] = 0.0f;
#pragma unroll
        for (int c = 0; c < kMaxNC; ++c) {
            if (c < nc) {
#pragma unroll
                for (int tt = 0; tt < kLgStageTok; ++tt) {
                    const float4 xa = xb[(size_t)tt * q4 + (c * 2 + 0) * 32 + lane];
                    const float4 xc = xb[(size_t)tt * q4 + (c * 2 + 1) * 32 + lane];
#pragma unroll
                    for (int i = 0; i < kLgExpertsPerWarp; ++i) {
                        const uint4 v = wr[i][c];
                        float a = acc[tt][i];
                        a = __fmaf_rn(bf16_lo(v.x), xa.x, a);
                        a = __fmaf_rn(bf16_hi(v.x), xa.y, a);
                        a = __fmaf_rn(bf16_lo(v.y), xa.z, a);
                        a = __fmaf_rn(bf16_hi(v.y), xa.w, a);
                        a = __fmaf_rn(bf16_lo(v.z), xc.x, a);
                        a = __fmaf_rn(bf16_hi(v.z), xc.y, a);
                        a = __fmaf_rn(bf16_lo(v.w), xc.z, a);
                        a = __fmaf_rn(bf16_hi(v.w), xc.w, a);
                        acc[tt][i] = a;
                    }
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < kLgStageTok; ++tt) {
            const int t = t0 + st * kLgStageTok + tt;
#pragma unroll
            for (int i = 0; i < kLgExpertsPerWarp; ++i) {
                const float v = __fadd_rn(warp_sum(acc[tt][i]), be[i]);
                if (lane == i && t < T && e0 + i < E) logits[(size_t)t * E + e0 + i] = v;
            }
        }
        __syncthreads();  // the stage is refilled by the next iteration's load
    }
}

// ---------------------------------------------------------------------------
// 2. per token: top-k, weights, shared gate, bf16(x), y := 0.  One warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) select_kernel(const float* __restrict__ logits, const float* __restrict__ x,
                                                     const uint16_t* __restrict__ w_sg, int T, int H, int E, int k,
                                                     int norm_topk, int32_t* __restrict__ idx, float* __restrict__ w,
                                                     float* __restrict__ sigma, int32_t* __restrict__ user_idx,
                                                     float* __restrict__ user_w, uint16_t* __restrict__ x_bf,
                                                     float* __restrict__ y) {
    __shared__ int32_t s_idx[8][16];
    __shared__ float s_val[8][16], s_w[8][16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    const float* lg = logits + (size_t)t * E;
    const float* xt = x + (size_t)t * H;
    warp_topk(lg, E, k, norm_topk, lane, s_idx[warp], s_val[warp], s_w[warp]);
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
    uint2* xo = reinterpret_cast<uint2*>(x_bf + (size_t)t * H);
    float4* yo = reinterpret_cast<float4*>(y + (size_t)t * H);
    for (int v = lane; v < H / 4; v += 32) {
        const float4 a = reinterpret_cast<const float4*>(xt)[v];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
        xo[v] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
        yo[v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
}

// ---------------------------------------------------------------------------
// 3. histogram of one block of 1024 pairs and each pair's rank among the
// block's pairs of the same expert (pairs in ascending id).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kHistThreads) hist_kernel(const int32_t* __restrict__ idx, int P, int E, int n_hist,
                                                            int32_t* __restrict__ local_rank,
                                                            int32_t* __restrict__ cnt) {
    extern __shared__ uint16_t cw[];  // [32 warps][E] pairs per warp, then their exclusive prefix over warps
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += kHistThreads) cw[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * kHistThreads + tid;
    const bool live = p < P;
    const int e = live ? idx[p] : -1;
    const unsigned act = __ballot_sync(kFullMask, live);
    int rank = 0;
    if (live) {
        const unsigned peers = __match_any_sync(act, e);
        rank = __popc(peers & ((1u << lane) - 1u));
        if (rank == 0) cw[warp * E + e] = (uint16_t)__popc(peers);
    }
    __syncthreads();
    // exclusive prefix over warps, per expert; block totals to cnt[e][block]
    for (int ex = tid; ex < E; ex += kHistThreads) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int v = cw[w * E + ex];
            cw[w * E + ex] = (uint16_t)run;
            run += v;
        }
        cnt[(size_t)ex * n_hist + blockIdx.x] = run;
    }
    __syncthreads();
    if (live) local_rank[p] = rank + cw[warp * E + e];
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFullMask, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// exclusive scan of v over the block (1024 threads); *total = sum
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int s = warp_incl_scan(ws[lane], lane);
        ws[lane] = s;
    }
    __syncthreads();
    const int r = incl - v + (warp ? ws[warp - 1] : 0);
    *total = ws[31];
    __syncthreads();
    return r;
}

// Stable rank of this thread's partial chunk among all partial chunks, by size
// r descending then owner (thread) ascending, sizes 1..nb-1 (0 = no partial
// chunk): a counting sort on r.  Every thread of the block calls it.  Shared
// scratch: wcnt[32 * nb], start[nb]; returns the rank (meaningful for r > 0)
// and the number of partial chunks in *n_part.
__device__ int partial_rank(int r, int nb, int* wcnt, int* start, int* ws, int* n_part) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 32 * nb; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const unsigned same = __match_any_sync(kFullMask, r);
    if (r > 0 && lane == __ffs(same) - 1) wcnt[warp * nb + r] = __popc(same);
    __syncthreads();
    // thread i < nb owns size nb-1-i: prefix of that size over the warps, then
    // a scan over the sizes in descending order gives each size's first rank
    const int sz = nb - 1 - tid;
    int tot_sz = 0;
    if (tid < nb && sz > 0)
        for (int w = 0; w < 32; ++w) {
            const int v = wcnt[w * nb + sz];
            wcnt[w * nb + sz] = tot_sz;
            tot_sz += v;
        }
    const int first = block_excl_scan(tot_sz, ws, n_part);
    if (tid < nb) start[sz] = first;
    __syncthreads();
    const unsigned below = same & ((1u << lane) - 1u);
    return r > 0 ? start[r] + wcnt[warp * nb + r] + __popc(below) : 0;
}

__device__ __forceinline__ void put_chunk(ChunkRec* list, int i, int e, int row0, int n, int hrow0,
                                          const uint8_t* blob) {
    ChunkRec c;
    c.e = e;
    c.row0 = row0;
    c.n = n;
    c.hrow0 = hrow0;
    c.blob = blob;
    c.pad[0] = c.pad[1] = 0;
    list[i] = c;
}

// full chunks of every owner in owner order, then the partial chunks by size
// descending (ties: lower owner first), so a static round-robin over the CTAs
// hands out the longest tiles first
template <int CL>
__device__ void chunk_list(int NE, const int* tot, const int* off, int hoff, const uint8_t* blob, int* wcnt,
                           int* start, int* ws, ChunkRec* list, int32_t* n_list) {
    const int tid = threadIdx.x;
    const int t = tid < NE ? tot[tid] : 0;
    const int nf = t / CL;
    int n_full = 0, n_part = 0;
    const int fpos = block_excl_scan(nf, ws, &n_full);
    for (int i = 0; i < nf; ++i) put_chunk(list, fpos + i, tid, off[tid] + i * CL, CL, hoff + i * CL, blob);
    const int r = t % CL;
    const int rank = partial_rank(r, CL, wcnt, start, ws, &n_part);
    if (r > 0) put_chunk(list, n_full + rank, tid, off[tid] + nf * CL, r, hoff + nf * CL, blob);
    if (tid == 0) *n_list = n_full + n_part;
}

// ---------------------------------------------------------------------------
// 4. scan: per-(expert, block) first positions, expert offsets, the two chunk
// lists (kChunk rows for gate/up, kChunk1 rows for down).  The shared expert
// (owner E) covers tokens 0..T-1 in order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ cnt, int E, int n_hist, int T,
                                                    const uint8_t* const* __restrict__ dir,
                                                    const uint8_t* __restrict__ shared_blob,
                                                    int32_t* __restrict__ offsets, ChunkRec* __restrict__ chunks,
                                                    ChunkRec* __restrict__ chunks1, int32_t* __restrict__ n_chunks) {
    __shared__ int tot[1025], off[1025];
    __shared__ int wcnt[32 * kChunk], start[kChunk];
    __shared__ int ws[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // block counts -> first positions within each expert: a warp takes 8 of its
    // experts at a time, 32 blocks per step, loads issued before the scans
    for (int e8 = warp * 8; e8 < E; e8 += 32 * 8) {
        int carry[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) carry[q] = 0;
        for (int cb = 0; cb < n_hist; cb += 32) {
            const int i = cb + lane;
            int v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = (e8 + q < E && i < n_hist) ? cnt[(size_t)(e8 + q) * n_hist + i] : 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int incl = warp_incl_scan(v[q], lane);
                if (e8 + q < E && i < n_hist) cnt[(size_t)(e8 + q) * n_hist + i] = carry[q] + incl - v[q];
                carry[q] += __shfl_sync(kFullMask, incl, 31);
            }
        }
        if (lane < 8 && e8 + lane < E) {
            int cl = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q == lane) cl = carry[q];
            tot[e8 + lane] = cl;
        }
    }
    __syncthreads();
    const int has_shared = shared_blob != nullptr;
    const int NE = E + has_shared;  // chunk owners
    int total = 0;
    {
        const int v = tid < E ? tot[tid] : 0;
        const int ex = block_excl_scan(v, ws, &total);
        if (tid < E) {
            off[tid] = ex;
            offsets[tid] = ex;
        }
        if (tid == 0) offsets[E] = total;
    }
    if (has_shared && tid == 0) {
        tot[E] = T;
        off[E] = 0;
    }
    __syncthreads();
    for (size_t i = tid; i < (size_t)E * n_hist; i += 1024) cnt[i] += off[i / n_hist];
    // first row of every owner in the SwiGLU buffers (segments padded to 16 rows)
    int h_used = 0;
    const int hoff = block_excl_scan(tid < NE ? (tot[tid] + 15) & ~15 : 0, ws, &h_used);
    const uint8_t* blob = tid < E ? dir[tid] : (tid == E ? shared_blob : nullptr);
    chunk_list<kChunk>(NE, tot, off, hoff, blob, wcnt, start, ws, chunks, n_chunks);
    chunk_list<kChunk1>(NE, tot, off, hoff, blob, wcnt, start, ws, chunks1, n_chunks + 1);
}

// ---------------------------------------------------------------------------
// 5. scatter: the pair at sorted position (first position of its (expert,
// block) + its rank in the block): its id, token and routing weight
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kHistThreads) scatter_kernel(const int32_t* __restrict__ idx,
                                                               const int32_t* __restrict__ local_rank,
                                                               const int32_t* __restrict__ cnt,
                                                               const float* __restrict__ w, int P, int k, int n_hist,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ tok_sorted,
                                                               float* __restrict__ w_sorted) {
    const int p = blockIdx.x * kHistThreads + threadIdx.x;
    if (p >= P) return;
    const int e = idx[p];
    const int pos = cnt[(size_t)e * n_hist + blockIdx.x] + local_rank[p];
    perm[pos] = p;
    tok_sorted[pos] = p / k;
    w_sorted[pos] = w[p];
}

// ---------------------------------------------------------------------------
// 6. gather: the bf16 token row of every sorted position, so that the gate/up
// GEMM loads each chunk's rows as one rectangular TMA box per k-block.  A warp
// copies one row of H/8 16-byte units per step.
// ---------------------------------------------------------------------------
constexpr int kGatherThreads = 512;
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const int32_t* __restrict__ tok_sorted,
                                                                const uint16_t* __restrict__ x, int x_stride, int P,
                                                                int H, uint16_t* __restrict__ xs) {
    const int lane = threadIdx.x & 31;
    const int units = H / 8;  // <= 256
    const int step = gridDim.x * (kGatherThreads / 32);
    for (int row = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); row < P; row += step) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)__ldg(tok_sorted + row) * x_stride);
        uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)row * H);
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (lane + 32 * i < units) v[i] = __ldg(src + lane + 32 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (lane + 32 * i < units) dst[lane + 32 * i] = v[i];
    }
}

template <class T>
cudaError_t dalloc(T** p, size_t n) {
    return cudaMalloc(reinterpret_cast<void**>(p), (n ? n : 1) * sizeof(T));
}

}  // namespace

cudaError_t launch_logits(const uint16_t* w_r, const float* bias, const float* x, int T, int H, int E, int tok_tile,
                          float* logits, cudaStream_t st) {
    const size_t smem = (size_t)kLgStages * kLgStageTok * H * sizeof(float);
    cudaError_t e = smem_limit(reinterpret_cast<const void*>(logits_kernel), (int)smem);
    if (e != cudaSuccess) return e;
    tok_tile = std::max(1, std::min(tok_tile, kLgTokens));
    dim3 grid((E + kLgExperts - 1) / kLgExperts, (T + tok_tile - 1) / tok_tile);
    logits_kernel<<<grid, kLgThreads, smem, st>>>(w_r, bias, x, T, H, E, tok_tile, logits);
    return cudaGetLastError();
}

// TMA maps of the gate/up GEMM's token operand (bf16, boxes of 64 x 64):
// x_map over bf16(x) [max_tokens][hidden] with row stride x_stride (x_bf, or
// the first third of each x3 row), xs_map over x_sorted [max_tokens * k][hidden]
static bool encode_x_maps(PrefillScratch& p, const Shapes& s, int max_tokens, std::string& err) {
    typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        !fn || q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        err = "the driver has no cuTensorMapEncodeTiled";
        return false;
    }
    auto encode = [&](CUtensorMap* m, void* base, size_t cols, size_t rows, size_t stride_elems, uint32_t box_rows,
                      CUtensorMapSwizzle swz) {
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)stride_elems * 2};
        const cuuint32_t box[2] = {64, box_rows}, estr[2] = {1, 1};
        return ((EncodeFn)fn)(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    const size_t x_stride = p.two_stage ? 3 * (size_t)s.hidden : (size_t)s.hidden;
    void* xb = p.two_stage ? (void*)p.x3 : (void*)p.x_bf;
    const size_t P = (size_t)max_tokens * s.top_k;
    const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult r = encode(&p.x_map, xb, s.hidden, max_tokens, x_stride, 64, SW);
    if (r == CUDA_SUCCESS) r = encode(&p.xs_map, p.x_sorted, s.hidden, P, s.hidden, 64, SW);
    if (r != CUDA_SUCCESS) {
        char buf[96];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        err = buf;
        return false;
    }
    return true;
}

std::string prefill_check(const Shapes& s) {
    if (s.hidden % 256 || s.hidden > 256 * kMaxNC) return "prefill needs hidden to be a multiple of 256, at most 2048";
    if (s.inter % 128 || s.shared_inter % 128) return "prefill needs inter and shared_inter to be multiples of 128";
    if (s.n_experts > 1023) return "prefill supports at most 1023 experts";
    return std::string();
}

int prefill_alloc(PrefillScratch& p, const Shapes& s, int max_tokens, int device, std::string& err) {
    const std::string why = prefill_check(s);
    if (!why.empty()) {
        err = why;
        return MOE_EINVAL;
    }
    const size_t T = max_tokens, k = s.top_k, E = s.n_experts, H = s.hidden, P = T * k;
    p.max_tokens = max_tokens;
    p.n_hist = (int)((P + kHistThreads - 1) / kHistThreads);
    p.max_chunks = (int)((P + T) / kChunk + E + 2);
    p.max_chunks1 = (int)((P + T) / kChunk1 + E + 2);
    p.h_rows = (int)((P + T + 16 * (E + 1) + 15) / 16 * 16);
    p.two_stage = router_two_stage_ok(s);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        err = "cudaGetDeviceProperties failed";
        return MOE_ECUDA;
    }
    p.sms = prop.multiProcessorCount;
    if (dalloc(&p.logits, T * E) || dalloc(&p.x_bf, T * H) || dalloc(&p.idx, P) || dalloc(&p.w, P) ||
        dalloc(&p.sigma, T) || dalloc(&p.local_rank, P) || dalloc(&p.cnt, E * p.n_hist) ||
        dalloc(&p.offsets, E + 1) || dalloc(&p.perm, P) || dalloc(&p.tok_sorted, P) || dalloc(&p.x_sorted, P * H) ||
        dalloc(&p.w_sorted, P) || dalloc(&p.chunks, (size_t)p.max_chunks) ||
        dalloc(&p.chunks1, (size_t)p.max_chunks1) || dalloc(&p.n_chunks, 2) || dalloc(&p.h_hi, (size_t)p.h_rows * s.h_stride) ||
        dalloc(&p.h_lo, (size_t)p.h_rows * s.h_stride) ||
        (router_two_stage_ok(s) && (dalloc(&p.x3, T * 3 * H) || dalloc(&p.xnorm, T) || dalloc(&p.wnorm, E)))) {
        cudaGetLastError();
        char buf[160];
        snprintf(buf, sizeof buf, "cudaMalloc of the prefill scratch for %d tokens failed", max_tokens);
        err = buf;
        prefill_free(p);
        return MOE_ENOMEM;
    }
    if (cudaHostAlloc(reinterpret_cast<void**>(&p.status_host), sizeof(int), cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(reinterpret_cast<void**>(&p.status_dev), p.status_host, 0) != cudaSuccess) {
        cudaGetLastError();
        err = "mapped status word allocation failed";
        prefill_free(p);
        return MOE_ENOMEM;
    }
    *p.status_host = 0;
    if (!encode_x_maps(p, s, max_tokens, err)) {
        prefill_free(p);
        return MOE_ECUDA;
    }
    // rows past an expert's last row (up to its 16-row padding) feed MMA columns
    // that are never read back; zero them once so they hold finite values
    if (cudaMemset(p.h_hi, 0, (size_t)p.h_rows * s.h_stride * 2) != cudaSuccess ||
        cudaMemset(p.h_lo, 0, (size_t)p.h_rows * s.h_stride * 2) != cudaSuccess) {
        cudaGetLastError();
        err = "cudaMemset failed";
        prefill_free(p);
        return MOE_ECUDA;
    }
    return MOE_OK;
}

void prefill_free(PrefillScratch& p) {
    cudaFree(p.logits);
    cudaFree(p.x_bf);
    cudaFree(p.idx);
    cudaFree(p.w);
    cudaFree(p.sigma);
    cudaFree(p.local_rank);
    cudaFree(p.cnt);
    cudaFree(p.offsets);
    cudaFree(p.perm);
    cudaFree(p.tok_sorted);
    cudaFree(p.x_sorted);
    cudaFree(p.w_sorted);
    cudaFree(p.chunks);
    cudaFree(p.chunks1);
    cudaFree(p.n_chunks);
    cudaFree(p.h_hi);
    cudaFree(p.h_lo);
    cudaFree(p.x3);
    cudaFree(p.xnorm);
    cudaFree(p.wnorm);
    if (p.status_host) cudaFreeHost(p.status_host);
    p = PrefillScratch{};
}

int prefill_last_status(const PrefillScratch& p) { return p.status_host ? *(volatile int*)p.status_host : 0; }

cudaError_t launch_prefill(const Shapes& s, PrefillScratch& p, const PrefillArgs& a, cudaStream_t st, int* launches,
                           cudaEvent_t* ev) {
    const int T = a.T, H = s.hidden, E = s.n_experts, k = s.top_k, P = T * k;
    const int n_hist = (P + kHistThreads - 1) / kHistThreads;
    *launches = 0;
    cudaError_t e;
    int mark = 0;
    auto stamp = [&]() -> cudaError_t { return ev ? cudaEventRecord(ev[mark++], st) : cudaSuccess; };
    if ((e = stamp())) return e;
    if (p.two_stage) {
        // approximate logits on the tensor cores, exact logits of the candidates
        if ((e = launch_router_two_stage(s, p, a, st, launches))) return e;
        if ((e = stamp())) return e;
    } else {
        if ((e = launch_logits(a.router_w, a.router_bias, a.x, T, H, E, kLgTokens, p.logits, st))) return e;
        ++*launches;
        if ((e = stamp())) return e;
        select_kernel<<<(T + 7) / 8, 256, 0, st>>>(p.logits, a.x, a.shared_blob ? a.shared_gate : nullptr, T, H, E,
                                                   k, s.norm_topk, p.idx, p.w, p.sigma, a.user_idx, a.user_w, p.x_bf,
                                                   a.y);
        ++*launches;
    }
    if ((e = stamp())) return e;
    {
        const size_t smem = (size_t)32 * E * sizeof(uint16_t);
        if ((e = smem_limit(reinterpret_cast<const void*>(hist_kernel), (int)smem))) return e;
        hist_kernel<<<n_hist, kHistThreads, smem, st>>>(p.idx, P, E, n_hist, p.local_rank, p.cnt);
        ++*launches;
    }
    if ((e = stamp())) return e;
    scan_kernel<<<1, 1024, 0, st>>>(p.cnt, E, n_hist, T, a.dir, a.shared_blob, p.offsets, p.chunks, p.chunks1,
                                    p.n_chunks);
    ++*launches;
    if ((e = stamp())) return e;
    scatter_kernel<<<n_hist, kHistThreads, 0, st>>>(p.idx, p.local_rank, p.cnt, p.w, P, k, n_hist, p.perm,
                                                    p.tok_sorted, p.w_sorted);
    ++*launches;
    if ((e = cudaGetLastError())) return e;
    if ((e = stamp())) return e;
    gather_kernel<<<4 * p.sms, kGatherThreads, 0, st>>>(p.tok_sorted, p.two_stage ? p.x3 : p.x_bf,
                                                        p.two_stage ? 3 * H : H, P, H, p.x_sorted);
    ++*launches;
    if ((e = cudaGetLastError())) return e;
    if ((e = stamp())) return e;
    if ((e = launch_prefill_gemm(0, s, p, a, st))) return e;
    ++*launches;
    if ((e = stamp())) return e;
    if ((e = launch_prefill_gemm(1, s, p, a, st))) return e;
    ++*launches;
    return stamp();
}

}  // namespace moe
