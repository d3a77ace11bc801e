// prefill_gemm.cu -- the two grouped GEMMs of the prefill path on the 5th
// generation tensor cores (tcgen05, fp32 accumulators in tensor memory).
//
// Work unit ("tile"): one chunk of <= 256 sorted rows of one expert (tokens for
// the gate/up GEMM, SwiGLU rows for the down GEMM) against 256 weight rows:
//   mode 0 (gate/up): weight rows s*128 .. s*128+127 of gate AND of up
//                     (two accumulators), K = hidden; epilogue
//                     h = silu(gate) * up in fp32, stored as the bf16 pair
//                     hi = bf16(h), lo = bf16(h - hi) (h to about 2^-17).
//   mode 1 (down):    output rows p*256 .. p*256+255 of the down matrix (two
//                     accumulators of 128 rows), K = inter, every k-block
//                     multiplied with both hi and lo; epilogue
//                     y[token] += weight * acc (fp32 reductions in L2).
// The MMA computes D[128 x N] = A[128 x 64] * B[N x 64]^T per 64-wide k-block,
// A = dequantised weights, B = activation rows, N = rows rounded up to 16.
//
// Warp roles of each persistent CTA (one per SM):
//   warp 0        one thread issues the MMAs and the commits
//   warps 1-4     epilogue: tensor memory -> registers -> global (warp w reads
//                 tensor-memory lanes 32*(w%4) .. +31)
//   warps 5-12    producers, two groups of four warps taking alternate
//                 k-blocks: load the packed codes and scale/bias, dequantise
//                 to bf16(fp32 fma(scale, q, bias)) and write them as
//                 128-byte-swizzled K-major tiles; mode 0 also gathers the
//                 token rows of bf16(x) the same way, mode 1 bulk-copies the
//                 SwiGLU rows, which the gate/up epilogue stored already
//                 swizzled (one copy per operand per k-block).
// Stage hand-off uses mbarriers (full: producers -> MMA, empty: MMA commit ->
// producers; accumulator full/empty between MMA and epilogue).  Every wait is
// bounded; a wait that runs out records a status word in mapped host memory
// and the CTA winds down, draining its MMAs and freeing its tensor memory.
//
// MLX affine group quantisation (Swiftlet README, "Relation to
// TurboFieldfare"): w = scale * q + bias per 64-column group.  The tensor-core
// operands are bf16 (weights dequantised in shared memory), accumulation fp32.
#include <cuda_bf16.h>

#include "gemv.cuh"
#include "prefill.h"
#include "umma.cuh"

namespace moe {
namespace {

using namespace umma;

constexpr int kGemmThreads = 416;
constexpr int kGroupThreads = 128;
constexpr int kTileBytes = 16 * 1024;  // 128 rows x 64 bf16 (one 256-row operand = 2 tiles)
constexpr int kTmemCols = 512;         // two accumulators of up to 256 columns

template <int MODE>
struct Cfg;
template <>
struct Cfg<0> {  // A0 | A1 | B
    static constexpr int kStages = 3, kStageBytes = 4 * kTileBytes;
};
template <>
struct Cfg<1> {  // A0 | A1 | B hi | B lo
    static constexpr int kStages = 2, kStageBytes = 6 * kTileBytes;
};

struct GemmArgs {
    int H, E, k, T, P;  // P = T * k
    int inter, shared_inter, slices0, h_rows;
    int x_stride;  // elements between token rows of x_bf
    const int4* chunks;
    const int32_t* n_chunks;
    const int32_t* perm;
    const uint16_t* x_bf;
    uint16_t* h_hi;
    uint16_t* h_lo;
    const float* w;
    const float* sigma;
    float* y;
    const uint8_t* const* dir;
    const uint8_t* shared_blob;
    int* status;
    unsigned long long timeout_ns;
};

struct Tile {
    int e, row0, n, hrow0, sub, kb;
    const uint8_t* blob;
};

template <int MODE>
__device__ __forceinline__ bool tile_at(const GemmArgs& a, int t, Tile& tl) {
    const int per = MODE == 0 ? a.slices0 : a.H / 256;
    const int4 c = a.chunks[t / per];
    tl.e = c.x;
    tl.row0 = c.y;
    tl.n = c.z;
    tl.hrow0 = c.w;
    tl.sub = t % per;
    const bool sh = tl.e == a.E;
    const int inter_e = sh ? a.shared_inter : a.inter;
    if (MODE == 0) {
        if (tl.sub * 128 >= inter_e) return false;
        tl.kb = a.H / 64;
    } else {
        tl.kb = inter_e / 64;
    }
    tl.blob = sh ? a.shared_blob : a.dir[tl.e];
    return tl.blob != nullptr;
}

__device__ __forceinline__ int n_pad(int n) { return n < 16 ? 16 : (n + 15) & ~15; }

__device__ __forceinline__ void fail(const GemmArgs& a, volatile int* abort, int code) {
    *abort = 1;
    *(volatile int*)a.status = code;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// code byte i of v as an exact float: bits 0x4B0000qq = 2^23 + q
__device__ __forceinline__ float code_f(uint32_t v, int i) {
    return __fsub_rn(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u | (uint32_t)i)), 8388608.0f);
}

// bf16(fma(s, q, b)) of 8 consecutive int4 columns (one code word)
__device__ __forceinline__ uint4 dq8_int4(uint32_t wd, float s, float b) {
    const uint32_t lo = wd & 0x0F0F0F0Fu, hi = (wd >> 4) & 0x0F0F0F0Fu;  // even / odd columns
    uint4 o;
    o.x = pack_bf16(__fmaf_rn(s, code_f(lo, 0), b), __fmaf_rn(s, code_f(hi, 0), b));
    o.y = pack_bf16(__fmaf_rn(s, code_f(lo, 1), b), __fmaf_rn(s, code_f(hi, 1), b));
    o.z = pack_bf16(__fmaf_rn(s, code_f(lo, 2), b), __fmaf_rn(s, code_f(hi, 2), b));
    o.w = pack_bf16(__fmaf_rn(s, code_f(lo, 3), b), __fmaf_rn(s, code_f(hi, 3), b));
    return o;
}

// ... of 8 consecutive int8 columns (two code words)
__device__ __forceinline__ uint4 dq8_int8(uint32_t w0, uint32_t w1, float s, float b) {
    uint4 o;
    o.x = pack_bf16(__fmaf_rn(s, code_f(w0, 0), b), __fmaf_rn(s, code_f(w0, 1), b));
    o.y = pack_bf16(__fmaf_rn(s, code_f(w0, 2), b), __fmaf_rn(s, code_f(w0, 3), b));
    o.z = pack_bf16(__fmaf_rn(s, code_f(w1, 0), b), __fmaf_rn(s, code_f(w1, 1), b));
    o.w = pack_bf16(__fmaf_rn(s, code_f(w1, 2), b), __fmaf_rn(s, code_f(w1, 3), b));
    return o;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Producer-side position in the CTA's sequence of (tile, k-block) iterations.
struct Cursor {
    int t;        // tile index (global), -1 = past the end
    int kb;       // k-block within the tile
    uint32_t it;  // iteration number within the CTA
    Tile tl;
};

template <int MODE>
__device__ __forceinline__ void cursor_first(const GemmArgs& a, int n_tiles, Cursor& c) {
    c.it = 0;
    c.kb = 0;
    for (c.t = blockIdx.x; c.t < n_tiles; c.t += gridDim.x)
        if (tile_at<MODE>(a, c.t, c.tl)) return;
    c.t = -1;
}

template <int MODE>
__device__ __forceinline__ void cursor_next(const GemmArgs& a, int n_tiles, Cursor& c) {
    if (c.t < 0) return;
    ++c.it;
    if (++c.kb < c.tl.kb) return;
    c.kb = 0;
    for (c.t += gridDim.x; c.t < n_tiles; c.t += gridDim.x)
        if (tile_at<MODE>(a, c.t, c.tl)) return;
    c.t = -1;
}

// Per producer thread: its 16-byte code units of the two 128-row weight tiles
// of one k-block (unit u = gt + 128 i: tile u / (128 U), row (u / U) % 128,
// part u % U, with U = 16-byte units per row per k-block) and their scale/bias.
template <int BITS>
struct ProdRegs {
    static constexpr int U = BITS / 2;
    static constexpr int kUnitsA = 2 * 128 * U / kGroupThreads;
    uint4 qa[kUnitsA];
    uint32_t sba[kUnitsA];
};

template <int MODE, int BITS>
__device__ __forceinline__ void prod_load(const GemmArgs& a, const Cursor& c, int gt, ProdRegs<BITS>& R) {
    using PR = ProdRegs<BITS>;
    const Tile& tl = c.tl;
    const int inter_e = tl.e == a.E ? a.shared_inter : a.inter;
    const BlobLayout L = blob_layout(a.H, inter_e, BITS);
    const int K = MODE == 0 ? a.H : inter_e;
    const size_t rowbytes = (size_t)K * BITS / 8;
    const int groups = K / 64;
#pragma unroll
    for (int i = 0; i < PR::kUnitsA; ++i) {
        const int u = gt + kGroupThreads * i;
        const int m = u / (128 * PR::U), r = (u / PR::U) % 128, part = u % PR::U;
        int row;
        uint64_t qoff, sboff;
        if (MODE == 0) {
            row = tl.sub * 128 + r;
            qoff = m ? L.up_q : L.gate_q;
            sboff = m ? L.up_sb : L.gate_sb;
        } else {
            row = tl.sub * 256 + m * 128 + r;
            qoff = L.down_q;
            sboff = L.down_sb;
        }
        R.qa[i] = ldg_nc(tl.blob + qoff + row * rowbytes + (size_t)c.kb * 64 * BITS / 8 + part * 16);
        R.sba[i] = __ldg(reinterpret_cast<const uint32_t*>(tl.blob + sboff) + (size_t)row * groups + c.kb);
    }
}

template <int BITS>
__device__ __forceinline__ void prod_store(int gt, uint32_t stage, const ProdRegs<BITS>& R) {
    using PR = ProdRegs<BITS>;
#pragma unroll
    for (int i = 0; i < PR::kUnitsA; ++i) {
        const int u = gt + kGroupThreads * i;
        const int m = u / (128 * PR::U), r = (u / PR::U) % 128, part = u % PR::U;
        const uint32_t tile = stage + m * kTileBytes;
        const float s = __half2float(__ushort_as_half((unsigned short)(R.sba[i] & 0xffffu)));
        const float b = __half2float(__ushort_as_half((unsigned short)(R.sba[i] >> 16)));
        if (BITS == 4) {
            sts128(tile + swz_chunk(r, part * 4 + 0), dq8_int4(R.qa[i].x, s, b));
            sts128(tile + swz_chunk(r, part * 4 + 1), dq8_int4(R.qa[i].y, s, b));
            sts128(tile + swz_chunk(r, part * 4 + 2), dq8_int4(R.qa[i].z, s, b));
            sts128(tile + swz_chunk(r, part * 4 + 3), dq8_int4(R.qa[i].w, s, b));
        } else {
            sts128(tile + swz_chunk(r, part * 2 + 0), dq8_int8(R.qa[i].x, R.qa[i].y, s, b));
            sts128(tile + swz_chunk(r, part * 2 + 1), dq8_int8(R.qa[i].z, R.qa[i].w, s, b));
        }
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// arrive on the mbarrier once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* b) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(b)) : "memory");
}

// token of sorted row j of a gate/up tile
__device__ __forceinline__ int token_row(const GemmArgs& a, const Tile& tl, int j) {
    if (j >= tl.n) return 0;
    return tl.e == a.E ? tl.row0 + j : a.perm[tl.row0 + j] / a.k;
}

// element offset of (row, col) in a pre-swizzled SwiGLU buffer: planes of 64
// columns, [plane][row][64], 16-byte chunks swizzled by row & 7
__device__ __forceinline__ size_t h_offset(int rows, int row, int col) {
    return ((size_t)(col >> 6) * rows + row) * 64 + ((((col >> 3) ^ row) & 7) << 3) + (col & 7);
}

template <int MODE, int BITS>
__global__ void __launch_bounds__(kGemmThreads, 1) grouped_gemm_kernel(GemmArgs a) {
    constexpr int S = Cfg<MODE>::kStages, SB = Cfg<MODE>::kStageBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[S], empty_bar[S], accf_bar, acce_bar, drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int n_tiles = *a.n_chunks * (MODE == 0 ? a.slices0 : a.H / 256);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            // four producer warps, plus (gate/up) one asynchronous arrival per
            // producer thread when its token-row copies have landed
            bar_init(&full_bar[s], MODE == 0 ? 4 + kGroupThreads : 4);
            bar_init(&empty_bar[s], 1);
        }
        bar_init(&accf_bar, 1);
        bar_init(&acce_bar, 4);
        bar_init(&drain_bar, 1);
        abort_s = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;

    if (warp == 0) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t it = 0, acc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                Tile tl;
                if (!tile_at<MODE>(a, t, tl)) continue;
                if (!bar_wait(&acce_bar, (acc & 1u) ^ 1u, a.timeout_ns, &abort_s)) {
                    fail(a, &abort_s, 2);
                    break;
                }
                fence_after_sync();
                const uint32_t idesc = idesc_bf16(128, n_pad(tl.n));
                for (int kb = 0; kb < tl.kb; ++kb, ++it) {
                    const uint32_t s = it % S;
                    if (!bar_wait(&full_bar[s], (it / S) & 1u, a.timeout_ns, &abort_s)) {
                        fail(a, &abort_s, 2);
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    fence_proxy_async_smem();  // the token rows were written by cp.async (generic proxy)
                    const uint32_t st = smem0 + s * SB;
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sdesc(st + m * kTileBytes + kk * 32);
                            mma_bf16(tmem + m * 256, ad, sdesc(st + 2 * kTileBytes + kk * 32), idesc,
                                     (kb | kk) ? 1u : 0u);
                            if (MODE == 1) mma_bf16(tmem + m * 256, ad, sdesc(st + 4 * kTileBytes + kk * 32), idesc, 1u);
                        }
                    mma_commit(&empty_bar[s]);
                }
                if (!ok) break;
                mma_commit(&accf_bar);
                ++acc;
            }
            // every MMA issued above has completed once this commit arrives
            mma_commit(&drain_bar);
            if (!bar_wait(&drain_bar, 0, a.timeout_ns, &abort_s)) fail(a, &abort_s, 2);
        }
        __syncwarp();
    } else if (warp <= 4) {
        // ------------------------------------------------------------- epilogue
        const int q = warp & 3;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t acc = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            Tile tl;
            if (!tile_at<MODE>(a, t, tl)) continue;
            if (!bar_wait(&accf_bar, acc & 1u, a.timeout_ns, &abort_s)) {
                fail(a, &abort_s, 3);
                break;
            }
            fence_after_sync();
            const bool sh = tl.e == a.E;
            for (int c0 = 0; c0 < tl.n; c0 += 32) {
                uint32_t d0[32], d1[32];
                tmem_ld32(trow + c0, d0);
                tmem_ld32(trow + 256 + c0, d1);
                tmem_ld_wait();
                const int nc = min(32, tl.n - c0);
                if constexpr (MODE == 0) {
                    const int col = tl.sub * 128 + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < nc) {
                            const float v = silu_mul(__uint_as_float(d0[j]), __uint_as_float(d1[j]));
                            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                            const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));
                            const size_t off = h_offset(a.h_rows, tl.hrow0 + c0 + j, col);
                            a.h_hi[off] = __bfloat16_as_ushort(hi);
                            a.h_lo[off] = __bfloat16_as_ushort(lo);
                        }
                    }
                } else {
                    int tok = 0;
                    float wt = 0.0f;
                    if (lane < nc) {
                        if (sh) {
                            tok = tl.row0 + c0 + lane;
                            wt = a.sigma[tok];
                        } else {
                            const int pair = a.perm[tl.row0 + c0 + lane];
                            tok = pair / a.k;
                            wt = a.w[pair];
                        }
                    }
                    float* y0 = a.y + tl.sub * 256 + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tj = __shfl_sync(kFullMask, tok, j);
                        const float wj = __shfl_sync(kFullMask, wt, j);
                        if (j < nc) {
                            float* yr = y0 + (size_t)tj * a.H;
                            atomicAdd(yr, wj * __uint_as_float(d0[j]));
                            atomicAdd(yr + 128, wj * __uint_as_float(d1[j]));
                        }
                    }
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) bar_arrive(&acce_bar);
            ++acc;
        }
    } else {
        // ------------------------------------------------------------ producers
        // Two register sets of packed codes, each loaded two own iterations
        // (four k-blocks) before it is dequantised.
        const int g = (warp - 5) >> 2, gt = tid - 160 - g * kGroupThreads;
        ProdRegs<BITS> R0, R1;
        int brow[16];
        int brow_tile = -1;
        Cursor c0, c1, tail;
        cursor_first<MODE>(a, n_tiles, c0);
        if (c0.t >= 0 && g == 1) cursor_next<MODE>(a, n_tiles, c0);
        c1 = c0;
        cursor_next<MODE>(a, n_tiles, c1);
        cursor_next<MODE>(a, n_tiles, c1);
        tail = c1;
        if (c0.t >= 0) prod_load<MODE, BITS>(a, c0, gt, R0);
        if (c1.t >= 0) prod_load<MODE, BITS>(a, c1, gt, R1);
        auto iterate = [&](const Cursor& c, const ProdRegs<BITS>& R) -> bool {
            const uint32_t s = c.it % S;
            if (!bar_wait(&empty_bar[s], ((c.it / S) & 1u) ^ 1u, a.timeout_ns, &abort_s)) {
                fail(a, &abort_s, 1);
                return false;
            }
            const uint32_t st = smem0 + s * SB;
            if constexpr (MODE == 0) {
                // token rows of bf16(x): 8 lanes per 128-byte row, copied straight into the swizzled tile
                if (c.t != brow_tile) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) brow[i] = token_row(a, c.tl, (gt >> 3) + 16 * i);
                    brow_tile = c.t;
                }
                const int np = n_pad(c.tl.n);
                const uint32_t btile = st + 2 * kTileBytes;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int j = (gt >> 3) + 16 * i;
                    if (j < c.tl.n)
                        cp_async16(btile + swz_chunk(j, gt & 7),
                                   a.x_bf + (size_t)brow[i] * a.x_stride + c.kb * 64 + (gt & 7) * 8);
                    else if (j < np)
                        sts128(btile + swz_chunk(j, gt & 7), make_uint4(0, 0, 0, 0));
                }
                cp_async_arrive(&full_bar[s]);
            } else {
                if (gt == 0) {
                    // the SwiGLU rows of this chunk and k-block, hi and lo, already swizzled
                    const uint32_t bytes = (uint32_t)n_pad(c.tl.n) * 128u;
                    const size_t src = ((size_t)c.kb * a.h_rows + c.tl.hrow0) * 64;
                    bar_expect_tx(&full_bar[s], 2 * bytes);
                    bulk_g2s(st + 2 * kTileBytes, a.h_hi + src, bytes, &full_bar[s]);
                    bulk_g2s(st + 4 * kTileBytes, a.h_lo + src, bytes, &full_bar[s]);
                }
            }
            prod_store<BITS>(gt, st, R);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(&full_bar[s]);
            return true;
        };
        for (;;) {
            if (c0.t < 0 || !iterate(c0, R0)) break;
            cursor_next<MODE>(a, n_tiles, tail);
            cursor_next<MODE>(a, n_tiles, tail);
            c0 = tail;
            if (c0.t >= 0) prod_load<MODE, BITS>(a, c0, gt, R0);
            if (c1.t < 0 || !iterate(c1, R1)) break;
            cursor_next<MODE>(a, n_tiles, tail);
            cursor_next<MODE>(a, n_tiles, tail);
            c1 = tail;
            if (c1.t >= 0) prod_load<MODE, BITS>(a, c1, gt, R1);
        }
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE, int BITS>
cudaError_t launch_mode(const GemmArgs& g, int grid, cudaStream_t st) {
    const size_t smem = (size_t)Cfg<MODE>::kStages * Cfg<MODE>::kStageBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<MODE, BITS><<<grid, kGemmThreads, smem, st>>>(g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gemm(int mode, const Shapes& s, const PrefillScratch& p, const PrefillArgs& a,
                                cudaStream_t st) {
    GemmArgs g{};
    g.H = s.hidden;
    g.E = s.n_experts;
    g.k = s.top_k;
    g.T = a.T;
    g.P = a.T * s.top_k;
    g.inter = s.inter;
    g.shared_inter = a.shared_blob ? s.shared_inter : 0;
    g.slices0 = s.h_stride / 128;
    g.h_rows = p.h_rows;
    g.chunks = p.chunks;
    g.n_chunks = p.n_chunks;
    g.perm = p.perm;
    g.x_bf = p.two_stage ? p.x3 : p.x_bf;
    g.x_stride = p.two_stage ? 3 * s.hidden : s.hidden;
    g.h_hi = p.h_hi;
    g.h_lo = p.h_lo;
    g.w = p.w;
    g.sigma = p.sigma;
    g.y = a.y;
    g.dir = a.dir;
    g.shared_blob = a.shared_blob;
    g.status = p.status_dev;
    g.timeout_ns = a.timeout_ns;
    if (mode == 0) return s.bits == 4 ? launch_mode<0, 4>(g, p.sms, st) : launch_mode<0, 8>(g, p.sms, st);
    return s.bits == 4 ? launch_mode<1, 4>(g, p.sms, st) : launch_mode<1, 8>(g, p.sms, st);
}

}  // namespace moe
