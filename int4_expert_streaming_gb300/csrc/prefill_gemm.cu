// prefill_gemm.cu -- the two grouped GEMMs of the prefill path on the 5th
// generation tensor cores (tcgen05, fp32 accumulators in tensor memory).
//
// Work unit ("tile"): one chunk of sorted rows of one expert against 256
// weight rows, K in blocks of 64:
//   mode 0 (gate/up): chunk of <= 256 token rows; weight rows s*128 .. +127 of
//                     gate AND of up (accumulators in tensor-memory columns
//                     0-255 and 256-511), K = hidden; epilogue
//                     h = silu(gate) * up in fp32, stored as the bf16 pair
//                     hi = bf16(h), lo = bf16(h - hi) (h to about 2^-17).
//   mode 1 (down):    chunk of <= 128 SwiGLU rows; output rows p*256 .. +255
//                     of the down matrix (two accumulators of 128 columns,
//                     double-buffered: columns 0-255 and 256-511), K = inter,
//                     every k-block multiplied with both hi and lo; epilogue
//                     y[token] += weight * acc (fp32 reductions in L2).
// The MMA computes D[128 x N] = A[128 x 64] * B[N x 64]^T per k-block, A =
// dequantised weights, B = activation rows, N = rows rounded up to 16.
//
// Warp roles of each persistent CTA (one per SM, 26 warps):
//   warp 0        one thread issues the MMAs and the commits
//   warp 1        B loader, a 3-stage ring ahead of the MMA: mode 0 copies
//                 the chunk's token rows (bf16(x) in sorted pair order, or in
//                 token order for the shared expert) with TMA, boxes of 64 rows
//                 x 64 columns landing 128-byte swizzled; mode 1 bulk-copies
//                 the SwiGLU rows, which the gate/up epilogue stored already
//                 swizzled
//   warps 2-9     epilogue: tensor memory -> registers -> global; warp w reads
//                 tensor-memory lanes 32*(w%4) .. +31, the two warps of a lane
//                 quarter take alternate 16-column groups
//   warps 10-25   dequantisers, two threads per weight row (32 columns each):
//                 each thread stages its own packed codes and scale/bias
//                 several k-blocks ahead with cp.async (a private ring, so no
//                 barrier), then writes bf16(fp32 fma(scale, q, bias)) into
//                 the swizzled A tile of a 3-stage ring (2 for int8)
// Stage hand-off uses mbarriers (A/B full: producers -> MMA; one "k-block
// done" commit per k-block into a ring of 6, on which the A producers wait two
// k-blocks later and the B loader three; accumulator full/empty between MMA
// and epilogue).  The MMA thread shares its issue slots with busy warps, so
// its loop is kept short: descriptors are a fixed high word and a low word
// stepped by adds, stage and phase counters advance without division.
// Every wait is bounded; a wait that runs out records a status word in mapped
// host memory and the CTA winds down, draining its MMAs and copies and freeing
// its tensor memory.
//
// MLX affine group quantisation (Swiftlet README, "Relation to
// TurboFieldfare"): w = scale * q + bias per 64-column group.  The tensor-core
// operands are bf16 (weights dequantised in shared memory), accumulation fp32.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "gemv.cuh"
#include "prefill.h"
#include "umma.cuh"

namespace moe {
namespace {

using namespace umma;
using namespace gemmc;

constexpr int kLoadWarp = 1;
constexpr int kEpiWarp0 = 2, kEpiWarps = 8;
constexpr int kDqWarp0 = 10, kDqWarps = 16;
constexpr int kThreads = 32 * (kDqWarp0 + kDqWarps);  // 832
constexpr int kDqThreads = 32 * kDqWarps;             // two per weight row
constexpr int kTileBytes = 16 * 1024;                  // 128 rows x 64 bf16
constexpr int kStageBytes = 2 * kTileBytes;            // two weight tiles, 256 token rows, or hi + lo of 128 rows
constexpr int kBStages = 3;
constexpr int kDone = 6;  // k-block done ring: a multiple of both stage counts
constexpr int kTmemCols = 512;
constexpr int kOffB = 0;  // shared-memory map from a 1024-byte aligned base: B ring, A ring, code ring

// Shared memory per code width: the A ring (3 stages for int4, 2 for int8) and
// the dequantisers' private code ring: per thread and k-block, 32 packed
// weights (16 bytes int4, 32 bytes int8 as two 16-byte parts) and the
// scale/bias word.
template <int BITS>
struct Ring {
    static constexpr int kAStages = BITS == 4 ? 3 : 2;
    static constexpr int kParts = BITS / 4;  // 16-byte parts per thread
    static constexpr int kSlotBytes = kDqThreads * (16 * kParts + 4);
    static constexpr int kSlots = 3;
    static constexpr int kOffA = kOffB + kBStages * kStageBytes;
    static constexpr int kOffCodes = kOffA + kAStages * kStageBytes;
    static constexpr int kSmem = kOffCodes + kSlots * kSlotBytes;
};
static_assert(kDone % 2 == 0 && kDone % 3 == 0, "done ring");
static_assert(Ring<4>::kSmem + 1024 + 512 <= 227 * 1024, "shared memory");
static_assert(Ring<8>::kSmem + 1024 + 512 <= 227 * 1024, "shared memory");

struct GemmArgs {
    int H, E, T;
    int inter, shared_inter;
    int per;  // tiles per chunk: mode 0 inter slices of 128, mode 1 output slices of 256
    int h_rows;
    const ChunkRec* chunks;
    const int32_t* n_chunks;
    const int32_t* tok_sorted;
    const float* w_sorted;
    uint16_t* h_hi;
    uint16_t* h_lo;
    const float* sigma;
    float* y;
    int* status;
    unsigned long long timeout_ns;
};

struct TileInfo {
    int e, row0, n, hrow0, sub;
    const uint8_t* blob;
};

__device__ __forceinline__ int n_pad(int n) { return n < 16 ? 16 : (n + 15) & ~15; }

// The CTA's tiles t = blockIdx.x + i * gridDim.x, each with its chunk record;
// the record of the following tile is loaded one tile ahead, so moving on does
// not wait for memory.
template <int MODE>
struct Tiles {
    int t, pref_t;
    int4 pc, pb;  // raw record of tile pref_t
    TileInfo cur;

    __device__ __forceinline__ static void load(const GemmArgs& a, int t, int4& c, int4& b) {
        const int4* r = reinterpret_cast<const int4*>(a.chunks + t / a.per);
        c = __ldg(r);
        b = __ldg(r + 1);
    }
    __device__ __forceinline__ bool decode(const GemmArgs& a, int4 c, int4 b) {
        cur.e = c.x;
        cur.row0 = c.y;
        cur.n = c.z;
        cur.hrow0 = c.w;
        cur.sub = t % a.per;
        cur.blob = reinterpret_cast<const uint8_t*>((unsigned long long)(uint32_t)b.x |
                                                    ((unsigned long long)(uint32_t)b.y << 32));
        if (!cur.blob) return false;
        if (MODE == 0) return cur.sub * 128 < (cur.e == a.E ? a.shared_inter : a.inter);
        return true;
    }
    // moves to the next valid tile; false past the end
    __device__ __forceinline__ bool next(const GemmArgs& a, int n_tiles) {
        for (;;) {
            t += gridDim.x;
            if (t >= n_tiles) return false;
            int4 c, b;
            if (pref_t == t) {
                c = pc;
                b = pb;
            } else {
                load(a, t, c, b);
            }
            pref_t = t + gridDim.x;
            if (pref_t < n_tiles) load(a, pref_t, pc, pb);
            if (decode(a, c, b)) return true;
        }
    }
    __device__ __forceinline__ bool first(const GemmArgs& a, int n_tiles) {
        t = (int)blockIdx.x - (int)gridDim.x;
        pref_t = -1;
        return next(a, n_tiles);
    }
    __device__ __forceinline__ int kblocks(const GemmArgs& a) const {
        return (MODE == 0 ? a.H : (cur.e == a.E ? a.shared_inter : a.inter)) / 64;
    }
};

__device__ __forceinline__ void fail(const GemmArgs& a, volatile int* abort, int code) {
    *abort = 1;
    *(volatile int*)a.status = code;
}

// D (+)= A * B^T with both descriptors given as (low, high) words
__device__ __forceinline__ void mma_bf16_w(uint32_t d, uint32_t alo, uint32_t blo, uint32_t dhi, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 ad, bd;\n mov.b64 ad, {%1, %3};\n mov.b64 bd, {%2, %3};\n setp.ne.b32 p, %5, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, p;\n}" ::"r"(d),
        "r"(alo), "r"(blo), "r"(dhi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// bounded wait taken by lane 0 for the whole warp
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, const GemmArgs& a, volatile int* abort,
                                          int lane) {
    int ok = 1;
    if (lane == 0) ok = bar_wait(b, parity, a.timeout_ns, abort) ? 1 : 0;
    return __shfl_sync(kFullMask, ok, 0) != 0;
}

// Dequantiser thread (weight row r of the tile, column half hf): the address
// of its codes and of its row's scale/bias words in the tile's expert blob.
template <int MODE, int BITS>
__device__ __forceinline__ void code_src(const GemmArgs& a, const TileInfo& ti, int r, int hf, const uint8_t*& q,
                                         const uint8_t*& sb) {
    const int inter_e = ti.e == a.E ? a.shared_inter : a.inter;
    const BlobLayout L = blob_layout(a.H, inter_e, BITS);
    const int K = MODE == 0 ? a.H : inter_e;
    const size_t rowbytes = (size_t)K * BITS / 8;
    int row;
    uint64_t qoff, sboff;
    if (MODE == 0) {
        const int m = r >> 7;
        row = ti.sub * 128 + (r & 127);
        qoff = m ? L.up_q : L.gate_q;
        sboff = m ? L.up_sb : L.gate_sb;
    } else {
        row = ti.sub * 256 + r;
        qoff = L.down_q;
        sboff = L.down_sb;
    }
    q = ti.blob + qoff + row * rowbytes + hf * 4 * BITS;
    sb = ti.blob + sboff + (size_t)row * (K / 64) * 4;
}

template <int MODE, int BITS>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap x_map,
                                                                   const __grid_constant__ CUtensorMap xs_map, GemmArgs a) {
    using RG = Ring<BITS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr int kAStages = RG::kAStages;
    __shared__ uint64_t a_full[kAStages], b_full[kBStages], kb_done[kDone];
    __shared__ uint64_t acc_full[2], acc_empty[2], drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s, never_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int n_tiles = a.n_chunks[MODE] * a.per;

    if (tid == 0) {
        for (int s = 0; s < kAStages; ++s) bar_init(&a_full[s], kDqWarps);
        for (int s = 0; s < kBStages; ++s) bar_init(&b_full[s], 1);
        for (int s = 0; s < kDone; ++s) bar_init(&kb_done[s], 1);
        for (int s = 0; s < 2; ++s) {
            bar_init(&acc_full[s], 1);
            bar_init(&acc_empty[s], kEpiWarps);
        }
        bar_init(&drain_bar, 1);
        abort_s = 0;
        never_s = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, kTmemCols);
    // operand rows past a chunk's last row are never written; keep them finite
    for (int i = tid; i < kBStages * kStageBytes / 16; i += kThreads)
        sts128(smem0 + kOffB + 16 * i, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;

    if (warp == 0) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t tc = 0, sa = 0, pa = 0, sb = 0, pb = 0, sd = 0;
            const uint32_t dhi = (uint32_t)(sdesc(smem0) >> 32);  // the same for every operand tile
            const uint32_t a_lo = (uint32_t)sdesc(smem0 + RG::kOffA), b_lo = (uint32_t)sdesc(smem0 + kOffB);
            constexpr uint32_t kTileLo = kTileBytes >> 4, kStageLo = kStageBytes >> 4;
            bool ok = true;
            Tiles<MODE> tiles;
            for (bool has = tiles.first(a, n_tiles); has && ok; has = tiles.next(a, n_tiles), ++tc) {
                const TileInfo& ti = tiles.cur;
                const uint32_t ab = MODE == 0 ? 0u : (tc & 1u);
                const uint32_t use = MODE == 0 ? tc : (tc >> 1);
                if (!bar_wait(&acc_empty[ab], (use & 1u) ^ 1u, a.timeout_ns, &abort_s)) {
                    fail(a, &abort_s, 2);
                    break;
                }
                fence_after_sync();
                const uint32_t idesc = idesc_bf16(128, n_pad(ti.n));
                const uint32_t d0 = tmem + (MODE == 0 ? 0u : ab * 256);
                const int nkb = tiles.kblocks(a);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!bar_wait(&a_full[sa], pa, a.timeout_ns, &abort_s) ||
                        !bar_wait(&b_full[sb], pb, a.timeout_ns, &abort_s)) {
                        fail(a, &abort_s, 2);
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t al = a_lo + sa * kStageLo, bl = b_lo + sb * kStageLo;
                    const uint32_t acc0 = kb ? 1u : 0u;
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t am = al + m * kTileLo + 2 * kk;
                            if (MODE == 0) {
                                mma_bf16_w(d0 + m * 256, am, bl + 2 * kk, dhi, idesc, kk ? 1u : acc0);
                            } else {
                                mma_bf16_w(d0 + m * 128, am, bl + 2 * kk, dhi, idesc, kk ? 1u : acc0);
                                mma_bf16_w(d0 + m * 128, am, bl + kTileLo + 2 * kk, dhi, idesc, 1u);
                            }
                        }
                    mma_commit(&kb_done[sd]);
                    sd = sd == kDone - 1 ? 0 : sd + 1;
                    if (++sa == kAStages) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == kBStages) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&acc_full[ab]);
            }
            // every MMA issued above has completed once this commit arrives
            mma_commit(&drain_bar);
            if (!bar_wait(&drain_bar, 0, a.timeout_ns, &never_s)) fail(a, &abort_s, 2);
        }
        __syncwarp();
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------- B loader
        uint32_t it = 0;
        Tiles<MODE> tiles;
        if constexpr (MODE == 0) {
            // one thread: per k-block, ceil(n / 64) boxes of 64 rows
            if (lane == 0) {
                for (bool has = tiles.first(a, n_tiles); has; has = tiles.next(a, n_tiles)) {
                    const TileInfo& ti = tiles.cur;
                    const CUtensorMap* map = ti.e == a.E ? &x_map : &xs_map;
                    const int nb = (ti.n + 63) >> 6;
                    const int nkb = tiles.kblocks(a);
                    bool ok = true;
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const uint32_t s = it % kBStages;
                        // stage s was last read by the MMAs of k-block it - kBStages
                        if (it >= kBStages && !bar_wait(&kb_done[(it - kBStages) % kDone],
                                                        ((it - kBStages) / kDone) & 1u, a.timeout_ns, &abort_s)) {
                            fail(a, &abort_s, 4);
                            ok = false;
                            break;
                        }
                        const uint32_t bs = smem0 + kOffB + s * kStageBytes;
                        bar_arrive_expect_tx(&b_full[s], (uint32_t)nb * 8192u);
                        for (int q = 0; q < nb; ++q) tma_load_2d(bs + q * 8192, map, kb * 64, ti.row0 + 64 * q, &b_full[s]);
                    }
                    if (!ok) break;
                }
                // copies still in flight land before the CTA exits
                for (uint32_t i = it > kBStages ? it - kBStages : 0; i < it; ++i)
                    bar_wait(&b_full[i % kBStages], (i / kBStages) & 1u, a.timeout_ns, &never_s);
            }
            __syncwarp();
        } else {
            // one thread: the hi and lo rows of a k-block, two bulk copies
            if (lane == 0) {
                for (bool has = tiles.first(a, n_tiles); has; has = tiles.next(a, n_tiles)) {
                    const TileInfo& ti = tiles.cur;
                    const uint32_t bytes = (uint32_t)n_pad(ti.n) * 128u;
                    const int nkb = tiles.kblocks(a);
                    bool ok = true;
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const uint32_t s = it % kBStages;
                        // stage s was last read by the MMAs of k-block it - kBStages
                        if (it >= kBStages && !bar_wait(&kb_done[(it - kBStages) % kDone],
                                                        ((it - kBStages) / kDone) & 1u, a.timeout_ns, &abort_s)) {
                            fail(a, &abort_s, 4);
                            ok = false;
                            break;
                        }
                        const uint32_t bs = smem0 + kOffB + s * kStageBytes;
                        const size_t src = ((size_t)kb * a.h_rows + ti.hrow0) * 64;
                        bar_arrive_expect_tx(&b_full[s], 2 * bytes);
                        bulk_g2s(bs, a.h_hi + src, bytes, &b_full[s]);
                        bulk_g2s(bs + kTileBytes, a.h_lo + src, bytes, &b_full[s]);
                    }
                    if (!ok) break;
                }
                // copies still in flight land before the CTA exits
                for (uint32_t i = it > kBStages ? it - kBStages : 0; i < it; ++i)
                    bar_wait(&b_full[i % kBStages], (i / kBStages) & 1u, a.timeout_ns, &never_s);
            }
            __syncwarp();
        }
    } else if (warp < kDqWarp0) {
        // ------------------------------------------------------------- epilogue
        const int q = warp & 3, hh = (warp - kEpiWarp0) >> 2;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t tc = 0;
        Tiles<MODE> tiles;
        for (bool has = tiles.first(a, n_tiles); has; has = tiles.next(a, n_tiles), ++tc) {
            const TileInfo& ti = tiles.cur;
            const uint32_t ab = MODE == 0 ? 0u : (tc & 1u);
            const uint32_t use = MODE == 0 ? tc : (tc >> 1);
            const bool sh = ti.e == a.E;
            // mode 1: token and weight of this warp's columns 16 hh + 32 s + i
            // (step s = 0..3, i = 0..15): lane l holds s = l >> 4 (set A) and
            // s = 2 + (l >> 4) (set B), column i = l & 15
            int tokA = 0, tokB = 0;
            float wA = 0.0f, wB = 0.0f;
            if constexpr (MODE == 1) {
                const int ca = 16 * hh + 32 * (lane >> 4) + (lane & 15), cb = ca + 64;
                if (ca < ti.n) {
                    tokA = sh ? ti.row0 + ca : __ldg(a.tok_sorted + ti.row0 + ca);
                    wA = sh ? __ldg(a.sigma + ti.row0 + ca) : __ldg(a.w_sorted + ti.row0 + ca);
                }
                if (cb < ti.n) {
                    tokB = sh ? ti.row0 + cb : __ldg(a.tok_sorted + ti.row0 + cb);
                    wB = sh ? __ldg(a.sigma + ti.row0 + cb) : __ldg(a.w_sorted + ti.row0 + cb);
                }
            }
            if (!warp_wait(&acc_full[ab], use & 1u, a, &abort_s, lane)) {
                fail(a, &abort_s, 3);
                break;
            }
            fence_after_sync();
            for (int c0 = 16 * hh, si = 0; c0 < ti.n; c0 += 32, ++si) {
                uint32_t d0[16], d1[16];
                const int nc = min(16, ti.n - c0);
                if constexpr (MODE == 0) {
                    tmem_ld16(trow + c0, d0);
                    tmem_ld16(trow + 256 + c0, d1);
                    tmem_ld_wait();
                    const int col = ti.sub * 128 + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j < nc) {
                            const float v = silu_mul(__uint_as_float(d0[j]), __uint_as_float(d1[j]));
                            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                            const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));
                            const size_t off = h_offset(a.h_rows, ti.hrow0 + c0 + j, col);
                            a.h_hi[off] = __bfloat16_as_ushort(hi);
                            a.h_lo[off] = __bfloat16_as_ushort(lo);
                        }
                    }
                } else {
                    tmem_ld16(trow + ab * 256 + c0, d0);
                    tmem_ld16(trow + ab * 256 + 128 + c0, d1);
                    tmem_ld_wait();
                    const int tsrc = (si >> 1) ? tokB : tokA;
                    const float wsrc = (si >> 1) ? wB : wA;
                    float* y0 = a.y + ti.sub * 256 + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tj = __shfl_sync(kFullMask, tsrc, 16 * (si & 1) + j);
                        const float wj = __shfl_sync(kFullMask, wsrc, 16 * (si & 1) + j);
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
            if (lane == 0) bar_arrive(&acc_empty[ab]);
        }
    } else {
        // ---------------------------------------------------------- dequantisers
        constexpr int D = RG::kSlots;
        const int dt = tid - 32 * kDqWarp0, r = dt >> 1, hf = dt & 1;
        const uint32_t codes0 = smem0 + RG::kOffCodes;
        // issue side: the (tile, k-block) D k-blocks ahead of the one consumed
        Tiles<MODE> ahead;
        bool ahas = ahead.first(a, n_tiles);
        int akb = 0, anb = ahas ? ahead.kblocks(a) : 0;
        const uint8_t *aq = nullptr, *asb = nullptr;
        if (ahas) code_src<MODE, BITS>(a, ahead.cur, r, hf, aq, asb);
        uint32_t iss = 0;
        auto issue = [&](uint32_t slot) {
            if (ahas) {
                const uint32_t base = codes0 + slot * RG::kSlotBytes;
#pragma unroll
                for (int p = 0; p < RG::kParts; ++p)
                    cp_async16(base + (p * kDqThreads + dt) * 16, aq + (size_t)akb * 8 * BITS + 16 * p);
                cp_async4(base + RG::kParts * kDqThreads * 16 + dt * 4, asb + (size_t)akb * 4);
                ++iss;
                if (++akb == anb) {
                    akb = 0;
                    ahas = ahead.next(a, n_tiles);
                    if (ahas) {
                        anb = ahead.kblocks(a);
                        code_src<MODE, BITS>(a, ahead.cur, r, hf, aq, asb);
                    }
                }
            }
            cp_async_commit();
        };
#pragma unroll 1
        for (int j = 0; j < D; ++j) issue(j);
        const uint64_t m2 = f2(__float_as_uint(-8388608.0f), __float_as_uint(-8388608.0f));
        const int m = r >> 7, rr = r & 127;
        for (uint32_t it = 0; it < iss; ++it) {
            cp_async_wait<D - 1>();
            const uint32_t slot = it % D;
            const uint32_t base = codes0 + slot * RG::kSlotBytes;
            const uint32_t sbw = lds32(base + RG::kParts * kDqThreads * 16 + dt * 4);
            const float s = __half2float(__ushort_as_half((unsigned short)(sbw & 0xffffu)));
            const float b = __half2float(__ushort_as_half((unsigned short)(sbw >> 16)));
            const uint64_t s2 = f2(__float_as_uint(s), __float_as_uint(s));
            const uint64_t b2 = f2(__float_as_uint(b), __float_as_uint(b));
            uint4 o[4];
            if (BITS == 4) {
                const uint4 w = lds128(base + dt * 16);
                float cb;
                if (shifted_bias(s, b, cb)) {
                    const uint64_t c2 = f2(__float_as_uint(cb), __float_as_uint(cb));
                    o[0] = dq8_int4_fast(w.x, s2, c2);
                    o[1] = dq8_int4_fast(w.y, s2, c2);
                    o[2] = dq8_int4_fast(w.z, s2, c2);
                    o[3] = dq8_int4_fast(w.w, s2, c2);
                } else {
                    o[0] = dq8_int4(w.x, s2, b2, m2);
                    o[1] = dq8_int4(w.y, s2, b2, m2);
                    o[2] = dq8_int4(w.z, s2, b2, m2);
                    o[3] = dq8_int4(w.w, s2, b2, m2);
                }
            } else {
                const uint4 w0 = lds128(base + dt * 16), w1 = lds128(base + (kDqThreads + dt) * 16);
                o[0] = dq8_int8(w0.x, w0.y, s2, b2, m2);
                o[1] = dq8_int8(w0.z, w0.w, s2, b2, m2);
                o[2] = dq8_int8(w1.x, w1.y, s2, b2, m2);
                o[3] = dq8_int8(w1.z, w1.w, s2, b2, m2);
            }
            const uint32_t sa = it % kAStages;
            // stage sa was last read by the MMAs of k-block it - kAStages
            if (it >= kAStages &&
                !warp_wait(&kb_done[(it - kAStages) % kDone], ((it - kAStages) / kDone) & 1u, a, &abort_s, lane)) {
                fail(a, &abort_s, 1);
                break;
            }
            const uint32_t tile = smem0 + RG::kOffA + sa * kStageBytes + m * kTileBytes;
#pragma unroll
            for (int i = 0; i < 4; ++i) sts128(tile + swz_chunk(rr, 4 * hf + i), o[i]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(&a_full[sa]);
            // this slot's codes are consumed: refill it D k-blocks ahead
            issue(slot);
        }
        cp_async_wait_all();
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE, int BITS>
cudaError_t launch_mode(const CUtensorMap& map, const CUtensorMap& smap, const GemmArgs& g, int grid, cudaStream_t st) {
    const size_t smem = (size_t)Ring<BITS>::kSmem + 1024;
    cudaError_t e = smem_limit(reinterpret_cast<const void*>(grouped_gemm_kernel<MODE, BITS>), (int)smem);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<MODE, BITS><<<grid, kThreads, smem, st>>>(map, smap, g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gemm(int mode, const Shapes& s, const PrefillScratch& p, const PrefillArgs& a,
                                cudaStream_t st) {
    GemmArgs g{};
    g.H = s.hidden;
    g.E = s.n_experts;
    g.T = a.T;
    g.inter = s.inter;
    g.shared_inter = a.shared_blob ? s.shared_inter : 0;
    g.per = mode == 0 ? s.h_stride / 128 : s.hidden / 256;
    g.h_rows = p.h_rows;
    g.chunks = mode == 0 ? p.chunks : p.chunks1;
    g.n_chunks = p.n_chunks;
    g.tok_sorted = p.tok_sorted;
    g.w_sorted = p.w_sorted;
    g.h_hi = p.h_hi;
    g.h_lo = p.h_lo;
    g.sigma = p.sigma;
    g.y = a.y;
    g.status = p.status_dev;
    g.timeout_ns = a.timeout_ns;
    const CUtensorMap &m = p.x_map, &ms = p.xs_map;
    if (mode == 0) return s.bits == 4 ? launch_mode<0, 4>(m, ms, g, p.sms, st) : launch_mode<0, 8>(m, ms, g, p.sms, st);
    return s.bits == 4 ? launch_mode<1, 4>(m, ms, g, p.sms, st) : launch_mode<1, 8>(m, ms, g, p.sms, st);
}

}  // namespace moe
