// stack_kernel.cu -- the persistent decode-stack kernel for sm_103a.
//
// One cooperative launch runs B tokens (B <= 8) through every MoE layer of a
// call, one CTA per SM.  Per layer and CTA:
//   A  x = renorm(y of the previous layer) (or the input) and its block-
//      fixed-point digits; router logits of this CTA's experts and the shared
//      expert's gate/up rows of this CTA, both from shared memory prefetched
//      during the previous layer.
//   B  top-k + routing weights + dispatch lists (computed redundantly, the
//      same bits in every CTA); this CTA's share of the routed gate/up rows
//      and of every active expert's down rows are fetched with cp.async.bulk
//      into shared-memory stages (mbarrier completion); the next layer's
//      router/shared rows are prefetched; gate/up + SwiGLU runs stage by stage.
//   C  this CTA's output rows: every active expert's down rows (already in
//      shared memory) times h, weighted and summed in ascending expert order.
// There is no grid barrier.  Values that cross CTAs (logits, h, y) travel as
// 8-byte words {value, epoch} written with one relaxed store each; a reader
// polls each word until it carries the epoch of the current layer, so the
// data itself is the synchronisation (one L2 round trip instead of a barrier
// and a load).  Each exchange buffer is double-buffered by layer parity; a
// CTA can be at most one layer ahead of any other, because every CTA produces
// y rows and gate/up rows that all others wait for (grid <= min(H, k*I)).
//
// This removes the per-layer launch chain that the Swiftlet pages identify
// as the limit of their decode loop ("dispatch-bound, not IO-bound": article
// section "Capability boundaries", README introduction) and keeps HBM busy
// with bulk copies issued as soon as routing is known.
//
// Every wait is bounded (%globaltimer): a poll or an mbarrier wait that does
// not complete within kWaitNs sets the status word; every CTA then stops at
// its next wait, drains its outstanding copies (again bounded) and exits.  The
// last CTA to leave publishes the status to mapped host memory and advances
// the epoch for the next launch.
#include <algorithm>

#include "gemv.cuh"
#include "stack.h"

namespace moe {
namespace {

constexpr int kST = 256, kSW = kST / 32;
constexpr int kEPT = (1024 + kST - 1) / kST;  // experts per thread in the dispatch scan (E <= 1024)
constexpr int kNSG = 4, kNSD = 2;  // gate/up stages, down stages
constexpr int kMaxB = 8;
constexpr int kNB = kNSG + kNSD + 2;  // mbarriers: G stages, D stages, prefetch[2]
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr int kStatusTimeout = 2;

struct Params {
    int H, E, k, I, Is, norm_topk, B, bits;
    int layer0, n_layers;
    float eps;
    const float* x_in;
    float* y_out;
    float* x_trace;
    int32_t* idx_trace;
    float* y_trace;
    const uint16_t* router_w;
    const float* router_bias;
    const uint16_t* shared_gate;
    const uint8_t* const* dir;
    const uint8_t* shared_pool;
    unsigned long long shared_stride;
    unsigned long long* lg_ll;  // [2][kMaxB*E]
    unsigned long long* h_ll;   // [2][hp*h_stride]
    unsigned long long* y_ll;   // [2][kMaxB*H]
    int h_stride, hp;           // hp = pairs per parity of h_ll
    unsigned* sync;             // [1] CTAs finished, [2] epoch base
    int* status;
    int* status_host;
    // shared-memory plan
    int rE, rS, jn;
    int p_bytes;
    int g_cap, g_unit;
    int d_cap, d_unit, d_rows_bytes;
    int amax, pmax;
    int off_disp, off_part, off_xs, off_xd, off_P, off_G, off_D;
    int smem_bytes;
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sptr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* m) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sptr(m)) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* m, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sptr(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* m, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(sptr(m)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     sptr(dst)),
                 "l"(src), "r"(bytes), "r"(sptr(m))
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_volatile(const int* p) { return *(volatile const int*)p; }

// Abort check for spin loops: the timer and the (shared, global) status word
// are looked at only every 256 spins, so thousands of waiting threads do not
// hammer one L2 line.
__device__ __forceinline__ bool spin_abort(int* status, unsigned& spins, unsigned long long t0) {
    if ((++spins & 255u) != 0u) return false;
    if (gtime() - t0 > kWaitNs) {
        atomicCAS(status, 0, kStatusTimeout);
        return true;
    }
    return ld_volatile(status) != 0;
}

// {value, epoch} words
__device__ __forceinline__ void ll_store(unsigned long long* p, float v, uint32_t ep) {
    const unsigned long long w = ((unsigned long long)ep << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void ll_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Re-poll one {value, epoch} pair until both carry ep (out of line: the slow
// path).  Returns the pair; ok = 0 on timeout or abort.
struct LLPair {
    unsigned long long a, b;
    int ok;
};

__device__ __noinline__ LLPair ll_wait_pair(const unsigned long long* src, uint32_t ep, int* status) {
    const unsigned long long t0 = gtime();
    unsigned spins = 0;
    LLPair r;
    r.ok = 1;
    for (;;) {
        ll_load2(src, r.a, r.b);
        if ((uint32_t)(r.a >> 32) == ep && (uint32_t)(r.b >> 32) == ep) return r;
        if (spin_abort(status, spins, t0)) {
            r.ok = 0;
            return r;
        }
        __nanosleep(32);
    }
}

// Poll n words (n even, 16-byte aligned) until each carries epoch ep; the
// values go to out[].  Loads are issued in batches of 8 before any is checked.
// Returns false on timeout or abort.
__device__ bool ll_read(const unsigned long long* src, int n, uint32_t ep, float* out, int tid,
                                     int nthreads, int* status) {
    for (int base = 2 * tid; base < n; base += 16 * nthreads) {
        unsigned long long a[8], b[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = base + 2 * nthreads * q;
            a[q] = b[q] = (unsigned long long)ep << 32;
            if (i < n) ll_load2(src + i, a[q], b[q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = base + 2 * nthreads * q;
            if ((uint32_t)(a[q] >> 32) != ep || (uint32_t)(b[q] >> 32) != ep) {
                const LLPair r = ll_wait_pair(src + i, ep, status);
                if (!r.ok) return false;
                a[q] = r.a;
                b[q] = r.b;
            }
            if (i < n) {
                out[i] = __uint_as_float((uint32_t)a[q]);
                out[i + 1] = __uint_as_float((uint32_t)b[q]);
            }
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// shared-memory state of one CTA
// ---------------------------------------------------------------------------
struct Disp {
    int32_t idx[kMaxB][16];
    float val[kMaxB][16];
    float w[kMaxB][16];
    float sig[kMaxB];
    float rs[kMaxB];
    int xe[kMaxB];         // block-fixed-point exponent of each token's x
    float xmax[kMaxB];     // max |x| of each token
    uint32_t keys[kMaxB][16];
    float red[2 * kRenormThreads / 32];
    int n_act, n_routed, n_pairs, pad;
};

struct Lists {
    int32_t* act_expert;
    const uint8_t** act_blob;
    int32_t* act_off;
    int32_t* pair_token;
    float* pair_w;
    int32_t* pair_act;
};

__host__ __device__ inline int r16i(int v) { return (v + 15) / 16 * 16; }

__device__ __forceinline__ Lists lists(uint8_t* base, int amax, int pmax) {
    Lists L;
    uint8_t* p = base + r16i((int)sizeof(Disp));
    L.act_blob = reinterpret_cast<const uint8_t**>(p);
    p += r16i(amax * 8);
    L.act_expert = reinterpret_cast<int32_t*>(p);
    p += r16i(amax * 4);
    L.act_off = reinterpret_cast<int32_t*>(p);
    p += r16i((amax + 1) * 4);
    L.pair_token = reinterpret_cast<int32_t*>(p);
    p += r16i(pmax * 4);
    L.pair_w = reinterpret_cast<float*>(p);
    p += r16i(pmax * 4);
    L.pair_act = reinterpret_cast<int32_t*>(p);
    return L;
}

__host__ __device__ inline int disp_bytes(int amax, int pmax) {
    return r16i((int)sizeof(Disp)) + r16i(amax * 8) + r16i(amax * 4) + r16i((amax + 1) * 4) + 3 * r16i(pmax * 4);
}

struct Waits {
    uint32_t phase;  // bit i = expected parity of mbarrier i
    uint32_t armed;  // bit i = mbarrier i has an outstanding phase
};

// bounded wait on mbarrier i; every thread calls it; false (everywhere) on abort
__device__ bool stage_wait(uint64_t* mb, int i, Waits& w, const Params& p) {
    const uint32_t par = (w.phase >> i) & 1u;
    const unsigned long long t0 = gtime();
    unsigned spins = 0;
    bool ok = true;
    while (!mbar_test(mb + i, par)) {
        if (spin_abort(p.status, spins, t0)) {
            ok = false;
            break;
        }
    }
    if (ok) {
        w.phase ^= 1u << i;
        w.armed &= ~(1u << i);
    }
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// ---------------------------------------------------------------------------
// copies (each stage issued by one lane)
// ---------------------------------------------------------------------------
// prefetch buffer: [router rows rE x 2H][shared gate q rS][shared up q rS][gate sb rS][up sb rS]
__device__ void issue_prefetch(const Params& p, int layer, uint8_t* buf, uint64_t* mb) {
    const int c = blockIdx.x, G = gridDim.x;
    const int e0 = (int)((long long)p.E * c / G), e1 = (int)((long long)p.E * (c + 1) / G);
    const int s0 = (int)((long long)p.Is * c / G), s1 = (int)((long long)p.Is * (c + 1) / G);
    const uint32_t rb = (uint32_t)p.H * 2, qb = (uint32_t)p.H * p.bits / 8, sbb = (uint32_t)p.H / 16;
    mbar_expect(mb, (e1 - e0) * rb + (s1 - s0) * 2 * (qb + sbb));
    if (e1 > e0) bulk_load(buf, p.router_w + ((size_t)layer * p.E + e0) * p.H, (e1 - e0) * rb, mb);
    if (s1 > s0) {
        const uint8_t* blob = p.shared_pool + (size_t)layer * p.shared_stride;
        const BlobLayout L = blob_layout(p.H, p.Is, p.bits);
        uint8_t* d = buf + p.rE * rb;
        const uint32_t n = s1 - s0;
        bulk_load(d, blob + L.gate_q + (size_t)s0 * qb, n * qb, mb);
        bulk_load(d + p.rS * qb, blob + L.up_q + (size_t)s0 * qb, n * qb, mb);
        bulk_load(d + 2 * p.rS * qb, blob + L.gate_sb + (size_t)s0 * sbb, n * sbb, mb);
        bulk_load(d + 2 * p.rS * qb + p.rS * sbb, blob + L.up_sb + (size_t)s0 * sbb, n * sbb, mb);
    }
}

// gate/up stage: [gate q g_cap rows][up q][gate sb][up sb]; units [ua, ub) of this layer's routed rows
__device__ void issue_gateup(const Params& p, const Lists& D, int ua, int ub, uint8_t* stage, uint64_t* mb) {
    const uint32_t qb = (uint32_t)p.H * p.bits / 8, sbb = (uint32_t)p.H / 16;
    mbar_expect(mb, (uint32_t)(ub - ua) * 2 * (qb + sbb));
    const BlobLayout L = blob_layout(p.H, p.I, p.bits);
    for (int u = ua; u < ub;) {
        const int a = u / p.I, r0 = u - a * p.I;
        const int n = min(ub - u, p.I - r0);
        const uint8_t* blob = D.act_blob[a];
        const int o = u - ua;
        bulk_load(stage + (size_t)o * qb, blob + L.gate_q + (size_t)r0 * qb, n * qb, mb);
        bulk_load(stage + (size_t)(p.g_cap + o) * qb, blob + L.up_q + (size_t)r0 * qb, n * qb, mb);
        uint8_t* sbase = stage + (size_t)2 * p.g_cap * qb;
        bulk_load(sbase + (size_t)o * sbb, blob + L.gate_sb + (size_t)r0 * sbb, n * sbb, mb);
        bulk_load(sbase + (size_t)(p.g_cap + o) * sbb, blob + L.up_sb + (size_t)r0 * sbb, n * sbb, mb);
        u += n;
    }
}

// down stage: per active expert a in [aa, ab): [jn rows x row bytes][aligned scale/bias superset]
__device__ void issue_down(const Params& p, const Lists& D, int aa, int ab, int j0, int jn, uint8_t* stage,
                           uint64_t* mb) {
    uint32_t total = 0;
    for (int a = aa; a < ab; ++a) {
        const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
        const uint32_t rb = (uint32_t)cols * p.bits / 8, sbb = (uint32_t)cols / 16;
        const uint32_t s_lo = (j0 * sbb) & ~15u, s_hi = ((j0 + jn) * sbb + 15u) & ~15u;
        total += jn * rb + (s_hi - s_lo);
    }
    mbar_expect(mb, total);
    for (int a = aa; a < ab; ++a) {
        const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
        const uint32_t rb = (uint32_t)cols * p.bits / 8, sbb = (uint32_t)cols / 16;
        const BlobLayout L = blob_layout(p.H, cols, p.bits);
        const uint8_t* blob = D.act_blob[a];
        uint8_t* u = stage + (size_t)(a - aa) * p.d_unit;
        bulk_load(u, blob + L.down_q + (size_t)j0 * rb, jn * rb, mb);
        const uint32_t s_lo = (j0 * sbb) & ~15u, s_hi = ((j0 + jn) * sbb + 15u) & ~15u;
        bulk_load(u + p.d_rows_bytes, blob + L.down_sb + s_lo, s_hi - s_lo, mb);
    }
}

// inclusive block scan of one int per thread (kST threads)
__device__ int block_scan(int v, int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int s = lane < kSW ? wsum[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFullMask, s, off);
            if (lane >= off) s += o;
        }
        if (lane < kSW) wsum[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += wsum[warp - 1];
    __syncthreads();
    return v;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BITS, int NPER>
__global__ void __launch_bounds__(kST, 1) stack_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t mbar[kNB];
    __shared__ int s_wsum[32];
    uint64_t* mbG = mbar;
    uint64_t* mbD = mbar + kNSG;
    uint64_t* mbP = mbar + kNSG + kNSD;

    static_assert(kST == kRenormThreads, "the renormalisation order is defined for kRenormThreads threads");
    static_assert((1024 + kSW - 1) / kSW <= 128, "top-k slices hold at most 128 logits");
    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int H = p.H, E = p.E, k = p.k, B = p.B;
    const int nc = H / CC;  // chunks of a gate/up row
    const uint32_t qb = (uint32_t)H * BITS / 8, sbb = (uint32_t)H / 16;
    Disp* ds = reinterpret_cast<Disp*>(smem + p.off_disp);
    const Lists D = lists(smem + p.off_disp, p.amax, p.pmax);
    float* part = reinterpret_cast<float*>(smem + p.off_part);
    float* xs = reinterpret_cast<float*>(smem + p.off_xs);
    uint32_t* xdw = reinterpret_cast<uint32_t*>(smem + p.off_xd);           // [B][nc][DW]
    int32_t* xS = reinterpret_cast<int32_t*>(xdw + (size_t)B * nc * DW);  // [B][nc]
    uint8_t* Pbuf = smem + p.off_P;
    uint8_t* Gbuf = smem + p.off_G;
    uint8_t* Dbuf = smem + p.off_D;
    const int gstage = p.g_cap * p.g_unit;
    const int dstage = p.d_cap * p.d_unit;
    const size_t h_par = (size_t)p.hp * p.h_stride;

    const uint32_t ep0 = *(volatile const unsigned*)&p.sync[2];
    Waits wt{0u, 0u};
    if (tid == 0) {
        for (int i = 0; i < kNB; ++i) mbar_init(&mbar[i]);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) issue_prefetch(p, p.layer0, Pbuf + (p.layer0 & 1) * p.p_bytes, &mbP[p.layer0 & 1]);
    wt.armed |= 1u << (kNSG + kNSD + (p.layer0 & 1));

    const int j0 = (int)((long long)H * c / G), jn = (int)((long long)H * (c + 1) / G) - j0;
    const int e0 = (int)((long long)E * c / G), ne = (int)((long long)E * (c + 1) / G) - e0;
    const int s0 = (int)((long long)p.Is * c / G), ns = (int)((long long)p.Is * (c + 1) / G) - s0;
    bool ok = true;
    const int lend = p.layer0 + p.n_layers;

    for (int l = p.layer0; l < lend && ok; ++l) {
        const int li = l - p.layer0, par = l & 1;
        const uint32_t ep = ep0 + (uint32_t)li;
        // the next layer's router and shared rows do not depend on this layer:
        // fetch them now (their buffer was last read in the previous layer)
        if (l + 1 < lend) {
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) issue_prefetch(p, l + 1, Pbuf + (par ^ 1) * p.p_bytes, &mbP[par ^ 1]);
            wt.armed |= 1u << (kNSG + kNSD + (par ^ 1));
        }
        // ------------------------------------------------------------ phase A
        if (l == p.layer0) {
            for (int i = tid; i < B * H / 4; i += kST)
                reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(p.x_in) + i);
            __syncthreads();
        } else {
            const bool got = ll_read(p.y_ll + (size_t)(par ^ 1) * kMaxB * H, B * H, ep - 1, xs, tid, kST, p.status);
            if (!__syncthreads_and(got ? 1 : 0)) {
                ok = false;
                break;
            }
        }
        // renormalisation (from the second layer on) and max |x| of each token
        for (int t = 0; t < B; ++t) {
            float my;
            const float r = renorm_block(xs + t * H, H, p.eps, ds->red, &my);
            if (tid == 0) {
                ds->rs[t] = r;
                ds->xmax[t] = l == p.layer0 ? my : __fmul_rn(my, r);  // max|x| = max|y| * r exactly (r > 0)
            }
        }
        __syncthreads();
        if (l != p.layer0)
            for (int i = tid; i < B * H; i += kST) xs[i] = __fmul_rn(xs[i], ds->rs[i / H]);
        // block fixed point of each token: exponent from max |x|, then digits
        {
            if (tid < B) ds->xe[tid] = bfp_exponent(ds->xmax[tid]);
            __syncthreads();
            uint8_t* xb = reinterpret_cast<uint8_t*>(xdw);
            for (int i = tid; i < B * H; i += kST) {
                const int t = i / H, col = i - t * H;
                const int V = bfp_int(xs[i], ds->xe[t]);
                uint32_t d0, d1, d2;
                bfp_digits(V, d0, d1, d2);
                const int ch = col / CC, pos = col - ch * CC;
                uint8_t* cw = xb + ((size_t)(t * nc + ch) * DW) * 4;
                if (BITS == 4) {
                    const int wi = pos >> 3, b8 = pos & 7, odd = b8 & 1, by = b8 >> 1;
                    cw[(6 * wi + 0 + odd) * 4 + by] = (uint8_t)d0;
                    cw[(6 * wi + 2 + odd) * 4 + by] = (uint8_t)d1;
                    cw[(6 * wi + 4 + odd) * 4 + by] = (uint8_t)d2;
                    const int S = __reduce_add_sync(kFullMask, V);
                    if (lane == 0) xS[t * nc + ch] = S;
                } else {
                    const int wi = pos >> 2, by = pos & 3;
                    cw[(3 * wi + 0) * 4 + by] = (uint8_t)d0;
                    cw[(3 * wi + 1) * 4 + by] = (uint8_t)d1;
                    cw[(3 * wi + 2) * 4 + by] = (uint8_t)d2;
                    const int S = lane < 16 ? __reduce_add_sync(0x0000ffffu, V) : __reduce_add_sync(0xffff0000u, V);
                    if ((lane & 15) == 0) xS[t * nc + ch] = S;
                }
            }
        }
        if (p.x_trace && c == 0)
            for (int i = tid; i < B * H; i += kST) p.x_trace[(size_t)li * B * H + i] = xs[i];
        if (!stage_wait(mbar, kNSG + kNSD + par, wt, p)) {
            ok = false;
            break;
        }
        // router rows and shared rows (prefetched), the shared gate
        {
            const uint8_t* pb = Pbuf + par * p.p_bytes;
            const int n_tasks = ne + ns + B;
            for (int task = warp; task < n_tasks; task += kSW) {
                if (task < ne) {
                    const int e = e0 + task;
                    const float bias = p.router_bias[(size_t)l * E + e];
                    const uint16_t* row = reinterpret_cast<const uint16_t*>(pb + (size_t)task * 2 * H);
                    for (int t = 0; t < B; ++t) {
                        const float v = router_logit(row, xs + t * H, H, bias, lane);
                        if (lane == 0) ll_store(p.lg_ll + (size_t)par * kMaxB * E + (size_t)t * E + e, v, ep);
                    }
                } else if (task < ne + ns) {
                    const int rr = task - ne;
                    const uint8_t* sq = pb + (size_t)p.rE * 2 * H;
                    const uint8_t* gq = sq + (size_t)rr * qb;
                    const uint8_t* uq = sq + (size_t)(p.rS + rr) * qb;
                    const uint32_t* gsb = reinterpret_cast<const uint32_t*>(sq + (size_t)2 * p.rS * qb + rr * sbb);
                    const uint32_t* usb =
                        reinterpret_cast<const uint32_t*>(sq + (size_t)2 * p.rS * qb + (p.rS + rr) * sbb);
                    for (int t = 0; t < B; ++t) {
                        XDigits<BITS, NPER> xr;
                        load_xdigits(xr, xdw + (size_t)t * nc * DW, xS + t * nc, nc, lane);
                        float g, u;
                        row_dot_x2(gq, gsb, uq, usb, xr, ds->xe[t], nc, lane, g, u);
                        if (lane == 0)
                            ll_store(p.h_ll + par * h_par + (size_t)(B * k + t) * p.h_stride + s0 + rr,
                                     silu_mul(g, u), ep);
                    }
                } else {
                    const int t = task - ne - ns;
                    const float sg =
                        p.Is > 0 ? shared_gate(p.shared_gate + (size_t)l * H, xs + t * H, H, lane) : 0.0f;
                    if (lane == 0) ds->sig[t] = sg;
                }
            }
        }
        // ------------------------------------------------------------ phase B
        float* s_lg = reinterpret_cast<float*>(Gbuf);  // temp area, before the stage copies
        int* s_cnt = reinterpret_cast<int*>(Gbuf + r16i(B * E * 4));
        unsigned long long* s_msk = reinterpret_cast<unsigned long long*>(Gbuf + r16i(B * E * 4) + r16i(E * 4));
        int* s_scan = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(s_msk) + (size_t)E * 8);
        for (int e = tid; e < E; e += kST) {
            s_cnt[e] = 0;
            s_msk[e] = 0ull;
        }
        {
            const bool got = ll_read(p.lg_ll + (size_t)par * kMaxB * E, B * E, ep, s_lg, tid, kST, p.status);
            if (!__syncthreads_and(got ? 1 : 0)) {
                ok = false;
                break;
            }
        }
        // top-k in two levels: every warp selects the k best of its slice of each
        // token's logits, then one warp per token selects among the candidates
        {
            uint32_t* ck = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(s_scan) + r16i(E * 4));
            int32_t* ci = reinterpret_cast<int32_t*>(ck + kMaxB * kSW * 16);
            uint32_t* kk_all = reinterpret_cast<uint32_t*>(ci + kMaxB * kSW * 16);
            int32_t* ii_all = reinterpret_cast<int32_t*>(kk_all + kSW * 128);
            const int eb = (int)((long long)E * warp / kSW), ee = (int)((long long)E * (warp + 1) / kSW);
            const int nsl = ee - eb, kk = min(k, nsl);
            for (int t = 0; t < B; ++t) {
                uint32_t keys[4];
                int32_t ids[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int i = lane + 32 * m;
                    keys[m] = i < nsl ? order_key(s_lg[t * E + eb + i]) : 0u;
                    ids[m] = eb + i;
                }
                // stage the slice as candidate arrays for warp_select
                uint32_t* sk = ck + (t * kSW + warp) * 16;
                int32_t* si = ci + (t * kSW + warp) * 16;
                uint32_t* wk = kk_all + warp * 128;
                int32_t* wi = ii_all + warp * 128;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    wk[lane + 32 * m] = keys[m];
                    wi[lane + 32 * m] = ids[m];
                }
                __syncwarp();
                warp_select<4>(wk, wi, nsl, kk, lane, si, sk);
                if (lane >= kk && lane < 16) {
                    sk[lane] = 0u;
                    si[lane] = 0x7fffffff;
                }
                __syncwarp();
            }
            __syncthreads();
            if (warp < B) {
                const int t = warp;
                warp_select<(kSW * 16 + 31) / 32>(ck + t * kSW * 16, ci + t * kSW * 16, kSW * 16, k, lane, ds->idx[t],
                                                   ds->keys[t]);
                if (lane < k) ds->val[t][lane] = s_lg[t * E + ds->idx[t][lane]];
                __syncwarp();
                topk_weights(s_lg + t * E, E, k, p.norm_topk, lane, ds->val[t], ds->w[t]);
            }
            __syncthreads();
        }
        if (p.idx_trace && c == 0 && tid < B * k) p.idx_trace[(size_t)li * B * k + tid] = ds->idx[tid / k][tid % k];
        for (int q = tid; q < B * k; q += kST) {
            const int e = ds->idx[q / k][q % k], t = q / k;
            atomicAdd(&s_cnt[e], 1);
            atomicOr(&s_msk[e], 1ull << t);
        }
        __syncthreads();
        {
            int v[kEPT], tot = 0;
#pragma unroll
            for (int q = 0; q < kEPT; ++q) {
                const int e = tid * kEPT + q;
                v[q] = e < E ? ((s_cnt[e] << 16) | (s_cnt[e] > 0 ? 1 : 0)) : 0;
                tot += v[q];
            }
            const int incl = block_scan(tot, s_wsum);
            int run = incl - tot;
#pragma unroll
            for (int q = 0; q < kEPT; ++q) {
                const int e = tid * kEPT + q;
                if (e < E) s_scan[e] = run;
                run += v[q];
            }
            if (tid == kST - 1) {
                ds->n_routed = incl & 0xffff;
                ds->n_pairs = B * k + (p.Is > 0 ? B : 0);
                ds->n_act = (incl & 0xffff) + (p.Is > 0 ? 1 : 0);
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kST) {
            if (s_cnt[e] > 0) {
                const int a = s_scan[e] & 0xffff;
                D.act_expert[a] = e;
                D.act_blob[a] = p.dir[(size_t)l * E + e];
                D.act_off[a] = s_scan[e] >> 16;
            }
        }
        for (int q = tid; q < B * k; q += kST) {
            const int e = ds->idx[q / k][q % k], t = q / k;
            const int rank = __popcll(s_msk[e] & ((1ull << t) - 1ull));
            const int pr = (s_scan[e] >> 16) + rank;
            D.pair_token[pr] = t;
            D.pair_w[pr] = ds->w[t][q % k];
            D.pair_act[pr] = s_scan[e] & 0xffff;
        }
        if (tid == 0) {
            const int nr = ds->n_routed;
            if (p.Is > 0) {
                D.act_expert[nr] = -1;
                D.act_blob[nr] = p.shared_pool + (size_t)l * p.shared_stride;
                D.act_off[nr] = B * k;
                D.act_off[nr + 1] = B * k + B;
            } else {
                D.act_off[nr] = B * k;
            }
        }
        if (p.Is > 0 && tid < B) {
            D.pair_token[B * k + tid] = tid;
            D.pair_w[B * k + tid] = ds->sig[tid];
            D.pair_act[B * k + tid] = ds->n_routed;
        }
        fence_proxy_async();  // generic accesses to the stages precede the bulk writes below
        __syncthreads();
        const int n_act = ds->n_act, n_pairs = ds->n_pairs;
        const int U = ds->n_routed * p.I;
        const int u0 = (int)((long long)U * c / G), u1 = (int)((long long)U * (c + 1) / G);
        const int mine = u1 - u0;
        const int gcs = mine > 0 ? min(p.g_cap, (mine + kNSG - 1) / kNSG) : 1;
        const int n_gch = (mine + gcs - 1) / gcs;
        const int dcs = min(p.d_cap, (n_act + kNSD - 1) / kNSD);
        const int n_dch = jn > 0 ? (n_act + dcs - 1) / dcs : 0;
        // one issuing lane per stage: warps 0..3 gate/up, 4..5 down, 6 next-layer prefetch
        if (lane == 0) {
            if (warp < kNSG) {
                if (warp < n_gch)
                    issue_gateup(p, D, u0 + warp * gcs, min(u1, u0 + (warp + 1) * gcs), Gbuf + (size_t)warp * gstage,
                                 &mbG[warp]);
            } else if (warp < kNSG + kNSD) {
                const int s = warp - kNSG;
                if (s < n_dch)
                    issue_down(p, D, s * dcs, min(n_act, (s + 1) * dcs), j0, jn, Dbuf + (size_t)s * dstage, &mbD[s]);
            }
        }
        for (int s = 0; s < min(n_gch, kNSG); ++s) wt.armed |= 1u << s;
        for (int s = 0; s < min(n_dch, kNSD); ++s) wt.armed |= 1u << (kNSG + s);
        // gate/up + SwiGLU, stage by stage
        unsigned long long* hll = p.h_ll + par * h_par;
        for (int ch = 0; ch < n_gch; ++ch) {
            const int s = ch % kNSG;
            if (!stage_wait(mbar, s, wt, p)) {
                ok = false;
                break;
            }
            const uint8_t* st = Gbuf + (size_t)s * gstage;
            const int ua = u0 + ch * gcs, n = min(u1, ua + gcs) - ua;
            const int w0 = n * warp / kSW, w1 = n * (warp + 1) / kSW;
            int cur_t = -1;
            XDigits<BITS, NPER> xr;
            for (int o = w0; o < w1; ++o) {
                const int u = ua + o, a = u / p.I, r = u - a * p.I;
                const uint8_t* gq = st + (size_t)o * qb;
                const uint8_t* uq = st + (size_t)(p.g_cap + o) * qb;
                const uint32_t* gsb = reinterpret_cast<const uint32_t*>(st + (size_t)2 * p.g_cap * qb + o * sbb);
                const uint32_t* usb =
                    reinterpret_cast<const uint32_t*>(st + (size_t)2 * p.g_cap * qb + (p.g_cap + o) * sbb);
                for (int pr = D.act_off[a]; pr < D.act_off[a + 1]; ++pr) {
                    const int t = D.pair_token[pr];
                    if (t != cur_t) {
                        load_xdigits(xr, xdw + (size_t)t * nc * DW, xS + t * nc, nc, lane);
                        cur_t = t;
                    }
                    float g, uu;
                    row_dot_x2(gq, gsb, uq, usb, xr, ds->xe[t], nc, lane, g, uu);
                    if (lane == 0) ll_store(hll + (size_t)pr * p.h_stride + r, silu_mul(g, uu), ep);
                }
            }
            fence_proxy_async();
            __syncthreads();
            if (ch + kNSG < n_gch) {
                if (tid == 0)
                    issue_gateup(p, D, u0 + (ch + kNSG) * gcs, min(u1, u0 + (ch + kNSG + 1) * gcs),
                                 Gbuf + (size_t)s * gstage, &mbG[s]);
                wt.armed |= 1u << s;
            }
        }
        if (!ok) break;
        // ------------------------------------------------------------ phase C
        const int half = (jn + 1) / 2;
        for (int ch = 0; ch < n_dch && ok; ++ch) {
            const int s = ch % kNSD;
            if (!stage_wait(mbar, kNSG + s, wt, p)) {
                ok = false;
                break;
            }
            const uint8_t* st = Dbuf + (size_t)s * dstage;
            const int aa = ch * dcs, ab = min(n_act, aa + dcs);
            const int pa = D.act_off[aa], pb = D.act_off[ab];
            bool okc = true;
            // tasks: (pair, half of this CTA's rows)
            for (int task = warp; task < 2 * (pb - pa); task += kSW) {
                const int pr = pa + (task >> 1), hf = task & 1;
                const int a = D.pair_act[pr];
                const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
                const uint32_t rb = (uint32_t)cols * BITS / 8, dsb = (uint32_t)cols / 16;
                const uint8_t* unit = st + (size_t)(a - aa) * p.d_unit;
                const uint8_t* sbase = unit + p.d_rows_bytes + ((j0 * dsb) & 15u);
                // h of the pair: lane L polls its chunk's CC words, 8 loads in flight at a time
                HF<BITS> hd;
                float* hv = hd.v;
                const bool mine_c = lane < cols / CC;
                const unsigned long long* src = hll + (size_t)pr * p.h_stride + lane * CC;
#pragma unroll
                for (int i0 = 0; i0 < CC; i0 += 16) {
                    unsigned long long wa[8], wb[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        wa[q] = wb[q] = (unsigned long long)ep << 32;
                        if (mine_c) ll_load2(src + i0 + 2 * q, wa[q], wb[q]);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (okc && ((uint32_t)(wa[q] >> 32) != ep || (uint32_t)(wb[q] >> 32) != ep)) {
                            const LLPair r = ll_wait_pair(src + i0 + 2 * q, ep, p.status);
                            okc = r.ok != 0;
                            wa[q] = r.a;
                            wb[q] = r.b;
                        }
                        hv[i0 + 2 * q] = mine_c ? __uint_as_float((uint32_t)wa[q]) : 0.0f;
                        hv[i0 + 2 * q + 1] = mine_c ? __uint_as_float((uint32_t)wb[q]) : 0.0f;
                    }
                }
                if (__any_sync(kFullMask, !okc)) {
                    okc = false;
                    break;
                }
                hf_sum(hd);
                const float wp = D.pair_w[pr];
                const int jb = hf * half, je = min(jn, jb + half);
                int jj = jb;
                for (; jj + 1 < je; jj += 2) {
                    float v0, v1;
                    row_dot_h2<BITS>(unit + (size_t)jj * rb, reinterpret_cast<const uint32_t*>(sbase + (size_t)jj * dsb),
                                     unit + (size_t)(jj + 1) * rb,
                                     reinterpret_cast<const uint32_t*>(sbase + (size_t)(jj + 1) * dsb), hd, cols, lane, v0,
                                     v1);
                    if (lane == 0) {
                        part[(size_t)pr * p.jn + jj] = __fmul_rn(wp, v0);
                        part[(size_t)pr * p.jn + jj + 1] = __fmul_rn(wp, v1);
                    }
                }
                if (jj < je) {
                    const float v = row_dot_h<BITS>(unit + (size_t)jj * rb,
                                                    reinterpret_cast<const uint32_t*>(sbase + (size_t)jj * dsb), hd,
                                                    cols, lane);
                    if (lane == 0) part[(size_t)pr * p.jn + jj] = __fmul_rn(wp, v);
                }
            }
            fence_proxy_async();
            if (!__syncthreads_and(okc ? 1 : 0)) {
                ok = false;
                break;
            }
            if (ch + kNSD < n_dch) {
                if (tid == 0)
                    issue_down(p, D, (ch + kNSD) * dcs, min(n_act, (ch + kNSD + 1) * dcs), j0, jn,
                               Dbuf + (size_t)s * dstage, &mbD[s]);
                wt.armed |= 1u << (kNSG + s);
            }
        }
        if (!ok) break;
        // y rows of this CTA: ascending expert order per token
        for (int i = tid; i < B * jn; i += kST) {
            const int t = i / jn, jj = i - t * jn;
            float acc = 0.0f;
            for (int pr = 0; pr < n_pairs; ++pr)
                if (D.pair_token[pr] == t) acc = __fadd_rn(acc, part[(size_t)pr * p.jn + jj]);
            const size_t o = (size_t)t * H + j0 + jj;
            ll_store(p.y_ll + (size_t)par * kMaxB * H + o, acc, ep);
            if (l == lend - 1) p.y_out[o] = acc;
            if (p.y_trace) p.y_trace[(size_t)li * B * H + o] = acc;
        }
        __syncthreads();
    }
    // drain outstanding copies (bounded) before the CTA's shared memory goes away
    __syncthreads();
    for (int i = 0; i < kNB; ++i) {
        if (wt.armed & (1u << i)) {
            const uint32_t par = (wt.phase >> i) & 1u;
            const unsigned long long t0 = gtime();
            while (!mbar_test(&mbar[i], par) && gtime() - t0 < kWaitNs) {
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.sync[1], 1u);
        if (prev == (unsigned)G - 1) {
            uint32_t next = ep0 + (uint32_t)p.n_layers + 1u;
            if (next == 0u) next = 1u;
            p.sync[2] = next;
            p.sync[1] = 0u;
            const int stt = ld_volatile(p.status);
            if (stt) *(volatile int*)p.status_host = stt;
            __threadfence_system();
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int nper_of(int hidden, int bits) {
    const int nchunk = hidden * bits / 128;
    return (nchunk + 31) / 32;
}

bool plan(const Shapes& sh, int B, int grid, int max_smem, Params& p) {
    const int H = sh.hidden, E = sh.n_experts, k = sh.top_k, bits = sh.bits;
    auto r128 = [](long long v) { return (int)((v + 127) / 128 * 128); };
    const int G = grid;
    p.rE = (E + G - 1) / G;
    p.rS = (sh.shared_inter + G - 1) / G;
    p.jn = (H + G - 1) / G;
    const int qb = H * bits / 8, sbb = H / 16;
    p.p_bytes = r128((long long)p.rE * 2 * H + (long long)p.rS * 2 * (qb + sbb));
    p.g_unit = 2 * (qb + sbb);
    const int cmax = std::max(sh.inter, sh.shared_inter);
    const int rbmax = cmax * bits / 8, sbmax = cmax / 16;
    p.d_rows_bytes = r16i(p.jn * rbmax);
    p.d_unit = p.d_rows_bytes + r16i(p.jn * sbmax) + 32;  // scale/bias copied as an aligned superset
    p.amax = std::min(E, B * k) + 1;
    p.pmax = B * (k + 1);
    const int CC = bits == 4 ? 32 : 16, DW = bits == 4 ? 24 : 12;
    const int nc = H / CC;
    int off = 0;
    p.off_disp = off;
    off += r128(disp_bytes(p.amax, p.pmax));
    p.off_part = off;
    off += r128((long long)p.pmax * p.jn * 4);
    p.off_xs = off;
    off += r128((long long)B * H * 4);
    p.off_xd = off;
    off += r128((long long)B * nc * (DW + 1) * 4);
    p.off_P = off;
    off += 2 * p.p_bytes;
    const int budget = max_smem - 1024;  // static shared memory of the kernel
    int left = budget - off;
    p.d_cap = std::max(1, std::min((k + 2 + kNSD - 1) / kNSD, left / 3 / (kNSD * p.d_unit)));
    const int dbytes = kNSD * p.d_cap * p.d_unit;
    left -= dbytes;
    p.g_cap = left / (kNSG * p.g_unit);
    if (p.g_cap < 1) return false;
    p.off_G = off;
    off += kNSG * p.g_cap * p.g_unit;
    off = r128(off);
    p.off_D = off;
    off += dbytes;
    p.smem_bytes = off;
    // the top-k temp area lives in the gate/up stages
    const long long tmp =
        r16i(B * E * 4) + r16i(E * 4) + (long long)E * 8 + r16i(E * 4) + 2LL * kMaxB * kSW * 16 * 4 + 2LL * kSW * 128 * 4;
    if (tmp > (long long)kNSG * p.g_cap * p.g_unit) return false;
    return off <= budget;
}

template <int BITS, int NPER>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&stack_kernel<BITS, NPER>);
}

void* select_kernel(int bits, int nper) {
    if (bits == 4) {
        if (nper == 1) return kernel_ptr<4, 1>();
        if (nper == 2) return kernel_ptr<4, 2>();
    } else {
        if (nper == 1) return kernel_ptr<8, 1>();
        if (nper == 2) return kernel_ptr<8, 2>();
        if (nper == 4) return kernel_ptr<8, 4>();
    }
    return nullptr;
}

}  // namespace

int stack_alloc(StackScratch& s, const Shapes& sh, int n_layers, int max_batch, int device, std::string& err) {
    (void)n_layers;
    (void)max_batch;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        err = "cudaGetDeviceProperties failed";
        return MOE_ECUDA;
    }
    // every CTA must own y rows and routed gate/up rows in every layer (see the header comment)
    s.grid = std::min(prop.multiProcessorCount, std::min(sh.hidden, sh.top_k * sh.inter));
    s.max_smem = (int)prop.sharedMemPerBlockOptin;
    s.hp = kMaxB * (sh.top_k + 1);
    const size_t bytes_lg = sizeof(unsigned long long) * 2 * kMaxB * (size_t)sh.n_experts;
    const size_t bytes_y = sizeof(unsigned long long) * 2 * kMaxB * (size_t)sh.hidden;
    const size_t bytes_h = sizeof(unsigned long long) * 2 * (size_t)s.hp * sh.h_stride;
    if (cudaMalloc(&s.lg_ll, bytes_lg) != cudaSuccess || cudaMalloc(&s.y_ll, bytes_y) != cudaSuccess ||
        cudaMalloc(&s.h_ll, bytes_h) != cudaSuccess || cudaMalloc(&s.sync, 4 * sizeof(unsigned)) != cudaSuccess ||
        cudaMalloc(&s.status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        err = "cudaMalloc of the stack scratch failed";
        return MOE_ENOMEM;
    }
    if (cudaHostAlloc(&s.status_host, sizeof(int), cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(&s.status_host_dev, s.status_host, 0) != cudaSuccess) {
        cudaGetLastError();
        err = "mapped status word allocation failed";
        return MOE_ENOMEM;
    }
    *s.status_host = 0;
    const unsigned init[4] = {0u, 0u, 1u, 0u};  // epoch base starts at 1 (zeroed buffers carry epoch 0)
    if (cudaMemset(s.lg_ll, 0, bytes_lg) != cudaSuccess || cudaMemset(s.y_ll, 0, bytes_y) != cudaSuccess ||
        cudaMemset(s.h_ll, 0, bytes_h) != cudaSuccess ||
        cudaMemcpy(s.sync, init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(s.status, 0, sizeof(int)) != cudaSuccess) {
        err = "stack scratch initialisation failed";
        return MOE_ECUDA;
    }
    const int nper = nper_of(sh.hidden, sh.bits);
    if (void* f = select_kernel(sh.bits, nper)) {
        if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, s.max_smem - 1024) != cudaSuccess) {
            cudaGetLastError();
            s.grid = 0;  // persistent kernel unavailable; per-layer kernels serve the stack
        }
    }
    return MOE_OK;
}

void stack_free(StackScratch& s) {
    cudaFree(s.lg_ll);
    cudaFree(s.y_ll);
    cudaFree(s.h_ll);
    cudaFree(s.sync);
    cudaFree(s.status);
    if (s.status_host) cudaFreeHost(s.status_host);
    s = StackScratch{};
}

bool stack_supported(const Shapes& sh, const StackScratch& s, int B) {
    if (s.grid <= 0 || !s.lg_ll || B < 1 || B > kMaxB || sh.hidden > 2048 || sh.top_k > 16) return false;
    const int nper = nper_of(sh.hidden, sh.bits);
    if (!select_kernel(sh.bits, nper)) return false;
    const int cmax = std::max(sh.inter, sh.shared_inter);
    if (cmax * sh.bits / 128 > 32) return false;  // one chunk per lane on down rows
    Params p{};
    return plan(sh, B, s.grid, s.max_smem, p);
}

int stack_last_status(const StackScratch& s) { return s.status_host ? *(volatile int*)s.status_host : 0; }

cudaError_t launch_stack(const Shapes& sh, StackScratch& s, const StackArgs& a, cudaStream_t st) {
    Params p{};
    if (!plan(sh, a.B, s.grid, s.max_smem, p)) return cudaErrorInvalidValue;
    p.H = sh.hidden, p.E = sh.n_experts, p.k = sh.top_k, p.I = sh.inter, p.Is = sh.shared_inter;
    p.norm_topk = sh.norm_topk, p.B = a.B, p.bits = sh.bits;
    p.layer0 = a.layer0, p.n_layers = a.n_layers, p.eps = a.eps;
    p.x_in = a.x, p.y_out = a.y, p.x_trace = a.x_trace, p.idx_trace = a.idx_trace, p.y_trace = a.y_trace;
    p.router_w = a.router_w, p.router_bias = a.router_bias, p.shared_gate = a.shared_gate, p.dir = a.dir;
    p.shared_pool = a.shared_pool, p.shared_stride = a.shared_stride;
    p.lg_ll = s.lg_ll, p.h_ll = s.h_ll, p.y_ll = s.y_ll, p.h_stride = sh.h_stride, p.hp = s.hp;
    p.sync = s.sync, p.status = s.status, p.status_host = s.status_host_dev;
    void* f = select_kernel(sh.bits, nper_of(sh.hidden, sh.bits));
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(f, dim3(s.grid), dim3(kST), args, (size_t)p.smem_bytes, st);
}

}  // namespace moe
