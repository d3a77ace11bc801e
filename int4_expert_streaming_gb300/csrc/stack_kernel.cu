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
// Streaming contexts use it with the host's slot pool behind it.  A launch's
// first layer takes its routing from a buffer (rin_*: written by the route
// kernels or by the launch before) instead of computing it.  Every later
// layer publishes its routing to mapped host memory, where the host runs the
// pool's bookkeeping in order, and then checks its experts against the
// device directory: when all are resident the launch simply goes on; at the
// first layer with an absent expert it leaves that layer's x and routing for
// the next launch, marks the layer as stopped and exits.  The host copies the
// missing experts on its side stream and launches again from that layer, so
// it is on the critical path only for layers that miss.
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
    // streaming launch (rin_idx non-null): the first layer's routing is given
    // (idx, w [B*k], sigma [B]); every later layer's routing is published to
    // mapped host memory (pub_idx row l, then pub_ready[l] = *pub_epoch).  A
    // layer whose experts are all resident (non-null directory entries) runs
    // on; at the first one that is not, the launch writes that layer's x and
    // routing for the next launch (x_out [B*H], rout_* like rin_*), sets
    // pub_stop[l] = *pub_epoch before the ready word, and stops.
    const int32_t* rin_idx;
    const float* rin_w;
    const float* rin_sig;
    float* x_out;
    int32_t* rout_idx;
    float* rout_w;
    float* rout_sig;
    int32_t* pub_idx;
    int pub_stride;
    volatile uint32_t* pub_ready;
    volatile uint32_t* pub_stop;
    const volatile uint32_t* pub_epoch;
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

// Poll the first `cols` words of rows row0 .. row0+nrows-1 of an exchange
// buffer (row stride `stride` words) until each carries epoch ep; the values
// go to dst[(row - row0) * stride + col].  cols and stride are even.  All
// threads take part; each polls batches of 8 word pairs, re-issuing the whole
// batch until every pair carries ep (a rolled loop: this runs once per
// exchange and its code size matters more than its arithmetic).  Returns false
// on timeout or abort.
__device__ bool ll_read_rows(const unsigned long long* base, int row0, int nrows, int stride, int cols, uint32_t ep,
                             float* dst, int tid, int nthreads, int* status) {
    const int n = nrows * cols;
    const unsigned long long* b0 = base + (size_t)row0 * stride;
    for (int b = 2 * tid; b < n; b += 16 * nthreads) {
        int off[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = b + 2 * nthreads * q;
            const int r = i / cols;
            off[q] = i < n ? r * stride + (i - r * cols) : -1;
        }
        unsigned long long a[8], c[8];
        unsigned spins = 0;
        unsigned long long t0 = 0;
        for (;;) {
            bool all = true;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                a[q] = c[q] = (unsigned long long)ep << 32;
                if (off[q] >= 0) ll_load2(b0 + off[q], a[q], c[q]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                all = all && (uint32_t)(a[q] >> 32) == ep && (uint32_t)(c[q] >> 32) == ep;
            if (all) break;
            if (!t0) t0 = gtime();
            if (spin_abort(status, spins, t0)) return false;
            __nanosleep(32);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (off[q] >= 0) {
                dst[off[q]] = __uint_as_float((uint32_t)a[q]);
                dst[off[q] + 1] = __uint_as_float((uint32_t)c[q]);
            }
        }
    }
    return true;
}

// n contiguous words (n even)
__device__ __forceinline__ bool ll_read(const unsigned long long* src, int n, uint32_t ep, float* out, int tid,
                                        int nthreads, int* status) {
    return ll_read_rows(src, 0, 1, n, n, ep, out, tid, nthreads, status);
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

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BITS, int NPER>
__global__ void __launch_bounds__(kST, 1) stack_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t mbar[kNB];
    uint64_t* mbG = mbar;
    uint64_t* mbD = mbar + kNSG;
    uint64_t* mbP = mbar + kNSG + kNSD;

    static_assert(kST == kRenormThreads, "the renormalisation order is defined for kRenormThreads threads");
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
        const bool given = l == p.layer0 && p.rin_idx != nullptr;  // routing from rin_*
        const bool streamed = l > p.layer0 && p.rin_idx != nullptr;  // routing published, residency checked
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
        // x = y * r (from the second layer on) and its block-fixed-point digits,
        // one pass: a warp covers 32 consecutive columns of one token (one int4
        // chunk, two int8 chunks); the digit words are assembled with shuffles
        // in the layout of bfp_chunk and stored whole.
        {
            if (tid < B) ds->xe[tid] = bfp_exponent(ds->xmax[tid]);
            __syncthreads();
            const bool scale = l != p.layer0;
            for (int i = tid; i < B * H; i += kST) {
                const int t = i / H, col = i - t * H;
                float xv = xs[i];
                if (scale) {
                    xv = __fmul_rn(xv, ds->rs[t]);
                    xs[i] = xv;
                }
                const int V = bfp_int(xv, ds->xe[t]);
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
        __syncthreads();
        if (p.x_trace && c == 0)
            for (int i = tid; i < B * H; i += kST) p.x_trace[(size_t)li * B * H + i] = xs[i];
        if (!stage_wait(mbar, kNSG + kNSD + par, wt, p)) {
            ok = false;
            break;
        }
        // router rows and shared rows (prefetched), the shared gate
        {
            const uint8_t* pb = Pbuf + par * p.p_bytes;
            // given routing: no router rows and no shared gate
            const int na = given ? 0 : ne, nb = ns;
            const int n_tasks = na + nb + (given ? 0 : B);
            for (int task = warp; task < n_tasks; task += kSW) {
                if (task < na) {
                    const int e = e0 + task;
                    const float bias = p.router_bias[(size_t)l * E + e];
                    const uint16_t* row = reinterpret_cast<const uint16_t*>(pb + (size_t)task * 2 * H);
                    for (int t = 0; t < B; ++t) {
                        const float v = router_logit(row, xs + t * H, H, bias, lane);
                        if (lane == 0) ll_store(p.lg_ll + (size_t)par * kMaxB * E + (size_t)t * E + e, v, ep);
                    }
                } else if (task < na + nb) {
                    const int rr = task - na;
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
                    const int t = task - na - nb;
                    const float sg =
                        p.Is > 0 ? shared_gate(p.shared_gate + (size_t)l * H, xs + t * H, H, lane) : 0.0f;
                    if (lane == 0) ds->sig[t] = sg;
                }
            }
        }
        // ------------------------------------------------------------ phase B
        // Routing by ranks (no serial selection loop).  Temp area in the
        // gate/up stages, before this layer's copies land there.
        const int C = kSW * k;  // top-k candidates per token (k from each warp's slice)
        uint8_t* tp = Gbuf;
        float* s_lg = reinterpret_cast<float*>(tp);  // [B][E] logits
        tp += r16i(B * E * 4);
        uint32_t* c_key = reinterpret_cast<uint32_t*>(tp);  // [B][C]
        tp += r16i(B * C * 4);
        int32_t* c_idx = reinterpret_cast<int32_t*>(tp);  // [B][C], -1 = empty
        if (given) {
            for (int i = tid; i < B * k; i += kST) {
                ds->idx[i / k][i % k] = p.rin_idx[i];
                ds->w[i / k][i % k] = p.rin_w[i];
            }
            if (tid < B) ds->sig[tid] = p.Is > 0 ? p.rin_sig[tid] : 0.0f;
        } else {
        {
            const bool got = ll_read(p.lg_ll + (size_t)par * kMaxB * E, B * E, ep, s_lg, tid, kST, p.status);
            if (!__syncthreads_and(got ? 1 : 0)) {
                ok = false;
                break;
            }
        }
        for (int i = tid; i < B * C; i += kST) c_idx[i] = -1;
        __syncthreads();
        // level 1: each warp selects the k best keys of its slice of every
        // token (key desc, index asc; <= 4 keys per lane), one per round: a
        // warp max of the lanes' best keys, then the lowest index among the
        // lanes holding it.  The slice's picks become candidates in order.
        {
            const int S = ((E + kSW - 1) / kSW + 31) / 32 * 32;  // slice of whole warp-rows
            const int sb = warp * S, se = min(E, sb + S), M1 = S / 32;
            for (int t = 0; t < B; ++t) {
                uint32_t key[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int j = sb + lane + 32 * m;
                    key[m] = (m < M1 && j < se) ? order_key(s_lg[t * E + j]) : 0u;
                }
#pragma unroll 1
                for (int r = 0; r < k; ++r) {
                    uint32_t best = key[0];
                    int bm = 0;
#pragma unroll
                    for (int m = 1; m < 4; ++m)
                        if (key[m] > best) best = key[m], bm = m;
                    const uint32_t mx = __reduce_max_sync(kFullMask, best);
                    const uint32_t jw = __reduce_min_sync(
                        kFullMask, (best == mx && mx != 0u) ? (uint32_t)(sb + lane + 32 * bm) : 0xffffffffu);
                    if (jw == 0xffffffffu) break;  // the slice has fewer than k keys
                    if (lane == 0) {
                        c_key[t * C + warp * k + r] = mx;
                        c_idx[t * C + warp * k + r] = (int)jw;
                    }
                    const int lw = (int)(jw - sb) & 31, mw = (int)(jw - sb) >> 5;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (lane == lw && m == mw) key[m] = 0u;
                }
            }
        }
        __syncthreads();
        // level 2 (one warp per token): the same selection over the token's
        // candidates (<= 4 per lane), ties to the lower expert index; then the
        // routing weights
        if (warp < B) {
            const int t = warp;
            uint32_t key[4];
            int id[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int j = lane + 32 * m;
                const int ij = j < C ? c_idx[t * C + j] : -1;
                key[m] = ij >= 0 ? c_key[t * C + j] : 0u;
                id[m] = ij >= 0 ? ij : 0x7fffffff;
            }
#pragma unroll 1
            for (int r = 0; r < k; ++r) {
                uint32_t best = key[0];
                int bi = id[0];
#pragma unroll
                for (int m = 1; m < 4; ++m)
                    if (key[m] > best || (key[m] == best && id[m] < bi)) best = key[m], bi = id[m];
                const uint32_t mx = __reduce_max_sync(kFullMask, best);
                const int w = (int)__reduce_min_sync(kFullMask, best == mx ? (uint32_t)bi : 0xffffffffu);
                if (lane == 0) {
                    ds->idx[t][r] = w;
                    ds->val[t][r] = s_lg[t * E + w];
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (id[m] == w) key[m] = 0u, id[m] = 0x7fffffff;
            }
            __syncwarp();
            topk_weights(s_lg + t * E, E, k, p.norm_topk, lane, ds->val[t], ds->w[t]);
        }
        }  // routing computed
        __syncthreads();
        if (streamed) {
            // residency of the layer's experts: the same answer in every CTA
            const bool absent = tid < B * k && p.dir[(size_t)l * E + ds->idx[tid / k][tid % k]] == nullptr;
            const bool stop = __syncthreads_or(absent ? 1 : 0) != 0;
            if (c == 0) {
                int32_t* row = p.pub_idx + (size_t)l * p.pub_stride;
                for (int i = tid; i < B * k; i += kST) row[i] = ds->idx[i / k][i % k];
                if (stop) {
                    for (int i = tid; i < B * H; i += kST) p.x_out[i] = xs[i];
                    for (int i = tid; i < B * k; i += kST) {
                        p.rout_idx[i] = ds->idx[i / k][i % k];
                        p.rout_w[i] = ds->w[i / k][i % k];
                    }
                    if (tid < B) p.rout_sig[tid] = ds->sig[tid];
                }
                __threadfence_system();
                __syncthreads();
                if (tid == 0) {
                    const uint32_t e = *p.pub_epoch;
                    if (stop) p.pub_stop[l] = e;
                    __threadfence_system();
                    p.pub_ready[l] = e;
                }
            }
            if (stop) break;  // the host fetches the missing experts and launches again from this layer
        }
        if (p.idx_trace && c == 0 && tid < B * k) p.idx_trace[(size_t)li * B * k + tid] = ds->idx[tid / k][tid % k];
        // dispatch (warp 0): pairs sorted by (expert, token) by rank (pair key
        // expert << 3 | token), then active experts in ascending id
        const int nq = B * k;
        if (warp == 0) {
            for (int m = 0; m * 32 < nq; ++m) {
                const int q = lane + 32 * m;
                const uint32_t kq = q < nq ? ((uint32_t)ds->idx[q / k][q % k] << 3) | (uint32_t)(q / k) : 0xffffffffu;
                int rank = 0;
                for (int mm = 0; mm * 32 < nq; ++mm) {
                    const int qb = lane + 32 * mm;
                    const uint32_t kb =
                        qb < nq ? ((uint32_t)ds->idx[qb / k][qb % k] << 3) | (uint32_t)(qb / k) : 0xffffffffu;
                    const int lim = min(32, nq - 32 * mm);
#pragma unroll 4
                    for (int s2 = 0; s2 < lim; ++s2) rank += __shfl_sync(kFullMask, kb, s2) < kq ? 1 : 0;
                }
                if (q < nq) {
                    D.pair_act[rank] = (int)kq;  // the sorted keys, replaced by active indices below
                    D.pair_w[rank] = ds->w[q / k][q % k];
                }
            }
            __syncwarp();
            int base = 0;
            uint32_t prev = 0xffffffffu;
            for (int m = 0; m * 32 < nq; ++m) {
                const int pr = lane + 32 * m;
                const uint32_t kq = pr < nq ? (uint32_t)D.pair_act[pr] : 0xffffffffu;
                uint32_t kp = __shfl_up_sync(kFullMask, kq, 1);
                if (lane == 0) kp = prev;
                const bool first = pr < nq && (kp == 0xffffffffu || (kp >> 3) != (kq >> 3));
                const unsigned bal = __ballot_sync(kFullMask, first);
                const int a = base + __popc(bal & (0xffffffffu >> (31 - lane))) - 1;
                prev = __shfl_sync(kFullMask, kq, 31);
                __syncwarp();
                if (pr < nq) {
                    const int e = (int)(kq >> 3);
                    D.pair_token[pr] = (int)(kq & 7u);
                    D.pair_act[pr] = a;
                    if (first) {
                        D.act_expert[a] = e;
                        D.act_blob[a] = p.dir[(size_t)l * E + e];
                        D.act_off[a] = pr;
                    }
                }
                base += __popc(bal);
            }
            if (lane == 0) ds->n_routed = base;
        }
        __syncthreads();
        if (tid == 0) {
            const int nr = ds->n_routed;
            ds->n_pairs = B * k + (p.Is > 0 ? B : 0);
            ds->n_act = nr + (p.Is > 0 ? 1 : 0);
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
        const int gcs = mine > 0 ? min(p.g_cap, max(2 * kSW, (mine + kNSG - 1) / kNSG)) : 1;
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
        for (int ch = 0; ch < n_dch && ok; ++ch) {
            const int s = ch % kNSD;
            if (!stage_wait(mbar, kNSG + s, wt, p)) {
                ok = false;
                break;
            }
            const uint8_t* st = Dbuf + (size_t)s * dstage;
            const int aa = ch * dcs, ab = min(n_act, aa + dcs);
            const int pa = D.act_off[aa], pb = D.act_off[ab];
            // h of the pairs, into the (idle) gate/up stage area: all pairs at the
            // first stage when they fit, else this stage's pairs
            const bool all_h = (long long)n_pairs * p.h_stride * 4 <= (long long)kNSG * gstage;
            const int ha = all_h ? 0 : pa, hb = all_h ? n_pairs : pb;
            float* hs = reinterpret_cast<float*>(Gbuf) - (size_t)ha * p.h_stride;  // hs[pr * h_stride + col]
            if (!all_h || ch == 0) {
                const int nrt = max(0, min(hb, B * k) - ha);  // routed pairs (cols I), then shared pairs (cols Is)
                bool okh = ll_read_rows(hll, ha, nrt, p.h_stride, p.I, ep, hs + (size_t)ha * p.h_stride, tid, kST,
                                        p.status);
                if (okh && hb > ha + nrt)
                    okh = ll_read_rows(hll, ha + nrt, hb - ha - nrt, p.h_stride, p.Is, ep,
                                       hs + (size_t)(ha + nrt) * p.h_stride, tid, kST, p.status);
                if (!__syncthreads_and(okh ? 1 : 0)) {
                    ok = false;
                    break;
                }
            }
            bool okc = true;
            // tasks: (pair, group of kRG of this CTA's rows)
            constexpr int kRG = 8;
            const int ngr = (jn + kRG - 1) / kRG;
            for (int task = warp; task < (pb - pa) * ngr; task += kSW) {
                const int pr = pa + task / ngr, g0 = (task % ngr) * kRG;
                const int a = D.pair_act[pr];
                const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
                const uint32_t rb = (uint32_t)cols * BITS / 8, dsb = (uint32_t)cols / 16;
                const uint8_t* unit = st + (size_t)(a - aa) * p.d_unit;
                const uint8_t* sbase = unit + p.d_rows_bytes + ((j0 * dsb) & 15u);
                HF<BITS> hd;
                const bool halves = BITS == 4 && cols == 16 * CC;
                const float* hrow = hs + (size_t)pr * p.h_stride + (halves ? (lane & 15) : lane) * CC;
                if (halves || lane < cols / CC) {
#pragma unroll
                    for (int i = 0; i < CC; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(hrow + i);
                        hd.v[i] = v.x, hd.v[i + 1] = v.y, hd.v[i + 2] = v.z, hd.v[i + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < CC; ++i) hd.v[i] = 0.0f;
                }
                hf_sum(hd);
                const float wp = D.pair_w[pr];
                const int je = min(jn, g0 + kRG);
                if (halves) {
                    // 16 chunks per row: two rows per pass, one per half-warp
#pragma unroll 1
                    for (int jj = g0; jj < je; jj += 2) {
                        const int j1 = min(jj + 1, je - 1);  // an odd tail repeats its row in the upper half
                        const float v = row_dot_h_halves<BITS>(
                            unit + (size_t)jj * rb, reinterpret_cast<const uint32_t*>(sbase + (size_t)jj * dsb),
                            unit + (size_t)j1 * rb, reinterpret_cast<const uint32_t*>(sbase + (size_t)j1 * dsb), hd,
                            lane);
                        const int jo = jj + (lane >> 4);
                        if ((lane & 15) == 0 && jo < je) part[(size_t)pr * p.jn + jo] = __fmul_rn(wp, v);
                    }
                } else {
#pragma unroll 1
                    for (int jj = g0; jj < je; ++jj) {
                        const float v = row_dot_h<BITS>(unit + (size_t)jj * rb,
                                                        reinterpret_cast<const uint32_t*>(sbase + (size_t)jj * dsb), hd,
                                                        cols, lane);
                        if (lane == 0) part[(size_t)pr * p.jn + jj] = __fmul_rn(wp, v);
                    }
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
    const int dbytes = kNSD * p.d_cap * p.d_unit;  // sized before any reduction of d_cap below
    left -= dbytes;
    p.g_cap = left / (kNSG * p.g_unit);
    if (p.g_cap < 1) return false;
    // phase C stages the h of a down stage's pairs (<= d_cap * B + B) in the gate/up area
    while (p.d_cap > 1 && (long long)(p.d_cap * B + B) * sh.h_stride * 4 > (long long)kNSG * p.g_cap * p.g_unit)
        --p.d_cap;
    if ((long long)(p.d_cap * B + B) * sh.h_stride * 4 > (long long)kNSG * p.g_cap * p.g_unit) return false;
    p.off_G = off;
    off += kNSG * p.g_cap * p.g_unit;
    off = r128(off);
    p.off_D = off;
    off += dbytes;
    p.smem_bytes = off;
    // the top-k temp area lives in the gate/up stages
    const long long tmp =
        r16i(B * E * 4) + 2LL * r16i(B * kSW * k * 4);
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
    if (a.rin_idx) {
        if (!a.rin_w || !a.rin_sig || !a.pub || !a.x_out || !a.rout_idx || !a.rout_w || !a.rout_sig)
            return cudaErrorInvalidValue;
        p.rin_idx = a.rin_idx, p.rin_w = a.rin_w, p.rin_sig = a.rin_sig;
        p.x_out = a.x_out, p.rout_idx = a.rout_idx, p.rout_w = a.rout_w, p.rout_sig = a.rout_sig;
        p.pub_idx = a.pub->idx, p.pub_stride = a.pub->idx_stride;
        p.pub_ready = a.pub->ready, p.pub_stop = a.pub->stop, p.pub_epoch = a.pub->epoch;
    }
    void* f = select_kernel(sh.bits, nper_of(sh.hidden, sh.bits));
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(f, dim3(s.grid), dim3(kST), args, (size_t)p.smem_bytes, st);
}

}  // namespace moe
