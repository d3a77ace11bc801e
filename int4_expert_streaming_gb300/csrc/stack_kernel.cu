// stack_kernel.cu -- the persistent decode-stack kernel for sm_103a.
//
// One cooperative launch runs B tokens (B <= 8) through every MoE layer of a
// call, one CTA of 16 warps per SM.  Per layer and CTA:
//   A  x = renorm(y of the previous layer) (or the input) and its block-
//      fixed-point digits; the router logits of this CTA's experts and the
//      shared expert's gate/up rows of this CTA, both from shared memory
//      prefetched during the previous layer; then the next layer's router and
//      shared rows are prefetched while HBM would otherwise idle.
//   B  top-k + routing weights + dispatch lists, computed redundantly (the
//      same bits in every CTA).  Top-k: each warp keeps the k best logits of
//      its 32-expert slice; every key below the largest of the warps' k-th
//      keys is out; the survivors are ranked in parallel.  Then every warp
//      fetches its own share of the routed gate/up rows with cp.async.bulk
//      into its own ring of shared-memory slots (one mbarrier per slot, so a
//      warp starts as soon as its rows land and nothing waits for the whole
//      CTA), and the down rows of every active expert for this CTA's output
//      rows are fetched behind them.
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
// Code size is a first-order cost here: each layer's code runs once per layer
// and is fetched again from L2 when it does not fit the instruction caches,
// so every outer loop stays rolled and each arithmetic helper has one call
// site per phase.
//
// This removes the per-layer launch chain that the Swiftlet pages identify
// as the limit of their decode loop ("dispatch-bound, not IO-bound": article
// section "Capability boundaries", README introduction) and keeps HBM busy
// with bulk copies issued as soon as routing is known.
//
// Streaming contexts use it with the host's slot pool behind it.  Every layer
// publishes its routing to mapped host memory, where the host runs the pool's
// bookkeeping in order, and checks its experts against the device directory:
// when all are resident the launch simply goes on.  A missing expert's rows
// are read straight from pinned host memory (the store, over the
// host-device link) by the same bulk copies that read resident rows from
// HBM, and used at once; no copy engine and no host call sits between the
// routing and the compute.  The CTA that read a row also writes it from
// shared memory into the HBM slot that the host's pool chose (the answer
// arrives in mapped memory while the rows are in flight), so the blob
// crosses the link once and the slot is filled when the launch ends.  With an
// expert container on disk the host first reads each missing blob into a
// pinned staging buffer and names it in the answer, which the layer then
// waits for.  One launch runs the whole call either way.
//
// Every wait is bounded (%globaltimer): a poll or an mbarrier wait that does
// not complete within wait_ns sets the status word; every CTA then stops at
// its next wait, drains its outstanding copies (again bounded) and exits.  The
// last CTA to leave publishes the status to mapped host memory and advances
// the epoch for the next launch.
#include <algorithm>

#include "gemv.cuh"
#include "stack.h"

namespace moe {
namespace {

constexpr int kST = 512, kSW = kST / 32;
constexpr int kMaxB = 8;
constexpr int kRing = 4;                              // gate/up slots per warp (at most)
constexpr int kNSD = 2;                               // down stages
constexpr int kMbD = kSW * kRing;                     // first down-stage mbarrier
constexpr int kMbP = kMbD + kNSD;                     // the prefetch mbarriers [2], by layer parity
constexpr int kNB = kMbP + 2;
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s
constexpr unsigned long long kFaultWaitNs = 1000000ull;  // 1 ms (the test-only fault mode)
constexpr int kStatusTimeout = 2;
constexpr int kStatusAbandoned = 3;  // the host abandoned the call at a gated layer

static_assert(kST == kRenormThreads, "the renormalisation order is defined for kRenormThreads threads");

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
    unsigned long long wait_ns;  // bound of every device-side wait
    int fault_cta;               // tests: this CTA withholds its y words of the launch's first layer (-1: none)
    // streaming launch (pub_idx non-null): every layer's routing is published
    // to mapped host memory (pub_idx row l, then pub_ready[l] = epoch).  A
    // layer whose experts are all resident (non-null directory entries) runs
    // on; one that is not sets pub_gated[l] = epoch before the ready word,
    // reads the missing experts' rows from host memory (store + (l E + e)
    // store_stride, or with a null store the staging buffer of the answer)
    // and, once served[l] = epoch, serve_n[l] and the layer's serve_tab row
    // give the missed experts' slots and the evicted experts, writes those
    // rows into the slots.  CTA 0 patches the device directory (dir_patch).
    int32_t* pub_idx;
    int pub_stride;
    volatile uint32_t* pub_ready;
    volatile uint32_t* pub_gated;
    const uint32_t* served;
    const int32_t* serve_n;
    const ServeEntry* serve_tab;
    int serve_stride;
    const uint8_t** dir_patch;
    const uint8_t* store;
    unsigned long long store_stride;
    uint32_t epoch;
    // shared-memory plan
    int rE, rS, jn;
    int p_bytes, off_sg;  // prefetch buffer size; offset of w_sg in it
    int g_unit, ring, g_bytes;
    int d_cap, d_unit, d_rows_bytes;
    int amax, pmax;
    int off_disp, off_part, off_xs, off_xd, off_P, off_dirs, off_G, off_D;
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
// the same test with a suspend-time hint: a thread whose phase has not
// completed sleeps (up to `ns`) until it does, instead of spinning on issue slots
__device__ __forceinline__ bool mbar_sleep(uint64_t* m, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(sptr(m)), "r"(parity), "r"(ns)
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

// Abort check for spin loops: the timer and the (global) status word are
// looked at only every 256 spins, so thousands of waiting threads do not
// hammer one L2 line.
__device__ __forceinline__ bool spin_abort(const Params& p, unsigned& spins, unsigned long long t0) {
    if ((++spins & 255u) != 0u) return false;
    if (gtime() - t0 > p.wait_ns) {
        atomicCAS(p.status, 0, kStatusTimeout);
        return true;
    }
    return ld_volatile(p.status) != 0;
}

// {value, epoch} words
__device__ __forceinline__ void ll_store(unsigned long long* p, float v, uint32_t ep) {
    const unsigned long long w = ((unsigned long long)ep << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ll_load(const unsigned long long* p) {
    unsigned long long a;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void ll_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Polls the word pairs of rows row0 .. row0+nrows-1 of an exchange buffer
// (row stride `stride` words, the first `cols` words of each row, cols even)
// until every word carries epoch ep; the value of (row, col) goes to
// dst[(row - row0) * dstride + col], or with swz = CC > 0 (chunks of CC
// columns, CC a multiple of 4) to the chunk-interleaved position
// dst[(row - row0) * dstride + ((i / 4) * (dstride / CC) + col / CC) * 4 + i % 4],
// i = col % CC, where the lanes that each read one chunk's float4s hit
// consecutive addresses.  Thread i takes pairs i, i + kST, ... in batches of
// up to four, re-issuing a batch until all of it is current.  Returns false
// (in the calling thread) on timeout or abort.
__device__ __forceinline__ bool poll_rows(const unsigned long long* base, int row0, int nrows, int stride, int cols,
                                          int dstride, uint32_t ep, float* dst, const Params& p, int swz = 0) {
    const int half = cols >> 1, n = nrows * half;
#pragma unroll 1
    for (int q0 = threadIdx.x; q0 < n; q0 += 4 * kST) {
        int so[4], d0[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int q = q0 + m * kST;
            const int r = q / half, cc = 2 * (q - r * half);
            so[m] = q < n ? (row0 + r) * stride + cc : -1;
            const int ci = swz ? cc % swz : 0;
            d0[m] = r * dstride + (swz ? ((ci >> 2) * (dstride / swz) + cc / swz) * 4 + (ci & 3) : cc);
        }
        unsigned long long a[4], b[4];
        unsigned spins = 0;
        unsigned long long t0 = 0;
#pragma unroll 1
        for (;;) {
            bool all = true;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                a[m] = b[m] = (unsigned long long)ep << 32;
                if (so[m] >= 0) ll_load2(base + so[m], a[m], b[m]);
                all = all && (uint32_t)(a[m] >> 32) == ep && (uint32_t)(b[m] >> 32) == ep;
            }
            if (all) break;
            if (!t0) t0 = gtime();
            if (spin_abort(p, spins, t0)) return false;
            __nanosleep(64);  // back off: thousands of pollers share L2 with the weight stream
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (so[m] >= 0) {
                dst[d0[m]] = __uint_as_float((uint32_t)a[m]);
                dst[d0[m] + 1] = __uint_as_float((uint32_t)b[m]);
            }
    }
    return true;
}

// bounded wait of one warp on an mbarrier phase; false (in every lane) on abort
__device__ __forceinline__ bool warp_wait(uint64_t* m, uint32_t parity, const Params& p) {
    unsigned spins = 0;
    unsigned long long t0 = 0;
#pragma unroll 1
    for (;;) {
        if (__all_sync(kFullMask, mbar_sleep(m, parity, 20000u))) return true;
        if (!t0) t0 = gtime();
        if (__any_sync(kFullMask, spin_abort(p, spins, t0))) return false;
    }
}

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int32_t ld_relaxed_sys(const int32_t* p) {
    int32_t v;
    asm volatile("ld.relaxed.sys.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_sys64(const void* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// streaming: the host's answer for layer l (served[l] = the call's epoch);
// one thread; false on timeout or abort
__device__ __forceinline__ bool served_wait(const Params& p, int l) {
    unsigned spins = 0;
    const unsigned long long t0 = gtime();
#pragma unroll 1
    while (ld_acquire_sys(p.served + l) != p.epoch) {
        if (spin_abort(p, spins, t0)) return false;
        __nanosleep(128);
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
    int xe[kMaxB];      // block-fixed-point exponent of each token's x
    float xmax[kMaxB];  // max |x| of each token
    float red[kMaxB][2][kSW];
    int n_act, n_routed, n_pairs, n_miss;
    // streaming, a gated layer: the missing experts and (once the host's
    // answer is in: ans = 2; 1 while a warp fetches it, 3 if it failed) their slots
    int ans, pad2;
    const uint8_t* miss_slot[kMaxMiss];
    int32_t miss_e[kMaxMiss];
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

// top-k scratch inside the gate/up area (free between the previous layer's
// down phase and this layer's copies): logits [B][E] and the warps' candidate
// lists [B][kSW][k] (key, index)
struct TopkTemp {
    float* lg;
    uint32_t* ck;
    int32_t* ci;
};

__host__ __device__ inline int topk_temp_bytes(int B, int E, int k) {
    return r16i(B * E * 4) + 2 * r16i(B * kSW * k * 4);
}

__device__ __forceinline__ TopkTemp topk_temp(uint8_t* base, int B, int E, int k) {
    TopkTemp T;
    uint8_t* q = base;
    T.lg = reinterpret_cast<float*>(q);
    q += r16i(B * E * 4);
    const int n = r16i(B * kSW * k * 4);
    T.ck = reinterpret_cast<uint32_t*>(q);
    T.ci = reinterpret_cast<int32_t*>(q + n);
    return T;
}

struct Waits {
    uint32_t phase;  // bit i = expected parity of mbarrier i
    uint32_t armed;  // bit i = mbarrier i has an outstanding phase
};

// bounded wait on CTA-wide mbarrier i (down stages, prefetch); every thread
// calls it; false (everywhere) on abort
__device__ bool stage_wait(uint64_t* mb, int i, Waits& w, const Params& p) {
    const uint32_t bit = 1u << (i - kMbD);
    const uint32_t par = (w.phase & bit) ? 1u : 0u;
    const unsigned long long t0 = gtime();
    unsigned spins = 0;
    bool ok = true;
    while (!mbar_sleep(mb + i, par, 20000u)) {
        if (spin_abort(p, spins, t0)) {
            ok = false;
            break;
        }
    }
    if (ok) {
        w.phase ^= bit;
        w.armed &= ~bit;
    }
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// This CTA's down rows j0 .. j0+jn-1 of a routed expert (H x I), as staged in
// shared memory ([jn rows of rb bytes][scale/bias words from the 16-byte
// boundary below row j0's]), into the expert's slot blob; one warp.
__device__ __forceinline__ void store_down(uint8_t* slot, const uint8_t* unit, int j0, int jn, int H, int I, int bits,
                                          uint32_t rb, uint32_t dsb, int rows_bytes, int lane) {
    const size_t q = (size_t)I * H * bits / 8, sq = (size_t)I * H / 16;  // down q at 2q, down sb at 3q + 2sq
    uint4* dq = reinterpret_cast<uint4*>(slot + 2 * q + (size_t)j0 * rb);
#pragma unroll 1
    for (int i = lane; i < (int)(jn * rb / 16); i += 32) dq[i] = reinterpret_cast<const uint4*>(unit)[i];
    const uint32_t* ss = reinterpret_cast<const uint32_t*>(unit + rows_bytes + ((j0 * dsb) & 15u));
    uint32_t* ds = reinterpret_cast<uint32_t*>(slot + 3 * q + 2 * sq + (size_t)j0 * dsb);
#pragma unroll 1
    for (int i = lane; i < (int)(jn * dsb / 4); i += 32) ds[i] = ss[i];
}

// streaming: the host's answer for gated layer l, fetched by the first warp
// of the CTA that needs it (the others wait for that warp): the missed
// experts' slots (and, without a store in host memory, their staging buffers,
// entered tagged into the CTA's directory row); CTA 0 also patches the device
// directory.  Warp-collective; false (in every lane) on timeout or abort.
__device__ __forceinline__ bool answer_wait(const Params& p, Disp* ds, int l, const uint8_t** dir_row, int lane) {
    volatile int* ans = &ds->ans;
    int s = 0;
    if (lane == 0) {
        s = *ans;
        if (s == 0) s = atomicCAS(&ds->ans, 0, 1) == 0 ? -1 : 1;
    }
    s = __shfl_sync(kFullMask, s, 0);
    if (s == 2) return true;
    if (s == 3) return false;
    bool ok = true;
    if (s == -1) {  // this warp fetches
        int sn = -1;
        if (lane == 0) {
            ok = served_wait(p, l);
            sn = ok ? ld_relaxed_sys(p.serve_n + l) : -1;
        }
        sn = __shfl_sync(kFullMask, sn, 0);
        const int nm = sn & 0xffff, nv = (sn >> 16) & 0x7fff;
        ok = sn >= 0 && nm == ds->n_miss && nm + nv <= p.serve_stride;
        bool bad = false;
        if (ok) {
            (void)ld_acquire_sys(p.served + l);  // this lane's own acquire of the answer
#pragma unroll 1
            for (int i = lane; i < nm + nv; i += 32) {
                const ServeEntry* en = p.serve_tab + (size_t)l * p.serve_stride + i;
                const int e = ld_relaxed_sys(&en->expert), ee = e < 0 ? -1 - e : e;
                if (ee >= p.E) {
                    bad = true;
                } else if (i < nm) {
                    const uint8_t* slot = reinterpret_cast<const uint8_t*>(ld_relaxed_sys64(&en->slot));
                    int j = -1;
#pragma unroll 1
                    for (int q = 0; q < nm; ++q)
                        if (ds->miss_e[q] == e) j = q;
                    if (j < 0 || !slot) {
                        bad = true;
                    } else {
                        ds->miss_slot[j] = slot;
                        if (!p.store) {
                            const uintptr_t src = (uintptr_t)ld_relaxed_sys64(&en->src);
                            dir_row[e] = reinterpret_cast<const uint8_t*>(src | 1u);
                        }
                        if (blockIdx.x == 0) p.dir_patch[(size_t)l * p.E + e] = slot;  // for later launches
                    }
                } else if (blockIdx.x == 0) {
                    p.dir_patch[(size_t)l * p.E + ee] = nullptr;
                }
            }
            ok = !__any_sync(kFullMask, bad);
        }
        __syncwarp();
        __threadfence_block();
        if (lane == 0) {
            if (!ok) atomicCAS(p.status, 0, kStatusAbandoned);
            *ans = ok ? 2 : 3;
        }
        return ok;
    }
    if (lane == 0) {  // another warp fetches
        unsigned spins = 0;
        const unsigned long long t0 = gtime();
#pragma unroll 1
        for (;;) {
            const int v = *ans;
            if (v == 2) break;
            if (v == 3 || spin_abort(p, spins, t0)) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
        __threadfence_block();
    }
    return __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
}

// the slot of missing expert e (after answer_wait); lane-parallel search
__device__ __forceinline__ uint8_t* miss_slot_of(const Disp* ds, int e, int lane) {
    const int n = ds->n_miss;
    int j = -1;
#pragma unroll 1
    for (int q = lane; q < n; q += 32)
        if (ds->miss_e[q] == e) j = q;
    const unsigned b = __ballot_sync(kFullMask, j >= 0);
    j = __shfl_sync(kFullMask, j, b ? __ffs(b) - 1 : 0);
    return j >= 0 ? const_cast<uint8_t*>(ds->miss_slot[j]) : nullptr;
}

// One gate/up unit in shared memory ([gate q][up q][gate sb][up sb], row r of
// an expert with I rows) into the expert's slot blob, in 16-byte pieces by one warp.
__device__ __forceinline__ void store_unit(uint8_t* slot, const uint8_t* unit, int r, int I, uint32_t qb, uint32_t sbb,
                                           int lane) {
    const int nq = (int)(qb / 16), ns = (int)(sbb / 16);
    const size_t q = (size_t)I * qb, sq = (size_t)I * sbb;  // blob layout: gate q, up q, down q, gate sb, up sb, down sb
#pragma unroll 1
    for (int i = lane; i < 2 * (nq + ns); i += 32) {
        size_t off;
        if (i < 2 * nq)
            off = (i < nq ? 0 : q) + (size_t)r * qb + 16 * (i < nq ? i : i - nq);
        else
            off = 3 * q + (i < 2 * nq + ns ? 0 : sq) + (size_t)r * sbb + 16 * (i < 2 * nq + ns ? i - 2 * nq : i - 2 * nq - ns);
        *reinterpret_cast<uint4*>(slot + off) = reinterpret_cast<const uint4*>(unit)[i];
    }
}

// ---------------------------------------------------------------------------
// copies (each issued by one lane)
// ---------------------------------------------------------------------------
// prefetch buffer: [router rows rE x 2H][shared gate q rS][shared up q rS][gate sb rS][up sb rS][w_sg 2H];
// and the layer's directory row into dirs[layer & 1] (the directory does not change during a launch)
__device__ __forceinline__ void issue_prefetch(const Params& p, int layer, uint8_t* buf, const uint8_t** dirs,
                                               uint64_t* mb) {
    const int c = blockIdx.x, G = gridDim.x;
    const int e0 = p.E * c / G, e1 = p.E * (c + 1) / G;  // 32-bit: E, Is <= 4096, G <= 1024
    const int s0 = p.Is * c / G, s1 = p.Is * (c + 1) / G;
    const uint32_t rb = (uint32_t)p.H * 2, qb = (uint32_t)p.H * p.bits / 8, sbb = (uint32_t)p.H / 16;
    const bool sg = p.Is > 0;
    mbar_expect(mb, (e1 - e0) * rb + (s1 - s0) * 2 * (qb + sbb) + (sg ? rb : 0u) + (uint32_t)p.E * 8u);
    bulk_load(dirs + (layer & 1) * p.E, p.dir + (size_t)layer * p.E, (uint32_t)p.E * 8u, mb);
    if (e1 > e0) bulk_load(buf, p.router_w + ((size_t)layer * p.E + e0) * p.H, (e1 - e0) * rb, mb);
    if (sg) bulk_load(buf + p.off_sg, p.shared_gate + (size_t)layer * p.H, rb, mb);
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

// one gate/up unit (row r of active routed expert a): [gate q][up q][gate sb][up sb]
__device__ __forceinline__ void issue_unit(const Params& p, const uint8_t* blob, int r, uint8_t* slot, uint64_t* mb) {
    const uint32_t qb = (uint32_t)p.H * p.bits / 8, sbb = (uint32_t)p.H / 16;
    const BlobLayout L = blob_layout(p.H, p.I, p.bits);
    mbar_expect(mb, 2 * (qb + sbb));
    bulk_load(slot, blob + L.gate_q + (size_t)r * qb, qb, mb);
    bulk_load(slot + qb, blob + L.up_q + (size_t)r * qb, qb, mb);
    bulk_load(slot + 2 * qb, blob + L.gate_sb + (size_t)r * sbb, sbb, mb);
    bulk_load(slot + 2 * qb + sbb, blob + L.up_sb + (size_t)r * sbb, sbb, mb);
}

// down stage: per active expert a in [aa, ab): [jn rows x row bytes][aligned scale/bias superset]
__device__ __forceinline__ void issue_down(const Params& p, const Lists& D, int aa, int ab, int j0, int jn,
                                        uint8_t* stage, uint64_t* mb) {
    uint32_t total = 0;
#pragma unroll 1
    for (int a = aa; a < ab; ++a) {
        const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
        const uint32_t rb = (uint32_t)cols * p.bits / 8, sbb = (uint32_t)cols / 16;
        const uint32_t s_lo = (j0 * sbb) & ~15u, s_hi = ((j0 + jn) * sbb + 15u) & ~15u;
        total += jn * rb + (s_hi - s_lo);
    }
    mbar_expect(mb, total);
#pragma unroll 1
    for (int a = aa; a < ab; ++a) {
        const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
        const uint32_t rb = (uint32_t)cols * p.bits / 8, sbb = (uint32_t)cols / 16;
        const BlobLayout L = blob_layout(p.H, cols, p.bits);
        const uint8_t* blob = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(D.act_blob[a]) & ~(uintptr_t)1);
        uint8_t* u = stage + (size_t)(a - aa) * p.d_unit;
        bulk_load(u, blob + L.down_q + (size_t)j0 * rb, jn * rb, mb);
        const uint32_t s_lo = (j0 * sbb) & ~15u, s_hi = ((j0 + jn) * sbb + 15u) & ~15u;
        bulk_load(u + p.d_rows_bytes, blob + L.down_sb + s_lo, s_hi - s_lo, mb);
    }
}

// ---------------------------------------------------------------------------
// top-k of every token: the warps' candidate lists, the threshold, the
// survivors' ranks.  Order: logit descending, ties to the lower expert id,
// the order of warp_topk in the per-layer kernels.
// ---------------------------------------------------------------------------
// Level 1 (warp w, token t): the k best of experts w*32*M + lane + 32 m
// (m < M), polled straight from the exchange buffer; also writes every
// polled logit to T.lg.  Returns false on abort.
__device__ __forceinline__ bool topk_lists(const Params& p, const unsigned long long* lgx, uint32_t ep, const TopkTemp& T,
                                        int M, int nlist) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, E = p.E, k = p.k;
#pragma unroll 1
    for (int t = 0; t < p.B; ++t) {
        uint32_t key0 = 0u, key1 = 0u;  // scalars: a runtime-indexed array would live in local memory
#pragma unroll 1
        for (int m = 0; m < M; ++m) {
            const int j = warp * 32 * M + 32 * m + lane;
            if (j >= E) continue;
            unsigned spins = 0;
            unsigned long long t0 = 0, wv;
#pragma unroll 1
            for (;;) {
                wv = ll_load(lgx + (size_t)t * E + j);
                if ((uint32_t)(wv >> 32) == ep) break;
                if (!t0) t0 = gtime();
                if (spin_abort(p, spins, t0)) return false;
                __nanosleep(64);
            }
            const float v = __uint_as_float((uint32_t)wv);
            T.lg[t * E + j] = v;
            if (m == 0)
                key0 = order_key(v);
            else
                key1 = order_key(v);
        }
        if (warp >= nlist) continue;
        uint32_t* ck = T.ck + (t * kSW + warp) * k;
        int32_t* ci = T.ci + (t * kSW + warp) * k;
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            const int bm = key1 > key0 ? 1 : 0;
            const uint32_t best = bm ? key1 : key0;
            const uint32_t mx = __reduce_max_sync(kFullMask, best);
            const uint32_t win = __reduce_min_sync(
                kFullMask, (best == mx && mx != 0u) ? (uint32_t)(warp * 32 * M + 32 * bm + lane) : 0xffffffffu);
            if (lane == 0) {
                ck[r] = mx;
                ci[r] = (int)win;  // 0xffffffff (-1): the slice has fewer than k keys
            }
            if (win == 0xffffffffu) break;
            const int wl = (int)(win & 31u), wm = (int)(win - (uint32_t)(warp * 32 * M)) >> 5;
            if (lane == wl) {
                if (wm == 0)
                    key0 = 0u;
                else
                    key1 = 0u;
            }
        }
    }
    return true;
}

// Level 2 for token t = warp: a merge of the warps' lists (each sorted by
// key descending, ties by index ascending, and holding its slice's k best, so
// together they hold the token's k best) in k rounds of a warp maximum over
// the list heads, ties to the lower expert id.  Lane i < nlist holds the head
// of list i and its next entry.  Then the routing weights.
__device__ __forceinline__ void topk_merge(const Params& p, const TopkTemp& T, Disp* ds, int nlist) {
    const int t = threadIdx.x >> 5, lane = threadIdx.x & 31, k = p.k;
    const uint32_t* ck = T.ck + (t * kSW + (lane < nlist ? lane : 0)) * k;
    const int32_t* ci = T.ci + (t * kSW + (lane < nlist ? lane : 0)) * k;
    uint32_t hk = 0u, hi = 0xffffffffu, nk = 0u, ni = 0xffffffffu;
    if (lane < nlist) {
        if (ci[0] >= 0) hk = ck[0], hi = (uint32_t)ci[0];
        if (k > 1 && ci[1] >= 0 && hi != 0xffffffffu) nk = ck[1], ni = (uint32_t)ci[1];
    }
    int pos = 1;  // index of the entry held in (nk, ni)
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        const uint32_t mx = __reduce_max_sync(kFullMask, hk);
        const uint32_t win = __reduce_min_sync(kFullMask, hk == mx ? hi : 0xffffffffu);
        if (lane == 0) {
            ds->idx[t][r] = (int)win;
            ds->val[t][r] = T.lg[t * p.E + (int)win];
        }
        if (hi == win) {  // this list's head was taken
            hk = nk, hi = ni;
            ++pos;
            nk = 0u, ni = 0xffffffffu;
            if (hi != 0xffffffffu && pos < k && ci[pos] >= 0) nk = ck[pos], ni = (uint32_t)ci[pos];
        }
    }
    __syncwarp();
    topk_weights(T.lg + t * p.E, p.E, k, p.norm_topk, lane, ds->val[t], ds->w[t]);
}

// Dispatch (warp 0): pairs sorted by (expert, token) by rank (key expert << 3 | token),
// then the active experts in ascending id with their blob addresses.
__device__ __forceinline__ void dispatch(const Params& p, const Lists& D, Disp* ds, int l,
                                         const uint8_t* const* dir_row) {
    const int lane = threadIdx.x & 31, k = p.k, nq = p.B * k;
#pragma unroll 1
    for (int m = 0; m * 32 < nq; ++m) {
        const int q = lane + 32 * m;
        const uint32_t kq = q < nq ? ((uint32_t)ds->idx[q / k][q % k] << 3) | (uint32_t)(q / k) : 0xffffffffu;
        int rank = 0;
#pragma unroll 1
        for (int mm = 0; mm * 32 < nq; ++mm) {
            const int qb = lane + 32 * mm;
            const uint32_t kb = qb < nq ? ((uint32_t)ds->idx[qb / k][qb % k] << 3) | (uint32_t)(qb / k) : 0xffffffffu;
            const int lim = min(32, nq - 32 * mm);
#pragma unroll 1
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
#pragma unroll 1
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
                D.act_blob[a] = dir_row[e];
                D.act_off[a] = pr;
            }
        }
        base += __popc(bal);
    }
    __syncwarp();
    if (lane == 0) {
        const int nr = base, B = p.B;
        ds->n_routed = nr;
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
    if (p.Is > 0 && lane < p.B) {
        D.pair_token[p.B * k + lane] = lane;
        D.pair_w[p.B * k + lane] = ds->sig[lane];
        D.pair_act[p.B * k + lane] = base;
    }
}

// gate and up rows (codes + scale/bias words in shared memory) against token
// t's digits; silu(g) * u
template <int BITS>
__device__ __forceinline__ float swiglu_row(const uint8_t* gq, const uint8_t* uq, const uint32_t* gsb,
                                            const uint32_t* usb, const uint32_t* xdw, const int32_t* xS, int xe, int nc) {
    float g, u;
    row_dot_x2_sm<BITS>(gq, gsb, uq, usb, xdw, xS, xe, nc, threadIdx.x & 31, g, u);
    return silu_mul(g, u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BITS, bool ONE, bool STREAM>
__global__ void __launch_bounds__(kST, 1) stack_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t mbar[kNB];

    constexpr int CC = Codes<BITS>::kCols, DW = Codes<BITS>::kDigitWords;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int H = p.H, E = p.E, k = p.k, B = ONE ? 1 : p.B;  // ONE: the batch-1 instance
    const int nc = H / CC;  // chunks of a gate/up row
    const uint32_t qb = (uint32_t)H * BITS / 8, sbb = (uint32_t)H / 16;
    Disp* ds = reinterpret_cast<Disp*>(smem + p.off_disp);
    const Lists D = lists(smem + p.off_disp, p.amax, p.pmax);
    float* part = reinterpret_cast<float*>(smem + p.off_part);
    float* xs = reinterpret_cast<float*>(smem + p.off_xs);
    uint32_t* xdw = reinterpret_cast<uint32_t*>(smem + p.off_xd);           // [B][nc][DW]
    int32_t* xS = reinterpret_cast<int32_t*>(xdw + (size_t)B * nc * DW);  // [B][nc]
    uint8_t* Pb = smem + p.off_P;                                           // [2][p_bytes], by layer parity
    const uint8_t** dirs = reinterpret_cast<const uint8_t**>(smem + p.off_dirs);
    uint8_t* Gbuf = smem + p.off_G;
    uint8_t* Dbuf = smem + p.off_D;
    const TopkTemp TT = topk_temp(Gbuf, B, E, k);
    const int dstage = p.d_cap * p.d_unit;
    const size_t h_par = (size_t)p.hp * p.h_stride;
    const int M = (E + kST - 1) / kST;              // keys per lane in the first top-k level
    const int nlist = (E + 32 * M - 1) / (32 * M);  // warps holding keys
    const int R = p.ring;
    uint8_t* wslots = Gbuf + (size_t)warp * R * p.g_unit;

    const uint32_t ep0 = *(volatile const unsigned*)&p.sync[2];
    Waits wt{0u, 0u};
    uint32_t wph = 0u, warm = 0u;  // this warp's slots: expected parity, outstanding
    if (tid == 0) {
        for (int i = 0; i < kNB; ++i) mbar_init(&mbar[i]);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) issue_prefetch(p, p.layer0, Pb + (p.layer0 & 1) * p.p_bytes, dirs, &mbar[kMbP + (p.layer0 & 1)]);
    wt.armed |= 1u << (kMbP + (p.layer0 & 1) - kMbD);

    // work splits in 32-bit arithmetic (every product stays below 2^31)
    const int j0 = H * c / G, jn = H * (c + 1) / G - j0;
    const int e0 = E * c / G, ne = E * (c + 1) / G - e0;
    const int s0 = p.Is * c / G, ns = p.Is * (c + 1) / G - s0;
    bool ok = true;
    const int lend = p.layer0 + p.n_layers;

#pragma unroll 1
    for (int l = p.layer0; l < lend && ok; ++l) {
        const int li = l - p.layer0, par = l & 1;
        const uint32_t ep = ep0 + (uint32_t)li;
        const bool streamed = STREAM && p.pub_idx != nullptr;  // routing published, residency checked
        uint8_t* Pbuf = Pb + par * p.p_bytes;
        unsigned long long* hll = p.h_ll + par * h_par;
        // the next layer's router rows, shared rows and directory row do not
        // depend on this layer: fetch them now (their buffer was last read in
        // the previous layer)
        if (l + 1 < lend) {
            if (tid == 0) issue_prefetch(p, l + 1, Pb + (par ^ 1) * p.p_bytes, dirs, &mbar[kMbP + (par ^ 1)]);
            wt.armed |= 1u << (kMbP + (par ^ 1) - kMbD);
        }
        // ------------------------------------------------------------ phase A
        // x: the call's input, or the previous layer's y from the exchange
        bool got = true;
        if (l == p.layer0) {
#pragma unroll 1
            for (int i = tid; i < B * H / 4; i += kST)
                reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(p.x_in) + i);
        } else {
            got = poll_rows(p.y_ll + (size_t)(par ^ 1) * kMaxB * H, 0, B, H, H, H, ep - 1, xs, p);
        }
        if (!__syncthreads_and(got ? 1 : 0)) {
            ok = false;
            break;
        }
#pragma unroll 1
        for (int t = 0; t < B; ++t) {
            float s, m;
            renorm_partial(xs + t * H, H, tid, s, m);
            s = warp_sum(s);
            m = warp_max(m);
            if (lane == 0) {
                ds->red[t][0][warp] = s;
                ds->red[t][1][warp] = m;
            }
        }
        __syncthreads();
        // every thread forms r and the digit exponent of each token itself
        // (the same bits everywhere), so no further barrier is needed before x = y * r
        float r_t[kMaxB];
        int xe_t[kMaxB];
#pragma unroll
        for (int t = 0; t < kMaxB; ++t) {
            if (t < B) {
                float mx = ds->red[t][1][0];
#pragma unroll 1
                for (int w = 1; w < kSW; ++w) mx = fmaxf(mx, ds->red[t][1][w]);
                r_t[t] = renorm_scale(ds->red[t][0], H, p.eps);
                const float xm = l == p.layer0 ? mx : __fmul_rn(mx, r_t[t]);  // max|x| = max|y| * r exactly (r > 0)
                xe_t[t] = bfp_exponent(xm);
            }
        }
        if (tid < B) {
#pragma unroll
            for (int t = 0; t < kMaxB; ++t)
                if (t == tid) ds->rs[t] = r_t[t], ds->xe[t] = xe_t[t];
        }
        if (l != p.layer0) {  // x = y * r
#pragma unroll
            for (int t = 0; t < kMaxB; ++t)
                if (t < B)
#pragma unroll 1
                    for (int i = tid; i < H; i += kST) xs[t * H + i] = __fmul_rn(xs[t * H + i], r_t[t]);
        }
        __syncthreads();
        if (p.x_trace && c == 0)
#pragma unroll 1
            for (int i = tid; i < B * H; i += kST) p.x_trace[(size_t)li * B * H + i] = xs[i];
        if (!stage_wait(mbar, kMbP + par, wt, p)) {
            ok = false;
            break;
        }
        // The router rows go first, on the top warps: their logits reach the
        // exchange while the other warps make the digits (which only the
        // expert rows need) and these warps the shared gate.
        {
            const int na = ne * B, ng = p.Is == 0 ? 0 : B;
            const int nr = min(kSW / 2, max(1, na + ng));  // router warps
            if (warp >= kSW - nr) {
                unsigned long long* lgx = p.lg_ll + (size_t)par * kMaxB * E;
#pragma unroll 1
                for (int task = kSW - 1 - warp; task < na + ng; task += nr) {
                    const bool gate = task >= na;
                    const int q = gate ? task - na : task;
                    const int t = gate ? q : q % B, e = gate ? 0 : e0 + q / B;
                    const uint16_t* row =
                        reinterpret_cast<const uint16_t*>(Pbuf + (gate ? (size_t)p.off_sg : (size_t)(e - e0) * 2 * H));
                    const float v =
                        router_logit(row, xs + t * H, H, gate ? 0.0f : p.router_bias[(size_t)l * E + e], lane);
                    if (gate) {
                        if (lane == 0) ds->sig[t] = __fdividef(1.0f, __fadd_rn(1.0f, __expf(-v)));
                    } else if (lane == 0) {
                        ll_store(lgx + (size_t)t * E + e, v, ep);
                    }
                }
            } else {
                make_digits<BITS>(B, H, xs, xdw, xS, ds->xe, 0, kSW - nr);
            }
        }
        __syncthreads();
        // ------------------------------------------------------------ phase B
        {
            const bool okl = topk_lists(p, p.lg_ll + (size_t)par * kMaxB * E, ep, TT, M, nlist);
            if (!__syncthreads_and(okl ? 1 : 0)) {
                ok = false;
                break;
            }
            if (warp < B) topk_merge(p, TT, ds, nlist);
        }
        fence_proxy_async();  // the top-k scratch shares the area the copies below write
        __syncthreads();
        bool gated = false;
        if (streamed) {
            // residency of the layer's experts: the same answer in every CTA
            const bool absent = tid < B * k && dirs[(l & 1) * E + ds->idx[tid / k][tid % k]] == nullptr;
            gated = __syncthreads_or(absent ? 1 : 0) != 0;
            // the routing goes to the host from one warp of CTA 0 (the others go on)
            if (c == 0 && warp == kSW - 1) {
                int32_t* row = p.pub_idx + (size_t)l * p.pub_stride;
#pragma unroll 1
                for (int i = lane; i < B * k; i += 32) row[i] = ds->idx[i / k][i % k];
                __threadfence_system();
                __syncwarp();
                if (lane == 0) {
                    if (gated) p.pub_gated[l] = p.epoch;
                    __threadfence_system();
                    p.pub_ready[l] = p.epoch;
                }
            }
            if (gated) {
                // the layer's missing experts (the same list in every CTA);
                // their rows are read from host memory, through directory
                // entries tagged in bit 0 (blob addresses are 4096-aligned)
                if (warp == 0) {
                    int n = 0;
#pragma unroll 1
                    for (int q0 = 0; q0 < B * k; q0 += 32) {
                        const int q = q0 + lane;
                        int e = -1;
                        if (q < B * k) {
                            e = ds->idx[q / k][q % k];
                            if (dirs[(l & 1) * E + e] != nullptr) e = -1;
#pragma unroll 1
                            for (int q2 = 0; q2 < q && e >= 0; ++q2)
                                if (ds->idx[q2 / k][q2 % k] == e) e = -1;
                        }
                        const unsigned bal = __ballot_sync(kFullMask, e >= 0);
                        if (e >= 0) ds->miss_e[n + __popc(bal & ((1u << lane) - 1u))] = e;
                        n += __popc(bal);
                    }
                    if (lane == 0) {
                        ds->n_miss = n;
                        ds->ans = 0;
                    }
                }
                __syncthreads();
                if (p.store) {  // the pinned store
                    if (tid < ds->n_miss) {
                        const int e = ds->miss_e[tid];
                        dirs[(l & 1) * E + e] = reinterpret_cast<const uint8_t*>(
                            reinterpret_cast<uintptr_t>(p.store + ((size_t)l * E + e) * p.store_stride) | 1u);
                    }
                } else {  // staging buffers named in the host's answer
                    bool oka = true;
                    if (warp == 0) oka = answer_wait(p, ds, l, dirs + (l & 1) * E, lane);
                    if (!__syncthreads_and(oka ? 1 : 0)) {
                        ok = false;
                        break;
                    }
                }
                __syncthreads();
            }
        }
        if (p.idx_trace && c == 0 && tid < B * k) p.idx_trace[(size_t)li * B * k + tid] = ds->idx[tid / k][tid % k];
        const uint8_t* const* dir_l = dirs + (l & 1) * E;
        const uint8_t** dir_l_w = dirs + (l & 1) * E;
        int n_act, n_pairs, n_routed;
        int el = 0x7fffffff, rk = 0;  // one token: this lane's expert (lanes < k) and its rank among the k
        // blob of active expert a (every lane calls it; ONE: from the ranks, before
        // the lists are visible), tagged in bit 0 when it is read from host memory
        auto blob_of = [&](int a) -> const uint8_t* {
            if (ONE) {
                const int src = __ffs(__ballot_sync(kFullMask, rk == a && lane < k)) - 1;
                return dir_l[__shfl_sync(kFullMask, el, src)];
            }
            return D.act_blob[a];
        };
        auto expert_of = [&](int a) -> int {
            if (ONE) return __shfl_sync(kFullMask, el, __ffs(__ballot_sync(kFullMask, rk == a && lane < k)) - 1);
            return D.act_expert[a];
        };
        auto untag = [](const uint8_t* b) {
            return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(b) & ~(uintptr_t)1);
        };
        if (ONE) {
            // one token: the active experts are its k experts in ascending id
            // and pair a is active expert a.  Every warp ranks them itself and
            // issues its copies at once; warp 0 also writes the lists that
            // phase C and the combine read (after later barriers).
            n_routed = k;
            n_act = n_pairs = k + (p.Is > 0 ? 1 : 0);
            el = lane < k ? ds->idx[0][lane] : 0x7fffffff;
#pragma unroll 1
            for (int s2 = 0; s2 < k; ++s2) rk += __shfl_sync(kFullMask, el, s2) < el ? 1 : 0;
            if (warp == 0) {
                if (lane < k) {
                    D.act_expert[rk] = el;
                    D.act_blob[rk] = dir_l[el];
                    D.act_off[rk] = rk;
                    D.pair_token[rk] = 0;
                    D.pair_w[rk] = ds->w[0][lane];
                    D.pair_act[rk] = rk;
                }
                if (lane == 0) {
                    if (p.Is > 0) {
                        D.act_expert[k] = -1;
                        D.act_blob[k] = p.shared_pool + (size_t)l * p.shared_stride;
                        D.pair_token[k] = 0;
                        D.pair_w[k] = ds->sig[0];
                        D.pair_act[k] = k;
                    }
                    D.act_off[k] = k;
                    D.act_off[k + 1] = k + 1;
                }
            }
            const int U = k * p.I, u0 = U * c / G, u1 = U * (c + 1) / G;
            const int mine = u1 - u0;
            const int wu0 = u0 + mine * warp / kSW, wn = u0 + mine * (warp + 1) / kSW - wu0;
#pragma unroll 1
            for (int j = 0; j < min(R, wn); ++j) {
                const int u = wu0 + j, a = u / p.I;
                const uint8_t* blob = untag(blob_of(a));
                if (lane == 0) issue_unit(p, blob, u - a * p.I, wslots + (size_t)j * p.g_unit, &mbar[warp * kRing + j]);
                warm |= 1u << j;
            }
        } else {
            if (warp == 0) dispatch(p, D, ds, l, dir_l);
            __syncthreads();
            n_act = ds->n_act, n_pairs = ds->n_pairs, n_routed = ds->n_routed;
            const int U = n_routed * p.I, u0 = U * c / G, u1 = U * (c + 1) / G;  // U <= 129 * 4096
            const int mine = u1 - u0;
            const int wu0 = u0 + mine * warp / kSW, wn = u0 + mine * (warp + 1) / kSW - wu0;
            if (lane == 0) {
#pragma unroll 1
                for (int j = 0; j < min(R, wn); ++j) {
                    const int u = wu0 + j, a = u / p.I;
                    issue_unit(p, untag(D.act_blob[a]), u - a * p.I, wslots + (size_t)j * p.g_unit, &mbar[warp * kRing + j]);
                }
            }
#pragma unroll 1
            for (int j = 0; j < min(R, wn); ++j) warm |= 1u << j;
        }
        const int U = n_routed * p.I, u0 = U * c / G, u1 = U * (c + 1) / G;
        const int mine = u1 - u0;
        const int wu0 = u0 + mine * warp / kSW, wn = u0 + mine * (warp + 1) / kSW - wu0;  // this warp's units
        const int dcs = min(p.d_cap, n_act);
        const int n_dch = jn > 0 ? (n_act + dcs - 1) / dcs : 0;
        // the shared expert's rows of this CTA (in shared memory since the
        // previous layer) while the routed rows are in flight
#pragma unroll 1
        for (int task = warp; task < ns * B; task += kSW) {
            const int rr = task / B, t = task - rr * B;
            const uint8_t* sq = Pbuf + (size_t)p.rE * 2 * H;
            const uint8_t* sbase = sq + (size_t)2 * p.rS * qb;
            const float h = swiglu_row<BITS>(sq + (size_t)rr * qb, sq + (size_t)(p.rS + rr) * qb,
                                             reinterpret_cast<const uint32_t*>(sbase + rr * sbb),
                                             reinterpret_cast<const uint32_t*>(sbase + (p.rS + rr) * sbb),
                                             xdw + (size_t)t * nc * DW, xS + t * nc, ds->xe[t], nc);
            if (lane == 0) ll_store(hll + (size_t)(B * k + t) * p.h_stride + s0 + rr, h, ep);
        }
        // gate/up + SwiGLU: this warp's units as they land
        {
            bool okw = true;
#pragma unroll 1
            for (int j = 0; j < wn; ++j) {
                const int s = j % R;
                if (!warp_wait(&mbar[warp * kRing + s], (wph >> s) & 1u, p)) {
                    okw = false;
                    break;
                }
                wph ^= 1u << s;
                warm &= ~(1u << s);
                const uint8_t* st = wslots + (size_t)s * p.g_unit;
                const int u = wu0 + j, a = u / p.I, r = u - a * p.I;
                const int pr0 = ONE ? a : D.act_off[a], pr1 = ONE ? a + 1 : D.act_off[a + 1];
#pragma unroll 1
                for (int pr = pr0; pr < pr1; ++pr) {
                    const int t = ONE ? 0 : D.pair_token[pr];
                    const float h = swiglu_row<BITS>(st, st + qb, reinterpret_cast<const uint32_t*>(st + 2 * qb),
                                                     reinterpret_cast<const uint32_t*>(st + 2 * qb + sbb),
                                                     xdw + (size_t)t * nc * DW, xS + t * nc, ds->xe[t], nc);
                    if (lane == 0) ll_store(hll + (size_t)pr * p.h_stride + r, h, ep);
                }
                if (gated && (reinterpret_cast<uintptr_t>(blob_of(a)) & 1u)) {
                    // a row read from host memory: into the expert's new slot
                    const int e = expert_of(a);
                    uint8_t* slot = answer_wait(p, ds, l, dir_l_w, lane) ? miss_slot_of(ds, e, lane) : nullptr;
                    if (!slot) {
                        okw = false;
                        break;
                    }
                    store_unit(slot, st, r, p.I, qb, sbb, lane);
                }
                if (j + R < wn) {
                    const int un = wu0 + j + R, an = un / p.I;
                    const uint8_t* blob = untag(blob_of(an));
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) issue_unit(p, blob, un - an * p.I, wslots + (size_t)s * p.g_unit, &mbar[warp * kRing + s]);
                    warm |= 1u << s;
                }
            }
            if (!__syncthreads_and(okw ? 1 : 0)) {
                ok = false;
                break;
            }
        }
        // ------------------------------------------------------------ phase C
        // The down rows are fetched now, behind the gate/up rows: they stream
        // while the SwiGLU vectors travel between CTAs.  Then every pair's h is
        // polled block-wide into the (idle) gate/up area, and each warp takes
        // whole pairs: this CTA's down rows of the pair's expert.  The down
        // stages are used in rounds of kNSD (one round when every active
        // expert fits).
        {
            if (lane == 0) {
                const int s = kSW - 1 - warp;
                if (s < min(n_dch, kNSD))
                    issue_down(p, D, s * dcs, min(n_act, (s + 1) * dcs), j0, jn, Dbuf + (size_t)s * dstage,
                               &mbar[kMbD + s]);
            }
#pragma unroll 1
            for (int s = 0; s < min(n_dch, kNSD); ++s) wt.armed |= 1u << s;
            const bool all_h = n_pairs * p.h_stride * 4 <= p.g_bytes;
            float* hs = reinterpret_cast<float*>(Gbuf);  // all pairs, or the round's pairs from the first
            const int rounds = (n_dch + kNSD - 1) / kNSD;
#pragma unroll 1
            for (int rd = 0; rd < rounds && ok; ++rd) {
                const int aa = rd * kNSD * dcs, ab = min(n_act, aa + kNSD * dcs);
                const int pa = D.act_off[aa], pb = D.act_off[ab];
                const int ha = all_h ? 0 : pa, hb = all_h ? n_pairs : pb;
                if (!all_h || rd == 0) {
                    const int nrt = max(0, min(hb, B * k) - ha);  // routed pairs (cols I), then shared pairs (cols Is)
                    bool okh = poll_rows(hll, ha, nrt, p.h_stride, p.I, p.h_stride, ep, hs, p, CC);
                    if (okh && hb > ha + nrt)
                        okh = poll_rows(hll, ha + nrt, hb - ha - nrt, p.h_stride, p.Is, p.h_stride, ep,
                                        hs + (size_t)nrt * p.h_stride, p, CC);
                    if (!__syncthreads_and(okh ? 1 : 0)) {
                        ok = false;
                        break;
                    }
                }
                bool okc = true;
#pragma unroll 1
                for (int pr = pa + warp; pr < pb; pr += kSW) {
                    const int a = D.pair_act[pr];
                    const int s = (a - aa) / dcs;
                    if (!warp_wait(&mbar[kMbD + s], (wt.phase >> s) & 1u, p)) {
                        okc = false;
                        break;
                    }
                    const int cols = D.act_expert[a] < 0 ? p.Is : p.I;
                    const bool halves = BITS == 4 && cols == 16 * CC;
                    const int ch = halves ? (lane & 15) : lane;
                    HF<BITS> hd;
                    if (halves || ch < cols / CC) {
                        const int nch = p.h_stride / CC;  // chunk-interleaved: float4 i/4 of chunk ch
                        const float* hrow = hs + (size_t)(pr - ha) * p.h_stride + ch * 4;
#pragma unroll
                        for (int i = 0; i < CC; i += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(hrow + (i >> 2) * nch * 4);
                            hd.v[i] = v.x, hd.v[i + 1] = v.y, hd.v[i + 2] = v.z, hd.v[i + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < CC; ++i) hd.v[i] = 0.0f;
                    }
                    hf_sum(hd);
                    const uint32_t rb = (uint32_t)cols * BITS / 8, dsb = (uint32_t)cols / 16;
                    const uint8_t* unit = Dbuf + (size_t)s * dstage + (size_t)(a - aa - s * dcs) * p.d_unit;
                    const uint8_t* sbase = unit + p.d_rows_bytes + ((j0 * dsb) & 15u);
                    const float wp = D.pair_w[pr];
                    if (halves) {
                        // 16 chunks per row: eight rows per pass as four row pairs of
                        // half-warps, their butterflies interleaved (rows past the end
                        // repeat the last row and are dropped)
#pragma unroll 1
                        for (int jj = 0; jj < jn; jj += 8) {
                            const uint8_t* q8[8];
                            const uint32_t* sb8[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int jr = min(jj + i, jn - 1);
                                q8[i] = unit + (size_t)jr * rb;
                                sb8[i] = reinterpret_cast<const uint32_t*>(sbase + (size_t)jr * dsb);
                            }
                            float v[4];
                            row_dot_h_halves_n<BITS, 4>(q8, sb8, hd, lane, v);
                            if ((lane & 15) == 0) {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int jo = jj + 2 * i + (lane >> 4);
                                    if (jo < jn) part[(size_t)pr * p.jn + jo] = __fmul_rn(wp, v[i]);
                                }
                            }
                        }
                    } else {
#pragma unroll 1
                        for (int jj = 0; jj < jn; ++jj) {
                            const float v = row_dot_h<BITS>(unit + (size_t)jj * rb,
                                                            reinterpret_cast<const uint32_t*>(sbase + (size_t)jj * dsb),
                                                            hd, cols, lane);
                            if (lane == 0) part[(size_t)pr * p.jn + jj] = __fmul_rn(wp, v);
                        }
                    }
                    if (gated && pr == D.act_off[a] && (reinterpret_cast<uintptr_t>(D.act_blob[a]) & 1u)) {
                        // an expert read from host memory: this CTA's down rows of it into its new slot
                        uint8_t* slot = answer_wait(p, ds, l, dir_l_w, lane) ? miss_slot_of(ds, D.act_expert[a], lane) : nullptr;
                        if (!slot) {
                            okc = false;
                            break;
                        }
                        store_down(slot, unit, j0, jn, H, p.I, BITS, rb, dsb, p.d_rows_bytes, lane);
                    }
                }
                fence_proxy_async();
                if (!__syncthreads_and(okc ? 1 : 0)) {
                    ok = false;
                    break;
                }
                // every stage of the round has completed (each holds an expert some warp waited for)
                const int ns_r = (ab - aa + dcs - 1) / dcs;
#pragma unroll 1
                for (int s = 0; s < ns_r; ++s) {
                    wt.phase ^= 1u << s;
                    wt.armed &= ~(1u << s);
                }
                if (rd + 1 < rounds) {
                    const int na0 = (rd + 1) * kNSD * dcs;
#pragma unroll 1
                    for (int s = 0; s < kNSD && na0 + s * dcs < n_act; ++s) {
                        if (tid == 0)
                            issue_down(p, D, na0 + s * dcs, min(n_act, na0 + (s + 1) * dcs), j0, jn,
                                       Dbuf + (size_t)s * dstage, &mbar[kMbD + s]);
                        wt.armed |= 1u << s;
                    }
                }
            }
            if (!ok) break;
        }
        // y rows of this CTA: ascending expert order per token
        const bool withhold = c == p.fault_cta && li == 0 && p.n_layers > 1;
#pragma unroll 1
        for (int i = tid; i < B * jn; i += kST) {
            const int t = i / jn, jj = i - t * jn;
            float acc = 0.0f;
#pragma unroll 1
            for (int pr = 0; pr < n_pairs; ++pr)
                if (D.pair_token[pr] == t) acc = __fadd_rn(acc, part[(size_t)pr * p.jn + jj]);
            const size_t o = (size_t)t * H + j0 + jj;
            if (!withhold) ll_store(p.y_ll + (size_t)par * kMaxB * H + o, acc, ep);
            if (l == lend - 1) p.y_out[o] = acc;
            if (p.y_trace) p.y_trace[(size_t)li * B * H + o] = acc;
        }
        __syncthreads();
    }
    // drain outstanding copies (bounded) before the CTA's shared memory goes away
    __syncthreads();
#pragma unroll 1
    for (int s = 0; s < kRing; ++s)
        if (warm & (1u << s)) {
            const unsigned long long t0 = gtime();
            while (!mbar_test(&mbar[warp * kRing + s], (wph >> s) & 1u) && gtime() - t0 < p.wait_ns) {
            }
        }
#pragma unroll 1
    for (int i = kMbD; i < kNB; ++i) {
        const uint32_t bit = 1u << (i - kMbD);
        if (wt.armed & bit) {
            const unsigned long long t0 = gtime();
            while (!mbar_test(&mbar[i], (wt.phase & bit) ? 1u : 0u) && gtime() - t0 < p.wait_ns) {
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
bool plan(const Shapes& sh, int B, int grid, int max_smem, Params& p) {
    const int H = sh.hidden, E = sh.n_experts, k = sh.top_k, bits = sh.bits;
    auto r128 = [](long long v) { return (int)((v + 127) / 128 * 128); };
    const int G = grid;
    p.rE = (E + G - 1) / G;
    p.rS = (sh.shared_inter + G - 1) / G;
    p.jn = (H + G - 1) / G;
    const int qb = H * bits / 8, sbb = H / 16;
    p.off_sg = p.rE * 2 * H + p.rS * 2 * (qb + sbb);  // a multiple of 16
    p.p_bytes = r128((long long)p.off_sg + 2 * H);
    p.g_unit = r16i(2 * (qb + sbb));
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
    p.off_P = off;  // [2][p_bytes], by layer parity
    off += 2 * p.p_bytes;
    p.off_dirs = off;  // [2][E] blob addresses
    off += r128(2LL * E * 8);
    const int budget = max_smem - 1024;  // static shared memory of the kernel
    const int left = budget - off;
    // down stages: every active expert in the two stages if that leaves each
    // warp two gate/up slots, else fewer experts per stage
    int d_cap = (p.amax + kNSD - 1) / kNSD;
    auto ring_for = [&](int dc) { return (left - kNSD * dc * p.d_unit) / (kSW * p.g_unit); };
    while (d_cap > 1 && ring_for(d_cap) < 2) --d_cap;
    p.d_cap = d_cap;
    p.ring = std::min(kRing, ring_for(d_cap));
    if (p.ring < 1) return false;
    p.g_bytes = kSW * p.ring * p.g_unit;
    // the gate/up area also holds the top-k scratch
    if (topk_temp_bytes(B, E, k) > p.g_bytes) return false;
    p.off_G = off;
    off += p.g_bytes;
    off = r128(off);
    p.off_D = off;
    off += kNSD * p.d_cap * p.d_unit;
    p.smem_bytes = off;
    return off <= budget;
}

// ONE: the batch-1 instance; STREAM: the instance of streaming contexts (all
// the residency and slot-filling code lives only there)
void* select_kernel(int bits, bool one, bool stream) {
    if (bits == 4) {
        if (stream)
            return one ? reinterpret_cast<void*>(&stack_kernel<4, true, true>)
                       : reinterpret_cast<void*>(&stack_kernel<4, false, true>);
        return one ? reinterpret_cast<void*>(&stack_kernel<4, true, false>)
                   : reinterpret_cast<void*>(&stack_kernel<4, false, false>);
    }
    if (bits == 8) {
        if (stream)
            return one ? reinterpret_cast<void*>(&stack_kernel<8, true, true>)
                       : reinterpret_cast<void*>(&stack_kernel<8, false, true>);
        return one ? reinterpret_cast<void*>(&stack_kernel<8, true, false>)
                   : reinterpret_cast<void*>(&stack_kernel<8, false, false>);
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
    for (int v = 0; v < 4; ++v)
        if (void* f = select_kernel(sh.bits, (v & 1) != 0, (v & 2) != 0)) {
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
    if (sh.n_experts > 2 * kST) return false;  // two keys per lane in the first top-k level
    if (sh.n_experts % 2) return false;        // directory rows are bulk-copied: 16-byte aligned rows
    if (!select_kernel(sh.bits, B == 1, false)) return false;
    const int cmax = std::max(sh.inter, sh.shared_inter);
    if (cmax * sh.bits / 128 > 32) return false;  // one chunk per lane on down rows
    Params p{};
    return plan(sh, B, s.grid, s.max_smem, p);
}

int stack_last_status(const StackScratch& s) { return s.status_host ? *(volatile int*)s.status_host : 0; }

cudaError_t stack_clear_abandoned(StackScratch& s) {
    if (!s.status_host || *(volatile int*)s.status_host != kStatusAbandoned) return cudaSuccess;
    const cudaError_t e = cudaMemset(s.status, 0, sizeof(int));
    if (e == cudaSuccess) *(volatile int*)s.status_host = 0;
    return e;
}

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
    p.wait_ns = a.fault ? kFaultWaitNs : kWaitNs;
    p.fault_cta = a.fault ? s.grid - 1 : -1;
    if (a.pub) {
        if (!a.dir_patch || a.B * sh.top_k > kMaxMiss) return cudaErrorInvalidValue;
        p.pub_idx = a.pub->idx, p.pub_stride = a.pub->idx_stride;
        p.pub_ready = a.pub->ready, p.pub_gated = a.pub->gated;
        p.served = const_cast<const uint32_t*>(a.pub->served);
        p.serve_n = const_cast<const int32_t*>(a.pub->serve_n);
        p.serve_tab = a.pub->serve_tab, p.serve_stride = a.pub->serve_stride;
        p.dir_patch = a.dir_patch, p.store = a.store, p.store_stride = a.store_stride, p.epoch = a.epoch;
    }
    void* f = select_kernel(sh.bits, a.B == 1, a.pub != nullptr);
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(f, dim3(s.grid), dim3(kST), args, (size_t)p.smem_bytes, st);
}

}  // namespace moe
