// api.cu -- the C ABI of libmoe.so (see include/moe.h): context, expert store,
// HBM slot pool, miss engine and the forward entry points.
//
// Data layout in HBM (64-bit offsets throughout, the "byte-addressed kernels
// with 64-bit offsets" of the Swiftlet README, "Relation to TurboFieldfare"):
//   pool        [n_layers][pool_slots][stride] routed expert blobs
//   shared_pool [n_layers][shared_stride]      shared expert blobs
//   router_w    [n_layers][E][H] bf16, router_bias [n_layers][E] fp32,
//   shared_gate [n_layers][H] bf16
//   dir         [n_layers][E] blob address of each resident expert, NULL if not
// Streaming contexts keep the full store in pinned host memory
//   store       [n_layers][E][stride]
// and fetch a missed expert with one cudaMemcpyAsync of one stride on a side
// stream -- the CUDA counterpart of Swiftlet's one pread per expert from the
// fixed-stride container (article section 2; explainer "Flujo de Inferencia"
// steps 3-6).  Behind the per-layer kernels the compute stream waits on an
// event recorded after the copies, which is this library's explicit hazard
// management between slot refills and the kernels that read them.  Behind the
// persistent decode kernel (a few tokens) there is no copy at all: the store
// is mapped pinned memory, the kernel reads a missing expert's rows straight
// from it over the host-device link and writes them into the slot the pool
// chose, which the host names in mapped memory while the rows are in flight.  A streaming context can instead take its
// routed blobs from an expert container on disk (store.cpp): a miss is then
// one positioned read of the blob into a pinned staging buffer followed by the
// same copy, which is Swiftlet's own fetch path.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "moe_internal.h"
#include "store.h"
#include "prefill.h"
#include "stack.h"

int32_t moe_slotpool_resident(const moe_slotpool* p);

namespace {

thread_local std::string g_create_error;

struct LayerStats {
    uint64_t hits = 0, misses = 0, evictions = 0, h2d_bytes = 0;
    double h2d_ms = 0.0;
    int32_t calls = 0;
};

}  // namespace

struct moe_ctx {
    moe_config cfg{};
    moe::Shapes sh{};
    size_t stride = 0, shared_stride = 0;  // slot pitches: the widest layer's blob strides
    // per layer: bits, shapes handed to the per-layer kernels, blob strides
    std::vector<int32_t> lbits;
    std::vector<moe::Shapes> lsh;
    std::vector<size_t> lstride, lsstride;
    bool mixed = false;  // layers of different widths
    bool resident = false, poisoned = false;
    std::string err;

    // device
    uint8_t* pool = nullptr;
    uint8_t* shared_pool = nullptr;
    uint16_t* router_w = nullptr;
    float* router_bias = nullptr;
    uint16_t* shared_gate = nullptr;
    const uint8_t** dir = nullptr;
    unsigned long long* hits_dev = nullptr;
    float* logits = nullptr;
    float* sigma = nullptr;
    int32_t* idx = nullptr;
    float* w = nullptr;
    float* h = nullptr;
    float* part = nullptr;  // [max_pairs][H] weighted down rows of each pair
    float* xbuf = nullptr;  // [2][max_batch][H]
    float* ybuf = nullptr;  // [max_batch][H]
    // streaming, whole-stack calls: each layer's input [n_layers][max_batch][H],
    // the last layer's output, and one CUDA graph per layer (and one for the
    // first routing) for the call's batch size
    float* xring = nullptr;
    float* yout = nullptr;
    std::vector<cudaGraphExec_t> graphs;  // [0] first routing, [1 + l] layer l's dispatch .. next routing
    int graph_B = 0;
    float graph_eps = 0.0f;
    bool graphs_off = false;
    cudaStream_t cap = nullptr;
    void* disp_mem = nullptr;
    moe::Dispatch disp{};
    moe::TokenDigits xd{};
    moe::StackScratch stack{};
    moe::PrefillScratch pre{};
    // prefill kernel timing: a ring of event sets, harvested lazily
    static constexpr int kProfRing = 32;
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;  // [kProfRing][kPrefillKernels + 1]
    int64_t prof_calls = 0, prof_harvested = 0;
    double prof_ms[moe::kPrefillKernels] = {};

    // host
    uint8_t* store = nullptr;      // mapped pinned store [n_layers][E][stride]
    uint8_t* store_dev = nullptr;  // its device alias
    // streaming from an expert container: the open file and a pinned staging
    // ring, each buffer reused only after its copy to the slot has run
    moe::StoreFile file{};
    std::string store_path;
    // (mapped: the persistent kernel reads a staged blob during its layer, so a
    // buffer is reused within a call only for a later layer; kStage > kMaxMiss)
    static constexpr int kStage = 64;
    uint8_t* stage = nullptr;  // [kStage][stride]
    uint8_t* stage_dev = nullptr;
    cudaEvent_t stage_ev[kStage] = {};  // completes when the buffer's last reader has
    bool stage_used[kStage] = {};
    uint32_t stage_epoch[kStage] = {};  // call (epoch) and layer of a persistent launch's read, 0: none
    int stage_layer[kStage] = {};
    int stage_next = 0;
    const uint8_t** dir_host = nullptr;  // streaming: the host's directory (pinned), copied to dir on misses
    // streaming: mapped pinned block: ready [n_layers] (uint32, written by the
    // publish kernel), the call's epoch (written by the host), then the
    // published routing [max_batch * top_k]
    void* gate_mem = nullptr;
    moe::HostGate gate_host{}, gate_dev{};
    uint32_t epoch = 0;
    // router-bias updates go through a pinned ring, so they never synchronise
    static constexpr int kBiasSlots = 8;
    float* bias_stage = nullptr;  // [kBiasSlots][n_layers * n_experts]
    cudaEvent_t bias_ev[kBiasSlots] = {};
    bool bias_used[kBiasSlots] = {};
    int bias_next = 0;
    // miss-copy timing: one event pair per served layer with misses, harvested once complete
    static constexpr int kTimeRing = 64;
    cudaEvent_t tev[kTimeRing][2] = {};
    int tlayer[kTimeRing] = {};
    int64_t t_rec = 0, t_harv = 0;
    std::vector<uint8_t> loaded;
    std::vector<moe_slotpool*> pools;
    int32_t active_slots = 0;  // slots in use per layer (<= cfg.pool_slots, the reserved stride)
    std::vector<LayerStats> stats;
    std::vector<int32_t> trace;
    cudaStream_t side = nullptr;
    int64_t miss_copies = 0;
    bool fault_timeout_armed = false;
    bool fault_device_armed = false;  // MOE_FAULT_DEVICE_WAIT, not yet spent
    uint64_t launches = 0;
};

namespace {

int fail(moe_ctx* c, int code, const char* fmt, ...) __attribute__((format(printf, 3, 4)));

int fail(moe_ctx* c, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) {
        c->err = buf;
        if (code == MOE_ECUDA) c->poisoned = true;
    } else {
        g_create_error = buf;
    }
    return code;
}

#define CUDA_TRY(ctx, expr)                                                                          \
    do {                                                                                             \
        cudaError_t e_ = (expr);                                                                     \
        if (e_ != cudaSuccess)                                                                       \
            return fail((ctx), MOE_ECUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                                         \
    } while (0)

int timeout_ms(const moe_ctx* c) { return c->cfg.timeout_ms > 0 ? c->cfg.timeout_ms : 10000; }

// Bounded host wait on an event: polls cudaEventQuery until the deadline.
int wait_event(moe_ctx* c, cudaEvent_t ev) {
    if (c->fault_timeout_armed) {
        c->fault_timeout_armed = false;
        return fail(c, MOE_ETIMEOUT, "host wait timed out (injected)");
    }
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms(c));
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorNotReady)
            return fail(c, MOE_ECUDA, "cudaEventQuery failed: %s", cudaGetErrorString(e));
        if (std::chrono::steady_clock::now() > deadline)
            return fail(c, MOE_ETIMEOUT, "host wait exceeded %d ms", timeout_ms(c));
        std::this_thread::yield();
    }
}

int check_config(const moe_config* g) {
    if (!g) return fail(nullptr, MOE_EINVAL, "cfg is NULL");
    if (g->n_layers < 1) return fail(nullptr, MOE_EINVAL, "n_layers must be >= 1");
    if (g->hidden < 256 || g->hidden % 256) return fail(nullptr, MOE_EINVAL, "hidden must be a multiple of 256");
    if (g->n_experts < 1 || g->n_experts > 1024) return fail(nullptr, MOE_EINVAL, "n_experts must be in 1..1024");
    if (g->top_k < 1 || g->top_k > 16 || g->top_k > g->n_experts)
        return fail(nullptr, MOE_EINVAL, "top_k must be in 1..min(16, n_experts)");
    if (g->inter < 64 || g->inter % 64) return fail(nullptr, MOE_EINVAL, "inter must be a positive multiple of 64");
    if (g->shared_inter < 0 || g->shared_inter % 64)
        return fail(nullptr, MOE_EINVAL, "shared_inter must be a multiple of 64");
    if (g->bits != 4 && g->bits != 8) return fail(nullptr, MOE_EINVAL, "bits must be 4 or 8");
    // with layer_bits every layer's own width bounds its rows; `bits` alone otherwise
    if (!g->layer_bits && (g->inter * g->bits > 4096 || g->shared_inter * g->bits > 4096))
        return fail(nullptr, MOE_EINVAL, "inter * bits must be <= 4096 (inter <= 1024 for int4, <= 512 for int8)");
    if (g->layer_bits) {
        bool mixed = false;
        for (int l = 0; l < g->n_layers; ++l) {
            const int b = g->layer_bits[l];
            if (b != 4 && b != 8) return fail(nullptr, MOE_EINVAL, "layer_bits[%d] = %d: must be 4 or 8", l, b);
            if (g->inter * b > 4096 || g->shared_inter * b > 4096)
                return fail(nullptr, MOE_EINVAL, "layer_bits[%d]: inter * bits must be <= 4096", l);
            mixed |= b != g->layer_bits[0];
        }
        if (mixed && g->store_path)
            return fail(nullptr, MOE_EINVAL, "an expert container holds one width: no store_path with mixed layer_bits");
    }
    if (g->group_size != 64) return fail(nullptr, MOE_EINVAL, "group_size must be 64");
    if (g->pool_slots < g->top_k || g->pool_slots > g->n_experts)
        return fail(nullptr, MOE_EINVAL, "pool_slots must be in top_k..n_experts");
    if (g->policy < MOE_EVICT_LFU_RECENCY || g->policy > MOE_EVICT_LFU_AGED)
        return fail(nullptr, MOE_EINVAL, "unknown eviction policy");
    if (g->max_batch < 1 || g->max_batch > 64) return fail(nullptr, MOE_EINVAL, "max_batch must be in 1..64");
    if (g->store_flags & ~MOE_STORE_DIRECT) return fail(nullptr, MOE_EINVAL, "unknown store_flags");
    if (g->store_path && g->pool_slots == g->n_experts)
        return fail(nullptr, MOE_EINVAL, "store_path needs a streaming context (pool_slots < n_experts)");
    if (g->max_tokens < 0 || g->max_tokens > (1 << 20)) return fail(nullptr, MOE_EINVAL, "max_tokens out of range");
    return MOE_OK;
}

template <class T>
int dev_alloc(moe_ctx* c, T** p, size_t n, const char* what) {
    if (n == 0) n = 1;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(c, MOE_ENOMEM, "cudaMalloc(%s, %zu bytes) failed: %s", what, n * sizeof(T),
                    cudaGetErrorString(e));
    }
    return MOE_OK;
}

int check_layer(moe_ctx* c, int32_t layer) {
    if (c->poisoned) return fail(c, MOE_ESTATE, "context poisoned by an earlier CUDA error");
    if (layer < 0 || layer >= c->cfg.n_layers) return fail(c, MOE_EINVAL, "layer %d out of range", layer);
    if (!c->loaded[layer]) return fail(c, MOE_ESTATE, "layer %d has not been loaded", layer);
    return MOE_OK;
}

const uint8_t* shared_blob(moe_ctx* c, int layer) {
    return c->cfg.shared_inter > 0 ? c->shared_pool + (size_t)layer * c->shared_stride : nullptr;
}

// Account the device time of served layers' miss copies, oldest first: those
// already complete, or (wait) all of them.
void harvest_copy_timing(moe_ctx* c, bool wait) {
    for (; c->t_harv < c->t_rec; ++c->t_harv) {
        const int i = (int)(c->t_harv % moe_ctx::kTimeRing);
        if (wait)
            cudaEventSynchronize(c->tev[i][1]);
        else if (cudaEventQuery(c->tev[i][1]) != cudaSuccess)
            break;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, c->tev[i][0], c->tev[i][1]) == cudaSuccess) c->stats[c->tlayer[i]].h2d_ms += ms;
        cudaGetLastError();
    }
}

// Streaming through the persistent kernel: the host gives up the call from
// layer l on.  A layer the kernel waits at (now or later) reads serve_n < 0
// and the kernel ends within microseconds; the host waits for that (bounded).
// A launch that merely ended this way leaves the context usable (its status
// word is cleared); failures that left the pool ahead of the slots (a copy or
// a read that never ran) have poisoned the context already, and so does a
// stream that does not drain.
void abandon_layers(moe_ctx* c, int l, int lend, uint32_t epoch, cudaStream_t st) {
    for (int i = l; i < lend; ++i) c->gate_host.serve_n[i] = -1;
    std::atomic_thread_fence(std::memory_order_seq_cst);
    for (int i = l; i < lend; ++i) c->gate_host.served[i] = epoch;
    std::atomic_thread_fence(std::memory_order_seq_cst);
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms(c));
    for (;;) {
        const cudaError_t e = cudaStreamQuery(st);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady || std::chrono::steady_clock::now() > deadline) {
            cudaGetLastError();
            c->poisoned = true;
            return;
        }
        std::this_thread::yield();
    }
    if (moe::stack_clear_abandoned(c->stack) != cudaSuccess) c->poisoned = true;
}

// Streaming, host side of one layer: wait until the layer's routing has been
// published (mapped memory, polled) and run the slot pool policy on it.
// Behind the per-layer kernels (gated_launch false) each missed expert's blob
// is copied into its slot with cudaMemcpyAsync on the side stream, the compute
// stream waits on an event after the copies, and the layer's device directory
// is rewritten before the dispatch enqueued next.  Behind the persistent
// kernel (gated_launch true) nothing is copied: the kernel, which found the
// same experts absent, reads their rows from host memory (the mapped store,
// or a staging buffer that the blob is first read into from the container)
// and needs only the answer -- slots, staging buffers, evictions -- to fill
// the slots and patch the device directory itself.
int serve_layer(moe_ctx* c, int layer, int B, uint32_t epoch, cudaStream_t st, bool gated_launch) {
    const int k = c->cfg.top_k, E = c->cfg.n_experts;
    if (c->fault_timeout_armed) {
        c->fault_timeout_armed = false;
        return fail(c, MOE_ETIMEOUT, "host wait timed out (injected)");
    }
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms(c));
    for (uint32_t spin = 0; c->gate_host.ready[layer] != epoch; ++spin) {
        if ((spin & 255u) == 255u) {
            if (std::chrono::steady_clock::now() > deadline)
                return fail(c, MOE_ETIMEOUT, "the routing of layer %d was not published within %d ms", layer,
                            timeout_ms(c));
            const cudaError_t e = cudaStreamQuery(st);
            if (e != cudaSuccess && e != cudaErrorNotReady)
                return fail(c, MOE_ECUDA, "compute stream failed: %s", cudaGetErrorString(e));
        }
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    const bool gated = gated_launch && c->gate_host.gated[layer] == epoch;  // the kernel waits for the answer
    harvest_copy_timing(c, false);
    const int32_t* pub = c->gate_host.idx + (size_t)layer * c->gate_host.idx_stride;
    std::vector<int32_t> req(pub, pub + B * k);
    std::sort(req.begin(), req.end());
    req.erase(std::unique(req.begin(), req.end()), req.end());
    std::vector<int32_t> ev(4 * req.size());
    int rc = moe_slotpool_request(c->pools[layer], req.data(), (int32_t)req.size(), ev.data());
    if (rc < 0)
        return fail(c, rc, "slot pool request of %zu experts failed (pool has %d slots)", req.size(),
                    c->active_slots);
    LayerStats& S = c->stats[layer];
    const int64_t call_no = S.calls;
    const uint8_t** dirh = c->dir_host + (size_t)layer * E;
    size_t n_miss = 0;
    for (size_t i = 0; i < req.size(); ++i) n_miss += ev[4 * i + 1] != 0 ? 1 : 0;
    if (gated_launch && (n_miss > 0) != gated) {  // pool and device directory disagree: nothing later can be trusted
        fail(c, MOE_ESTATE, "layer %d: the pool %s while the device found every expert %s", layer,
             n_miss ? "misses" : "hits", n_miss ? "resident" : "but one");
        c->poisoned = true;
        return MOE_ESTATE;
    }
    // the pool has decided the slots: the host directory first
    struct Miss {
        int32_t e;
        uint8_t* dst;
    };
    std::vector<Miss> miss;
    std::vector<int32_t> evicted;
    for (size_t i = 0; i < req.size(); ++i) {
        const int32_t e = ev[4 * i], kind = ev[4 * i + 1], slot = ev[4 * i + 2], out = ev[4 * i + 3];
        c->trace.insert(c->trace.end(), {(int32_t)call_no, layer, e, kind, slot, out});
        if (kind == 0) {
            S.hits++;
            continue;
        }
        S.misses++;
        if (out >= 0) {
            S.evictions++;
            dirh[out] = nullptr;
            evicted.push_back(out);
        }
        uint8_t* dst = c->pool + ((size_t)layer * c->cfg.pool_slots + slot) * c->stride;
        miss.push_back({e, dst});
        dirh[e] = dst;
    }
    if (gated_launch) {
        moe::ServeEntry* tab = c->gate_host.serve_tab + (size_t)layer * c->gate_host.serve_stride;
        size_t n = 0;
        for (const Miss& m : miss) {
            const uint8_t* src = nullptr;  // the kernel reads the mapped store itself
            if (!c->store) {               // expert container: one positioned read into a staging buffer
                const int si = c->stage_next;
                c->stage_next = (si + 1) % moe_ctx::kStage;
                if (c->stage_used[si] && !(c->stage_epoch[si] == epoch && c->stage_layer[si] < layer)) {
                    if (c->stage_epoch[si] == epoch)  // (kStage > misses of one layer)
                        return fail(c, MOE_ESTATE, "staging ring overrun at layer %d", layer);
                    CUDA_TRY(c, cudaEventSynchronize(c->stage_ev[si]));  // an earlier call's reader
                }
                uint8_t* buf = c->stage + (size_t)si * c->stride;
                if (moe::store_read_blob(c->file, layer, m.e, buf) != MOE_OK) {
                    fail(c, MOE_EIO, "reading expert %d of layer %d from %s failed", m.e, layer,
                         c->store_path.c_str());
                    c->poisoned = true;  // the pool already counts the expert as resident
                    return MOE_EIO;
                }
                CUDA_TRY(c, cudaEventRecord(c->stage_ev[si], st));  // completes with the kernel reading it
                c->stage_used[si] = true;
                c->stage_epoch[si] = epoch;
                c->stage_layer[si] = layer;
                src = c->stage_dev + (size_t)si * c->stride;
            }
            if ((c->cfg.fault_flags & MOE_FAULT_MISS_COPY) && c->miss_copies == c->cfg.fault_arg) {
                c->miss_copies++;
                return fail(c, MOE_ECUDA, "miss copy %d failed (injected)", c->cfg.fault_arg);
            }
            c->miss_copies++;
            tab[n++] = moe::ServeEntry{m.e, 0, m.dst, src};
            S.h2d_bytes += c->lstride[layer];  // the blob crosses the link once, read by the kernel
        }
        for (int32_t o : evicted) tab[n++] = moe::ServeEntry{-1 - o, 0, nullptr, nullptr};
        if (gated) {
            c->gate_host.serve_n[layer] = (int32_t)(miss.size() | evicted.size() << 16);
            std::atomic_thread_fence(std::memory_order_seq_cst);
            c->gate_host.served[layer] = epoch;
            std::atomic_thread_fence(std::memory_order_seq_cst);
        }
        S.calls++;
        return MOE_OK;
    }
    if (miss.empty()) {
        S.calls++;
        return MOE_OK;
    }
    const int64_t ti = c->t_rec % moe_ctx::kTimeRing;
    if (c->t_rec - c->t_harv == moe_ctx::kTimeRing) harvest_copy_timing(c, true);
    CUDA_TRY(c, cudaEventRecord(c->tev[ti][0], c->side));
    for (const Miss& m : miss) {
        const uint8_t* src = c->store ? c->store + ((size_t)layer * E + m.e) * c->stride : nullptr;
        int stage_i = -1;
        if (!src) {  // expert container: one positioned read into the next staging buffer
            stage_i = c->stage_next;
            c->stage_next = (stage_i + 1) % moe_ctx::kStage;
            if (c->stage_used[stage_i]) CUDA_TRY(c, cudaEventSynchronize(c->stage_ev[stage_i]));
            uint8_t* buf = c->stage + (size_t)stage_i * c->stride;
            if (moe::store_read_blob(c->file, layer, m.e, buf) != MOE_OK) {
                fail(c, MOE_EIO, "reading expert %d of layer %d from %s failed", m.e, layer, c->store_path.c_str());
                c->poisoned = true;  // the pool already counts the expert as resident
                return MOE_EIO;
            }
            src = buf;
        }
        if ((c->cfg.fault_flags & MOE_FAULT_MISS_COPY) && c->miss_copies == c->cfg.fault_arg) {
            c->miss_copies++;
            return fail(c, MOE_ECUDA, "miss copy %d failed (injected)", c->cfg.fault_arg);
        }
        c->miss_copies++;
        // the slot's previous expert was last read before this routing was published
        CUDA_TRY(c, cudaMemcpyAsync(m.dst, src, c->lstride[layer], cudaMemcpyHostToDevice, c->side));
        if (stage_i >= 0) {
            CUDA_TRY(c, cudaEventRecord(c->stage_ev[stage_i], c->side));
            c->stage_used[stage_i] = true;
            c->stage_epoch[stage_i] = 0;
        }
        S.h2d_bytes += c->lstride[layer];
    }
    CUDA_TRY(c, cudaEventRecord(c->tev[ti][1], c->side));
    c->tlayer[ti] = layer;
    c->t_rec++;
    CUDA_TRY(c, cudaStreamWaitEvent(st, c->tev[ti][1], 0));
    // the layer's device directory, read by the dispatch enqueued next (the
    // source is pinned; the host rewrites it only after a later routing of
    // this layer has been published, i.e. after this copy has run)
    CUDA_TRY(c, cudaMemcpyAsync(c->dir + (size_t)layer * E, dirh, sizeof(void*) * E, cudaMemcpyHostToDevice, st));
    std::atomic_thread_fence(std::memory_order_release);
    S.calls++;
    return MOE_OK;
}

// Enqueues one layer of an all-resident context.
int decode_layer(moe_ctx* c, int layer, const float* x, int B, float* y, int32_t* uidx, float* uw,
                 cudaStream_t st) {
    const moe::Shapes& s = c->lsh[layer];
    const int E = c->cfg.n_experts;
    const uint16_t* wr = c->router_w + (size_t)layer * E * c->cfg.hidden;
    const float* bias = c->router_bias + (size_t)layer * E;
    const uint16_t* wsg = c->cfg.shared_inter > 0 ? c->shared_gate + (size_t)layer * c->cfg.hidden : nullptr;
    const uint8_t* const* dir = c->dir + (size_t)layer * E;
    CUDA_TRY(c, moe::launch_router(s, wr, bias, x, B, c->logits, st));
    c->launches += 6;  // router, top-k (per token), dispatch, gate/up, down, combine
    CUDA_TRY(c, moe::launch_route_dispatch(s, 3, c->logits, x, wsg, B, c->idx, c->w, c->sigma, uidx, uw, dir,
                                           shared_blob(c, layer), c->disp, c->xd, c->hits_dev + layer, st));
    CUDA_TRY(c, moe::launch_gateup_batched(s, c->disp, c->xd, c->h, st));
    CUDA_TRY(c, moe::launch_down_batched(s, c->disp, c->h, c->part, st));
    CUDA_TRY(c, moe::launch_combine(s, c->disp, c->part, y, B, c->cfg.shared_inter > 0, st));
    c->stats[layer].calls++;
    return MOE_OK;
}

// Streaming, enqueue helpers.  Routing of layer l: router, top-k and the
// publication of the routing to the host (a separate publish kernel above 8
// tokens): this many kernels.
int route_launches(int B) { return B > 8 ? 3 : 2; }

int enq_route(moe_ctx* c, int l, const float* xin, int B, int32_t* uidx, float* uw, cudaStream_t st) {
    const moe::Shapes& s = c->lsh[l];
    const int H = c->cfg.hidden, k = c->cfg.top_k, E = c->cfg.n_experts;
    const uint16_t* wr = c->router_w + (size_t)l * E * H;
    const float* bias = c->router_bias + (size_t)l * E;
    const uint16_t* wsg = c->cfg.shared_inter > 0 ? c->shared_gate + (size_t)l * H : nullptr;
    CUDA_TRY(c, moe::launch_router(s, wr, bias, xin, B, c->logits, st));
    CUDA_TRY(c, moe::launch_route_dispatch(s, 1, c->logits, xin, wsg, B, c->idx, c->w, c->sigma, uidx, uw, nullptr,
                                           nullptr, c->disp, c->xd, nullptr, st, &c->gate_dev, l));
    (void)k;
    return MOE_OK;
}

// ... and the rest of layer l once the host has served it: dispatch (reading
// the directory the host has just written), gate/up, down, combine into yl.
int enq_post(moe_ctx* c, int l, const float* xin, int B, float* yl, cudaStream_t st) {
    const moe::Shapes& s = c->lsh[l];
    const int H = c->cfg.hidden, E = c->cfg.n_experts;
    const uint16_t* wsg = c->cfg.shared_inter > 0 ? c->shared_gate + (size_t)l * H : nullptr;
    CUDA_TRY(c, moe::launch_route_dispatch(s, 2, c->logits, xin, wsg, B, c->idx, c->w, c->sigma, nullptr, nullptr,
                                           c->dir + (size_t)l * E, shared_blob(c, l), c->disp, c->xd, nullptr, st));
    CUDA_TRY(c, moe::launch_gateup_batched(s, c->disp, c->xd, c->h, st));
    CUDA_TRY(c, moe::launch_down_batched(s, c->disp, c->h, c->part, st));
    CUDA_TRY(c, moe::launch_combine(s, c->disp, c->part, yl, B, c->cfg.shared_inter > 0, st));
    return MOE_OK;
}

// Streaming stacks of a few tokens run as one persistent launch per call: the
// kernel publishes every layer's routing, reads a missing expert's rows from
// host memory itself and needs the host's answer only to fill the slots (see
// serve_layer).  Results are bitwise those of the all-resident persistent
// kernel.
bool stream_stack_ok(const moe_ctx* c, int B) {
    return !c->resident && !c->mixed && B <= moe::kStackPreferMaxB &&
           c->active_slots >= B * c->cfg.top_k && moe::stack_supported(c->sh, c->stack, B);
}

int enq_stack_streaming(moe_ctx* c, int l, int lend, const float* x, int B, float eps, float* y, uint32_t epoch,
                        cudaStream_t st) {
    moe::StackArgs a{};
    a.layer0 = l;
    a.n_layers = lend - l;
    a.B = B;
    a.eps = eps;
    a.x = x;
    a.y = y;
    a.router_w = c->router_w;
    a.router_bias = c->router_bias;
    a.shared_gate = c->cfg.shared_inter > 0 ? c->shared_gate : nullptr;
    a.dir = c->dir;
    a.shared_pool = c->cfg.shared_inter > 0 ? c->shared_pool : nullptr;
    a.shared_stride = c->shared_stride;
    a.pub = &c->gate_dev;
    a.dir_patch = c->dir;
    a.store = c->store ? c->store_dev : nullptr;
    a.store_stride = c->stride;
    a.epoch = epoch;
    const cudaError_t e = moe::launch_stack(c->sh, c->stack, a, st);
    if (e != cudaSuccess) return fail(c, MOE_ECUDA, "decode stack launch failed: %s", cudaGetErrorString(e));
    c->launches += 1;
    return MOE_OK;
}

// One CUDA graph per layer for whole-stack calls of B tokens: [0] routes layer
// 0 from xring[0]; [1 + l] runs layer l's dispatch .. combine and, below the
// last layer, renormalises into xring[l + 1] and routes layer l + 1.
int build_graphs(moe_ctx* c, int B, float eps) {
    const int L = c->cfg.n_layers, H = c->cfg.hidden;
    const size_t tok = (size_t)c->cfg.max_batch * H;
    for (cudaGraphExec_t g : c->graphs)
        if (g) cudaGraphExecDestroy(g);
    c->graphs.assign(L + 1, nullptr);
    c->graph_B = 0;
    auto capture = [&](int idx, auto&& body) -> int {
        cudaGraph_t g = nullptr;
        CUDA_TRY(c, cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
        const int rc = body();
        const cudaError_t e = cudaStreamEndCapture(c->cap, &g);
        if (rc || e != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            cudaGetLastError();
            return rc ? rc : fail(c, MOE_ECUDA, "graph capture failed: %s", cudaGetErrorString(e));
        }
        const cudaError_t ei = cudaGraphInstantiate(&c->graphs[idx], g, 0);
        cudaGraphDestroy(g);
        if (ei != cudaSuccess) return fail(c, MOE_ECUDA, "cudaGraphInstantiate failed: %s", cudaGetErrorString(ei));
        return MOE_OK;
    };
    int rc = capture(0, [&] { return enq_route(c, 0, c->xring, B, nullptr, nullptr, c->cap); });
    for (int l = 0; l < L && !rc; ++l) {
        rc = capture(1 + l, [&]() -> int {
            const float* xl = c->xring + (size_t)l * tok;
            if (l == L - 1) return enq_post(c, l, xl, B, c->yout, c->cap);
            int r = enq_post(c, l, xl, B, c->ybuf, c->cap);
            if (r) return r;
            float* xn = c->xring + (size_t)(l + 1) * tok;
            CUDA_TRY(c, moe::launch_renorm(c->ybuf, xn, B, H, eps, c->cap));
            return enq_route(c, l + 1, xn, B, nullptr, nullptr, c->cap);
        });
    }
    if (!rc) {
        c->graph_B = B;
        c->graph_eps = eps;
    }
    return rc;
}

// Streaming: layers layer0 .. layer0+n-1 of one call.  Per layer, the routing
// (router, top-k, publication) is enqueued; the host polls for it, serves the
// slot pool (miss copies on the side stream, the compute stream ordered after
// them by an event) and then enqueues the dispatch, gate/up, down, combine and
// the next layer's routing -- one graph launch per layer for whole-stack calls.
// No kernel ever waits on the host or on another stream.
int stream_layers(moe_ctx* c, int layer0, int n, const float* x, int B, float* y, float eps, float* x_trace,
                  int32_t* idx_trace, float* y_trace, int32_t* uidx, float* uw, cudaStream_t st) {
    const int H = c->cfg.hidden, k = c->cfg.top_k, L = c->cfg.n_layers;
    const size_t tok = (size_t)B * H;
    const uint32_t epoch = ++c->epoch ? c->epoch : ++c->epoch;  // never 0
    *const_cast<volatile uint32_t*>(c->gate_host.epoch) = epoch;
    std::atomic_thread_fence(std::memory_order_seq_cst);
    const bool plain = !x_trace && !idx_trace && !y_trace && !uidx && !uw;
    if (plain && stream_stack_ok(c, B)) {
        // one persistent launch; the host answers each layer as it is published
        if (moe::stack_last_status(c->stack))
            return fail(c, MOE_ETIMEOUT, "a device-side wait of an earlier decode-stack launch ran out (status %d)",
                        moe::stack_last_status(c->stack)) == MOE_ETIMEOUT
                       ? (c->poisoned = true, MOE_ETIMEOUT)
                       : MOE_ETIMEOUT;
        int rc = enq_stack_streaming(c, layer0, layer0 + n, x, B, eps, y, epoch, st);
        for (int l = layer0; l < layer0 + n && !rc; ++l) {
            rc = serve_layer(c, l, B, epoch, st, true);
            if (rc) abandon_layers(c, l, layer0 + n, epoch, st);
        }
        return rc;
    }
    const bool whole = layer0 == 0 && n == L && !x_trace && !idx_trace && !y_trace && !uidx && !uw;
    if (whole && !c->graphs_off && (c->graph_B != B || c->graph_eps != eps)) {
        const bool was_poisoned = c->poisoned;
        if (build_graphs(c, B, eps)) {
            // a launch that cannot be captured failed on the capture stream
            // only: fall back to plain launches for the rest of the context's life
            c->graphs_off = true;
            c->poisoned = was_poisoned;
            c->err.clear();
        }
    }
    if (whole && !c->graphs_off) {
        CUDA_TRY(c, cudaMemcpyAsync(c->xring, x, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
        CUDA_TRY(c, cudaGraphLaunch(c->graphs[0], st));
        c->launches += route_launches(B);
        for (int l = 0; l < n; ++l) {
            int rc = serve_layer(c, l, B, epoch, st, false);
            if (rc) return rc;
            CUDA_TRY(c, cudaGraphLaunch(c->graphs[1 + l], st));
            c->launches += 4 + (l == L - 1 ? 0 : 1 + route_launches(B));  // post, renorm, next routing
        }
        CUDA_TRY(c, cudaMemcpyAsync(y, c->yout, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
        return MOE_OK;
    }
    const float* xin = x;
    auto route = [&](int i) -> int {
        if (x_trace) CUDA_TRY(c, cudaMemcpyAsync(x_trace + i * tok, xin, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
        c->launches += route_launches(B);
        return enq_route(c, layer0 + i, xin, B, idx_trace ? idx_trace + (size_t)i * B * k : uidx, idx_trace ? nullptr : uw,
                         st);
    };
    int rc = route(0);
    for (int i = 0; i < n && !rc; ++i) {
        const int l = layer0 + i;
        if ((rc = serve_layer(c, l, B, epoch, st, false))) break;
        const bool last = i == n - 1;
        float* yl = last ? y : (y_trace ? y_trace + i * tok : c->ybuf);
        if ((rc = enq_post(c, l, xin, B, yl, st))) break;
        c->launches += 4;
        if (last) {
            if (y_trace) CUDA_TRY(c, cudaMemcpyAsync(y_trace + i * tok, y, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
            break;
        }
        float* xn = c->xbuf + (size_t)(i & 1) * c->cfg.max_batch * H;
        CUDA_TRY(c, moe::launch_renorm(yl, xn, B, H, eps, st));
        c->launches += 1;
        xin = xn;
        rc = route(i + 1);
    }
    return rc;
}

// Adds the kernel times of recorded prefill call i (ring slot i % kProfRing).
int prof_harvest_one(moe_ctx* c, int64_t i) {
    cudaEvent_t* ev = c->prof_ev.data() + (size_t)(i % moe_ctx::kProfRing) * (moe::kPrefillKernels + 1);
    CUDA_TRY(c, cudaEventSynchronize(ev[moe::kPrefillKernels]));
    for (int k = 0; k < moe::kPrefillKernels; ++k) {
        float ms = 0.0f;
        CUDA_TRY(c, cudaEventElapsedTime(&ms, ev[k], ev[k + 1]));
        c->prof_ms[k] += ms;
    }
    return MOE_OK;
}

int prof_harvest_all(moe_ctx* c) {
    for (; c->prof_harvested < c->prof_calls; ++c->prof_harvested) {
        int rc = prof_harvest_one(c, c->prof_harvested);
        if (rc) return rc;
    }
    return MOE_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" const char* moe_last_error(moe_ctx* ctx) {
    return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

extern "C" void moe_destroy(moe_ctx* c) {
    if (!c) return;
    if (c->cfg.device >= 0) cudaSetDevice(c->cfg.device);
    if (c->side) cudaStreamSynchronize(c->side);
    cudaDeviceSynchronize();
    cudaFree(c->pool);
    cudaFree(c->shared_pool);
    cudaFree(c->router_w);
    cudaFree(c->router_bias);
    cudaFree(c->shared_gate);
    cudaFree(c->dir);
    cudaFree(c->hits_dev);
    cudaFree(c->logits);
    cudaFree(c->sigma);
    cudaFree(c->idx);
    cudaFree(c->w);
    cudaFree(c->h);
    cudaFree(c->part);
    cudaFree(c->xbuf);
    cudaFree(c->ybuf);
    for (cudaGraphExec_t g : c->graphs)
        if (g) cudaGraphExecDestroy(g);
    cudaFree(c->xring);
    cudaFree(c->yout);
    if (c->cap) cudaStreamDestroy(c->cap);
    cudaFree(c->disp_mem);
    cudaFree(c->xd.words);
    cudaFree(c->xd.sums);
    cudaFree(c->xd.exps);
    moe::stack_free(c->stack);
    moe::prefill_free(c->pre);
    for (cudaEvent_t e : c->prof_ev) cudaEventDestroy(e);
    if (c->store) cudaFreeHost(c->store);
    moe::store_close(c->file);
    if (c->stage) cudaFreeHost(c->stage);
    for (cudaEvent_t e : c->stage_ev)
        if (e) cudaEventDestroy(e);
    if (c->dir_host) cudaFreeHost(c->dir_host);
    if (c->gate_mem) cudaFreeHost(c->gate_mem);
    for (auto* p : c->pools) moe_slotpool_destroy(p);
    if (c->side) cudaStreamDestroy(c->side);
    for (auto& pr : c->tev)
        for (cudaEvent_t e : pr)
            if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : c->bias_ev)
        if (e) cudaEventDestroy(e);
    if (c->bias_stage) cudaFreeHost(c->bias_stage);
    cudaGetLastError();
    delete c;
}

extern "C" int moe_create(const moe_config* cfg, moe_ctx** out) {
    if (!out) return fail(nullptr, MOE_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc) return rc;
    moe_ctx* c = new (std::nothrow) moe_ctx;
    if (!c) return fail(nullptr, MOE_ENOMEM, "host allocation failed");
    c->cfg = *cfg;
    if (cfg->store_path) {
        c->store_path = cfg->store_path;
        c->cfg.store_path = c->store_path.c_str();
    }
    const int L = cfg->n_layers;
    if (cfg->layer_bits)
        c->lbits.assign(cfg->layer_bits, cfg->layer_bits + L);
    else
        c->lbits.assign(L, cfg->bits);
    c->cfg.layer_bits = c->lbits.data();
    c->cfg.bits = c->lbits[0];  // the width of a uniform stack (mixed stacks do not use it)
    const moe_config& g = c->cfg;
    c->resident = g.pool_slots == g.n_experts;
    c->fault_timeout_armed = (g.fault_flags & MOE_FAULT_WAIT_TIMEOUT) != 0;
    c->fault_device_armed = (g.fault_flags & MOE_FAULT_DEVICE_WAIT) != 0;
    const int E = g.n_experts, H = g.hidden, Bm = g.max_batch, k = g.top_k;
    moe::Shapes& s = c->sh;
    s.hidden = H, s.n_experts = E, s.top_k = k, s.inter = g.inter, s.shared_inter = g.shared_inter;
    s.bits = g.bits, s.norm_topk = g.norm_topk ? 1 : 0;
    s.max_act = std::min(E, Bm * k) + 1;
    s.max_pairs = Bm * (k + 1);
    s.h_stride = std::max(g.inter, g.shared_inter);
    s.max_work = s.max_act + s.max_pairs / 8 + 1;
    c->lsh.assign(L, s);
    c->lstride.assign(L, 0);
    c->lsstride.assign(L, 0);
    for (int l = 0; l < L; ++l) {
        c->lsh[l].bits = c->lbits[l];
        c->mixed |= c->lbits[l] != c->lbits[0];
        c->lstride[l] = moe_blob_stride(H, g.inter, c->lbits[l]);
        c->lsstride[l] = g.shared_inter > 0 ? moe_blob_stride(H, g.shared_inter, c->lbits[l]) : 0;
        c->stride = std::max(c->stride, c->lstride[l]);
        c->shared_stride = std::max(c->shared_stride, c->lsstride[l]);
    }
    c->loaded.assign(L, 0);
    c->stats.assign(L, LayerStats{});

    auto bail = [&](int code) {
        std::string msg = c->err;
        moe_destroy(c);
        g_create_error = msg;
        return code;
    };
    if (cudaSetDevice(g.device) != cudaSuccess) {
        cudaGetLastError();
        c->err = "cudaSetDevice failed";
        return bail(MOE_ECUDA);
    }
    if ((rc = dev_alloc(c, &c->pool, (size_t)L * g.pool_slots * c->stride, "slot pool")) ||
        (rc = dev_alloc(c, &c->shared_pool, (size_t)L * c->shared_stride, "shared pool")) ||
        (rc = dev_alloc(c, &c->router_w, (size_t)L * E * H, "router weights")) ||
        (rc = dev_alloc(c, &c->router_bias, (size_t)L * E, "router bias")) ||
        (rc = dev_alloc(c, &c->shared_gate, (size_t)L * H, "shared gate")) ||
        (rc = dev_alloc(c, &c->dir, (size_t)L * E, "directory")) ||
        (rc = dev_alloc(c, &c->hits_dev, (size_t)L, "hit counters")) ||
        (rc = dev_alloc(c, &c->logits, (size_t)Bm * E, "logits")) ||
        (rc = dev_alloc(c, &c->sigma, (size_t)Bm, "sigma")) ||
        (rc = dev_alloc(c, &c->idx, (size_t)Bm * k, "idx")) || (rc = dev_alloc(c, &c->w, (size_t)Bm * k, "w")) ||
        (rc = dev_alloc(c, &c->h, (size_t)s.max_pairs * s.h_stride, "h")) ||
        (rc = dev_alloc(c, &c->part, (size_t)s.max_pairs * H, "down partials")) ||
        (rc = dev_alloc(c, &c->xbuf, (size_t)2 * Bm * H, "xbuf")) ||
        (rc = dev_alloc(c, &c->ybuf, (size_t)Bm * H, "ybuf")) ||
        (rc = dev_alloc(c, &c->xd.words, (size_t)Bm * H * 3 / 4, "token digits")) ||
        (rc = dev_alloc(c, &c->xd.sums, (size_t)Bm * H / 16, "token digit sums")) ||
        (rc = dev_alloc(c, &c->xd.exps, (size_t)Bm, "token exponents")))
        return bail(rc);
    // dispatch scratch in one allocation
    {
        const size_t A = s.max_act, P = s.max_pairs;
        const size_t W = s.max_work;
        const size_t bytes = 16 + A * 4 + A * 8 + (A + 1) * 4 + P * 4 + P * 4 + (size_t)Bm * 17 * 4 + W * 16 + 16 + 256;
        if ((rc = dev_alloc(c, reinterpret_cast<uint8_t**>(&c->disp_mem), bytes, "dispatch"))) return bail(rc);
        uint8_t* p = static_cast<uint8_t*>(c->disp_mem);
        auto take = [&](size_t n) {
            uint8_t* q = p;
            p += (n + 15) / 16 * 16;
            return q;
        };
        c->disp.n_act = reinterpret_cast<int32_t*>(take(4));
        c->disp.status = reinterpret_cast<int32_t*>(take(4));
        c->disp.act_blob = reinterpret_cast<const uint8_t**>(take(A * 8));
        c->disp.act_expert = reinterpret_cast<int32_t*>(take(A * 4));
        c->disp.act_off = reinterpret_cast<int32_t*>(take((A + 1) * 4));
        c->disp.pair_token = reinterpret_cast<int32_t*>(take(P * 4));
        c->disp.pair_w = reinterpret_cast<float*>(take(P * 4));
        c->disp.tok_pairs = reinterpret_cast<int32_t*>(take((size_t)Bm * 17 * 4));
        c->disp.work = reinterpret_cast<int4*>(take(W * 16));
        c->disp.n_work = reinterpret_cast<int32_t*>(take(4));
        if (cudaMemset(c->disp_mem, 0, bytes) != cudaSuccess) {
            c->err = "cudaMemset failed";
            return bail(MOE_ECUDA);
        }
    }
    if (cudaMemset(c->dir, 0, sizeof(void*) * (size_t)L * E) != cudaSuccess ||
        cudaMemset(c->hits_dev, 0, sizeof(unsigned long long) * L) != cudaSuccess ||
        cudaMemset(c->router_bias, 0, sizeof(float) * (size_t)L * E) != cudaSuccess) {
        c->err = "cudaMemset failed";
        return bail(MOE_ECUDA);
    }
    if (g.max_tokens > 0) {
        if (!c->resident) {
            c->err = "prefill (max_tokens > 0) needs an all-resident context (pool_slots == n_experts)";
            return bail(MOE_EINVAL);
        }
        rc = moe::prefill_alloc(c->pre, s, g.max_tokens, g.device, c->err);
        if (rc) return bail(rc);
    }
    // the persistent kernel serves all-resident stacks and, one layer per
    // launch, streaming stacks of a few tokens
    rc = moe::stack_alloc(c->stack, s, L, Bm, g.device, c->err);
    if (rc) return bail(rc);
    if (!c->resident) {
        if (g.fault_flags & MOE_FAULT_PINNED_ALLOC) {
            c->err = "pinned store allocation failed (injected)";
            return bail(MOE_ENOMEM);
        }
        if (g.store_path) {
            if (moe::store_open(g.store_path, (g.store_flags & MOE_STORE_DIRECT) != 0, c->file) != MOE_OK) {
                c->err = "cannot open the expert container " + c->store_path;
                return bail(MOE_EIO);
            }
            const moe::StoreShape& f = c->file.shape;
            if (f.n_layers != L || f.n_experts != E || f.hidden != H || f.inter != g.inter || f.bits != g.bits ||
                f.stride != c->stride) {  // (a container context is uniform: g.bits is every layer's width)
                c->err = "the expert container " + c->store_path + " does not match the config";
                return bail(MOE_EIO);
            }
            if (cudaHostAlloc(reinterpret_cast<void**>(&c->stage), (size_t)moe_ctx::kStage * c->stride,
                              cudaHostAllocMapped) != cudaSuccess ||
                cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->stage_dev), c->stage, 0) != cudaSuccess) {
                cudaGetLastError();
                if (c->stage) cudaFreeHost(c->stage);
                c->stage = nullptr;
                c->err = "cudaHostAlloc of the staging ring failed";
                return bail(MOE_ENOMEM);
            }
            if (c->file.direct && reinterpret_cast<uintptr_t>(c->stage) % 4096 != 0) {
                moe::store_close(c->file);  // direct reads want page-aligned buffers: read through the page cache
                if (moe::store_open(g.store_path, false, c->file) != MOE_OK) {
                    c->err = "cannot open the expert container " + c->store_path;
                    return bail(MOE_EIO);
                }
            }
            for (auto& e : c->stage_ev)
                if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
                    c->err = "cudaEventCreate failed";
                    return bail(MOE_ECUDA);
                }
        } else {
            const size_t store_bytes = (size_t)L * E * c->stride;
            if (cudaHostAlloc(reinterpret_cast<void**>(&c->store), store_bytes, cudaHostAllocMapped) != cudaSuccess ||
                cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->store_dev), c->store, 0) != cudaSuccess) {
                cudaGetLastError();
                if (c->store) cudaFreeHost(c->store);
                c->store = nullptr;
                char buf[160];
                snprintf(buf, sizeof buf, "cudaHostAlloc of the %zu-byte pinned store failed", store_bytes);
                c->err = buf;
                return bail(MOE_ENOMEM);
            }
        }
        // ready, epoch, gated, served, serve_n, idx; then the answer table (16-byte entries)
        const size_t words = 4 * (size_t)L + 1 + (size_t)L * Bm * k;
        const size_t tab_off = (words * 4 + 15) / 16 * 16, tab_stride = 2 * (size_t)Bm * k;
        const size_t gate_bytes = tab_off + sizeof(moe::ServeEntry) * (size_t)L * tab_stride;
        if (cudaHostAlloc(reinterpret_cast<void**>(&c->dir_host), sizeof(void*) * (size_t)L * E,
                          cudaHostAllocDefault) != cudaSuccess ||
            cudaHostAlloc(&c->gate_mem, gate_bytes, cudaHostAllocMapped) != cudaSuccess) {
            cudaGetLastError();
            c->err = "cudaHostAlloc failed";
            return bail(MOE_ENOMEM);
        }
        std::memset(c->dir_host, 0, sizeof(void*) * (size_t)L * E);
        std::memset(c->gate_mem, 0, gate_bytes);
        void* gate_dev = nullptr;
        if (cudaHostGetDevicePointer(&gate_dev, c->gate_mem, 0) != cudaSuccess) {
            cudaGetLastError();
            c->err = "cudaHostGetDevicePointer failed";
            return bail(MOE_ECUDA);
        }
        auto carve = [&](void* base, moe::HostGate& g) {
            uint32_t* w = static_cast<uint32_t*>(base);
            g.ready = w;
            g.epoch = w + L;
            g.gated = w + L + 1;
            g.served = w + 2 * L + 1;
            g.serve_n = reinterpret_cast<int32_t*>(w + 3 * L + 1);
            g.idx = reinterpret_cast<int32_t*>(w + 4 * L + 1);
            g.idx_stride = Bm * k;
            g.serve_tab = reinterpret_cast<moe::ServeEntry*>(static_cast<uint8_t*>(base) + tab_off);
            g.serve_stride = (int)tab_stride;
        };
        carve(c->gate_mem, c->gate_host);
        carve(gate_dev, c->gate_dev);
        c->pools.assign(L, nullptr);
        c->active_slots = g.pool_slots;
        for (int l = 0; l < L; ++l)
            if ((rc = moe_slotpool_create(g.pool_slots, E, g.policy, g.aging_period, &c->pools[l]))) {
                c->err = "slot pool creation failed";
                return bail(rc);
            }
        if (cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess) {
            c->err = "cudaStreamCreate failed";
            return bail(MOE_ECUDA);
        }
        if ((rc = dev_alloc(c, &c->xring, (size_t)L * Bm * H, "xring")) ||
            (rc = dev_alloc(c, &c->yout, (size_t)Bm * H, "yout")))
            return bail(rc);
    }
    for (auto& pr : c->tev)
        for (cudaEvent_t& e : pr)
            if (cudaEventCreate(&e) != cudaSuccess) {
                c->err = "cudaEventCreate failed";
                return bail(MOE_ECUDA);
            }
    *out = c;
    return MOE_OK;
}

extern "C" int moe_load_experts(moe_ctx* c, int32_t layer, const void* blobs, size_t stride,
                                const void* shared_blob_host, const uint16_t* router_w_host,
                                const uint16_t* shared_gate_host, const float* router_bias_host) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    if (c->poisoned) return fail(c, MOE_ESTATE, "context poisoned by an earlier CUDA error");
    const moe_config& g = c->cfg;
    if (layer < 0 || layer >= g.n_layers) return fail(c, MOE_EINVAL, "layer %d out of range", layer);
    const bool from_file = c->file.fd >= 0;
    if (!router_w_host) return fail(c, MOE_EINVAL, "router weights are required");
    if (from_file != (blobs == nullptr))
        return fail(c, MOE_EINVAL, from_file ? "blobs must be NULL: the expert container holds them"
                                             : "blobs are required");
    const size_t ls = c->lstride[layer];  // the layer's blob stride; slots are c->stride apart
    if (!from_file && stride != ls) return fail(c, MOE_EINVAL, "stride %zu != the layer's %zu", stride, ls);
    if ((g.shared_inter > 0) != (shared_blob_host != nullptr) || (g.shared_inter > 0) != (shared_gate_host != nullptr))
        return fail(c, MOE_EINVAL, "shared blob and shared gate are required iff shared_inter > 0");
    CUDA_TRY(c, cudaSetDevice(g.device));
    const int E = g.n_experts, H = g.hidden;
    const size_t layer_bytes = (size_t)E * c->stride;
    if (c->resident) {
        uint8_t* dst = c->pool + (size_t)layer * layer_bytes;
        if (ls == c->stride)
            CUDA_TRY(c, cudaMemcpy(dst, blobs, layer_bytes, cudaMemcpyHostToDevice));
        else  // a narrower layer of a mixed stack: one blob per (wider) slot
            CUDA_TRY(c, cudaMemcpy2D(dst, c->stride, blobs, ls, ls, E, cudaMemcpyHostToDevice));
        std::vector<const uint8_t*> d(E);
        for (int e = 0; e < E; ++e) d[e] = c->pool + ((size_t)layer * E + e) * c->stride;
        CUDA_TRY(c, cudaMemcpy(c->dir + (size_t)layer * E, d.data(), sizeof(void*) * E, cudaMemcpyHostToDevice));
    } else if (!from_file) {
        uint8_t* dst = c->store + (size_t)layer * layer_bytes;
        if (ls == c->stride)
            std::memcpy(dst, blobs, layer_bytes);
        else
            for (int e = 0; e < E; ++e)
                std::memcpy(dst + (size_t)e * c->stride, static_cast<const uint8_t*>(blobs) + (size_t)e * ls, ls);
    }
    if (g.shared_inter > 0) {
        CUDA_TRY(c, cudaMemcpy(c->shared_pool + (size_t)layer * c->shared_stride, shared_blob_host,
                               c->lsstride[layer], cudaMemcpyHostToDevice));
        CUDA_TRY(c, cudaMemcpy(c->shared_gate + (size_t)layer * H, shared_gate_host, sizeof(uint16_t) * H,
                               cudaMemcpyHostToDevice));
    }
    CUDA_TRY(c, cudaMemcpy(c->router_w + (size_t)layer * E * H, router_w_host, sizeof(uint16_t) * (size_t)E * H,
                           cudaMemcpyHostToDevice));
    if (router_bias_host)
        CUDA_TRY(c, cudaMemcpy(c->router_bias + (size_t)layer * E, router_bias_host, sizeof(float) * E,
                               cudaMemcpyHostToDevice));
    else
        CUDA_TRY(c, cudaMemset(c->router_bias + (size_t)layer * E, 0, sizeof(float) * E));
    c->loaded[layer] = 1;
    return MOE_OK;
}

namespace {
// Copies n floats of router bias from (any) host memory to dst through the
// next pinned staging slot, asynchronously on the stream.
int stage_bias(moe_ctx* c, float* dst, const float* src, size_t n, cudaStream_t st) {
    const size_t slot_floats = (size_t)c->cfg.n_layers * c->cfg.n_experts;
    if (!c->bias_stage) {
        if (cudaHostAlloc(reinterpret_cast<void**>(&c->bias_stage), sizeof(float) * slot_floats * moe_ctx::kBiasSlots,
                          cudaHostAllocDefault) != cudaSuccess) {
            cudaGetLastError();
            c->bias_stage = nullptr;
            return fail(c, MOE_ENOMEM, "cudaHostAlloc of the router-bias staging ring failed");
        }
        for (auto& e : c->bias_ev) CUDA_TRY(c, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    }
    const int slot = c->bias_next;
    c->bias_next = (c->bias_next + 1) % moe_ctx::kBiasSlots;
    if (c->bias_used[slot]) {
        int rc = wait_event(c, c->bias_ev[slot]);  // the copy that last used the slot (long done)
        if (rc) return rc;
    }
    float* stage = c->bias_stage + (size_t)slot * slot_floats;
    std::memcpy(stage, src, sizeof(float) * n);
    CUDA_TRY(c, cudaMemcpyAsync(dst, stage, sizeof(float) * n, cudaMemcpyHostToDevice, st));
    CUDA_TRY(c, cudaEventRecord(c->bias_ev[slot], st));
    c->bias_used[slot] = true;
    return MOE_OK;
}
}  // namespace

extern "C" int moe_set_router_bias(moe_ctx* c, int32_t layer, const float* bias_host, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    int rc = check_layer(c, layer);
    if (rc) return rc;
    if (!bias_host) return fail(c, MOE_EINVAL, "bias is NULL");
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    return stage_bias(c, c->router_bias + (size_t)layer * c->cfg.n_experts, bias_host, c->cfg.n_experts,
                      static_cast<cudaStream_t>(stream));
}

extern "C" int moe_set_router_bias_all(moe_ctx* c, const float* bias_host, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    if (c->poisoned) return fail(c, MOE_ESTATE, "context is poisoned by an earlier CUDA error");
    if (!bias_host) return fail(c, MOE_EINVAL, "bias is NULL");
    for (int l = 0; l < c->cfg.n_layers; ++l)
        if (!c->loaded[l]) return fail(c, MOE_ESTATE, "layer %d has not been loaded", l);
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    return stage_bias(c, c->router_bias, bias_host, (size_t)c->cfg.n_layers * c->cfg.n_experts,
                      static_cast<cudaStream_t>(stream));
}

extern "C" int moe_forward_decode(moe_ctx* c, int32_t layer, const float* x, int32_t B, float* y,
                                  int32_t* topk_idx, float* topk_w, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    int rc = check_layer(c, layer);
    if (rc) return rc;
    if (!x || !y || x == y) return fail(c, MOE_EINVAL, "x and y must be distinct device buffers");
    if (B < 1 || B > c->cfg.max_batch) return fail(c, MOE_EINVAL, "B=%d outside 1..max_batch", B);
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!c->resident) return stream_layers(c, layer, 1, x, B, y, 1.0f, nullptr, nullptr, nullptr, topk_idx, topk_w, st);
    return decode_layer(c, layer, x, B, y, topk_idx, topk_w, st);
}

extern "C" int moe_forward_decode_stack(moe_ctx* c, int32_t layer0, int32_t n, const float* x, int32_t B,
                                        float* y, float eps, float* x_trace, int32_t* idx_trace, float* y_trace,
                                        void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    if (n < 1 || layer0 < 0 || layer0 + n > c->cfg.n_layers)
        return fail(c, MOE_EINVAL, "layers %d..%d out of range", layer0, layer0 + n - 1);
    for (int l = layer0; l < layer0 + n; ++l) {
        int rc = check_layer(c, l);
        if (rc) return rc;
    }
    if (!x || !y || x == y) return fail(c, MOE_EINVAL, "x and y must be distinct device buffers");
    if (B < 1 || B > c->cfg.max_batch) return fail(c, MOE_EINVAL, "B=%d outside 1..max_batch", B);
    if (!(eps > 0.0f)) return fail(c, MOE_EINVAL, "renorm_eps must be > 0");
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int H = c->cfg.hidden, k = c->cfg.top_k;
    const size_t tok = (size_t)B * H;
    if (moe::stack_last_status(c->stack))
        return fail(c, MOE_ETIMEOUT, "a device-side wait of an earlier decode-stack launch ran out (status %d)",
                    moe::stack_last_status(c->stack)) == MOE_ETIMEOUT
                   ? (c->poisoned = true, MOE_ETIMEOUT)
                   : MOE_ETIMEOUT;
    // the persistent kernel wins for a few tokens; from 4 tokens on, the batched
    // per-layer kernels (each expert's rows read once for all of its tokens) are faster
    if (c->resident && !c->mixed && B <= moe::kStackPreferMaxB && moe::stack_supported(c->sh, c->stack, B)) {
        moe::StackArgs a{};
        a.layer0 = layer0;
        a.n_layers = n;
        a.B = B;
        a.eps = eps;
        a.x = x;
        a.y = y;
        a.x_trace = x_trace;
        a.idx_trace = idx_trace;
        a.y_trace = y_trace;
        a.router_w = c->router_w;
        a.router_bias = c->router_bias;
        a.shared_gate = c->cfg.shared_inter > 0 ? c->shared_gate : nullptr;
        a.dir = c->dir;
        a.shared_pool = c->cfg.shared_inter > 0 ? c->shared_pool : nullptr;
        a.shared_stride = c->shared_stride;
        a.fault = c->fault_device_armed && n > 1;
        if (a.fault) c->fault_device_armed = false;
        cudaError_t e = moe::launch_stack(c->sh, c->stack, a, st);
        if (e != cudaSuccess) return fail(c, MOE_ECUDA, "decode stack launch failed: %s", cudaGetErrorString(e));
        for (int l = layer0; l < layer0 + n; ++l) c->stats[l].calls++;
        c->launches += 1;
        return MOE_OK;
    }
    if (!c->resident) return stream_layers(c, layer0, n, x, B, y, eps, x_trace, idx_trace, y_trace, nullptr, nullptr, st);
    const float* xin = x;
    for (int l = layer0; l < layer0 + n; ++l) {
        const int i = l - layer0;
        if (x_trace) {
            CUDA_TRY(c, cudaMemcpyAsync(x_trace + i * tok, xin, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
        }
        float* yl = (l == layer0 + n - 1) ? y : (y_trace ? y_trace + i * tok : c->ybuf);
        int rc = decode_layer(c, l, xin, B, yl, idx_trace ? idx_trace + (size_t)i * B * k : nullptr, nullptr, st);
        if (rc) return rc;
        if (l == layer0 + n - 1) {
            if (y_trace) {
                CUDA_TRY(c, cudaMemcpyAsync(y_trace + i * tok, y, tok * sizeof(float), cudaMemcpyDeviceToDevice, st));
            }
            break;
        }
        float* xn = c->xbuf + (size_t)(i & 1) * c->cfg.max_batch * H;
        CUDA_TRY(c, moe::launch_renorm(yl, xn, B, H, eps, st));
        c->launches += 1;
        xin = xn;
    }
    return MOE_OK;
}

extern "C" int moe_route_noalloc(moe_ctx* c, int32_t layer, const float* x, int32_t B, int32_t* topk_idx,
                                 float* topk_w, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    int rc = check_layer(c, layer);
    if (rc) return rc;
    if (!x || !topk_idx || !topk_w) return fail(c, MOE_EINVAL, "x, topk_idx and topk_w are required");
    if (B < 1 || B > c->cfg.max_batch) return fail(c, MOE_EINVAL, "B=%d outside 1..max_batch", B);
    const int E = c->cfg.n_experts, k = c->cfg.top_k, H = c->cfg.hidden;
    // scratch: logits [B][E], idx [B][k], w [B][k], sigma [B]; each part 256-byte aligned
    auto up = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t lg_b = up(sizeof(float) * (size_t)B * E), ix_b = up(sizeof(int32_t) * (size_t)B * k),
                 w_b = up(sizeof(float) * (size_t)B * k), sg_b = up(sizeof(float) * (size_t)B);
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    void* base = nullptr;
    size_t cap = 0;
    CUDA_TRY(c, moe::noalloc_scratch(c->cfg.device, &base, &cap));
    if (lg_b + ix_b + w_b + sg_b > cap)
        return fail(c, MOE_EINVAL, "routing scratch of %zu bytes exceeds the fixed %zu-byte array", lg_b + ix_b + w_b + sg_b,
                    cap);
    uint8_t* p = static_cast<uint8_t*>(base);
    float* lg = reinterpret_cast<float*>(p);
    int32_t* ix = reinterpret_cast<int32_t*>(p + lg_b);
    float* wt = reinterpret_cast<float*>(p + lg_b + ix_b);
    float* sg = reinterpret_cast<float*>(p + lg_b + ix_b + w_b);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* wr = c->router_w + (size_t)layer * E * H;
    const float* bias = c->router_bias + (size_t)layer * E;
    const uint16_t* wsg = c->cfg.shared_inter > 0 ? c->shared_gate + (size_t)layer * H : nullptr;
    CUDA_TRY(c, moe::launch_router(c->lsh[layer], wr, bias, x, B, lg, st));
    CUDA_TRY(c, moe::launch_route_dispatch(c->lsh[layer], 1 | 4, lg, x, wsg, B, ix, wt, sg, topk_idx, topk_w, nullptr,
                                           nullptr, c->disp, c->xd, nullptr, st));
    c->launches += 2;
    return MOE_OK;
}

extern "C" int moe_forward_prefill(moe_ctx* c, int32_t layer, const float* x, int32_t T, float* y,
                                   int32_t* topk_idx, float* topk_w, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    int rc = check_layer(c, layer);
    if (rc) return rc;
    if (c->cfg.max_tokens <= 0) return fail(c, MOE_ESTATE, "context created without prefill (max_tokens = 0)");
    if (T < 1 || T > c->cfg.max_tokens) return fail(c, MOE_EINVAL, "T=%d outside 1..max_tokens", T);
    if (!x || !y || x == y) return fail(c, MOE_EINVAL, "x and y must be distinct device buffers");
    if (const int st = moe::prefill_last_status(c->pre)) {
        c->poisoned = true;
        return fail(c, MOE_ETIMEOUT,
                    "a device-side check of an earlier prefill failed (status %d: 1-4 a wait ran out, 8 the router "
                    "bound)",
                    st);
    }
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    const int E = c->cfg.n_experts, H = c->cfg.hidden;
    moe::PrefillArgs a{};
    a.T = T;
    a.x = x;
    a.y = y;
    a.user_idx = topk_idx;
    a.user_w = topk_w;
    a.router_w = c->router_w + (size_t)layer * E * H;
    a.router_bias = c->router_bias + (size_t)layer * E;
    a.shared_gate = c->cfg.shared_inter > 0 ? c->shared_gate + (size_t)layer * H : nullptr;
    a.dir = c->dir + (size_t)layer * E;
    a.shared_blob = shared_blob(c, layer);
    a.timeout_ns = (unsigned long long)std::min(timeout_ms(c), 1000) * 1000000ull;  // per device-side wait
    cudaEvent_t* ev = nullptr;
    if (c->prof_on) {
        if (c->prof_calls - c->prof_harvested >= moe_ctx::kProfRing) {  // the slot about to be reused
            int rc2 = prof_harvest_one(c, c->prof_harvested++);
            if (rc2) return rc2;
        }
        ev = c->prof_ev.data() + (size_t)(c->prof_calls % moe_ctx::kProfRing) * (moe::kPrefillKernels + 1);
        c->prof_calls++;
    }
    int n = 0;
    cudaError_t e = moe::launch_prefill(c->lsh[layer], c->pre, a, static_cast<cudaStream_t>(stream), &n, ev);
    c->launches += n;
    if (e != cudaSuccess) return fail(c, MOE_ECUDA, "prefill launch failed: %s", cudaGetErrorString(e));
    c->stats[layer].calls++;
    return MOE_OK;
}

extern "C" int moe_pool_stats(moe_ctx* c, int32_t layer, moe_pool_stats_t* out) {
    if (!c || !out) return fail(c, MOE_EINVAL, "NULL argument");
    const moe_config& g = c->cfg;
    if (layer < -1 || layer >= g.n_layers) return fail(c, MOE_EINVAL, "layer %d out of range", layer);
    std::memset(out, 0, sizeof *out);
    std::vector<unsigned long long> hits(g.n_layers, 0);
    if (c->resident && !c->poisoned) {
        CUDA_TRY(c, cudaSetDevice(g.device));
        CUDA_TRY(c, cudaDeviceSynchronize());
        CUDA_TRY(c, cudaMemcpy(hits.data(), c->hits_dev, sizeof(unsigned long long) * g.n_layers,
                               cudaMemcpyDeviceToHost));
    }
    if (!c->resident && c->side && !c->poisoned) {
        CUDA_TRY(c, cudaStreamSynchronize(c->side));
        harvest_copy_timing(c, true);
    }
    for (int l = 0; l < g.n_layers; ++l) {
        if (layer >= 0 && l != layer) continue;
        const LayerStats& S = c->stats[l];
        out->hits += c->resident ? hits[l] : S.hits;
        out->misses += S.misses;
        out->evictions += S.evictions;
        out->h2d_bytes += S.h2d_bytes;
        out->h2d_ms += S.h2d_ms;
        out->calls += S.calls;
        out->resident += c->resident ? (c->loaded[l] ? g.n_experts : 0) : moe_slotpool_resident(c->pools[l]);
    }
    return MOE_OK;
}

extern "C" int moe_pool_reset(moe_ctx* c, int32_t slots, int32_t policy, int32_t aging_period, void* stream) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    if (c->poisoned) return fail(c, MOE_ESTATE, "context poisoned by an earlier CUDA error");
    const moe_config& g = c->cfg;
    if (c->resident) return fail(c, MOE_ESTATE, "an all-resident context has no pool to reset");
    if (slots < g.top_k || slots > g.pool_slots)
        return fail(c, MOE_EINVAL, "slots %d outside top_k..pool_slots (%d..%d)", slots, g.top_k, g.pool_slots);
    if (policy < MOE_EVICT_LFU_RECENCY || policy > MOE_EVICT_LFU_AGED)
        return fail(c, MOE_EINVAL, "unknown eviction policy %d", policy);
    CUDA_TRY(c, cudaSetDevice(g.device));
    CUDA_TRY(c, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    CUDA_TRY(c, cudaStreamSynchronize(c->side));
    harvest_copy_timing(c, true);
    const int L = g.n_layers, E = g.n_experts;
    std::vector<moe_slotpool*> fresh(L, nullptr);
    for (int l = 0; l < L; ++l) {
        const int rc = moe_slotpool_create(slots, E, policy, aging_period, &fresh[l]);
        if (rc) {
            for (auto* p : fresh) moe_slotpool_destroy(p);
            return fail(c, rc, "slot pool creation failed");
        }
    }
    for (auto* p : c->pools) moe_slotpool_destroy(p);
    c->pools = fresh;
    c->active_slots = slots;
    c->cfg.policy = policy;
    c->cfg.aging_period = aging_period;
    std::memset(c->dir_host, 0, sizeof(void*) * (size_t)L * E);
    CUDA_TRY(c, cudaMemset(c->dir, 0, sizeof(void*) * (size_t)L * E));
    c->stats.assign(L, LayerStats{});
    c->trace.clear();
    return MOE_OK;
}

extern "C" int moe_prefill_profile(moe_ctx* c, int32_t enable) {
    if (!c) return fail(nullptr, MOE_EINVAL, "ctx is NULL");
    if (c->poisoned) return fail(c, MOE_ESTATE, "context poisoned by an earlier CUDA error");
    CUDA_TRY(c, cudaSetDevice(c->cfg.device));
    if (enable && c->prof_ev.empty()) {
        c->prof_ev.assign((size_t)moe_ctx::kProfRing * (moe::kPrefillKernels + 1), nullptr);
        for (auto& e : c->prof_ev) CUDA_TRY(c, cudaEventCreate(&e));
    }
    if (enable && !c->prof_on) {  // a fresh accumulation
        int rc = prof_harvest_all(c);
        if (rc) return rc;
        for (double& v : c->prof_ms) v = 0.0;
        c->prof_calls = c->prof_harvested = 0;
    }
    c->prof_on = enable != 0;
    return MOE_OK;
}

extern "C" int moe_prefill_kernel_ms(moe_ctx* c, double* ms_out, int64_t* calls) {
    if (!c || !ms_out || !calls) return fail(c, MOE_EINVAL, "NULL argument");
    if (c->poisoned) return fail(c, MOE_ESTATE, "context poisoned by an earlier CUDA error");
    int rc = prof_harvest_all(c);
    if (rc) return rc;
    for (int k = 0; k < moe::kPrefillKernels; ++k) ms_out[k] = c->prof_ms[k];
    *calls = c->prof_calls;
    return MOE_OK;
}

extern "C" int moe_launch_count(moe_ctx* c, uint64_t* out) {
    if (!c || !out) return fail(c, MOE_EINVAL, "NULL argument");
    *out = c->launches;
    return MOE_OK;
}

extern "C" int moe_pool_trace(moe_ctx* c, int32_t* buf, size_t cap, size_t* n_out) {
    if (!c || !n_out) return fail(c, MOE_EINVAL, "NULL argument");
    const size_t rows = c->trace.size() / 6;
    *n_out = rows;
    if (buf) std::memcpy(buf, c->trace.data(), sizeof(int32_t) * 6 * std::min(rows, cap));
    return MOE_OK;
}
