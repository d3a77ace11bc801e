/*
 * moe.h -- C ABI of libmoe.so: the routed sparse-MoE layer with expert
 * streaming, for one NVIDIA GB300 (sm_103a).
 *
 * What the layer computes (the Swiftlet pages describe the system; they give
 * no formulas, the readings below are this library's):
 *   For each token x (fp32, length hidden) of one MoE layer:
 *     l      = W_r x + beta                    router logits, W_r bf16 [E x H]
 *     idx    = top-k of l (descending, ties -> lower expert id)
 *     w_i    = softmax over the k chosen logits (norm_topk = 1)
 *     E_e(x) = D_e (silu(G_e x) * (U_e x))     SwiGLU expert, int4/int8 weights
 *     y      = sum_i w_i E_{idx_i}(x) + sigmoid(w_sg . x) * S(x)
 *   S is the always-resident shared expert.  Each expert matrix is MLX affine
 *   group-quantised: w = scale * q + bias per 64 consecutive columns of a row,
 *   scale and bias fp16.
 *   [Swiftlet article (linlog.top), "Why MoE architectures can be streamed":
 *    512 routed experts choose 10 per token (80B), 256 choose 8 (35B), plus
 *    one shared expert; README translation (news.paixiangai.cn), "How it
 *    works" and "Relation to TurboFieldfare": MLX affine int4/int8 group
 *    quantisation computed on the GPU, byte-addressed kernels with 64-bit
 *    offsets, a cooperative SIMD-group GEMV fast path.]
 *
 * Expert storage: every routed expert is one fixed-stride blob, so fetching
 * an expert is one contiguous copy [article, section 2 "Fixed-stride pread
 * reads"].  A bounded per-layer slot pool in HBM caches experts and evicts by
 * use count with recency as the tie-break [article, section 3 "Expert cache
 * pool and LFU+LRU eviction"; README, "How it works": "LFU plus recency"].
 * A miss is served from a mapped pinned host store (or from an expert
 * container on disk through pinned staging buffers): the persistent decode
 * kernel reads the missing rows over the host link itself and fills the
 * slot; the per-layer kernels get the blob by one copy on a side stream.
 *
 * Blob layout v1 (little-endian; offsets in bytes, rows x cols per matrix):
 *   gate.q  [inter  x hidden*bits/32] u32   element c of a row in word
 *   up.q    [inter  x hidden*bits/32] u32     c/(32/bits), bit (c%(32/bits))*bits
 *   down.q  [hidden x inter*bits/32]  u32     (low bits first)
 *   gate.sb [inter  x hidden/64] u32     low half fp16 scale, high half fp16 bias
 *   up.sb   [inter  x hidden/64] u32
 *   down.sb [hidden x inter/64]  u32
 *   zero padding up to stride = round_up(bytes, 4096).
 *
 * Conventions.
 *   - Every call returns MOE_OK (0) or a negative MOE_E* code; moe_last_error()
 *     gives the message of the last failure on that context (or of a failed
 *     moe_create when ctx is NULL, per host thread).
 *   - Pointers named *_dev are device pointers owned by the caller (fp32 /
 *     int32, contiguous, row-major).  Pointers named *_host are host memory
 *     owned by the caller and only read during the call.
 *   - `stream` is the caller's cudaStream_t (NULL = legacy default stream).
 *   - The library owns the context, the HBM slot pool, the pinned host store,
 *     its side stream and all scratch.  One host thread per context.
 *   - A CUDA error poisons the context: later calls return MOE_ESTATE.
 *   - All-resident contexts (pool_slots == n_experts) never synchronise the
 *     host in forward calls.  Streaming contexts wait (bounded by timeout_ms)
 *     for each layer's routing, published by the GPU to mapped host memory,
 *     and run the slot pool on it; the call returns once the last layer has
 *     been served, with that layer's work still queued on the stream.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_EINVAL -1   /* invalid argument or shape; no GPU work was issued */
#define MOE_ENOMEM -2   /* device, pinned or host allocation failed */
#define MOE_ECUDA -3    /* a CUDA call failed; the context is poisoned */
#define MOE_EPOOL -4    /* a call needs more distinct experts than the pool has slots */
#define MOE_ETIMEOUT -5 /* a bounded host or device wait ran out */
#define MOE_ESTATE -6   /* wrong call order, unloaded layer, or poisoned context */
#define MOE_EIO -7      /* an expert container could not be opened, read or written, or is malformed */

#define MOE_EVICT_LFU_RECENCY 0 /* victim = min (use count, last use, slot) */
#define MOE_EVICT_LRU 1         /* victim = min (last use, slot) */
#define MOE_EVICT_LFU_PERSIST 2 /* min (all-time request count of the expert, last use, slot) */
#define MOE_EVICT_LFU_AGED 3    /* MOE_EVICT_LFU_RECENCY, counts halved every aging_period calls */

/* fault_flags: fault injection for tests (0 in production); no flag makes the GPU fault. */
#define MOE_FAULT_PINNED_ALLOC 0x1u /* pretend the pinned store allocation failed */
#define MOE_FAULT_MISS_COPY 0x2u    /* fail the fault_arg-th miss copy (0-based), without issuing it */
#define MOE_FAULT_WAIT_TIMEOUT 0x4u /* treat the next host wait as timed out */
#define MOE_FAULT_DEVICE_WAIT 0x8u  /* the next multi-layer persistent decode-stack launch of an all-resident
                                       context: one CTA withholds its outputs of the launch's first layer and
                                       every device-side wait is bounded by 1 ms, so the other CTAs' waits run
                                       out; the kernel ends normally with its status word set, and the next
                                       call reports MOE_ETIMEOUT and poisons the context */

/* store_flags */
#define MOE_STORE_DIRECT 0x1u /* read blobs with O_DIRECT (buffered where the file system has none) */

typedef struct moe_ctx moe_ctx;

typedef struct {
    int32_t n_layers;     /* MoE layers held by the context (>= 1) */
    int32_t hidden;       /* H, multiple of 256 */
    int32_t n_experts;    /* E routed experts per layer, 1..1024 */
    int32_t top_k;        /* k, 1..min(E, 16) */
    int32_t inter;        /* I, expert intermediate size, multiple of 64 */
    int32_t shared_inter; /* shared expert intermediate, multiple of 64 (0 = no shared expert) */
    int32_t bits;         /* 4 or 8 (with layer_bits: the widths come from there, `bits` is not used) */
    int32_t group_size;   /* 64 only */
    int32_t pool_slots;   /* slots per layer; == n_experts => all resident, no host sync */
    int32_t norm_topk;    /* 1 = renormalise the k weights (softmax over chosen), 0 = full softmax */
    int32_t policy;       /* MOE_EVICT_* */
    int32_t device;       /* CUDA device ordinal */
    int32_t max_batch;    /* largest B of a decode call, 1..64 */
    int32_t max_tokens;   /* largest T of a prefill call (0 = no prefill) */
    uint32_t fault_flags; /* MOE_FAULT_* (tests only) */
    int32_t fault_arg;
    int32_t timeout_ms;   /* bound on every host wait (<= 0: 10000) */
    int32_t aging_period; /* MOE_EVICT_LFU_AGED: layer calls between halvings (<= 0: 64) */
    uint32_t store_flags; /* MOE_STORE_* */
    const char* store_path; /* streaming only: expert container (moe_store_create) that holds the routed
                               blobs; NULL = a pinned host store filled by moe_load_experts */
    const int32_t* layer_bits; /* [n_layers] 4 or 8 per layer, a mixed store (NULL = every layer `bits`).
                                  Blobs of layer l are packed for layer_bits[l]; every slot is sized for the
                                  widest layer.  Mixed stacks run on the per-layer kernels; no expert
                                  container (it holds one width).  Copied by moe_create. */
} moe_config;

typedef struct {
    uint64_t hits;      /* expert lookups served from the pool */
    uint64_t misses;    /* lookups that needed a host->HBM copy */
    uint64_t evictions; /* misses that displaced a resident expert */
    uint64_t h2d_bytes; /* bytes copied for misses */
    double h2d_ms;      /* device time of those copies (CUDA events; with an expert container it
                           also spans the positioned reads between the copies) */
    int32_t resident;   /* experts currently resident */
    int32_t calls;      /* forward calls that routed through this layer */
} moe_pool_stats_t;

/* ------------------------------------------------------------------ */
/* blobs                                                                */
/* ------------------------------------------------------------------ */

/* Packed bytes of one expert (before padding) and its fixed stride. 0 on bad shape. */
size_t moe_blob_bytes(int32_t hidden, int32_t inter, int32_t bits);
size_t moe_blob_stride(int32_t hidden, int32_t inter, int32_t bits);

/*
 * Pack one expert's quantised tensors into its blob (host only, pure).
 * q_*_host: one code per byte, values < 2^bits; gate/up [inter x hidden],
 * down [hidden x inter].  sb_*_host: fp16 bit patterns, (scale, bias) pairs
 * per 64-column group, [rows x cols/64 x 2].  blob_host must hold
 * moe_blob_stride() bytes; padding is zeroed.
 * Errors: MOE_EINVAL for bad shape, short buffer or an out-of-range code.
 */
int moe_pack_expert(int32_t hidden, int32_t inter, int32_t bits, const uint8_t* q_gate_host,
                    const uint16_t* sb_gate_host, const uint8_t* q_up_host, const uint16_t* sb_up_host,
                    const uint8_t* q_down_host, const uint16_t* sb_down_host, void* blob_host, size_t blob_bytes);

/* ------------------------------------------------------------------ */
/* context                                                              */
/* ------------------------------------------------------------------ */

/*
 * [Swiftlet article (linlog.top), section 1 "Dense core resident, experts read
 * on demand": router, shared expert and the other dense weights stay
 * resident while routed experts are fetched when chosen; section 3 "Expert
 * cache pool and LFU+LRU eviction": a bounded pool of experts in memory.]
 * Validate cfg, allocate the HBM slot pool (n_layers x pool_slots x stride,
 * 64-bit offsets), the device directory, scratch and, when streaming, the
 * mapped pinned host store (n_layers x n_experts x stride) and the side stream.
 * Errors: MOE_EINVAL (bad config, nothing allocated), MOE_ENOMEM, MOE_ECUDA,
 * MOE_EIO (store_path cannot be opened, or its header does not match the
 * config's n_layers, n_experts, hidden, inter and bits).
 */
int moe_create(const moe_config* cfg, moe_ctx** out);

/* Synchronise the library's streams and free everything.  NULL is ignored. */
void moe_destroy(moe_ctx* ctx);

/*
 * [Swiftlet article, section 2 "Fixed-stride pread reads": every routed
 * expert is one fixed-stride blob, fetched by one read; README translation
 * (news.paixiangai.cn), "How it works": router and shared expert are part of
 * the resident dense weights.]
 * Load one layer (call once per layer before its first forward).  Copies:
 *   blobs_host      [n_experts x stride] routed expert blobs (stride as returned
 *                   by moe_blob_stride for (hidden, inter, the layer's bits))
 *   shared_blob_host one blob of the shared expert (stride for shared_inter and
 *                   the layer's bits),
 *                   NULL iff shared_inter == 0
 *   router_w_host   bf16 bits [n_experts x hidden]
 *   shared_gate_host bf16 bits [hidden] (NULL iff shared_inter == 0)
 *   router_bias_host fp32 [n_experts] or NULL (= zeros)
 * All-resident: blobs go straight to their HBM slots (slot = expert id).
 * Streaming: blobs go to the pinned store; the layer's pool starts empty.
 * Streaming from an expert container (store_path): blobs_host must be NULL
 * (the container holds them; each miss is one positioned read of it into a
 * pinned staging buffer, then the copy to the slot).
 * Synchronous (returns when the copies are done).
 */
int moe_load_experts(moe_ctx* ctx, int32_t layer, const void* blobs_host, size_t stride,
                     const void* shared_blob_host, const uint16_t* router_w_host,
                     const uint16_t* shared_gate_host, const float* router_bias_host);

/* Replace one layer's router bias (fp32 [n_experts], host).  Ordered on
 * `stream` and asynchronous: the values are staged in a pinned ring of the
 * context (the call waits only if the copy that last used the staging slot,
 * eight updates earlier, has not yet run).  The caller may reuse bias_host
 * as soon as the call returns. */
int moe_set_router_bias(moe_ctx* ctx, int32_t layer, const float* router_bias_host, void* stream);
/* The same for every layer at once: fp32 [n_layers x n_experts], host, one copy.
 * MOE_ESTATE if a layer has not been loaded.  (The pages have no counterpart:
 * a benchmark with drifting expert popularity sets all biases per step.) */
int moe_set_router_bias_all(moe_ctx* ctx, const float* router_bias_host, void* stream);

/* ------------------------------------------------------------------ */
/* forward                                                              */
/* ------------------------------------------------------------------ */

/*
 * [README translation, "How it works": each layer routes each token to 10 of
 * 512 experts (80B) or 8 of 256 (35B); Swiftlet article, "Why MoE
 * architectures can be streamed": the router picks the routed experts, one
 * shared expert always runs.]
 * Decode: one layer for B tokens (1 <= B <= max_batch).
 *   x_dev   fp32 [B x hidden] in, y_dev fp32 [B x hidden] out (may not alias x).
 *   topk_idx_dev int32 [B x top_k] / topk_w_dev fp32 [B x top_k]: the chosen
 *   experts in descending-logit order and their weights, or NULL.
 * Asynchronous on `stream` when all experts are resident.  A streaming context
 * reads the routing back once per call: with topk_idx_dev and topk_w_dev NULL
 * and B <= 3 the layer runs on the persistent kernel, which reads missed
 * blobs from host memory itself (see moe_forward_decode_stack); otherwise the
 * missed blobs are copied on the side stream and `stream` is ordered after
 * them.  Errors: MOE_EINVAL, MOE_ESTATE (layer not loaded),
 * MOE_EPOOL, MOE_ETIMEOUT, MOE_ECUDA.
 */
int moe_forward_decode(moe_ctx* ctx, int32_t layer, const float* x_dev, int32_t B, float* y_dev,
                       int32_t* topk_idx_dev, float* topk_w_dev, void* stream);

/*
 * [Swiftlet article, "Capability boundaries": the decode loop is limited by
 * dispatch, not by I/O; one launch here runs every layer of the call.]
 * Decode through consecutive layers layer0 .. layer0+n_layers-1 for B tokens:
 *   y_l = MoE_l(x_l);  x_{l+1} = y_l / sqrt(mean(y_l^2) + renorm_eps)
 * (the renormalisation stands in for the attention/norm layers that sit
 * between MoE layers in the full model).  y_dev receives y of the last layer.
 * Optional traces (NULL to skip), all device, for every layer l of the call:
 *   x_trace_dev fp32 [n_layers x B x hidden]   layer inputs x_l
 *   idx_trace_dev int32 [n_layers x B x top_k] chosen experts
 *   y_trace_dev fp32 [n_layers x B x hidden]   layer outputs y_l
 * All-resident contexts run the whole stack as one persistent kernel.
 * Streaming contexts run up to 3 tokens on the same kernel (when the pool has
 * at least B x top_k slots), one launch per call: it publishes each layer's
 * routing to the host, which runs the slot pool on it, and never stops.  A
 * missing expert's rows are read straight from the pinned store in host
 * memory (or from the staging buffer the host reads it into from an expert
 * container) and written into the slot the pool chose by the CTAs that read
 * them, so misses cost link bandwidth inside the layer rather than a copy and
 * a relaunch [Swiftlet article, section 3: misses hidden behind compute].
 * The call returns once the host has served every layer; if the host has to
 * give up mid-call (an I/O error, an injected fault) the kernel ends early
 * and the context is poisoned.  Calls with traces use the
 * per-layer kernels.  From 4 tokens on: per-layer kernels with the host's pool
 * decision between routing and dispatch of every layer.  All paths give the
 * same bits.
 */
int moe_forward_decode_stack(moe_ctx* ctx, int32_t layer0, int32_t n_layers, const float* x_dev, int32_t B,
                             float* y_dev, float renorm_eps, float* x_trace_dev, int32_t* idx_trace_dev,
                             float* y_trace_dev, void* stream);

/*
 * [README translation, "Correctness": incremental decode is verified against
 * full-sequence processing; "Four ways to use it": a conversation cache with
 * incremental prefill.  The pages give no prefill kernel design.]
 * Prefill: one layer for T tokens (1 <= T <= max_tokens), all experts of the
 * layer resident.  Tokens are sorted per expert and the experts run as a
 * grouped GEMM on the tensor cores: weights dequantised to bf16
 * (bf16(fp32 fma(scale, q, bias))), token activations rounded to bf16 for the
 * gate/up projections, fp32 accumulation.  The SwiGLU output h is NOT rounded
 * to one bf16: it enters the down projection as the bf16 pair hi = bf16(h),
 * lo = bf16(h - hi) (h to about 2^-17 relative), both multiplied by the bf16
 * down weights.  Routing is computed exactly as in decode (fp32 x).
 *   x_dev fp32 [T x hidden], y_dev fp32 [T x hidden],
 *   topk_idx_dev int32 [T x top_k] / topk_w_dev fp32 [T x top_k] or NULL.
 */
int moe_forward_prefill(moe_ctx* ctx, int32_t layer, const float* x_dev, int32_t T, float* y_dev,
                        int32_t* topk_idx_dev, float* topk_w_dev, void* stream);

/*
 * Routing only, allocation-free: router logits, top-k and routing weights of
 * B decode tokens of one layer (the same kernels and results as the routing
 * inside moe_forward_decode), with all of its scratch in one fixed device
 * array inside the library (256 KiB; no cudaMalloc or other allocation by
 * the call).  The Swiftlet pages have no counterpart of this call.
 *   x_dev fp32 [B x hidden]; topk_idx_dev int32 [B x top_k] and topk_w_dev
 *   fp32 [B x top_k] receive the result (device, caller-owned, required).
 * The scratch needs B*(n_experts + 2*top_k + 1)*4 bytes (each part rounded up
 * to 256); a larger request fails with MOE_EINVAL before any GPU work.
 * Nothing in the array has to start at zero: every element the kernels read
 * is written earlier in the same call.  The first call on a device looks up
 * the array's address (cudaGetSymbolAddress) and should therefore come before
 * any stream capture.  The looked-up address is kept for the life of the
 * process and assumes the device's primary context stays alive: after a
 * cudaDeviceReset, or under a non-primary context, it is stale.  The array is
 * shared by all contexts of a device: calls that may overlap in time (other
 * streams, other host threads) race on it.
 */
int moe_route_noalloc(moe_ctx* ctx, int32_t layer, const float* x_dev, int32_t B, int32_t* topk_idx_dev,
                      float* topk_w_dev, void* stream);

/* ------------------------------------------------------------------ */
/* pool introspection                                                   */
/* ------------------------------------------------------------------ */

/* [Swiftlet article, section 3 "Expert cache pool and LFU+LRU eviction":
 * the pages report the pool's hit rate (43-70 %).]
 * Counters of one layer, or the sum over layers (layer = -1).  Synchronises. */
int moe_pool_stats(moe_ctx* ctx, int32_t layer, moe_pool_stats_t* out);

/*
 * Streaming contexts only: empty every layer's pool (the next call of each
 * layer starts cold), use the first `slots` of the pool_slots slots that
 * moe_create reserved, and evict by `policy` (MOE_EVICT_*; aging_period as in
 * moe_config).  Zeroes the counters of moe_pool_stats and the trace; the
 * per-layer clock restarts at 0.  Synchronises the caller's stream and the
 * side stream first, so no copy into a slot is in flight.  The size and
 * policy sweep of the pages' cache section (hit rate moves with pool size
 * while throughput barely does) runs on one loaded store this way.
 * MOE_EINVAL: slots outside top_k..pool_slots or unknown policy;
 * MOE_ESTATE: all-resident context or poisoned context.
 */
int moe_pool_reset(moe_ctx* ctx, int32_t slots, int32_t policy, int32_t aging_period, void* stream);

/*
 * [README translation, "Correctness": streaming placement never changes the
 * model's semantics, an expert answers the same from the cache or from disk;
 * the trace lets a checker replay every pool decision.]
 * Streaming contexts: copy the pool event trace, oldest first, as rows of six
 * int32 (call number of that layer, layer, expert, kind 0 = HIT / 1 = MISS,
 * slot, evicted expert or -1), at most `cap` rows into buf_host; *n_out = rows
 * available in total.  All-resident contexts record no trace (*n_out = 0):
 * every lookup is a hit in slot = expert id.
 */
int moe_pool_trace(moe_ctx* ctx, int32_t* buf_host, size_t cap, size_t* n_out);

/*
 * Prefill kernel timing (diagnostics).  enable = 1: every later prefill call
 * records a CUDA event on its stream before and after each of its kernels;
 * enable = 0 stops recording.  moe_prefill_kernel_ms adds up, over the calls
 * recorded since profiling was enabled, the device milliseconds of each
 * kernel, in launch order:
 *   [0] router logits  [1] top-k / weights / shared gate  [2] pair histogram
 *   [3] scan + chunk lists  [4] scatter  [5] token rows in sorted order
 *   [6] gate/up grouped GEMM  [7] down grouped GEMM
 * into ms_out[MOE_PREFILL_KERNELS] and the number of calls into *calls.
 * Synchronises with the recorded events.
 */
#define MOE_PREFILL_KERNELS 8
int moe_prefill_profile(moe_ctx* ctx, int32_t enable);
int moe_prefill_kernel_ms(moe_ctx* ctx, double* ms_out, int64_t* calls);

/* Number of CUDA kernels this context has launched so far (all entry points). */
int moe_launch_count(moe_ctx* ctx, uint64_t* out);

const char* moe_last_error(moe_ctx* ctx);

/* ------------------------------------------------------------------ */
/* expert container: routed blobs on disk, one positioned read per blob  */
/* ------------------------------------------------------------------ */
/*
 * [Swiftlet article, section 2 "Fixed-stride pread reads"; README, "How it
 * works": routed experts repacked into a container of fixed-stride blobs, one
 * pread per expert, no mmap.]  Layout (this library's): a 4096-byte little-
 * endian header (magic "MOEXPRT1", version 1, n_layers, n_experts, hidden,
 * inter, bits, group size 64, stride, data offset 4096), then blob (l, e) at
 * 4096 + (l * n_experts + e) * stride, stride = moe_blob_stride(hidden,
 * inter, bits).  Host only; MOE_EIO on any I/O failure, a bad header or a
 * file shorter than its header says.
 */
/* Create (or truncate) a container sized for every blob (unwritten blobs read as zeros). */
int moe_store_create(const char* path, int32_t n_layers, int32_t n_experts, int32_t hidden, int32_t inter,
                     int32_t bits);
/* Write all blobs of one layer: blobs_host [n_experts][stride]. */
int moe_store_write_layer(const char* path, int32_t layer, const void* blobs_host, size_t stride);
/* shape_out[5] = {n_layers, n_experts, hidden, inter, bits}; *stride_out = stride. */
int moe_store_info(const char* path, int32_t* shape_out, uint64_t* stride_out);
/* Read one blob (stride bytes) into dst_host (cap >= stride). */
int moe_store_read(const char* path, int32_t layer, int32_t expert, void* dst_host, size_t cap);

/* ------------------------------------------------------------------ */
/* the slot-pool policy on its own (host only; used by the context)      */
/* ------------------------------------------------------------------ */

typedef struct moe_slotpool moe_slotpool;

/* aging_period: calls between count halvings of MOE_EVICT_LFU_AGED (<= 0: 64) */
int moe_slotpool_create(int32_t slots, int32_t n_experts, int32_t policy, int32_t aging_period,
                        moe_slotpool** out);
void moe_slotpool_destroy(moe_slotpool* p);

/*
 * One request of distinct expert ids, ascending (req_host[n]).  Hits update
 * use count and recency; each miss takes the lowest free slot or evicts the
 * policy's victim among slots not requested in this call.  Counts are kept
 * per slot while resident (LFU_RECENCY, LFU_AGED: a call whose clock is a
 * positive multiple of the aging period first halves every occupied slot's
 * count, rounding down) or per expert over all calls (LFU_PERSIST: every
 * request of the call raises its expert's count before any victim is
 * chosen).  events_host
 * receives n rows of (expert, kind 0 = HIT / 1 = MISS, slot, evicted or -1)
 * in ascending expert order.  Returns n, or MOE_EPOOL if n > slots,
 * MOE_EINVAL if req is not ascending and in range.
 */
int moe_slotpool_request(moe_slotpool* p, const int32_t* req_host, int32_t n, int32_t* events_host);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
