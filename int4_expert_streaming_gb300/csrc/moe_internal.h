// moe_internal.h -- shared between the host runtime and the CUDA kernels.
#pragma once

#include <mutex>
#include <tuple>
#include <vector>

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, once: the call costs host time on every launch otherwise,
// and the launches of the streaming path are also captured into graphs.
inline cudaError_t smem_limit(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::vector<std::tuple<const void*, int, int>> done;  // (kernel, device, bytes)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (auto& d : done)
        if (std::get<0>(d) == kernel && std::get<1>(d) == dev && std::get<2>(d) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.emplace_back(kernel, dev, bytes);
    return e;
}

// Byte offsets of the six sections of one blob (layout v1, see moe.h).
struct BlobLayout {
    uint64_t gate_q, up_q, down_q, gate_sb, up_sb, down_sb, bytes;
};

__host__ __device__ inline BlobLayout blob_layout(int hidden, int rows, int bits) {
    BlobLayout L;
    uint64_t q = (uint64_t)rows * hidden * bits / 8;
    uint64_t sb = (uint64_t)rows * (hidden / 64) * 4;
    L.gate_q = 0;
    L.up_q = q;
    L.down_q = 2 * q;
    L.gate_sb = 3 * q;
    L.up_sb = 3 * q + sb;
    L.down_sb = 3 * q + 2 * sb;
    L.bytes = 3 * q + 3 * sb;
    return L;
}

// Device-side routing/dispatch scratch of one decode call.  "Active experts"
// are the distinct routed experts chosen by any token of the call (ascending
// id) followed by the shared expert; each owns a contiguous run of "pairs"
// (token, weight), tokens ascending within the run.
struct Dispatch {
    int32_t* n_act;        // [1]  routed active + 1 (shared)
    int32_t* act_expert;   // [max_act] expert id, -1 = shared
    const uint8_t** act_blob;  // [max_act] blob base address in HBM
    int32_t* act_off;      // [max_act + 1] first pair of each active expert
    int32_t* pair_token;   // [max_pairs]
    float* pair_w;         // [max_pairs] routing weight (sigmoid gate for the shared expert)
    int32_t* status;       // [1] device error word (0 = ok, 1 = routed to a non-resident expert)
    int32_t* tok_pairs;    // [max_batch][17] each token's pairs, ascending (the shared pair last)
    int4* work;            // [max_work] {active expert, first pair, pairs (<= 8), 0} of the batched kernels
    int32_t* n_work;       // [1]
};

// One entry of the host's answer to a streaming layer with absent experts:
// a missed expert (expert >= 0) with the slot the pool gave it and, for an
// expert container, the pinned staging buffer its blob has been read into
// (null when the whole store is in pinned host memory), or an evicted one
// (expert = -1 - id, slot null).
struct ServeEntry {
    int32_t expert;
    int32_t pad;
    const uint8_t* slot;
    const uint8_t* src;
};

// Publication of a streaming layer's routing to the host and the host's
// answer (device aliases of mapped pinned host memory).  The device writes
// idx, then ready[layer] = the call's epoch (and gated[layer] first when some
// expert of the layer is absent); the host runs the slot pool on idx.  For a
// gated layer it writes the layer's entries (misses first), serve_n[layer] =
// misses | evictions << 16 (or -1: the call is abandoned), then
// served[layer] = epoch.
struct HostGate {
    volatile uint32_t* ready;        // [n_layers] epoch of the last routing published per layer
    const volatile uint32_t* epoch;  // [1] the epoch of the current call, written by the host
    volatile uint32_t* gated;        // [n_layers] epoch of the call whose persistent launch found an absent expert there
    int32_t* idx;                    // [n_layers][idx_stride] the published routing of each layer
    int idx_stride;                  // max_batch * top_k
    volatile uint32_t* served;       // [n_layers] epoch of the call whose layer has been answered
    volatile int32_t* serve_n;       // [n_layers]
    ServeEntry* serve_tab;           // [n_layers][serve_stride]
    int serve_stride;                // 2 * max_batch * top_k
};

struct Shapes {
    int hidden, n_experts, top_k, inter, shared_inter, bits, norm_topk;
    int max_act, max_pairs, h_stride;  // h_stride = max(inter, shared_inter)
    int max_work;                      // max_act + max_pairs / 8 + 1 work items of the batched kernels
};

// Block-fixed-point digits of the decode tokens (see gemv.cuh), written by the
// top-k kernel and read by the gate/up kernel.
struct TokenDigits {
    uint32_t* words;  // [max_batch][hidden/cols_per_chunk][digit words per chunk]
    int32_t* sums;    // [max_batch][hidden/cols_per_chunk]
    int32_t* exps;    // [max_batch]
};

// kernels (decode_kernels.cu)
cudaError_t launch_router(const Shapes& s, const uint16_t* w_r, const float* bias, const float* x, int B,
                          float* logits, cudaStream_t st);
// mode bit 1 = top-k, bit 2 = dispatch, bit 4 = skip the token digits (routing only)
cudaError_t launch_route_dispatch(const Shapes& s, int mode, const float* logits, const float* x,
                                  const uint16_t* shared_gate_w, int B, int32_t* idx, float* w, float* sigma,
                                  int32_t* user_idx, float* user_w, const uint8_t* const* dir_layer,
                                  const uint8_t* shared_blob, Dispatch d, TokenDigits xd,
                                  unsigned long long* hit_counter, cudaStream_t st,
                                  const HostGate* publish = nullptr, int publish_layer = 0);
cudaError_t launch_renorm(const float* y, float* x_next, int B, int hidden, float eps, cudaStream_t st);
// batched per-layer path: gate/up per (expert, row block) with staged token digits,
// down per (expert, row block) into part[pair][H], then the per-token combine
cudaError_t launch_gateup_batched(const Shapes& s, Dispatch d, TokenDigits xd, float* h, cudaStream_t st);
cudaError_t launch_down_batched(const Shapes& s, Dispatch d, const float* h, float* part, cudaStream_t st);
cudaError_t launch_combine(const Shapes& s, Dispatch d, const float* part, float* y, int B, bool has_shared,
                           cudaStream_t st);

// prefill_route.cu: router logits of T tokens in the fixed fp32 order, register
// tiled (hidden <= 2048, a multiple of 256); tok_tile tokens per CTA (<= 64)
cudaError_t launch_logits(const uint16_t* w_r, const float* bias, const float* x, int T, int H, int E, int tok_tile,
                          float* logits, cudaStream_t st);

// noalloc.cu: the fixed scratch array of moe_route_noalloc on `device`
cudaError_t noalloc_scratch(int device, void** ptr, size_t* bytes);

}  // namespace moe
