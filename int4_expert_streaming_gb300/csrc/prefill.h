// prefill.h -- the prefill path: exact routing of T tokens, a counting sort of
// the T*top_k (token, expert) pairs by expert, and two grouped GEMMs on the
// tensor cores (gate/up + SwiGLU, then down + weighted scatter into y).
#pragma once

#include <cuda.h>

#include <string>

#include "moe_internal.h"

namespace moe {

// Chunk of sorted rows handled by one GEMM tile column block: expert e (E =
// the shared expert), first row row0 (sorted position for a routed expert,
// token index for the shared one), n rows (1..chunk size), first row in the
// SwiGLU buffers (each expert's rows start on a multiple of 16 there) and the
// expert's blob, so that a tile needs no second, dependent load.  The gate/up
// GEMM takes chunks of up to kChunk rows, the down GEMM chunks of up to
// kChunk1 rows (its two accumulators of 128 columns are double-buffered).
constexpr int kChunk = 256;
constexpr int kChunk1 = 128;

struct alignas(16) ChunkRec {
    int e, row0, n, hrow0;
    const uint8_t* blob;
    int pad[2];
};

struct PrefillScratch {
    int max_tokens = 0, n_hist = 0, max_chunks = 0, max_chunks1 = 0;
    float* logits = nullptr;      // [T][E]
    uint16_t* x_bf = nullptr;     // [T][H] bf16(x)
    int32_t* idx = nullptr;       // [T][k]
    float* w = nullptr;           // [T][k]
    float* sigma = nullptr;       // [T]
    int32_t* local_rank = nullptr;  // [T*k] rank of a pair among the same expert's pairs of its histogram block
    int32_t* cnt = nullptr;       // [E][n_hist] pairs per (expert, block), then their first sorted position
    int32_t* offsets = nullptr;   // [E + 1]
    int32_t* perm = nullptr;      // [T*k] sorted position -> pair id (token * k + slot)
    int32_t* tok_sorted = nullptr;  // [T*k] sorted position -> token
    float* w_sorted = nullptr;    // [T*k] sorted position -> routing weight
    ChunkRec* chunks = nullptr;   // [max_chunks] chunks of up to kChunk rows
    ChunkRec* chunks1 = nullptr;  // [max_chunks1] chunks of up to kChunk1 rows
    int32_t* n_chunks = nullptr;  // [2] lengths of the two chunk lists
    // SwiGLU output h = hi + lo (two bf16), rows: routed experts in sorted
    // order then the shared expert, each expert padded to 16 rows; stored in
    // planes of 64 columns [h_stride / 64][h_rows][64], each 128-byte row
    // swizzled like a shared-memory MMA tile (chunk c at c ^ (row & 7)).
    uint16_t* h_hi = nullptr;
    uint16_t* h_lo = nullptr;
    int h_rows = 0;
    // two-stage router (norm_topk, E a multiple of 128): x as three bf16 pieces
    // [T][3H] (the first H columns are bf16(x), the operand of the expert GEMMs),
    // norm bounds of x_t and of the router rows
    uint16_t* x3 = nullptr;
    float* xnorm = nullptr;
    float* wnorm = nullptr;
    bool two_stage = false;
    uint16_t* x_sorted = nullptr;   // [T*k][H] bf16 token row of every sorted position
    // TMA maps of the gate/up GEMM's token operand, boxes of 64 columns x 64
    // rows landing 128-byte swizzled: the token rows in token order (shared
    // expert) and in sorted pair order (routed experts)
    CUtensorMap x_map, xs_map;
    int* status_host = nullptr;   // pinned, mapped: 0 = ok, else a device-side wait ran out
    int* status_dev = nullptr;    // device alias of status_host
    int sms = 0;
};

struct PrefillArgs {
    int T;
    const float* x;              // [T][H]
    float* y;                    // [T][H]
    int32_t* user_idx;           // optional [T][k]
    float* user_w;               // optional [T][k]
    const uint16_t* router_w;    // [E][H] of the layer
    const float* router_bias;    // [E]
    const uint16_t* shared_gate; // [H] or NULL
    const uint8_t* const* dir;   // [E] blob addresses of the layer
    const uint8_t* shared_blob;  // or NULL
    unsigned long long timeout_ns;
};

// Shapes the prefill kernels support (hidden <= 2048, multiples of 256;
// inter and shared_inter multiples of 128).  Returns an empty string if ok.
std::string prefill_check(const Shapes& s);
int prefill_alloc(PrefillScratch& p, const Shapes& s, int max_tokens, int device, std::string& err);
void prefill_free(PrefillScratch& p);
int prefill_last_status(const PrefillScratch& p);
// Enqueues the whole layer; returns the first launch error and the number of
// kernels launched through *launches.  ev (optional, kPrefillKernels + 1
// events) is recorded before the first kernel and after each kernel.
constexpr int kPrefillKernels = 8;
cudaError_t launch_prefill(const Shapes& s, PrefillScratch& p, const PrefillArgs& a, cudaStream_t st,
                           int* launches, cudaEvent_t* ev = nullptr);

// router_gemm.cu
bool router_two_stage_ok(const Shapes& s);
cudaError_t launch_router_two_stage(const Shapes& s, const PrefillScratch& p, const PrefillArgs& a, cudaStream_t st,
                                    int* launches);

}  // namespace moe
