// stack.h -- the persistent decode-stack kernel (all-resident stacks, and
// streaming stacks that wait for the host only at layers that miss).
#pragma once

#include <string>

#include "moe_internal.h"

namespace moe {

struct StackScratch {
    unsigned long long* lg_ll = nullptr;  // logits {value, epoch} words [2][8][E]
    unsigned long long* h_ll = nullptr;   // SwiGLU outputs [2][hp][h_stride]
    unsigned long long* y_ll = nullptr;   // layer outputs [2][8][H]
    unsigned* sync = nullptr;             // [1] CTAs finished, [2] epoch base
    int* status = nullptr;                // device status word (0 = ok)
    int* status_host = nullptr;           // pinned, mapped: status of the last finished launch
    int* status_host_dev = nullptr;       // device alias of status_host
    int grid = 0;                         // CTAs of the cooperative launch
    int max_smem = 0;                     // opt-in shared memory per CTA
    int hp = 0;                           // pairs per parity of h_ll
};

struct StackArgs {
    int layer0, n_layers, B;
    float eps;
    const float* x;
    float* y;
    float* x_trace;
    int32_t* idx_trace;
    float* y_trace;
    const uint16_t* router_w;
    const float* router_bias;
    const uint16_t* shared_gate;
    const uint8_t* const* dir;
    const uint8_t* shared_pool;
    size_t shared_stride;
    // streaming: every layer's routing is published through `pub`.  A layer
    // with absent experts reads their rows straight from host memory (the
    // pinned store `store`, blob stride store_stride, or, when store is null,
    // the staging buffers named in the host's answer), and each CTA writes
    // the rows it read into the slots of the host's answer; CTA 0 patches the
    // device directory `dir_patch` (the array `dir` points to).
    const HostGate* pub;
    const uint8_t** dir_patch;
    const uint8_t* store;
    size_t store_stride;
    uint32_t epoch;  // the call's epoch (what ready/gated/served carry)
    // tests: one CTA withholds its outputs of the launch's first layer and every
    // device-side wait is bounded by 1 ms, so the others' waits run out
    int fault;
};

// largest batch the decode stack sends to the persistent kernel (measured crossover)
constexpr int kStackPreferMaxB = 3;
// missed experts per layer of a streaming launch (kStackPreferMaxB tokens x top_k <= 16)
constexpr int kMaxMiss = 48;

int stack_alloc(StackScratch& s, const Shapes& sh, int n_layers, int max_batch, int device, std::string& err);
void stack_free(StackScratch& s);
bool stack_supported(const Shapes& sh, const StackScratch& s, int B);
// Status of the last finished launch (read from mapped host memory, no sync):
// 0 = ok, otherwise a device-side wait ran out.
int stack_last_status(const StackScratch& s);
// After a finished launch that the host abandoned (and nothing worse): clears
// the device and host status words so that later launches run.
cudaError_t stack_clear_abandoned(StackScratch& s);
cudaError_t launch_stack(const Shapes& sh, StackScratch& s, const StackArgs& a, cudaStream_t st);

}  // namespace moe
