// stack.h -- the persistent decode-stack kernel (all experts resident).
#pragma once

#include <string>

#include "moe_internal.h"

namespace moe {

struct StackScratch {
    void* mem = nullptr;
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
};

int stack_alloc(StackScratch& s, const Shapes& sh, int n_layers, int max_batch, std::string& err);
void stack_free(StackScratch& s);
bool stack_supported(const Shapes& sh, int B);
cudaError_t launch_stack(const Shapes& sh, StackScratch& s, const StackArgs& a, cudaStream_t st);

}  // namespace moe
