// stack_kernel.cu -- persistent decode-stack kernel (placeholder: the per-layer
// kernels serve every stack until this kernel exists).
#include "stack.h"

namespace moe {

int stack_alloc(StackScratch& s, const Shapes&, int, int, std::string&) {
    s.mem = nullptr;
    return MOE_OK;
}

void stack_free(StackScratch& s) {
    if (s.mem) cudaFree(s.mem);
    s.mem = nullptr;
}

bool stack_supported(const Shapes&, int) { return false; }

cudaError_t launch_stack(const Shapes&, StackScratch&, const StackArgs&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace moe
