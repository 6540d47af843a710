// stack_fill.cu - the device-fill variants of the fused decode stack (moe_decode_stack_fill),
// instantiated apart from the common ones so that both compile in parallel.
#include "stack_kernel.cuh"

namespace rl {

rl_status launch_stack_fill(const StackArgs &a, cudaStream_t s) { return launch_stack_any<true>(a, s); }

}  // namespace rl
