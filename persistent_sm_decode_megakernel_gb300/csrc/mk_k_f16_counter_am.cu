// Step-kernel instantiation: f16 weights/KV, counter synchronisation, one step per launch,
// with the tensor-core attention only (max_batch <= 2, long KV capacity).
#include "mk_kernel.cuh"

namespace mk {
template __global__ void mk_step_kernel<__half, 0, false, false, true>(const __grid_constant__ DevState,
                                                                const __grid_constant__ StepArgs);
const void* step_kernel_entry_f16_counter_am() {
  return reinterpret_cast<const void*>(&mk_step_kernel<__half, 0, false, false, true>);
}
}  // namespace mk
