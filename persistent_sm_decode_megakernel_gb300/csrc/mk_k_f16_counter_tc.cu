// Step-kernel instantiation: f16 weights/KV, counter synchronisation, one step per launch,
// with the tensor-core GEMV and attention (contexts of max_batch >= 3).
#include "mk_kernel.cuh"

namespace mk {
template __global__ void mk_step_kernel<__half, 0, false, true, true>(const __grid_constant__ DevState,
                                                                const __grid_constant__ StepArgs);
const void* step_kernel_entry_f16_counter_tc() {
  return reinterpret_cast<const void*>(&mk_step_kernel<__half, 0, false, true, true>);
}
}  // namespace mk
