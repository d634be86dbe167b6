// Step-kernel instantiation: bf16 weights/KV, counter synchronisation, several steps per launch,
// without the tensor-core code (short contexts of max_batch <= 2).
#include "mk_kernel.cuh"

namespace mk {
template __global__ void mk_step_kernel<__nv_bfloat16, 0, true, false, false>(const __grid_constant__ DevState,
                                                                const __grid_constant__ StepArgs);
const void* step_kernel_entry_bf16_counter_ms() {
  return reinterpret_cast<const void*>(&mk_step_kernel<__nv_bfloat16, 0, true, false, false>);
}
}  // namespace mk
