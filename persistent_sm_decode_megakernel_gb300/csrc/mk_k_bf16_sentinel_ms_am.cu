// Step-kernel instantiation: bf16 weights/KV, sentinel synchronisation, several steps per launch,
// with the tensor-core attention only (max_batch <= 2, long KV capacity).
#include "mk_kernel.cuh"

namespace mk {
template __global__ void mk_step_kernel<__nv_bfloat16, 1, true, false, true>(const __grid_constant__ DevState,
                                                                const __grid_constant__ StepArgs);
const void* step_kernel_entry_bf16_sentinel_ms_am() {
  return reinterpret_cast<const void*>(&mk_step_kernel<__nv_bfloat16, 1, true, false, true>);
}
}  // namespace mk
