// Entry points of the device code, for the host runtime.
#pragma once

namespace mk {
// persistent step kernel instantiation for (weight dtype, sync mode); multi_step: the
// instance that runs several greedy steps per launch (one step: the other instance);
// variant (Geometry::instance()): 0 without tensor-core code, 1 with the tensor-core
// attention, 2 with the tensor-core GEMV and attention (geometries for max_batch >= 3)
const void* step_kernel_entry(int dtype, int sync_mode, bool multi_step, int variant);
// grid-barrier latency microbenchmark kernel
const void* barrier_kernel_entry();
// SM round-trip probe kernel (SM -> die map)
const void* rtt_kernel_entry();
// page-stream microbenchmark kernel
const void* stream_kernel_entry();
// L2 line latency probe (address -> die interleave)
const void* line_lat_kernel_entry();
}  // namespace mk
