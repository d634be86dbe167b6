// Entry points of the device code, for the host runtime.
#pragma once

namespace mk {
// persistent step kernel instantiation for (weight dtype, sync mode); multi_step: the
// instance that runs several greedy steps per launch (one step: the other instance); tc:
// the instance with the tensor-core GEMV, for geometries set up for it (max_batch >= 3) --
// contexts of batches 1..2 run the instance without that code
const void* step_kernel_entry(int dtype, int sync_mode, bool multi_step, bool tc);
// grid-barrier latency microbenchmark kernel
const void* barrier_kernel_entry();
// SM round-trip probe kernel (SM -> die map)
const void* rtt_kernel_entry();
// page-stream microbenchmark kernel
const void* stream_kernel_entry();
// L2 line latency probe (address -> die interleave)
const void* line_lat_kernel_entry();
}  // namespace mk
