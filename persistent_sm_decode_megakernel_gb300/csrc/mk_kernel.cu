// One-wave grid-barrier microbenchmark and the table of step-kernel instantiations.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mk_internal.h"
#include "mk_device.cuh"
#include "mk_kernels.h"
#include "mk_kernel.cuh"  // the step kernel's GEMV inner loops, for the stream benchmark

namespace mk {

// ---------------------------------------------------------------- barrier microbenchmark
// One-wave kernel doing n all-CTA barriers (§7.3 measurement).  mode 0: thread 0 of each
// CTA release-adds a counter and polls it (acquire) until every CTA has arrived; mode 1:
// every CTA overwrites its own NaN slot of the round and polls all slots of the round.
__global__ void __launch_bounds__(256, 1) mk_barrier_kernel(uint32_t* ctr, float* slots, int n_bar, int mode,
                                                            int64_t timeout_ns, uint64_t* out) {
  const int tid = threadIdx.x, nct = gridDim.x;
  __shared__ int bad;
  if (tid == 0) bad = 0;
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  for (int i = 0; i < n_bar; ++i) {
    if (mode == 0) {
      __syncthreads();
      if (tid == 0) {
        red_release_add_u32(ctr, 1u);
        const uint32_t target = (uint32_t)(i + 1) * nct;
        while ((int32_t)(ld_acquire_u32(ctr) - target) < 0) {
          if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
            bad = 1;
            break;
          }
        }
      }
    } else {
      __syncthreads();
      if (tid == 0) slots[(size_t)i * nct + blockIdx.x] = 1.0f;
      for (int k = tid; k < nct; k += blockDim.x) {
        while (isnan(ld_poll_f32(slots + (size_t)i * nct + k))) {
          if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
            bad = 1;
            break;
          }
        }
      }
    }
    if (__syncthreads_or(bad)) break;
  }
  if (blockIdx.x == 0 && tid == 0) {
    out[0] = globaltimer_ns() - t0;
    out[1] = bad;
  }
}

// ---------------------------------------------------------------- SM round-trip probe
// Die locality (P1 §7.4): CUDA does not say which SM sits on which die, so it is measured.
// A one-wave grid, one CTA per SM.  CTA 0 plays ping-pong with every other CTA in turn
// through the same two words (one 128-byte line, so every pair meets at the same L2
// home): it stores (partner, sequence number) into ping, the partner echoes it into pong,
// and CTA 0 times the round trip in SM cycles.  Partners sleep on a separate turn word
// until their turn, so that only the pair under test loads the memory system.  Every
// wait is bounded by timeout_ns and raises *bad instead of hanging.
__global__ void __launch_bounds__(32, 1) mk_rtt_kernel(uint32_t* words, int reps, int64_t timeout_ns,
                                                       uint32_t* smid_out, uint64_t* cyc_out, uint32_t* bad) {
  if (threadIdx.x != 0) return;
  const int me = blockIdx.x, n = gridDim.x;
  uint32_t sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  smid_out[me] = sm;
  uint32_t* turn = words;         // line 0
  uint32_t* ping = words + 32;    // line 1
  uint32_t* pong = words + 33;
  const uint64_t t0 = globaltimer_ns();
  if (me == 0) {
    cyc_out[0] = 0;
    for (int j = 1; j < n; ++j) {
      st_relaxed_u32(turn, (uint32_t)j);
      uint64_t sum = 0;
      for (int r = 1; r <= reps; ++r) {
        const uint32_t v = ((uint32_t)j << 16) | (uint32_t)r;
        const long long a = clock64();
        st_relaxed_u32(ping, v);
        while (ld_relaxed_u32(pong) != v) {
          if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
            st_relaxed_u32(bad, 1u);
            st_relaxed_u32(turn, (uint32_t)n);
            return;
          }
        }
        if (r > 2) sum += (uint64_t)(clock64() - a);  // the first two cover the partner's wake-up
      }
      cyc_out[j] = sum / (uint64_t)(reps - 2);
    }
    st_relaxed_u32(turn, (uint32_t)n);
    return;
  }
  while (ld_relaxed_u32(turn) < (uint32_t)me) {
    __nanosleep(2000);
    if (globaltimer_ns() - t0 > (uint64_t)timeout_ns || ld_relaxed_u32(bad)) return;
  }
  for (int r = 1; r <= reps; ++r) {
    const uint32_t v = ((uint32_t)me << 16) | (uint32_t)r;
    while (ld_relaxed_u32(ping) != v) {
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns || ld_relaxed_u32(bad)) return;
    }
    st_relaxed_u32(pong, v);
  }
}

// ---------------------------------------------------------------- L2 line latency from two SMs
// Which die's L2 holds a line (the address -> die interleave): one CTA per SM; the CTAs on
// sm_a and sm_b each time, for every offset, a chain of reps (>= 2) dependent L2-only loads
// of that line and store the mean cycles per load.  The buffer is all zeros (the host
// clears it and nothing writes it), so each next address -- the line plus the value just
// loaded -- is the line itself, yet the hardware cannot issue a load before the previous
// one returns.  No waits.
__global__ void __launch_bounds__(32, 1) mk_line_lat_kernel(const uint32_t* buf, const long long* offs, int n,
                                                            int sm_a, int sm_b, int reps, float* lat) {
  if (threadIdx.x != 0) return;
  uint32_t sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  const int which = sm == (uint32_t)sm_a ? 0 : (sm == (uint32_t)sm_b ? 1 : -1);
  if (which < 0) return;
  uint32_t acc = 0;
  for (int i = 0; i < n; ++i) {
    const uint32_t* p = buf + offs[i] / 4;
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");  // into L2
    const uint32_t* q = p + v;
    long long t0, t1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0) :: "memory");
    for (int r = 0; r < reps; ++r) {
      asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(q) : "memory");
      q = p + v;
    }
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1) :: "memory");
    acc += v;
    // the last load is issued, not completed, by t1: reps - 1 full latencies
    lat[which * n + i] = (float)(t1 - t0) / (float)(reps - 1);
  }
  if (acc) lat[which * n] = -1.f;  // never: the buffer is zeros (keeps the chain's last load)
}

// ---------------------------------------------------------------- page-stream microbenchmark
// The decode kernel's loader / compute-warp structure with nothing else: one lane of the
// loader warp streams bytes_per_cta of contiguous HBM through a ring of n_pages pages
// with TMA bulk copies; the 8 compute warps either hand each page straight back
// (mode 0) or first run the B=1 fp16 GEMV slice product on their eighth of it (mode 1).
// hint bit 0: L2 evict-first policy; bit 1: all CTAs read the same bytes.
__global__ void __launch_bounds__(kThreads, 1) mk_stream_kernel(const uint8_t* src, long long bytes_per_cta,
                                                                int page_bytes, int n_pages, int mode, int hint,
                                                                float* sink) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full[kMaxPages], empty[kMaxPages];
  __shared__ int bad;
  uint8_t* pages = smem;
  float* x = reinterpret_cast<float*>(smem + (size_t)n_pages * page_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ws = page_bytes / 16;  // slice elements per warp
  if (tid == 0) {
    for (int i = 0; i < n_pages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    bad = 0;
    mbar_fence_init();
  }
  for (int i = tid; i < ws; i += kThreads) x[i] = 1.0f / (1 + (i & 7));
  __syncthreads();
  const long long n = bytes_per_cta / page_bytes;
  // hint bit 1: every CTA streams the same bytes (the GEMV inputs' access pattern: all SMs
  // read one vector), else each its own slice
  const uint8_t* base = (hint & 2) ? src : src + (long long)blockIdx.x * bytes_per_cta;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = 2000000000ull;
  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    for (long long c = 0; c < n; ++c) {
      const int slot = (int)(c % n_pages);
      const uint32_t ph = (uint32_t)((c / n_pages) & 1);
      while (!mbar_try_wait(&empty[slot], ph ^ 1u)) {
        if (globaltimer_ns() - t0 > limit) {
          bad = 1;
          return;
        }
      }
      mbar_arrive_expect_tx(&full[slot], (uint32_t)page_bytes);
      if (hint & 1)
        tma_load_1d(pages + (size_t)slot * page_bytes, base + c * page_bytes, (uint32_t)page_bytes, &full[slot], pol);
      else
        tma_load_1d_plain(pages + (size_t)slot * page_bytes, base + c * page_bytes, (uint32_t)page_bytes, &full[slot]);
    }
    return;
  }
  float acc = 0.f;
  __shared__ float lanep[8 * kThreads];
  float xr[1][64];
#pragma unroll
  for (int j = 0; j < 64; ++j) xr[0][j] = (mode == 2 || mode >= 4) ? x[(lane + 32 * (j / 8)) * 8 + (j & 7)] : 0.f;
  for (long long c = 0; c < n; ++c) {
    const int slot = (int)(c % n_pages);
    const uint32_t ph = (uint32_t)((c / n_pages) & 1);
    bool timed_out = false;
    while (!mbar_try_wait(&full[slot], ph)) {
      if (bad || globaltimer_ns() - t0 > limit) {
        timed_out = true;
        break;
      }
    }
    if (timed_out) {
      bad = 1;
      break;
    }
    if (mode == 2 || mode == 3) {  // the step kernel's own slice products (B = 1)
      const uint8_t* wp = pages + (size_t)slot * page_bytes + (size_t)warp * ws * 2;
      float a[1];
      if (mode == 2) {
        slice_dot_xreg<__half, 1, 8>(wp, xr, ws / 8, lane, a);
      } else {
        slice_dot_smem<__half, 1>(wp, x, ws, ws, lane, a);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
      acc += a[0];
    }
    if (mode == 4 || mode == 5) {  // four accumulator chains; 4: lane partial to smem, 5: shuffles
      const uint4* w = reinterpret_cast<const uint4*>(pages + (size_t)slot * page_bytes + (size_t)warp * ws * 2);
      uint4 wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) wv[j] = w[lane + 32 * j];
      float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float f[8];
        Unpack<__half>::u8(wv[j], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) a4[(j * 8 + e) & 3] = fmaf(f[e], xr[0][j * 8 + e], a4[(j * 8 + e) & 3]);
      }
      float t = (a4[0] + a4[1]) + (a4[2] + a4[3]);
      if (mode == 5) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        acc += t;
      } else {
        lanep[(c & 7) * kThreads + warp * 32 + lane] = t;
        acc += t;
      }
    }
    if (mode == 1) {
      const uint4* w = reinterpret_cast<const uint4*>(pages + (size_t)slot * page_bytes + (size_t)warp * ws * 2);
      float a = 0.f;
      for (int v = lane; v < ws / 8; v += 32) {
        float f[8];
        Unpack<__half>::u8(w[v], f);
        const float4 x0 = reinterpret_cast<const float4*>(x + v * 8)[0];
        const float4 x1 = reinterpret_cast<const float4*>(x + v * 8)[1];
        a = fmaf(f[0], x0.x, a); a = fmaf(f[1], x0.y, a); a = fmaf(f[2], x0.z, a); a = fmaf(f[3], x0.w, a);
        a = fmaf(f[4], x1.x, a); a = fmaf(f[5], x1.y, a); a = fmaf(f[6], x1.z, a); a = fmaf(f[7], x1.w, a);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      acc += a;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (lane == 0) sink[blockIdx.x * kConsumerWarps + warp] = bad ? CUDART_NAN_F : acc;
}

// ---------------------------------------------------------------- launch table
#define MK_ENTRY(n) const void* step_kernel_entry_##n();
#define MK_ENTRIES(d, s)                                                                         \
  MK_ENTRY(d##_##s) MK_ENTRY(d##_##s##_am) MK_ENTRY(d##_##s##_tc) MK_ENTRY(d##_##s##_ms) MK_ENTRY(d##_##s##_ms_am) \
      MK_ENTRY(d##_##s##_ms_tc)
MK_ENTRIES(f16, counter)
MK_ENTRIES(f16, sentinel)
MK_ENTRIES(bf16, counter)
MK_ENTRIES(bf16, sentinel)
#undef MK_ENTRIES
#undef MK_ENTRY

const void* step_kernel_entry(int dtype, int sync_mode, bool multi_step, int variant) {
  using Fn = const void* (*)();
  // [dtype][sync][multi_step][variant]
#define MK_ROW(d, s) {{step_kernel_entry_##d##_##s, step_kernel_entry_##d##_##s##_am, step_kernel_entry_##d##_##s##_tc}, \
                      {step_kernel_entry_##d##_##s##_ms, step_kernel_entry_##d##_##s##_ms_am,                         \
                       step_kernel_entry_##d##_##s##_ms_tc}}
  static const Fn table[2][2][2][3] = {{MK_ROW(f16, counter), MK_ROW(f16, sentinel)},
                                       {MK_ROW(bf16, counter), MK_ROW(bf16, sentinel)}};
#undef MK_ROW
  const int v = variant < 0 ? 0 : (variant > 2 ? 2 : variant);
  return table[dtype == 0 ? 0 : 1][sync_mode == 0 ? 0 : 1][multi_step ? 1 : 0][v]();
}

const void* barrier_kernel_entry() { return reinterpret_cast<const void*>(&mk_barrier_kernel); }
const void* rtt_kernel_entry() { return reinterpret_cast<const void*>(&mk_rtt_kernel); }
const void* stream_kernel_entry() { return reinterpret_cast<const void*>(&mk_stream_kernel); }
const void* line_lat_kernel_entry() { return reinterpret_cast<const void*>(&mk_line_lat_kernel); }

}  // namespace mk
