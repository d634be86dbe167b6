// The persistent decode megakernel for sm_103a (templates; instantiated per weight
// dtype, sync mode and one-step / multi-step launch in mk_k_*.cu).
//
// Structure ("8 · Écrire son megakernel", §8.2): one CTA per SM walks its own queue of
// 64-byte instructions; for each one it waits for its dependency counter, executes the
// opcode, and signals the counter of its output.  Roles (§7.5, §8.2 classer_role): warp
// 8 is the loader -- one lane streams every weight/KV tile of the CTA's whole queue into a
// ring of shared-memory pages with TMA bulk copies, running ahead across instruction
// boundaries (weights never depend on activations, so the HBM stream does not stop at a
// dependency wait); warps 0-7 compute.  A page is handed back the moment its last reader
// is done with it (§8.4), which is what lets the loader start the next instruction's
// tiles while the current one still computes.
#pragma once
#include <cuda_runtime.h>

#include <type_traits>
#include <math_constants.h>

#include "mk_internal.h"
#include "mk_device.cuh"

namespace mk {
namespace {  // internal linkage: every instantiation unit gets its own copy

constexpr int kPoolSlots = 2;  // claimed attention units the loader may hold ahead of the compute warps

struct SmemCtl {
  uint64_t full[kMaxPages];
  uint64_t empty[kMaxPages];
  uint64_t pool_full[kPoolSlots];   // attention pool: the loader's claimed units, in claim order
  uint64_t pool_empty[kPoolSlots];
  int pool_fifo[kPoolSlots];        // unit index within the layer's pool, -1: the pool is empty
  int pool_slot;                    // compute side: next FIFO slot and its phase (thread 0)
  uint32_t pool_ph;
  int pool_unit;                    // the unit thread 0 took, for the other compute threads
  uint64_t xfull[2];                // tensor-core GEMV: bulk copies of the x staging, per half
  uint32_t xph[2];                  // their phases between ops
  int lm_staged;                    // the x buffer holds the LM head's whole input (and 1/rms)
  unsigned long long wbest[kConsumerWarps * kMaxBatch];  // LM head: each warp's best keys
  unsigned long long best[kMaxBatch];
  float inv_rms[kMaxBatch];
  float red[kConsumerWarps * kMaxBatch];
  int last_issue_phase[kMaxPages];
  uint64_t tmark[6];  // journal marks inside an op
  volatile int abort;
  StepArgs args;  // the step's arguments (from the launch, or from device memory for graphs)
  StepArgs largs; // the loader's copy: it runs ahead into the next step of a multi-step launch
  int ms_step;      // multi-step launches: the step being run
  float* step_act;  // multi-step launches: the current step's activation arena, batch tile and
  int step_nb;      // GQA group (kept here rather than in registers across the op calls)
  int step_G;
  DevState S;     // the context's state, copied from the launch parameters
  Instr cur[kConsumerWarps];  // each compute warp's copy of its current instruction
};
static_assert(sizeof(SmemCtl) <= kCtlSmem, "control block fits");

// The dynamic shared memory: control block | pages | x buffer | scratch.  The control
// block holds copies of the kernel's state and step arguments.  Functions that are not
// inlined into the kernel take those copies and their pointers from this symbol, so that
// the compiler emits shared-space accesses: a pointer or reference passed in as an
// argument is a generic address, and generic loads measured ~50x slower than ld.shared
// here while the loader's bulk copies stream into the same SM.
extern __shared__ __align__(1024) uint8_t mk_smem[];
__device__ __forceinline__ SmemCtl* smem_ctl() { return reinterpret_cast<SmemCtl*>(mk_smem); }
__device__ __forceinline__ uint8_t* smem_pages() { return mk_smem + kCtlSmem; }
__device__ __forceinline__ float* smem_xbuf(const DevState& S) {
  return reinterpret_cast<float*>(mk_smem + kCtlSmem + (size_t)S.n_pages * S.page_stride);
}
__device__ __forceinline__ float* smem_scratch(const DevState& S) {
  return reinterpret_cast<float*>(mk_smem + kCtlSmem + (size_t)S.n_pages * S.page_stride + S.xbuf_bytes);
}

enum { SYNC_COUNTER = 0, SYNC_SENTINEL = 1 };

// ---------------------------------------------------------------- errors
__device__ __noinline__ void set_err(const DevState& S, uint32_t code, int pc, int ctr) {
  if (atomicCAS(&S.ctl->err.code, 0u, code) == 0u) {
    S.ctl->err.cta = blockIdx.x;
    S.ctl->err.pc = pc;
    S.ctl->err.ctr = ctr;
  }
}
__device__ __forceinline__ bool global_err(const DevState& S) {
  return ld_relaxed_u32(&S.ctl->err.code) != 0u;
}

// Bounded wait on a dependency counter (§8.5): acquire load, exponential __nanosleep
// backoff, gives up after the timeout and records where.  Wrap-safe comparison.
__device__ __noinline__ bool wait_counter(const DevState& S_arg, int ctr, uint32_t target, int pc) {
  const DevState& S = smem_ctl()->S;
  const uint32_t* p = S.counters + ctr;
  if ((int32_t)(ld_acquire_u32(p) - target) >= 0) return true;
  const uint64_t t0 = globaltimer_ns();
  int k = 0;
  while (true) {
    int ns = 20 << (k < 8 ? k : 8);
    __nanosleep(ns < S.backoff_max_ns ? ns : S.backoff_max_ns);
    ++k;
    if ((int32_t)(ld_acquire_u32(p) - target) >= 0) return true;
    if (global_err(S)) return false;
    if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
      set_err(S, 4u /*MK_ERR_TIMEOUT*/, pc, ctr);
      return false;
    }
  }
}

// The other parity's activations back to NaN sentinels, this CTA's share of the grid
// (threads t < nthr of every CTA take part).
__device__ __forceinline__ void nan_fill(float* base, int64_t n_floats, int t, int nthr) {
  const int64_t n4 = n_floats / 4;
  float4* o4 = reinterpret_cast<float4*>(base);
  const float4 nan4 = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
  for (int64_t i = (int64_t)blockIdx.x * nthr + t; i < n4; i += (int64_t)gridDim.x * nthr) o4[i] = nan4;
}

// Multi-step launches: wait (acquire) until the token sequence word reaches `target`, i.e.
// the step before has published its tokens -- every CTA has finished that step.
__device__ __noinline__ bool wait_seq(const uint32_t* p, uint32_t target, int pc) {
  const DevState& S = smem_ctl()->S;
  if ((int32_t)(ld_acquire_u32(p) - target) >= 0) return true;
  const uint64_t t0 = globaltimer_ns();
  int k = 0;
  while (true) {
    int ns = 20 << (k < 8 ? k : 8);
    __nanosleep(ns < S.backoff_max_ns ? ns : S.backoff_max_ns);
    ++k;
    if ((int32_t)(ld_acquire_u32(p) - target) >= 0) return true;
    if (global_err(S) || smem_ctl()->abort) return false;
    if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
      set_err(S, 4u /*MK_ERR_TIMEOUT*/, pc, -1);
      return false;
    }
  }
}

// Sentinel read: the value itself is the signal (§7.3) -- poll with an L1-bypassing
// gpu-scope load until it is no longer NaN.
__device__ __noinline__ float poll_slow(const float* p, const DevState& S, SmemCtl* c) {
  const uint64_t t0 = globaltimer_ns();
  int k = 0;
  while (true) {
    int ns = 20 << (k < 8 ? k : 8);
    __nanosleep(ns < S.backoff_max_ns ? ns : S.backoff_max_ns);
    ++k;
    float v = ld_poll_f32(p);
    if (!isnan(v)) return v;
    if (c->abort || global_err(S)) {
      c->abort = 1;
      return 0.f;
    }
    if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
      set_err(S, 4u, -1, -1);
      c->abort = 1;
      return 0.f;
    }
  }
}
template <int SYNC>
__device__ __forceinline__ float load_act(const float* p, const DevState& S, SmemCtl* c) {
  if (SYNC == SYNC_COUNTER) return __ldcg(p);
  float v = ld_poll_f32(p);
  if (!isnan(v)) return v;
  return poll_slow(p, S, c);
}

// a device pointer the host wrote into the instruction (pK at a[2K], a[2K+1])
__device__ __forceinline__ const uint16_t* iptr(const Instr& in, int at) {
  return reinterpret_cast<const uint16_t*>(((uint64_t)(uint32_t)in.a[at + 1] << 32) | (uint32_t)in.a[at]);
}
// instructions are read-only for the whole launch: 4 x 16-byte non-coherent loads
__device__ __forceinline__ Instr load_instr(const Instr* p) {
  Instr in;
  const uint4* s = reinterpret_cast<const uint4*>(p);
  uint4* d = reinterpret_cast<uint4*>(&in);
  d[0] = __ldg(s);
  d[1] = __ldg(s + 1);
  d[2] = __ldg(s + 2);
  d[3] = __ldg(s + 3);
  return in;
}
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- tile geometry
// A GEMV instruction covers one or two row segments of a row-major [rows, K] matrix.
// Its tiles are "slices": WS consecutive elements of one row; a page holds
// kConsumerWarps consecutive slices, one per compute warp.  Loader and compute warps
// derive the same slice sequence from the instruction.
struct Gemv {
  const uint16_t* seg[2];
  int segr[2];
  int K, WS;
  __device__ __forceinline__ int rows() const { return segr[0] + segr[1]; }
  __device__ __forceinline__ int spr() const { return K / WS; }
  __device__ __forceinline__ int nslices() const { return rows() * spr(); }
};

__device__ __forceinline__ Gemv make_gemv(const DevState& S, const Instr& in) {
  Gemv g;
  g.seg[0] = iptr(in, kP4);
  g.seg[1] = iptr(in, kP5);
  g.segr[1] = 0;
  switch (in.op) {
    case OP_QKV:
      g.segr[0] = g.segr[1] = in.a[3];
      g.K = S.d;
      g.WS = S.ws_qkv;
      break;
    case OP_OPROJ:
      g.segr[0] = in.a[1];
      g.K = S.Hq * S.hd;
      g.WS = S.ws_o;
      break;
    case OP_UPGATE:
      g.segr[0] = g.segr[1] = in.a[1];
      g.K = S.d;
      g.WS = S.ws_up;
      break;
    case OP_DOWN:
      g.segr[0] = in.a[1];
      g.K = S.F;
      g.WS = S.ws_down;
      break;
    default:  // OP_LMHEAD
      g.segr[0] = in.a[1];
      g.K = S.d;
      g.WS = S.ws_lm;
      break;
  }
  return g;
}

// Fragment form of a tensor-core GEMV input x[b][k] (batch tile of MT * 8 sequences): the
// 16-bit halves in the order of the m16n8k16 A fragments -- per k-step of 16 columns and
// tile of 8 sequences, 32 lanes x 4 words, lane g * 4 + c holding sequence g's columns
// (2c, 2c + 1) in word 0 (hi halves) and 1 (lo halves) and (2c + 8, 2c + 9) in words 2
// and 3.  Returns the index of x[b][k]'s hi half; its lo half is 2 further.
__device__ __forceinline__ size_t frag_index(int b, int k, int MT) {
  const int ks = k >> 4, kk = k & 15, c = (kk & 7) >> 1;
  return ((((size_t)(ks * MT + (b >> 3)) * 32 + (b & 7) * 4 + c) * 4 + ((kk >> 3) << 1)) << 1) + (kk & 1);
}
template <typename WT>
__device__ __forceinline__ void put_frag(uint16_t* f, int b, int k, int MT, float v) {
  uint16_t hi, lo;
  Mma<WT>::split(v, hi, lo);
  const size_t i = frag_index(b, k, MT);
  f[i] = hi;
  f[i + 2] = lo;
}
// the batch tiles of 8 sequences of the tensor-core GEMV at a padded batch of NB
template <int NB>
constexpr int kFragMT = NB > 8 ? 2 : 1;
// a word still holding a half of the NaN sentinel (0x7FFF or 0xFFFF: all 15 low bits set,
// which no finite 16-bit float has)
__device__ __forceinline__ bool frag_pending(uint32_t w) {
  const uint32_t x = (w & 0x7FFF7FFFu) ^ 0x7FFF7FFFu;  // a half is zero iff it was a sentinel
  return ((x - 0x00010001u) & ~x & 0x80008000u) != 0u;
}

// Split-KV unit (§8.2 ATTENTION): row b (position pos_b of cache sequence seq_b), kv head
// j, split s of S over positions 0..p0_b.  Cached positions [t0, min(t1, p0_b)) stream
// through pages as K, V blocks; the split holding position p0_b takes the keys/values of
// this launch's positions p0_b..pos_b (n_new rows: one for a decode step, the row's
// earlier rows of a prompt chunk plus its own) from the QKV op's fp32 copies.
struct Attn {
  int b, j, s, nsp, t0, t1, n_cached, pb, nblocks, n_new;
  bool has_new, active;
  const uint16_t* kb;
  const uint16_t* vb;
};
// Splits in use this step for sequence b: at most the schedule's S, and at least
// split_min_positions positions per split (short contexts: a few splits, a cheap merge).
// Within that, about one unit per CTA: a split costs a fixed ~2-3 us (q staging, the
// epilogue, its share of the merge) besides its positions, so a batch of B sequences
// uses n_cta / (B Hkv) splits -- unless a split would then hold more than
// kSplitLongPositions positions, where streaming the cache dominates and all S splits
// keep every CTA busy.
__device__ __forceinline__ int active_splits(const DevState& S, const StepArgs& A, int b) {
  const int npos = A.p0[b] + 1;
  const int pmin = S.split_min_positions;
  const int per_cta = max(1, S.n_cta / (A.B * S.Hkv));
  int want = max(per_cta, (npos + kSplitLongPositions - 1) / kSplitLongPositions);
  // a long context that needs more than half the schedule's splits takes all of them: the
  // schedule deals S units per (sequence, head) evenly over the CTAs, so a step whose
  // sequences all do that leaves no CTA a unit more than another
  if (2 * want > S.S) want = S.S;
  return max(1, min(S.S, min((npos + pmin - 1) / pmin, want)));
}
__device__ __forceinline__ Attn make_attn(const DevState& S, const StepArgs& A, const Instr& in) {
  Attn a;
  a.b = in.a[0];
  a.j = in.a[1];
  a.s = in.a[2];
  a.active = a.b < A.B;
  const int npos = a.active ? A.p0[a.b] + 1 : 1;
  a.nsp = a.active ? active_splits(S, A, a.b) : 1;
  a.active = a.active && a.s < a.nsp;
  a.t0 = (int)((uint32_t)(a.s * npos) / (uint32_t)a.nsp);  // s * npos < 2^31 (S <= 256, npos < 2^23)
  a.t1 = (int)((uint32_t)((a.s + 1) * npos) / (uint32_t)a.nsp);
  const int tc = min(a.t1, npos - 1);
  a.n_cached = max(0, tc - a.t0);
  a.has_new = (a.t1 == npos);
  a.n_new = a.active ? A.pos[a.b] - A.p0[a.b] + 1 : 0;
  a.pb = S.page_bytes / (S.hd * 2);
  a.nblocks = (a.n_cached + a.pb - 1) / a.pb;
  if (!a.active) {  // no such sequence, or a split beyond this step's count
    a.n_cached = 0;
    a.nblocks = 0;
    a.has_new = false;
  }
  // the baked pointer addresses cache sequence b; row b reads sequence seq_b
  const int64_t rows = a.active ? (int64_t)(A.seq[a.b] - a.b) * S.Hkv * S.max_ctx : 0;
  a.kb = iptr(in, kP4) + (rows + a.t0) * S.hd;
  a.vb = iptr(in, kP5) + (rows + a.t0) * S.hd;
  return a;
}

// The tensor-core attention takes the units of at least half a page of cached positions
// (both roles decide alike).  Its page blk is the box of pb positions from attn_box_pos: the
// block's own positions are the box rows [lo, pb) -- all of them but in the last block, whose
// box ends at the unit's last cached position, so that its first rows hold earlier positions
// of the sequence (or zeros before position 0): finite values, masked by the consumer.
__device__ __forceinline__ bool attn_mma_unit(const DevState& S, const Attn& a) {
  return S.attn_mma && a.n_cached * 2 >= a.pb;
}
__device__ __noinline__ bool attn_use_mma(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  return attn_mma_unit(smem_ctl()->S, make_attn(smem_ctl()->S, smem_ctl()->args, in));
}
__device__ __forceinline__ int attn_box_pos(const Attn& a, int blk, int* lo) {
  const int start = blk * a.pb, np = min(a.pb, a.n_cached - start);
  *lo = a.pb - np;
  return a.t0 + start - *lo;
}

// a split-KV unit with work this step: its sequence is in the batch and its split below the
// sequence's active count (uniform over the CTA)
__device__ __forceinline__ bool attn_unit_active(const DevState& S, const StepArgs& A, const Instr& in) {
  return in.a[0] < A.B && in.a[2] < active_splits(S, A, in.a[0]);
}
// how many queued units to skip after an inactive one: all of its run (a5) when its split is
// past every sequence's active count -- the run's later units have no smaller split
__device__ __noinline__ int attn_run_skip(const DevState& S, const StepArgs& A, const Instr& in) {
  if (in.a[5] <= 0) return 0;
  int mx = 0;
  for (int b = 0; b < A.B; ++b) mx = max(mx, active_splits(S, A, b));
  return in.a[2] >= mx ? in.a[5] : 0;
}

// first (cos, sin) of sequence b's RoPE row: the table's row of its position, or row b of a
// table that holds one row per sequence of the step
__device__ __forceinline__ size_t rope_row(const DevState& S, const StepArgs& A, int b) {
  return (size_t)(S.rope_by_seq ? b : A.pos[b]) * (size_t)(S.hd / 2);
}

__device__ __forceinline__ float* act_ptr(const DevState& S, float* act, int kind, int layer) {
  return act + S.act_off[kind] + (int64_t)layer * S.act_stride[kind];
}


// ---------------------------------------------------------------- loader warp
// A free slot for the next page: its previous page handed back by every compute warp,
// and -- when the in-flight limit is set -- the page issued `inflight` copies earlier
// landed, so that at most that many copies of this CTA queue in the memory system (the
// ring still holds n_pages of landed pages as slack; fewer copies in flight shorten the
// queues that the dependency-carrying loads and stores wait in).
__device__ __noinline__ bool producer_wait(const DevState& S_arg, SmemCtl* c, uint64_t* bar, uint32_t parity) {
  const DevState& S = smem_ctl()->S;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_wait_hint(bar, parity, 2000u)) {
    if (c->abort) return false;
    if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
      set_err(S, 4u, -3, -1);
      c->abort = 1;
      return false;
    }
  }
  return true;
}
// fmin: the in-flight limit raised to at least this for the pages being issued
__device__ __noinline__ bool producer_acquire(const DevState& S_arg, SmemCtl* c, int slot, uint32_t ph, long long issued,
                                              int fmin = 0) {
  const DevState& S = smem_ctl()->S;
  if (!producer_wait(S, c, &c->empty[slot], ph ^ 1)) return false;
  const int F = S.inflight_pages > 0 ? max(S.inflight_pages, fmin) : 0;
  if (F > 0 && F < S.n_pages && issued >= F) {
    const int ps = slot - F < 0 ? slot - F + S.n_pages : slot - F;
    const uint32_t pp = slot - F < 0 ? ph ^ 1u : ph;
    if (!producer_wait(S, c, &c->full[ps], pp)) return false;
  }
  return true;
}

template <bool MS, bool TC, bool AM>
__device__ __noinline__ void producer(const DevState& S_arg, const StepArgs& A_arg, SmemCtl* c, uint8_t* pages) {
  const DevState& S = smem_ctl()->S;
  StepArgs& A = MS ? smem_ctl()->largs : smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  const uint64_t pol = l2_evict_first_policy();
  int slot = 0;
  uint32_t ph = 0;
  long long issued = 0;
  const int cta = blockIdx.x;
  const int end = A.q_start[cta + 1];
  const int n_steps = (MS && A.n_steps > 1) ? A.n_steps : 1;
  bool ok = true;
  // A multi-step launch walks the queue once per step.  The weights of a step do not depend
  // on the one before, so they stream ahead across the boundary; the KV blocks do (the
  // previous step appended its key/value rows): before the first of them the loader waits
  // for the previous step's tokens, which every CTA's whole step precedes.
  int ps = 0;          // attention pool FIFO slot and phase
  uint32_t pph = 0;
  for (int st = 0; st < n_steps && ok; ++st) {
  bool kv_ready = st == 0;
  // the K, V blocks of one split-KV unit (before the first of a multi-step launch's later
  // steps, wait for the previous step's tokens: that step appended its key/value rows)
  auto stream_attn = [&](const Instr& un) {
    if (MS && !kv_ready) {
      if (!wait_seq(&S.ctl->tok_seq, A.step, -10)) {
        c->abort = 1;
        ok = false;
        return;
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes before bulk reads
      kv_ready = true;
    }
    const Attn at = make_attn(S, A, un);
    if (AM && attn_mma_unit(S, at)) {  // one tensor-map box per K / V page (key map, value map after it)
      const uint8_t* km = reinterpret_cast<const uint8_t*>(iptr(un, kP3));
      const int bh = A.seq[at.b] * S.Hkv + at.j;
      for (int blk = 0; blk < at.nblocks && ok; ++blk) {
        int lo;
        const int p0 = attn_box_pos(at, blk, &lo);
        for (int kv = 0; kv < 2; ++kv) {
          // a long unit's K / V boxes are the step's bulk stream here: more of them in flight
          if (!producer_acquire(S, c, slot, ph, issued++, kKvInflight)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&c->full[slot], (uint32_t)S.page_bytes);
          tma_load_4d(pages + (size_t)slot * S.page_stride, km + kv * kTmapBytes, 0, p0, 0, bh,
                      &c->full[slot], pol);
          c->last_issue_phase[slot] = (int)ph;
          if (++slot == S.n_pages) { slot = 0; ph ^= 1u; }
        }
      }
      return;
    }
    for (int blk = 0; blk < at.nblocks && ok; ++blk) {
      const int p0 = blk * at.pb;
      const int np = min(at.pb, at.n_cached - p0);
      const uint32_t bytes = (uint32_t)np * S.hd * 2u;
      for (int kv = 0; kv < 2; ++kv) {
        if (!producer_acquire(S, c, slot, ph, issued++)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c->full[slot], bytes);
        tma_load_1d(pages + (size_t)slot * S.page_stride, (kv ? at.vb : at.kb) + (size_t)p0 * S.hd, bytes,
                    &c->full[slot], pol);
        c->last_issue_phase[slot] = (int)ph;
        if (++slot == S.n_pages) { slot = 0; ph ^= 1u; }
      }
    }
  };
  if (MS && st > 0) {
    A.step += 1u;
    A.epoch += 1u;
    for (int b = 0; b < A.B; ++b) {
      A.pos[b] += 1;
      A.p0[b] += 1;
    }
  }
  for (int pc = A.q_start[cta]; pc < end && ok; ++pc) {
    const Instr in = load_instr(A.instr + pc);
    if (pc + 2 < end) prefetch_l1(A.instr + pc + 2);  // the next instructions, for both roles
    if (in.op == OP_END) break;
    switch (in.op) {
      case OP_QKV:
      case OP_OPROJ:
      case OP_UPGATE:
      case OP_DOWN:
      case OP_LMHEAD: {
        const Gemv g = make_gemv(S, in);
        const int ns = g.nslices();
        const uint32_t sb = (uint32_t)g.WS * 2u;
        // the compute warps will read the RMSNorm gain and the RoPE rows of this
        // instruction right after its dependency: pull them into L1 now
        if (in.op == OP_QKV || in.op == OP_UPGATE || in.op == OP_LMHEAD) {
          const char* gp = reinterpret_cast<const char*>(iptr(in, kP2));
          for (int off = 0; off < S.d * 2; off += 128) prefetch_l1(gp + off);
        }
        if (in.op == OP_QKV && in.a[0] < 2) {
          for (int b = 0; b < A.B; ++b) {
            const char* rp = reinterpret_cast<const char*>(S.rope + rope_row(S, A, b) + in.a[2]);
            for (int off = 0; off < in.a[3] * 8 + 128; off += 128) prefetch_l1(rp + off);
          }
        }
        if (TC && S.tc && A.B >= 3) {
          // tensor-core pages: for each window of kTcKw columns, the 16-row blocks of
          // segment 0, then of segment 1, each one tensor-map copy (p4 / p5 hold the
          // segments' maps; rows and columns past the segment land as zeros)
          const int nw = (g.K + kTcKw - 1) / kTcKw;
          for (int w = 0; w < nw && ok; ++w) {
            for (int sg = 0; sg < 2 && ok; ++sg) {
              const void* tm = iptr(in, sg ? kP5 : kP4);
              const int nrs = (g.segr[sg] + kTcRows - 1) / kTcRows;
              for (int j = 0; j < nrs; ++j) {
                if (!producer_acquire(S, c, slot, ph, issued++)) {
                  ok = false;
                  break;
                }
                mbar_arrive_expect_tx(&c->full[slot], (uint32_t)kTcPageBytes);
                tma_load_3d(pages + (size_t)slot * S.page_stride, tm, 0, j * kTcRows, w * (kTcKw / kTcChunkCols),
                            &c->full[slot], pol);
                c->last_issue_phase[slot] = (int)ph;
                if (++slot == S.n_pages) { slot = 0; ph ^= 1u; }
              }
            }
          }
          break;
        }
        // rows of a segment are contiguous and a row is spr slices, so slice j of
        // segment k starts at seg[k] + j * WS: a page is at most two bulk copies
        const int n0 = g.segr[0] * g.spr();
        for (int i0 = 0; i0 < ns; i0 += kConsumerWarps) {
          if (!producer_acquire(S, c, slot, ph, issued++)) {
            ok = false;
            break;
          }
          const int i1 = min(ns, i0 + kConsumerWarps);
          mbar_arrive_expect_tx(&c->full[slot], (uint32_t)(i1 - i0) * sb);
          uint8_t* dst = pages + (size_t)slot * S.page_stride;
          if (i0 < n0) {
            const int e = min(i1, n0);
            tma_load_1d(dst, g.seg[0] + (size_t)i0 * g.WS, (uint32_t)(e - i0) * sb, &c->full[slot], pol);
          }
          if (i1 > n0) {
            const int b0 = max(i0, n0);
            tma_load_1d(dst + (size_t)(b0 - i0) * sb, g.seg[1] + (size_t)(b0 - n0) * g.WS, (uint32_t)(i1 - b0) * sb,
                        &c->full[slot], pol);
          }
          c->last_issue_phase[slot] = (int)ph;
          if (++slot == S.n_pages) { slot = 0; ph ^= 1u; }
        }
        break;
      }
      case OP_ATTN:
        stream_attn(in);
        // the compute warps skip the rest of an inactive run; so does the loader
        if (TC && !attn_unit_active(S, A, in)) pc += attn_run_skip(S, A, in);
        break;
      case OP_ATTN_POOL: {
        // dynamic work queue (§8.8): claim the layer's units one at a time while the ring
        // frees -- a CTA that reaches its attention early takes more of them -- and hand
        // each unit to the compute warps (in claim order) before streaming its K, V blocks.
        // A step makes a1 + a3 claims on the counter: every CTA's last one comes back empty.
        // In a multi-step launch a later step claims only once the step before has published
        // its tokens (every CTA is through all its claims of that step): a claim taken earlier
        // could land in the previous step's range of the counter.
        const uint32_t per_step = (uint32_t)(in.a[1] + in.a[3]);
        if (MS && !kv_ready) {
          if (!wait_seq(&S.ctl->tok_seq, A.step, -10)) {
            c->abort = 1;
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes before bulk reads
          kv_ready = true;
        }
        for (;;) {
          if (!producer_wait(S, c, &c->pool_empty[ps], pph ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t k = atomicAdd(&S.counters[in.a[2]], 1u);
          const uint32_t u = k - A.epoch * per_step;
          const int unit = u < (uint32_t)in.a[1] ? (int)u : -1;
          c->pool_fifo[ps] = unit;
          mbar_arrive(&c->pool_full[ps]);
          if (++ps == kPoolSlots) { ps = 0; pph ^= 1u; }
          if (unit < 0) break;
          stream_attn(load_instr(A.instr + in.a[0] + unit));
          if (!ok) break;
        }
        break;
      }
      case OP_T_PAGES: {
        const int n = in.a[1];
        const int64_t words = S.page_bytes / 8;
        for (int k = 0; k < n; ++k) {
          if (!producer_acquire(S, c, slot, ph, issued++)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&c->full[slot], (uint32_t)S.page_bytes);
          tma_load_1d(pages + (size_t)slot * S.page_stride, S.test_buf + in.a[0] + (int64_t)k * words,
                      (uint32_t)S.page_bytes, &c->full[slot], pol);
          c->last_issue_phase[slot] = (int)ph;
          if (++slot == S.n_pages) { slot = 0; ph ^= 1u; }
        }
        break;
      }
      default:
        break;
    }
  }
  }  // steps
  // Drain: every issued copy must land before the CTA exits, and -- unless the step was
  // abandoned -- every page must have been handed back (no leak, §8.9).
  const uint64_t t0 = globaltimer_ns();
  for (int s = 0; s < S.n_pages; ++s) {
    const int p = c->last_issue_phase[s];
    if (p < 0) continue;
    while (!mbar_try_wait(&c->full[s], (uint32_t)p)) {
      if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
        set_err(S, 4u, -4, s);
        return;
      }
    }
    if (c->abort) continue;
    while (!mbar_try_wait(&c->empty[s], (uint32_t)p)) {
      if (c->abort) break;
      if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
        set_err(S, 5u /*MK_ERR_STATE: page never released*/, -5, s);
        return;
      }
    }
  }
}

// ---------------------------------------------------------------- compute warps: pages
struct Ring {
  int slot;
  uint32_t ph;
};
// an op works on a register copy of the caller's ring position and writes it back when it
// returns (the caller's copy lives in local memory: reached through a generic pointer)
struct RingCopy {
  Ring& io;
  Ring r;
  __device__ __forceinline__ explicit RingCopy(Ring& ring) : io(ring), r(ring) {}
  __device__ __forceinline__ ~RingCopy() { io = r; }
};

__device__ __noinline__ void page_wait_slow(const DevState& S, SmemCtl* c, const Ring& r) {
  {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_wait_hint(&c->full[r.slot], r.ph, 2000u)) {
      if (c->abort) break;
      if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
        set_err(S, 4u, -6, r.slot);
        c->abort = 1;
        break;
      }
    }
  }
}
__device__ __forceinline__ const uint8_t* page_wait(const DevState& S, SmemCtl* c, uint8_t* pages, const Ring& r) {
  if (!mbar_try_wait(&c->full[r.slot], r.ph)) page_wait_slow(S, c, r);
  return pages + (size_t)r.slot * S.page_stride;
}
// "free at last read" (§8.4): each compute warp hands the page back as soon as its own
// reads are done; the loader refills it when all warps have done so.
__device__ __forceinline__ void page_release(const DevState& S, SmemCtl* c, Ring& r) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c->empty[r.slot]);
  if (++r.slot == S.n_pages) {
    r.slot = 0;
    r.ph ^= 1u;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// This CTA's share of the sums of squares of an RMSNorm input (the tensor-core GEMV's
// consumer adds the slots of all CTAs): ssp[b] per compute thread, summed over the threads
// in a fixed order into slot blockIdx.x of kMaxBatch floats (zeros past NB).  All compute
// threads call it; it uses the control block's reduction array.
template <int NB>
__device__ __forceinline__ void put_ssq_slot(SmemCtl* c, const float (&ssp)[NB], float* slots) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float t = warp_sum(ssp[b]);
    if (lane == 0) c->red[warp * NB + b] = t;
  }
  consumer_sync();
  if (tid < kMaxBatch) {
    float t = 0.f;
    if (tid < NB)
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) t += c->red[w * NB + tid];
    slots[(size_t)blockIdx.x * kMaxBatch + tid] = t;
  }
  consumer_sync();
}

// ---------------------------------------------------------------- input staging
// A producer's fp32 output reaches shared memory through 16-byte loads by every consumer
// thread, U vectors in flight per thread: one L2 round trip.  With counters the loads
// follow the acquire; with NaN sentinels the loads are the polls -- vectors that still
// hold a sentinel are re-read together (all of a thread's pending vectors in one round
// trip) until the producer's values land.  put(i, v) stores vector i.
__device__ __noinline__ float4 poll_slow_v4(const float4* p, const DevState& S, SmemCtl* c) {
  const uint64_t t0 = globaltimer_ns();
  int k = 0;
  while (true) {
    const int ns = 20 << (k < 8 ? k : 8);
    __nanosleep(ns < S.backoff_max_ns ? ns : S.backoff_max_ns);
    ++k;
    const float4 v = ld_poll_v4(p);
    if (!any_nan4(v)) return v;
    if (c->abort || global_err(S)) {
      c->abort = 1;
      return make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
      set_err(S, 4u, -1, -1);
      c->abort = 1;
      return make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}
template <int SYNC>
__device__ __forceinline__ float4 load_v4(const float4* p, const DevState& S, SmemCtl* c) {
  if (SYNC == SYNC_COUNTER) return __ldcg(p);
  const float4 v = ld_poll_v4(p);
  return any_nan4(v) ? poll_slow_v4(p, S, c) : v;
}

// One pause of a sentinel re-poll loop: backs off (exponentially, up to the configured
// cap) and returns false once the wait has run past the timeout or another party
// aborted (the abort flag is set and, if nothing was recorded yet, MK_ERR_TIMEOUT).
__device__ __forceinline__ bool poll_pause(const DevState& S, SmemCtl* c, int k, uint64_t t0) {
  const int ns = 20 << (k < 8 ? k : 8);
  __nanosleep(ns < S.backoff_max_ns ? ns : S.backoff_max_ns);
  if (c->abort || global_err(S) || globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
    if (!global_err(S)) set_err(S, 4u, -1, -1);
    c->abort = 1;
    return false;
  }
  return true;
}

// Up to U 16-byte loads in flight (entries with p[u] == nullptr are skipped and read as
// zeros); with sentinels, the vectors still holding one are re-read together until the
// producers' values land (bounded, sets the abort flag on timeout).
template <int SYNC, int U>
__device__ __forceinline__ void load_vecs(const DevState& S, SmemCtl* c, const float4* const (&p)[U], float4 (&v)[U]) {
  if (SYNC == SYNC_COUNTER) {
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = p[u] != nullptr ? __ldcg(p[u]) : make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  // sentinels: every vector is read, then those still holding one are re-read together
  // until none does; a pass issues all of its loads before testing any of them
#pragma unroll
  for (int u = 0; u < U; ++u) v[u] = p[u] != nullptr ? ld_poll_v4(p[u]) : make_float4(0.f, 0.f, 0.f, 0.f);
  uint64_t t0 = 0;
  for (int k = 0;; ++k) {
    bool pend = false;
#pragma unroll
    for (int u = 0; u < U; ++u) pend |= any_nan4(v[u]);
    if (!pend) break;
    if (k == 0) t0 = globaltimer_ns();
    if (!poll_pause(S, c, k, t0)) break;
    bool need[U];
#pragma unroll
    for (int u = 0; u < U; ++u) need[u] = any_nan4(v[u]);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (need[u]) v[u] = ld_poll_v4(p[u]);
  }
}

// Up to U 16-byte fragment vectors of a tensor-core input: vector i (base + u * threads +
// tid, below n) belongs to sequence ((i / 32) % MT) * 8 + (i % 32) / 4; vectors of
// sequences >= B are not read and come back as zeros.  With sentinels, vectors still
// holding a sentinel half are re-read together until the producers' values land
// (bounded, sets the abort flag on timeout).
template <int SYNC, int U>
__device__ __forceinline__ void load_frags(const DevState& S, SmemCtl* c, const uint4* src, int base, int n, int B,
                                           int MT, uint4 (&v)[U]) {
  const int tid = threadIdx.x;
  bool live[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = base + u * kConsumerThreads + tid;
    live[u] = i < n && ((((i >> 5) & (MT - 1)) << 3) + ((i & 31) >> 2)) < B;
    if (SYNC == SYNC_COUNTER) {
      v[u] = live[u] ? __ldcg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    } else {
      const float4 f = live[u] ? ld_poll_v4(reinterpret_cast<const float4*>(src + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[u] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
    }
  }
  if (SYNC == SYNC_COUNTER) return;
  uint64_t t0 = 0;
  for (int k = 0;; ++k) {
    bool need[U], pend = false;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      need[u] = live[u] && (frag_pending(v[u].x) || frag_pending(v[u].y) || frag_pending(v[u].z) ||
                            frag_pending(v[u].w));
      pend |= need[u];
    }
    if (!pend) break;
    if (k == 0) t0 = globaltimer_ns();
    if (!poll_pause(S, c, k, t0)) break;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (need[u]) {
        const float4 f = ld_poll_v4(reinterpret_cast<const float4*>(src + base + u * kConsumerThreads + tid));
        v[u] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
      }
  }
}


template <int SYNC, int U = 4, typename Put>
__device__ __forceinline__ void stage_vec(const DevState& S, const float4* src, int n4, SmemCtl* c, Put&& put) {
  const int tid = threadIdx.x;
  for (int base = 0; base < n4; base += U * kConsumerThreads) {
    const float4* p[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kConsumerThreads + tid;
      p[u] = i < n4 ? src + i : nullptr;
    }
    float4 v[U];
    load_vecs<SYNC, U>(S, c, p, v);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kConsumerThreads + tid;
      if (i < n4) put(i, v[u]);
    }
  }
}

// The O-proj input merged from the KV-split partials while it is staged (the §8.2
// ATTN_REDUCE folded into O_PROJ): for every (b, kv head j, group head g),
//   o = sum_s w_s o_s,  w_s = 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s',  M = max_s m_s,
// over the splits s < NS_b that ran this step (o_s, m_s, l_s: split s's weighted value
// sum, running max and exp-sum, in log2 units).  Every O-proj unit merges all heads, so
// none waits on a merge step.  Fixed summation order (s ascending).  The unit holding O-proj
// row 0 also publishes o (for mk_read_activation).
template <int SYNC, int NB>
__device__ void stage_merge(const DevState& S, const StepArgs& A, int l, float* xbuf, float* scratch, SmemCtl* c,
                            float* act, bool publish) {
  const int tid = threadIdx.x, B = A.B;
  const int HD = S.hd, G = S.Hq / S.Hkv, RW = HD + kPartExtra, Hkv = S.Hkv, SS = S.S, K = S.Hq * HD;
  const float* part = act_ptr(S, act, ACT_PART, l);  // [b][j][s][g][RW]
  const int nrec = B * Hkv * SS * G;
  float2* ml = reinterpret_cast<float2*>(scratch);         // [b][j][s][g] (max, sum)
  float* wts = scratch + 2 * nrec;                          // [b][j][g][s] merge weights
  // 1. (max, sum) of every record that was written this step
  {
    constexpr int U = 4;
    for (int base = 0; base < nrec; base += U * kConsumerThreads) {
      const float4* p[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kConsumerThreads + tid;
        p[u] = nullptr;
        if (r < nrec) {
          const int s = (r / G) % SS, b = r / (G * SS * Hkv);
          if (s < active_splits(S, A, b)) p[u] = reinterpret_cast<const float4*>(part + (size_t)r * RW + HD);
        }
      }
      float4 v[U];
      load_vecs<SYNC, U>(S, c, p, v);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = base + u * kConsumerThreads + tid;
        if (r < nrec) ml[r] = make_float2(v[u].x, v[u].y);
      }
    }
  }
  consumer_sync();
  // 2. weights per (b, j, g)
  for (int t = tid; t < B * Hkv * G; t += kConsumerThreads) {
    const int g = t % G, bj = t / G, b = bj / Hkv;
    const int NS = active_splits(S, A, b);
    float M = -CUDART_INF_F;
    for (int s = 0; s < NS; ++s) M = fmaxf(M, ml[(bj * SS + s) * G + g].x);
    float den = 0.f;
    for (int s = 0; s < NS; ++s) {
      const float2 r = ml[(bj * SS + s) * G + g];
      den = fmaf(exp2f(r.x - M), r.y, den);
    }
    const float inv = 1.0f / den;
    for (int s = 0; s < NS; ++s) wts[t * SS + s] = exp2f(ml[(bj * SS + s) * G + g].x - M) * inv;
  }
  consumer_sync();
  // 3. the merged vectors, four splits in flight per output vector
  const int n_out = B * K / 4, per_b = K / 4, per_h = HD / 4;
  float4* x4 = reinterpret_cast<float4*>(xbuf);
  float4* o4 = reinterpret_cast<float4*>(act_ptr(S, act, ACT_O, l));
  for (int i = tid; i < n_out; i += kConsumerThreads) {
    const int b = i / per_b, h = (i % per_b) / per_h, e4 = i % per_h;
    const int j = h / G, g = h % G, NS = active_splits(S, A, b);
    const float* w = wts + ((b * Hkv + j) * G + g) * SS;
    const float* base = part + (((size_t)(b * Hkv + j) * SS) * G + g) * RW + 4 * e4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < NS; s0 += 4) {
      const float4* p[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        p[u] = s0 + u < NS ? reinterpret_cast<const float4*>(base + (size_t)(s0 + u) * G * RW) : nullptr;
      float4 v[4];
      load_vecs<SYNC, 4>(S, c, p, v);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s0 + u < NS) {
          const float ws = w[s0 + u];
          acc.x = fmaf(ws, v[u].x, acc.x);
          acc.y = fmaf(ws, v[u].y, acc.y);
          acc.z = fmaf(ws, v[u].z, acc.z);
          acc.w = fmaf(ws, v[u].w, acc.w);
        }
      }
    }
    x4[i] = acc;
    if (publish) o4[i] = acc;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = n_out + tid; i < NB * per_b; i += kConsumerThreads) x4[i] = z;
}

// B rows of K fp32 values ([B][K], 16-byte aligned) into the x buffer; padding rows up
// to NB are zeroed.
template <int SYNC, int NB>
__device__ void stage_copy(const DevState& S, const float* src, int K, int B, float* xbuf, SmemCtl* c) {
  float4* x4 = reinterpret_cast<float4*>(xbuf);
  const int k4 = K / 4;
  stage_vec<SYNC, 8>(S, reinterpret_cast<const float4*>(src), B * k4, c, [&](int i, const float4& v) { x4[i] = v; });
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = B * k4 + threadIdx.x; i < NB * k4; i += kConsumerThreads) x4[i] = z;
}

// RMSNorm, folded: W (g . h / rms) = (W (g . h)) / rms.  The residual is staged scaled by
// the gain while each thread accumulates its share of sum(h^2); the per-warp sums go to
// c->red and the epilogue turns them into 1/rms (fixed order, same in every thread), so
// no CTA-wide pass sits between staging and the weight pages.  The gains do not depend on
// the producer: their loads are issued ahead of the polls of h and land while those wait.
template <typename WT, int SYNC, int NB>
__device__ void stage_rmsnorm(const DevState& S, const float* h, const uint16_t* gain, int B, float* xbuf,
                              SmemCtl* c) {
  constexpr int U = 4;
  const int d = S.d, d4 = d / 4, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, n4 = B * d4;
  float4* x4 = reinterpret_cast<float4*>(xbuf);
  const float4* h4 = reinterpret_cast<const float4*>(h);
  const uint2* g4 = reinterpret_cast<const uint2*>(gain);  // 4 gains per vector
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
  for (int base = 0; base < n4; base += U * kConsumerThreads) {
    const float4* p[U];
    uint2 gb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kConsumerThreads + tid;
      p[u] = i < n4 ? h4 + i : nullptr;
      gb[u] = i < n4 ? __ldg(g4 + (i % d4)) : make_uint2(0u, 0u);
    }
    float4 v[U];
    load_vecs<SYNC, U>(S, c, p, v);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kConsumerThreads + tid;
      if (i >= n4) continue;
      const int b = i / d4;
      float4 w = v[u];
      const float sq = w.x * w.x + w.y * w.y + w.z * w.z + w.w * w.w;
#pragma unroll
      for (int bb = 0; bb < NB; ++bb)
        if (bb == b) ss[bb] += sq;
      w.x *= Unpack<WT>::one((uint16_t)(gb[u].x & 0xFFFFu));
      w.y *= Unpack<WT>::one((uint16_t)(gb[u].x >> 16));
      w.z *= Unpack<WT>::one((uint16_t)(gb[u].y & 0xFFFFu));
      w.w *= Unpack<WT>::one((uint16_t)(gb[u].y >> 16));
      x4[i] = w;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = B * d4 + tid; i < NB * d4; i += kConsumerThreads) x4[i] = z;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float t = warp_sum(ss[b]);
    if (lane == 0) c->red[warp * NB + b] = t;
  }
}

// 1/rms of sequence b from the per-warp sums stage_rmsnorm left (after a barrier)
template <int NB>
__device__ __forceinline__ float inv_rms_of(const DevState& S, const SmemCtl* c, int b) {
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) t += c->red[w * NB + b];
  return 1.0f / sqrtf(t / (float)S.d + S.eps);
}

// ---------------------------------------------------------------- GEMV slice
// One warp, one slice (WS consecutive weights of one row) per page.  Shared memory is
// the limit here: fp32 x costs twice the bytes of the fp16/bf16 weights, so
//  * slice_dot_xreg (B <= 2, each warp always on the same slice of a row): the warp's
//    x segment sits in registers for the whole instruction; only weights are read from
//    the page, 16 bytes per lane, all loads in flight, four accumulator chains;
//  * slice_dot_smem (otherwise): 8-byte weight loads and 16-byte x loads, both
//    contiguous across the warp (no bank conflicts), two accumulator chains.
template <typename WT, int NB, int J>
__device__ __forceinline__ void slice_dot_xreg(const uint8_t* wp, const float (&xr)[NB][8 * J], int nv, int lane,
                                               float (&acc)[NB]) {
  const uint4* w = reinterpret_cast<const uint4*>(wp);
  uint4 wv[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int v = lane + 32 * j;
    wv[j] = v < nv ? w[v] : make_uint4(0u, 0u, 0u, 0u);
  }
  float a[NB][4];
#pragma unroll
  for (int b = 0; b < NB; ++b) a[b][0] = a[b][1] = a[b][2] = a[b][3] = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    float f[8];
    Unpack<WT>::u8(wv[j], f);
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int e = 0; e < 8; ++e) a[b][j & 3] = fmaf(f[e], xr[b][j * 8 + e], a[b][j & 3]);
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b] = (a[b][0] + a[b][1]) + (a[b][2] + a[b][3]);
}

template <typename WT, int NB>
__device__ __forceinline__ void slice_dot_smem(const uint8_t* wp, const float* x, int K, int WS, int lane,
                                               float (&acc)[NB]) {
  const uint2* w = reinterpret_cast<const uint2*>(wp);
  const int nq = WS >> 2;  // groups of four weights
  float a0[NB], a1[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) a0[b] = a1[b] = 0.f;
  int q = lane;
  for (; q + 32 < nq; q += 64) {
    const uint2 w0 = w[q], w1 = w[q + 32];
    float f0[4], f1[4];
    Unpack<WT>::u4(w0, f0);
    Unpack<WT>::u4(w1, f1);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float4 x0 = *reinterpret_cast<const float4*>(x + (size_t)b * K + q * 4);
      const float4 x1 = *reinterpret_cast<const float4*>(x + (size_t)b * K + (q + 32) * 4);
      a0[b] = fmaf(f0[0], x0.x, a0[b]);
      a0[b] = fmaf(f0[1], x0.y, a0[b]);
      a0[b] = fmaf(f0[2], x0.z, a0[b]);
      a0[b] = fmaf(f0[3], x0.w, a0[b]);
      a1[b] = fmaf(f1[0], x1.x, a1[b]);
      a1[b] = fmaf(f1[1], x1.y, a1[b]);
      a1[b] = fmaf(f1[2], x1.z, a1[b]);
      a1[b] = fmaf(f1[3], x1.w, a1[b]);
    }
  }
  if (q < nq) {
    float f0[4];
    Unpack<WT>::u4(w[q], f0);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float4 x0 = *reinterpret_cast<const float4*>(x + (size_t)b * K + q * 4);
      a0[b] = fmaf(f0[0], x0.x, a0[b]);
      a0[b] = fmaf(f0[1], x0.y, a0[b]);
      a0[b] = fmaf(f0[2], x0.z, a0[b]);
      a0[b] = fmaf(f0[3], x0.w, a0[b]);
    }
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b] = a0[b] + a1[b];
}

// silu(u) = u / (1 + e^-u); the fast exponential (a few ulp) is far inside the tolerance
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

// The GEMV epilogue (after the barrier that ends the pages): each row is finished from its
// row parts in a fixed order and the op's output is written.  rowpart [rows][spr][NB];
// hres / cs0 are the thread's prefetched residual and RoPE row (its first row).
template <typename WT, int SYNC, int NB>
__device__ __forceinline__ void gemv_epilogue(const DevState& S, const StepArgs& A, const Instr& in, SmemCtl* c,
                                              float* act, const float* rowpart, int spr, int R, float hres,
                                              float2 cs0) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = A.B, l = in.layer;
  auto rowsum = [&](int r, int b) {
    float t = 0.f;
    for (int s = 0; s < spr; ++s) t += rowpart[((size_t)r * spr + s) * NB + b];
    return t;
  };
  switch (in.op) {
    case OP_QKV: {
      const int mat = in.a[0], head = in.a[1], i0 = in.a[2], n = in.a[3];
      const int hd = S.hd, half = hd / 2;
      for (int t = tid; t < n * B; t += kConsumerThreads) {
        const int r = t % n, b = t / n;
        const float ir = c->inv_rms[b];
        float va = rowsum(r, b) * ir, vb = rowsum(r + n, b) * ir;
        const int i = i0 + r;
        const int pos = A.pos[b];
        if (mat < 2) {  // rotate-half RoPE on the pair (i, i + hd/2)
          const float2 cs = t == tid ? cs0 : S.rope[rope_row(S, A, b) + i];
          const float xa = va * cs.x - vb * cs.y;
          const float xb = vb * cs.x + va * cs.y;
          va = xa;
          vb = xb;
        }
        if (mat == 0) {
          float* q = act_ptr(S, act, ACT_Q, l) + (size_t)b * S.Hq * hd + (size_t)head * hd;
          q[i] = va;
          q[i + half] = vb;
        } else {
          const uint16_t ra = Unpack<WT>::round(va), rb = Unpack<WT>::round(vb);
          uint16_t* cache =
              const_cast<uint16_t*>(iptr(in, kP3)) + (((size_t)A.seq[b] * S.Hkv + head) * S.max_ctx + pos) * hd;
          cache[i] = ra;
          cache[i + half] = rb;
          float* kvn = act_ptr(S, act, ACT_KVN, l) + ((size_t)b * 2 + (mat - 1)) * S.Hkv * hd + (size_t)head * hd;
          kvn[i] = Unpack<WT>::one(ra);
          kvn[i + half] = Unpack<WT>::one(rb);
        }
      }
      break;
    }
    case OP_OPROJ: {
      const int row0 = in.a[0];
      const float* hin = act_ptr(S, act, ACT_H, l);
      float* hout = act_ptr(S, act, ACT_HMID, l);
      uint16_t* fo = reinterpret_cast<uint16_t*>(act_ptr(S, act, ACT_HMF, l));
      const uint16_t* gn = iptr(in, kP2);
      float ssp[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) ssp[b] = 0.f;
      for (int t = tid; t < R * B; t += kConsumerThreads) {
        const int r = t % R, b = t / R;
        const size_t idx = (size_t)b * S.d + row0 + r;
        float hv = t == tid ? hres : load_act<SYNC>(hin + idx, S, c);
        if (SYNC == SYNC_SENTINEL && isnan(hv)) hv = poll_slow(hin + idx, S, c);
        const float y = hv + rowsum(r, b);
        hout[idx] = y;
        if (NB >= 4) {
          put_frag<WT>(fo, b, row0 + r, kFragMT<NB>, y * Unpack<WT>::one(gn[row0 + r]));
#pragma unroll
          for (int bb = 0; bb < NB; ++bb)
            if (bb == b) ssp[bb] += y * y;
        }
      }
      if (NB >= 4) put_ssq_slot<NB>(c, ssp, act_ptr(S, act, ACT_SSM, l));
      break;
    }
    case OP_UPGATE: {
      const int row0 = in.a[0], n = in.a[1];
      float* a = act_ptr(S, act, ACT_A, l);
      uint16_t* fo = reinterpret_cast<uint16_t*>(act_ptr(S, act, ACT_AF, l));
      for (int t = tid; t < n * B; t += kConsumerThreads) {
        const int r = t % n, b = t / n;
        const float ir = c->inv_rms[b];
        const float y = silu_f(rowsum(r, b) * ir) * (rowsum(r + n, b) * ir);
        a[(size_t)b * S.F + row0 + r] = y;
        if (NB >= 4) put_frag<WT>(fo, b, row0 + r, kFragMT<NB>, y);
      }
      break;
    }
    case OP_DOWN: {
      const int row0 = in.a[0];
      const float* hin = act_ptr(S, act, ACT_HMID, l);
      float* hout = act_ptr(S, act, ACT_H, l + 1);
      uint16_t* fo = reinterpret_cast<uint16_t*>(act_ptr(S, act, ACT_HF, l + 1));
      const uint16_t* gn = iptr(in, kP2);
      float ssp[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) ssp[b] = 0.f;
      for (int t = tid; t < R * B; t += kConsumerThreads) {
        const int r = t % R, b = t / R;
        const size_t idx = (size_t)b * S.d + row0 + r;
        float hv = t == tid ? hres : load_act<SYNC>(hin + idx, S, c);
        if (SYNC == SYNC_SENTINEL && isnan(hv)) hv = poll_slow(hin + idx, S, c);
        const float y = hv + rowsum(r, b);
        hout[idx] = y;
        if (NB >= 4) {
          put_frag<WT>(fo, b, row0 + r, kFragMT<NB>, y * Unpack<WT>::one(gn[row0 + r]));
#pragma unroll
          for (int bb = 0; bb < NB; ++bb)
            if (bb == b) ssp[bb] += y * y;
        }
      }
      if (NB >= 4) put_ssq_slot<NB>(c, ssp, act_ptr(S, act, ACT_SSH, l + 1));
      break;
    }
    default: {  // OP_LMHEAD: logits and the running argmax (packed key, lowest index wins ties)
      const int row0 = in.a[0];
      unsigned long long best[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) best[b] = 0ull;
      for (int t = tid; t < R * NB; t += kConsumerThreads) {
        const int r = t % R, b = t / R;
        if (b >= B) continue;
        const float z = rowsum(r, b) * c->inv_rms[b];
        const int row = row0 + r;
        if (A.logits) A.logits[(size_t)b * S.V + row] = z;
        if (isnan(z)) atomicOr(&S.ctl->nan_seen, 1u);
        const unsigned long long key =
            ((unsigned long long)orderable(z) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
          if (bb == b && key > best[bb]) best[bb] = key;
      }
      // each warp's best per sequence, then one thread per sequence over the warps (fixed
      // order) and one atomic on the CTA's running best
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        unsigned long long v = best[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
          v = w > v ? w : v;
        }
        if (lane == 0) c->wbest[(tid >> 5) * NB + b] = v;
      }
      consumer_sync();
      if (tid < B) {
        unsigned long long v = 0ull;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const unsigned long long x = c->wbest[w * NB + tid];
          v = x > v ? x : v;
        }
        if (v) atomicMax(&c->best[tid], v);
      }
      break;
    }
  }
}

template <typename WT, int SYNC, int NB>
__device__ __noinline__ void op_gemv(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c, uint8_t* pages,
                        float* xbuf, float* scratch, Ring& ring_io, float* act) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  RingCopy ring_copy(ring_io);
  Ring& ring = ring_copy.r;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = A.B, l = in.layer;
  const Gemv g = make_gemv(S, in);

  // 1. inputs (one inlined copy of each staging routine: the op only picks the source)
  const float* src;
  switch (in.op) {
    case OP_QKV: src = act_ptr(S, act, ACT_H, l); break;
    case OP_UPGATE: src = act_ptr(S, act, ACT_HMID, l); break;
    case OP_LMHEAD: src = act_ptr(S, act, ACT_H, S.L); break;
    case OP_OPROJ: src = act_ptr(S, act, ACT_O, l); break;
    default: src = act_ptr(S, act, ACT_A, l); break;  // OP_DOWN
  }
  if (in.op == OP_QKV || in.op == OP_UPGATE || in.op == OP_LMHEAD)
    stage_rmsnorm<WT, SYNC, NB>(S, src, iptr(in, kP2), B, xbuf, c);
  else if (in.flags & F_MERGE_IN)
    stage_merge<SYNC, NB>(S, A, l, xbuf, scratch, c, act, in.a[0] == 0);
  else
    stage_copy<SYNC, NB>(S, src, g.K, B, xbuf, c);
  consumer_sync();
  if (tid == 0 && (A.flags & SF_TRACE)) c->tmark[0] = globaltimer_ns();
  // the residual this thread adds in the epilogue (its first row), loaded now so the
  // latency hides behind the pages: the load is only issued here -- a sentinel is
  // checked (and re-polled) in the epilogue, so no warp waits for it before its pages
  float hres = 0.f;
  if ((in.op == OP_OPROJ || in.op == OP_DOWN) && tid < g.rows() * B) {
    const int r = tid % g.rows(), b = tid / g.rows();
    const float* hp = act_ptr(S, act, in.op == OP_OPROJ ? ACT_H : ACT_HMID, l) + (size_t)b * S.d + in.a[0] + r;
    hres = SYNC == SYNC_COUNTER ? __ldcg(hp) : ld_poll_f32(hp);
  }
  // likewise the (cos, sin) of the thread's first RoPE pair, and 1/rms per sequence (read
  // by the epilogue after the barrier that ends the pages)
  float2 cs0 = make_float2(1.f, 0.f);
  if (in.op == OP_QKV && in.a[0] < 2 && tid < in.a[3] * B)
    cs0 = S.rope[rope_row(S, A, tid / in.a[3]) + in.a[2] + tid % in.a[3]];
  if ((in.op == OP_QKV || in.op == OP_UPGATE || in.op == OP_LMHEAD) && tid < B) c->inv_rms[tid] = inv_rms_of<NB>(S, c, tid);

  // 2. stream the slices: warp w takes slice i0 + w of every page of 8 slices
  float* rowpart = scratch;  // [rows][spr][NB]
  const int spr = g.spr(), ns = g.nslices();
  const bool trace = (A.flags & SF_TRACE) != 0;
  uint64_t page_wait_ns = 0, page_work_ns = 0;
  auto run_pages = [&](auto&& dot) {
    for (int i0 = 0; i0 < ns; i0 += kConsumerWarps) {
      const uint64_t tw = trace ? globaltimer_ns() : 0ull;
      const uint8_t* pg = page_wait(S, c, pages, ring);
      const uint64_t tr = trace ? globaltimer_ns() : 0ull;
      if (trace) page_wait_ns += tr - tw;
      const int i = i0 + warp;
      if (i < ns) {
        const int r = i / spr, s = i - r * spr;
        float acc[NB];
        dot(pg + (size_t)warp * g.WS * 2, s, acc);
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
        if (lane == 0) {
#pragma unroll
          for (int b = 0; b < NB; ++b) rowpart[((size_t)r * spr + s) * NB + b] = acc[b];
        }
      }
      page_release(S, c, ring);
      if (trace) page_work_ns += globaltimer_ns() - tr;
    }
  };
  bool done = false;
  // slices i = 8c + w: when spr divides 8, warp w always sees slice w % spr of a row and
  // keeps that segment of x in registers (J 16-byte vectors per lane)
  auto run_xreg = [&](auto jtag) {
    constexpr int J = decltype(jtag)::value;
    const int nv = g.WS >> 3, sw = warp % spr;
    float xr[NB][8 * J];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int v = lane + 32 * j;
        const float* xp = xbuf + (size_t)b * g.K + (size_t)sw * g.WS + v * 8;
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (v < nv) {
          x0 = reinterpret_cast<const float4*>(xp)[0];
          x1 = reinterpret_cast<const float4*>(xp)[1];
        }
        xr[b][j * 8 + 0] = x0.x; xr[b][j * 8 + 1] = x0.y; xr[b][j * 8 + 2] = x0.z; xr[b][j * 8 + 3] = x0.w;
        xr[b][j * 8 + 4] = x1.x; xr[b][j * 8 + 5] = x1.y; xr[b][j * 8 + 6] = x1.z; xr[b][j * 8 + 7] = x1.w;
      }
    run_pages([&](const uint8_t* wp, int, float(&acc)[NB]) { slice_dot_xreg<WT, NB, J>(wp, xr, nv, lane, acc); });
  };
  if constexpr (NB <= 2) {
    if (kConsumerWarps % spr == 0 && g.WS <= 32 * 8 * 4) {
      run_xreg(std::integral_constant<int, 4>{});
      done = true;
    }
  }
  if constexpr (NB == 1) {
    if (!done && kConsumerWarps % spr == 0 && g.WS <= 32 * 8 * 8) {
      run_xreg(std::integral_constant<int, 8>{});
      done = true;
    }
  }
  if (!done)
    run_pages([&](const uint8_t* wp, int s, float(&acc)[NB]) {
      slice_dot_smem<WT, NB>(wp, xbuf + (size_t)s * g.WS, g.K, g.WS, lane, acc);
    });
  consumer_sync();
  if (tid == 0 && trace) {
    c->tmark[1] = globaltimer_ns();
    c->tmark[2] = page_wait_ns;
    c->tmark[4] = page_work_ns;
  }

  // 3. finalize rows in a fixed order and apply the op's epilogue
  const long long ck0 = trace ? clock64() : 0;
  gemv_epilogue<WT, SYNC, NB>(S, A, in, c, act, rowpart, spr, g.rows(), hres, cs0);
  if (tid == 0 && trace) {
    c->tmark[3] = globaltimer_ns();
    c->tmark[5] = (uint64_t)(clock64() - ck0);
  }
}

// ---------------------------------------------------------------- tensor-core GEMV
// Batches of 3..16: y[b] = W x[b] for 16-row blocks of
// weights at a time with mma.sync m16n8k16.  A = the inputs: each 16-row A tile holds 8
// sequences' inputs split into hi and lo 16-bit halves (rows 0-7 hi, rows 8-15 lo: the
// MMA's f32 accumulator sums both, so the inputs keep ~22 significant bits with fp16);
// B = 8 weight rows (a weight row is a column of B, its elements contiguous as in memory).
// The input is staged one window of kTcKw columns at a time, already in fragment order;
// the loader brings, per window, 16-row blocks of the instruction's rows.  Warps split a
// page's k-steps; their partials are summed in a fixed order into per-row accumulators,
// and the common epilogue finishes the rows.
// Tensor-core GEMV input staging through the copy engine: thread 0 issues one bulk copy of
// the staging's fragment vectors into shared memory, landing on half h's mbarrier.  The
// proxy fence orders this CTA's earlier generic accesses of the destination and the
// producers' writes it has acquired before the asynchronous copy.
__device__ __noinline__ void xstage_issue(SmemCtl* c, int h, void* dst, const void* src, uint32_t bytes) {
  asm volatile("fence.proxy.async;" ::: "memory");
  mbar_arrive_expect_tx(&c->xfull[h], bytes);
  tma_load_1d_plain(dst, src, bytes, &c->xfull[h]);
}
// a fragment vector still holding sentinel halves, re-read until its producers' values
// land (bounded: sets the abort flag and returns zeros on timeout)
__device__ __noinline__ uint4 poll_frag(const uint4* p, const DevState& S, SmemCtl* c) {
  const uint64_t t0 = globaltimer_ns();
  for (int k = 0;; ++k) {
    if (!poll_pause(S, c, k, t0)) return make_uint4(0u, 0u, 0u, 0u);
    const float4 f = ld_poll_v4(reinterpret_cast<const float4*>(p));
    const uint4 v = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
    if (!(frag_pending(v.x) || frag_pending(v.y) || frag_pending(v.z) || frag_pending(v.w))) return v;
  }
}
// All compute threads: wait (bounded) for half h's copy of n vectors, then, with sentinels,
// re-read from src the vectors of live sequences the copy caught before their producers
// wrote them; ends with a CTA barrier.
template <int SYNC>
__device__ __noinline__ void xstage_land(const DevState& S_arg, SmemCtl* c, int h, uint32_t ph, uint4* x, const uint4* src,
                                         int n, int B, int MT) {
  const DevState& S = smem_ctl()->S;
  c = smem_ctl();
  if (!mbar_try_wait(&c->xfull[h], ph)) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_wait_hint(&c->xfull[h], ph, 2000u)) {
      if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
        set_err(S, 4u, -12, h);
        c->abort = 1;
        break;
      }
    }
  }
  if (SYNC == SYNC_SENTINEL) {
    for (int i = threadIdx.x; i < n; i += kConsumerThreads) {
      if ((((i >> 5) & (MT - 1)) << 3) + ((i & 31) >> 2) >= B) continue;  // no such sequence
      const uint4 v = x[i];
      if (frag_pending(v.x) || frag_pending(v.y) || frag_pending(v.z) || frag_pending(v.w))
        x[i] = poll_frag(src + i, S, c);
    }
  }
  consumer_sync();
}

template <typename WT, int SYNC, int NB>
__device__ __noinline__ void op_gemv_tc(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c,
                                        uint8_t* pages, float* xbuf, float* scratch, Ring& ring_io, float* act) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  RingCopy ring_copy(ring_io);
  Ring& ring = ring_copy.r;
  constexpr int MT = (NB + 7) / 8;  // A tiles of 8 sequences
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  const int B = A.B, l = in.layer;
  const Gemv g = make_gemv(S, in);
  const int K = g.K, R = g.rows(), nw = (K + kTcKw - 1) / kTcKw;
  // row blocks: segment 0's, then segment 1's (a page never spans the two)
  const int nrb0 = (g.segr[0] + kTcRows - 1) / kTcRows, nrb = nrb0 + (g.segr[1] + kTcRows - 1) / kTcRows;
  const bool trace = (A.flags & SF_TRACE) != 0;
  float* part = scratch;                       // [2][warps][kTcRows][NB]
  float* rowacc = scratch + kTcPartialFloats;  // [R][NB]
  // the input in fragment form, written by its producers (gain x input for the ops after
  // an RMSNorm), and for those the producers' per-CTA sums of squares of the input
  const uint16_t* gain = nullptr;
  const uint4* frag;
  const float* ssq = nullptr;
  switch (in.op) {
    case OP_QKV:
      gain = iptr(in, kP2);
      frag = reinterpret_cast<const uint4*>(act_ptr(S, act, ACT_HF, l));
      ssq = act_ptr(S, act, ACT_SSH, l);
      break;
    case OP_UPGATE:
      gain = iptr(in, kP2);
      frag = reinterpret_cast<const uint4*>(act_ptr(S, act, ACT_HMF, l));
      ssq = act_ptr(S, act, ACT_SSM, l);
      break;
    case OP_LMHEAD:
      gain = iptr(in, kP2);
      frag = reinterpret_cast<const uint4*>(act_ptr(S, act, ACT_HF, S.L));
      ssq = act_ptr(S, act, ACT_SSH, S.L);
      break;
    case OP_OPROJ: frag = reinterpret_cast<const uint4*>(act_ptr(S, act, ACT_OF, l)); break;
    default: frag = reinterpret_cast<const uint4*>(act_ptr(S, act, ACT_AF, l)); break;  // OP_DOWN
  }

  for (int i = tid; i < R * NB; i += kConsumerThreads) rowacc[i] = 0.f;
  // epilogue inputs, prefetched as in the CUDA-core GEMV
  float hres = 0.f;
  if ((in.op == OP_OPROJ || in.op == OP_DOWN) && tid < R * B) {
    const int r = tid % R, b = tid / R;
    const float* hp = act_ptr(S, act, in.op == OP_OPROJ ? ACT_H : ACT_HMID, l) + (size_t)b * S.d + in.a[0] + r;
    hres = SYNC == SYNC_COUNTER ? __ldcg(hp) : ld_poll_f32(hp);
  }
  float2 cs0 = make_float2(1.f, 0.f);
  if (in.op == OP_QKV && in.a[0] < 2 && tid < in.a[3] * B)
    cs0 = S.rope[rope_row(S, A, tid / in.a[3]) + in.a[2] + tid % in.a[3]];
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
  uint64_t page_wait_ns = 0, page_work_ns = 0;
  int pcount = 0;
  // x staging.  With counters (the dependency wait has seen the producers done) by bulk
  // copies of the fragment form: every window at once when they fit the x buffer, else one
  // window per copy, double-buffered (the next window's copy in flight while this window's
  // pages run) when two windows fit, else one after the other.  With sentinels a copy could
  // catch the producers mid-write, so the compute threads poll the vectors in, SW windows
  // (as many as the buffer holds) per staging.
  const int wv = (kTcKw >> 4) * MT * 32;  // 16-byte vectors of a full window
  auto stage_n = [&](int w0, int nwin) { return ((min(K, (w0 + nwin) * kTcKw) - w0 * kTcKw) >> 4) * MT * 32; };
  const bool whole = stage_n(0, nw) * 16 <= S.xbuf_bytes;
  const bool dbl = SYNC == SYNC_COUNTER && !whole && 2 * wv * 16 <= S.xbuf_bytes;
  const int SW = whole ? nw : (dbl ? 1 : max(1, S.xbuf_bytes / (wv * 16)));
  uint4* xb = reinterpret_cast<uint4*>(xbuf);
  uint32_t xph[2] = {c->xph[0], c->xph[1]};
  // a CTA's LM head instructions follow each other with the same input: after the first
  // staged it whole (and set 1/rms), the others reuse it
  const bool reuse = in.op == OP_LMHEAD && whole && c->lm_staged;
  if (SYNC == SYNC_COUNTER && !reuse && tid == 0) xstage_issue(c, 0, xb, frag, (uint32_t)stage_n(0, SW) * 16u);
  // with an RMSNorm: the producers' per-CTA sums of squares of the input (one slot of
  // kMaxBatch floats per producing CTA), slot tid into this thread's ss[]
  if (gain != nullptr && !reuse && tid < S.n_cta) {
    const float4* sp = reinterpret_cast<const float4*>(ssq + (size_t)tid * kMaxBatch);
    const float4* pp[NB / 4];
#pragma unroll
    for (int q = 0; q < NB / 4; ++q) pp[q] = sp + q;
    float4 v[NB / 4];
    load_vecs<SYNC, NB / 4>(S, c, pp, v);
#pragma unroll
    for (int q = 0; q < NB / 4; ++q) {
      ss[4 * q] = v[q].x;
      ss[4 * q + 1] = v[q].y;
      ss[4 * q + 2] = v[q].z;
      ss[4 * q + 3] = v[q].w;
    }
  }
  for (int w = 0; w < nw; ++w) {
    const int k0 = w * kTcKw, kw = min(kTcKw, K - k0), nks = kw >> 4;
    // 1. this staging's inputs: the producers wrote them as hi/lo halves in fragment order
    //    (8 sequences per tile; slots of sequences >= B are not read).  A copy into a buffer
    //    the previous window read is issued after that window's last page barrier.
    const int h = dbl ? (w & 1) : 0;
    uint4* xw = xb + (dbl ? h * wv : 0);
    if (w % SW == 0 && !reuse) {
      const int n16 = stage_n(w, SW);
      if (SYNC == SYNC_COUNTER) {
        if (w > 0 && !dbl && tid == 0) xstage_issue(c, 0, xw, frag + (size_t)w * wv, (uint32_t)n16 * 16u);
        xstage_land<SYNC>(S, c, h, xph[h], xw, frag + (size_t)w * wv, n16, B, MT);
        xph[h] ^= 1u;
        if (dbl && w + 1 < nw && tid == 0)
          xstage_issue(c, h ^ 1, xb + (h ^ 1) * wv, frag + (size_t)(w + 1) * wv, (uint32_t)stage_n(w + 1, 1) * 16u);
      } else {
        constexpr int U = 8;
        const uint4* fs = frag + (size_t)w * wv;
        for (int base = 0; base < n16; base += U * kConsumerThreads) {
          uint4 v[U];
          load_frags<SYNC, U>(S, c, fs, base, n16, B, MT, v);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = base + u * kConsumerThreads + tid;
            if (i < n16) xw[i] = v[u];
          }
        }
        consumer_sync();
      }
    }
    const int kso = (w % SW) * (kTcKw >> 4);  // this window's first k-step in the staged tile
    const uint32_t* xtw = reinterpret_cast<const uint32_t*>(xw);
    if (tid == 0 && trace && w == 0) c->tmark[0] = globaltimer_ns();
    // 2. the window's row blocks
    const int per = (nks + kConsumerWarps - 1) / kConsumerWarps, ks0 = warp * per, ks1 = min(nks, ks0 + per);
    for (int rb = 0; rb < nrb; ++rb) {
      const uint64_t tw = trace ? globaltimer_ns() : 0ull;
      const uint8_t* pg = page_wait(S, c, pages, ring);
      const uint64_t tr = trace ? globaltimer_ns() : 0ull;
      if (trace) page_wait_ns += tr - tw;
      float d[MT][2][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) d[mt][nb][0] = d[mt][nb][1] = d[mt][nb][2] = d[mt][nb][3] = 0.f;
      for (int ks = ks0; ks < ks1; ++ks) {
        // k-step ks: columns 16 ks .. 16 ks + 15 = 16-byte granules 2 (ks % 4) and + 1 of
        // column chunk ks / 4; row r's granule g sits at g ^ (r % 8), and r % 8 = gq
        uint32_t bw[2][2];
        const uint8_t* cb = pg + (size_t)(ks >> 2) * kTcChunkBytes + cq * 4;
        const int g0 = ((ks & 3) * 2) ^ gq;
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const uint8_t* wr = cb + (nb * 8 + gq) * 128;
          bw[nb][0] = *reinterpret_cast<const uint32_t*>(wr + g0 * 16);
          bw[nb][1] = *reinterpret_cast<const uint32_t*>(wr + (g0 ^ 1) * 16);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint4 a = *reinterpret_cast<const uint4*>(xtw + ((size_t)((kso + ks) * MT + mt) * 32 + lane) * 4);
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) Mma<WT>::run(d[mt][nb], a, bw[nb][0], bw[nb][1]);
        }
      }
      page_release(S, c, ring);
      // hi + lo of (sequence mt*8 + g, weight rows nb*8 + 2c and + 1) into this warp's partial
      float* pb = part + ((size_t)((pcount & 1) * kConsumerWarps + warp) * kTcRows) * NB;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int sq = mt * 8 + gq;
        if (sq < NB) {
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            pb[(nb * 8 + 2 * cq) * NB + sq] = d[mt][nb][0] + d[mt][nb][2];
            pb[(nb * 8 + 2 * cq + 1) * NB + sq] = d[mt][nb][1] + d[mt][nb][3];
          }
        }
      }
      consumer_sync();
      if (tid < kTcRows * NB) {  // one (row, sequence) per thread: warps summed in a fixed order
        const int row = tid / NB, sq = tid - row * NB;
        const int sg = rb >= nrb0 ? 1 : 0, j = rb - sg * nrb0;
        const int fr = sg * g.segr[0] + j * kTcRows + row;
        if (j * kTcRows + row < g.segr[sg]) {
          const float* pr = part + ((size_t)(pcount & 1) * kConsumerWarps * kTcRows + row) * NB + sq;
          float t = 0.f;
#pragma unroll
          for (int ww = 0; ww < kConsumerWarps; ++ww) t += pr[(size_t)ww * kTcRows * NB];
          rowacc[(size_t)fr * NB + sq] += t;
        }
      }
      ++pcount;
      if (trace) page_work_ns += globaltimer_ns() - tr;
    }
  }
  // 1/rms from the sums of squares
  if (gain != nullptr) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float t = warp_sum(ss[b]);
      if (lane == 0) c->red[warp * NB + b] = t;
    }
  }
  consumer_sync();
  if (gain != nullptr && !reuse && tid < B) c->inv_rms[tid] = inv_rms_of<NB>(S, c, tid);
  if (tid == 0) {  // the staging copies' phases, for the next op (after the loop's barrier)
    c->xph[0] = xph[0];
    c->xph[1] = xph[1];
    c->lm_staged = in.op == OP_LMHEAD && whole;
  }
  consumer_sync();
  if (tid == 0 && trace) {
    c->tmark[1] = globaltimer_ns();
    c->tmark[2] = page_wait_ns;
    c->tmark[4] = page_work_ns;
  }
  const long long ck0 = trace ? clock64() : 0;
  gemv_epilogue<WT, SYNC, NB>(S, A, in, c, act, rowacc, 1, R, hres, cs0);
  if (tid == 0 && trace) {
    c->tmark[3] = globaltimer_ns();
    c->tmark[5] = (uint64_t)(clock64() - ck0);
  }
}

// ---------------------------------------------------------------- attention
// The split's partial record from the compute warps' partials in scratch ([warp][G][HD +
// kPartExtra]: G rows of HD weighted sums, then the warp's running max and sum): the warps'
// sums weighted by exp2(m_w - M) (a warp that saw no position has m_w = -inf and weight 0);
// the thread of element 0 of a head also writes M, the weighted sum and the two zero pads
template <int HD, int G>
__device__ __forceinline__ void attn_combine_warps(const DevState& S, float* act, const Attn& at, int l,
                                                   const float* scratch) {
  constexpr int RW = HD + kPartExtra;
  const int tid = threadIdx.x;
  float* part = act_ptr(S, act, ACT_PART, l) + (((size_t)at.b * S.Hkv + at.j) * S.S + at.s) * G * RW;
  for (int t = tid; t < G * HD; t += kConsumerThreads) {
    const int g = t / HD, e = t - g * HD;
    const float* sg = scratch + g * RW;
    float mw[kConsumerWarps], wt[kConsumerWarps];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      mw[w] = sg[w * G * RW + HD];
      M = fmaxf(M, mw[w]);
    }
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) wt[w] = mw[w] == -CUDART_INF_F ? 0.f : exp2f(mw[w] - M);
    float r0 = 0.f, r1 = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; w += 2) {
      r0 = fmaf(wt[w], sg[w * G * RW + e], r0);
      r1 = fmaf(wt[w + 1], sg[(w + 1) * G * RW + e], r1);
    }
    part[g * RW + e] = r0 + r1;
    if (e == 0) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) L = fmaf(wt[w], sg[w * G * RW + HD + 1], L);
      part[g * RW + HD] = M;
      part[g * RW + HD + 1] = L;
      part[g * RW + HD + 2] = 0.f;  // pads: written so that sentinel polls of the whole record end
      part[g * RW + HD + 3] = 0.f;
    }
  }
}

template <typename WT, int SYNC, int HD, int G>
__device__ __noinline__ void op_attn(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c, uint8_t* pages,
                        float* xbuf, float* scratch, Ring& ring_io, float* act) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  RingCopy ring_copy(ring_io);
  Ring& ring = ring_copy.r;
  // DPL dims per lane = DPL/8 16-byte row chunks, lane dl of a position group taking
  // chunks dl, dl + LPP, ... (each load instruction reads contiguous bytes across the
  // group: no bank conflicts).  16 dims per lane for G <= 2 (fewer shuffle stages per
  // score, more positions per pass); 8 for G = 4 keeps the heads' accumulators inside the
  // register budget (9 warps put 3 warps on one SM sub-partition of 16K registers, i.e.
  // 168 registers per thread)
  constexpr int DPL = G <= 2 ? 16 : 8;
  constexpr int LPP = HD / DPL;      // lanes per position
  constexpr int NGRP = 32 / LPP;     // positions per warp per pass
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int dl = lane & (LPP - 1), pgi = lane / LPP;
  const Attn at = make_attn(S, A, in);
  if (!at.active) return;  // uniform over the CTA
  const int l = in.layer;
  const float qscale = (1.0f / sqrtf((float)HD)) * 1.4426950408889634f;  // scores in log2 units

  const float* qsrc = act_ptr(S, act, ACT_Q, l) + ((size_t)at.b * S.Hq + (size_t)at.j * G) * HD;
  float4* q4 = reinterpret_cast<float4*>(xbuf);
  stage_vec<SYNC>(S, reinterpret_cast<const float4*>(qsrc), G * HD / 4, c, [&](int i, float4 v) {
    v.x *= qscale;
    v.y *= qscale;
    v.z *= qscale;
    v.w *= qscale;
    q4[i] = v;
  });
  // this launch's positions p0_b..pos_b (split holding p0_b): the keys and values of rows
  // b - n_new + 1 .. b, staged as storage-dtype rows [n][k | v] like a page (the values are
  // already rounded to that dtype, so this is exact)
  uint16_t* knew = reinterpret_cast<uint16_t*>(xbuf + G * HD);
  if (at.has_new) {
    const float* kn0 = act_ptr(S, act, ACT_KVN, l) + (size_t)(at.b - at.n_new + 1) * 2 * S.Hkv * HD + (size_t)at.j * HD;
    for (int t = tid; t < at.n_new * (HD / 2); t += kConsumerThreads) {
      const int r = t / (HD / 2), u = t % (HD / 2);
      const int kv = u / (HD / 4), e = (u % (HD / 4)) * 4;  // HD/4 vectors of k, then of v
      const float* kn = kn0 + (size_t)r * 2 * S.Hkv * HD;
      const float4 v = load_v4<SYNC>(reinterpret_cast<const float4*>(kn + (size_t)kv * S.Hkv * HD + e), S, c);
      uint16_t* dst = knew + (r * 2 + kv) * HD + e;
      dst[0] = Unpack<WT>::round(v.x);
      dst[1] = Unpack<WT>::round(v.y);
      dst[2] = Unpack<WT>::round(v.z);
      dst[3] = Unpack<WT>::round(v.w);
    }
  }
  consumer_sync();
  const bool mark = (A.flags & SF_TRACE) && tid == 0;
  if (mark) c->tmark[0] = globaltimer_ns();
  // q in registers when it fits beside the accumulators, else read (broadcast) from smem
  constexpr bool QREG = G * DPL <= 32;
  constexpr int QG = QREG ? G : 1, QD = QREG ? DPL : 1;
  float q[QG][QD];
  if (QREG) {
#pragma unroll
    for (int g = 0; g < QG; ++g)
#pragma unroll
      for (int i = 0; i < QD; ++i) q[g][i] = xbuf[g * HD + ((i / 8) * LPP + dl) * 8 + (i % 8)];
  }
  const float* qs = xbuf + dl * 8;  // + u * LPP * 8 for chunk u

  float m[G], lsum[G], o[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -CUDART_INF_F;
    lsum[g] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[g][i] = 0.f;
  }

  // One position per LPP-lane group: scores from its key row, online-softmax update,
  // then its value row.  Rows come from a page or, for the new position, from its copy
  // staged above (both in the storage dtype).
  // RC passes of the warp at once (RC positions per lane group): their scores are
  // independent, so they are computed together; one running-max update and one rescale of
  // the accumulators per chunk; then the value rows, each with its own weight.  RC is 4
  // while a block needs at least three more passes, else 1.
  auto chunk = [&](auto rct, int nvalid, const uint16_t* const* krow, const uint16_t* const* vrow) {
    constexpr int RC = decltype(rct)::value;
    float sc[RC][G];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
#pragma unroll
      for (int g = 0; g < G; ++g) sc[r][g] = 0.f;
      if (r < nvalid) {
#pragma unroll
        for (int u = 0; u < DPL / 8; ++u) {
          float kv[8];
          Unpack<WT>::u8(reinterpret_cast<const uint4*>(krow[r])[u * LPP + dl], kv);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float a = sc[r][g];
            if (QREG) {
#pragma unroll
              for (int e = 0; e < 8; ++e) a = fmaf(q[QREG ? g : 0][QREG ? u * 8 + e : 0], kv[e], a);
            } else {
              const float4 q0 = *reinterpret_cast<const float4*>(qs + g * HD + u * LPP * 8);
              const float4 q1 = *reinterpret_cast<const float4*>(qs + g * HD + u * LPP * 8 + 4);
              a = fmaf(q0.x, kv[0], a); a = fmaf(q0.y, kv[1], a); a = fmaf(q0.z, kv[2], a); a = fmaf(q0.w, kv[3], a);
              a = fmaf(q1.x, kv[4], a); a = fmaf(q1.y, kv[5], a); a = fmaf(q1.z, kv[6], a); a = fmaf(q1.w, kv[7], a);
            }
            sc[r][g] = a;
          }
        }
      }
    }
    // full scores within each lane group; invalid rows (beyond the block) at -inf
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = sc[r][g];
#pragma unroll
        for (int o2 = 1; o2 < LPP; o2 <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o2);
        sc[r][g] = r < nvalid ? a : -CUDART_INF_F;
      }
    float p[RC][G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = sc[0][g];
#pragma unroll
      for (int r = 1; r < RC; ++r) mx = fmaxf(mx, sc[r][g]);
#pragma unroll
      for (int o2 = LPP; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float mn = fmaxf(m[g], mx);  // warp-uniform
#pragma unroll
      for (int r = 0; r < RC; ++r) p[r][g] = 0.f;
      if (mn == -CUDART_INF_F) continue;
      if (mn != m[g]) {
        const float corr = exp2f(m[g] - mn);
        lsum[g] *= corr;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[g][i] *= corr;
        m[g] = mn;
      }
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        p[r][g] = r < nvalid ? exp2f(sc[r][g] - mn) : 0.f;
        lsum[g] += p[r][g];
      }
    }
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      if (r < nvalid) {
#pragma unroll
        for (int u = 0; u < DPL / 8; ++u) {
          float vv[8];
          Unpack<WT>::u8(reinterpret_cast<const uint4*>(vrow[r])[u * LPP + dl], vv);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][u * 8 + e] = fmaf(p[r][g], vv[e], o[g][u * 8 + e]);
        }
      }
    }
  };

  // the cached positions a page block at a time; this launch's positions p0_b..pos_b
  // (staged above) are n_new more rows of the last block
  const int nblk = at.nblocks > 0 ? at.nblocks : (at.has_new ? 1 : 0);
  for (int blk = 0; blk < nblk; ++blk) {
    const bool paged = blk < at.nblocks;
    const int np = paged ? min(at.pb, at.n_cached - blk * at.pb) : 0;
    const int nx = np + (blk == nblk - 1 && at.has_new ? at.n_new : 0);
    const uint8_t* kp = nullptr;
    const uint8_t* vp = nullptr;
    if (paged) {
      kp = page_wait(S, c, pages, ring);
      Ring rv = ring;
      if (++rv.slot == S.n_pages) { rv.slot = 0; rv.ph ^= 1u; }
      vp = page_wait(S, c, pages, rv);
    }
    // the block's rows dealt over (warp, lane group), RC passes per chunk: row
    // base + r * (warps x groups) + (warp, group) for r < RC; the bounds are uniform
    constexpr int PASS = kConsumerWarps * NGRP;
    auto run_chunk = [&](auto rct, int base) {
      constexpr int RC = decltype(rct)::value;
      {
        const uint16_t* kr[RC];
        const uint16_t* vr[RC];
        int nvalid = 0;  // rows r < nvalid exist for this lane group (a prefix)
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          const int t = base + r * PASS + warp * NGRP + pgi;
          const bool cached = t < np;
          const size_t off = (size_t)(cached ? t : 0) * HD * 2;
          const int nr = t < np ? 0 : min(t - np, at.n_new - 1);  // staged row (clamped: a valid address)
          kr[r] = cached ? reinterpret_cast<const uint16_t*>(kp + off) : knew + nr * 2 * HD;
          vr[r] = cached ? reinterpret_cast<const uint16_t*>(vp + off) : knew + nr * 2 * HD + HD;
          if (t < nx) nvalid = r + 1;
        }
        chunk(rct, nvalid, kr, vr);
      }
    };
    // chunks of 4 passes while at least 3 remain, then single passes: a chunk's rows past
    // the block still cost their shuffles
    if (nx <= PASS) {
      run_chunk(std::integral_constant<int, 1>{}, 0);
    } else {
      int base = 0;
      for (; nx - base > 2 * PASS; base += 4 * PASS) run_chunk(std::integral_constant<int, 4>{}, base);
      for (; base < nx; base += PASS) run_chunk(std::integral_constant<int, 1>{}, base);
    }
    if (paged) {
      page_release(S, c, ring);  // K page
      page_release(S, c, ring);  // V page
    }
  }
  if (mark) c->tmark[1] = globaltimer_ns();
  // Combine the NGRP position groups of the warp (they share the running max m[g]) with a
  // butterfly reduce-scatter: each round halves the values a lane holds, so the warp
  // shuffles V(1 - 1/NGRP) values instead of V log2(NGRP).  Lane group pgi ends with block
  // bitrev(pgi) of the G*DPL accumulators, reduced over the whole warp.
  constexpr int V = G * DPL;
  constexpr int R = NGRP == 1 ? 0 : (NGRP == 2 ? 1 : (NGRP == 4 ? 2 : (NGRP == 8 ? 3 : 4)));
  static_assert((1 << R) == NGRP && V % NGRP == 0, "reduce-scatter shape");
  float a[V];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < DPL; ++i) a[g * DPL + i] = o[g][i];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int n = V >> r, o2 = LPP << r;
    const bool upper = (lane & o2) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? a[i] : a[i + n / 2];
      const float keep = upper ? a[i + n / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int o2 = LPP; o2 < 32; o2 <<= 1) lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], o2);
  constexpr int RW = HD + kPartExtra;
  {
    constexpr int NH = V / NGRP;  // accumulators a lane holds after the rounds
    const int blk = R == 0 ? 0 : (int)(__brev((unsigned)pgi) >> (32 - R));
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const int v = blk * NH + k, g = v / DPL, i = v % DPL;
      scratch[(warp * G + g) * RW + ((i / 8) * LPP + dl) * 8 + (i % 8)] = a[k];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      scratch[(warp * G + g) * RW + HD] = m[g];
      scratch[(warp * G + g) * RW + HD + 1] = lsum[g];
    }
  }
  consumer_sync();
  attn_combine_warps<HD, G>(S, act, at, l, scratch);
}

// ---------------------------------------------------------------- attention on tensor cores
// The split-KV unit of op_attn (the same partial record) with its two contractions on
// mma.sync m16n8k16.  Warp w takes rows 16w .. 16w+15 of each 128-row pass of a page.
// Scores: the A tile holds head g's scaled query as 16-bit halves, hi in row g and lo in row
// g + 8 (heads g >= G: zeros); B is the 16 keys as columns; head g's score of a key is the
// sum of accumulator rows g and g + 8 -- both in the lane that holds it.  The online softmax
// runs on those accumulators (a lane group of 4 lanes per head, 4 keys per lane).  Values:
// the probabilities' hi/lo halves form the A tile of P V straight from the score
// accumulators' layout (rows g / g + 8 again), B the value rows read transposed by
// ldmatrix, and head g's output is the sum of accumulator rows g and g + 8.  K and V pages
// land as [64-element half][row][128 bytes] with 16-byte chunk c of row r at c ^ (r % 8)
// (the tensor map's 128-byte swizzle), so that ldmatrix's eight row reads of one chunk fall
// in eight bank groups.  The step's new rows sit in a 16-row page of the same layout.
template <typename WT, int SYNC, int HD, int G>
__device__ __noinline__ void op_attn_tc(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c,
                                        uint8_t* pages, float* xbuf, float* scratch, Ring& ring_io, float* act) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  RingCopy ring_copy(ring_io);
  Ring& ring = ring_copy.r;
  static_assert(G <= 8 && (HD == 64 || HD == 128), "tensor-core attention shape");
  constexpr int NKS = HD / 16;          // k-steps of q K^T
  constexpr int NDT = HD / 8;           // 8-column output tiles of P V
  constexpr int MINI = (HD / 64) * 16 * 128;  // bytes of one 16-row page of new rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  const Attn at = make_attn(S, A, in);
  if (!at.active) return;  // uniform over the CTA
  const int l = in.layer;
  const float qscale = (1.0f / sqrtf((float)HD)) * 1.4426950408889634f;  // scores in log2 units

  // the query's A fragments, one 16-byte vector per (k-step, lane), built straight from the
  // QKV op's output (scaled): rows fg (hi) and fg + 8 (lo) of head fg, zeros for fg >= G;
  // the page loop reads them back with one load per k-step
  const float* qsrc = act_ptr(S, act, ACT_Q, l) + ((size_t)at.b * S.Hq + (size_t)at.j * G) * HD;
  uint4* qf = reinterpret_cast<uint4*>(xbuf);
  if (tid < NKS * 32) {
    const int ks = tid >> 5, fg = (tid & 31) >> 2, fc = tid & 3;
    uint32_t f[4] = {0u, 0u, 0u, 0u};
    if (fg < G) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {  // k = 16 ks + 2 fc (+1), then + 8: one float4 holds the pair
        const int k = 16 * ks + 2 * fc + 8 * h2;
        const float4 v = load_v4<SYNC>(reinterpret_cast<const float4*>(qsrc + fg * HD + (k & ~3)), S, c);
        uint16_t h0, l0, h1, l1;
        Mma<WT>::split(((k & 2) ? v.z : v.x) * qscale, h0, l0);
        Mma<WT>::split(((k & 2) ? v.w : v.y) * qscale, h1, l1);
        f[2 * h2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        f[2 * h2 + 1] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
    }
    qf[tid] = make_uint4(f[0], f[1], f[2], f[3]);
  }
  // this launch's new rows (keys and values of positions p0_b..pos_b, rounded to the storage
  // dtype as the cache holds them): rows 0..n_new-1 of a key page and a value page, zeros after
  uint8_t* mini = reinterpret_cast<uint8_t*>(qf + NKS * 32);
  if (at.has_new) {
    const float* kn0 = act_ptr(S, act, ACT_KVN, l) + (size_t)(at.b - at.n_new + 1) * 2 * S.Hkv * HD + (size_t)at.j * HD;
    for (int t = tid; t < 2 * 16 * (HD / 4); t += kConsumerThreads) {
      const int kv = t / (16 * (HD / 4)), u = t - kv * (16 * (HD / 4)), r = u / (HD / 4), e = (u % (HD / 4)) * 4;
      uint2 w = make_uint2(0u, 0u);
      if (r < at.n_new) {
        const float* kn = kn0 + (size_t)r * 2 * S.Hkv * HD + (size_t)kv * S.Hkv * HD + e;
        const float4 v = load_v4<SYNC>(reinterpret_cast<const float4*>(kn), S, c);
        w.x = (uint32_t)Unpack<WT>::round(v.x) | ((uint32_t)Unpack<WT>::round(v.y) << 16);
        w.y = (uint32_t)Unpack<WT>::round(v.z) | ((uint32_t)Unpack<WT>::round(v.w) << 16);
      }
      const int ch = (e & 63) >> 3;
      *reinterpret_cast<uint2*>(mini + kv * MINI + (e >> 6) * 2048 + r * 128 + ((ch ^ (r & 7)) << 4) + (e & 7) * 2) = w;
    }
  }
  consumer_sync();
  const bool mark = (A.flags & SF_TRACE) && tid == 0;
  if (mark) c->tmark[0] = globaltimer_ns();
  uint64_t page_wait_ns = 0;  // journal: time spent waiting for K, V pages to land
  const uint4* qfl = qf + lane;  // this lane's fragment of k-step ks at qfl[32 ks]
  float o[NDT][4];
#pragma unroll
  for (int d = 0; d < NDT; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
  float mrun = -CUDART_INF_F, lrun = 0.f;  // head gq's running max and (this lane's) sum

  // rows [lo, hi) of a page whose halves hold rph rows each, npass passes of 128 rows
  auto block = [&](uint32_t kbase, uint32_t vbase, int rph, int npass, int lo, int hi) {
    const int mi = lane >> 3, ri = lane & 7;  // the matrix and the row this lane addresses
    for (int ps = 0; ps < npass; ++ps) {
      const int r0 = ps * 128 + warp * 16;
      if (r0 + 16 <= lo || r0 >= hi) continue;  // uniform over the warp
      // q K^T: key rows r0.. r0+7 and r0+8.. r0+15 (two column tiles), 16 dims per k-step;
      // even and odd k-steps in separate accumulators (two chains of dependent MMAs per tile)
      float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int row = r0 + ri + ((mi >> 1) << 3);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          const int ch = 2 * ks + (mi & 1);
          uint32_t b[4];
          ldsm_x4(kbase + (uint32_t)((ch >> 3) * rph * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)), b);
          const uint4 qa = qfl[32 * ks];
          float(&d0)[4] = (ks & 1) ? sb[0] : sa[0];
          float(&d1)[4] = (ks & 1) ? sb[1] : sa[1];
          Mma<WT>::run(d0, qa, b[0], b[1]);
          Mma<WT>::run(d1, qa, b[2], b[3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sa[0][e] += sb[0][e];
          sa[1][e] += sb[1][e];
        }
      }
      // online softmax over this lane group's head: 4 keys per lane, then the group's max
      float sc[2][2];
      float bm = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = r0 + 8 * nt + 2 * cq + e;
          const bool ok = gq < G && row >= lo && row < hi;
          sc[nt][e] = ok ? sa[nt][e] + sa[nt][e + 2] : -CUDART_INF_F;
          bm = fmaxf(bm, sc[nt][e]);
        }
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float mn = fmaxf(mrun, bm);
      float p[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      if (mn != -CUDART_INF_F) {
        if (mn != mrun) {
          const float corr = exp2f(mrun - mn);
          lrun *= corr;
#pragma unroll
          for (int d = 0; d < NDT; ++d) {
            o[d][0] *= corr;
            o[d][1] *= corr;
            o[d][2] *= corr;
            o[d][3] *= corr;
          }
          mrun = mn;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            p[nt][e] = exp2f(sc[nt][e] - mn);
            lrun += p[nt][e];
          }
      }
      __syncwarp();
      // P's A fragment: a0 / a2 the hi halves of keys 2cq.. / 8+2cq.., a1 / a3 the lo halves
      uint4 pa;
      {
        uint16_t h[2][2], lw[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) Mma<WT>::split(p[nt][e], h[nt][e], lw[nt][e]);
        pa.x = (uint32_t)h[0][0] | ((uint32_t)h[0][1] << 16);
        pa.y = (uint32_t)lw[0][0] | ((uint32_t)lw[0][1] << 16);
        pa.z = (uint32_t)h[1][0] | ((uint32_t)h[1][1] << 16);
        pa.w = (uint32_t)lw[1][0] | ((uint32_t)lw[1][1] << 16);
      }
      // P V: value rows r0.. r0+7 (k 0..7) and r0+8.. (k 8..15), two 8-column tiles per load
      {
        const int row = r0 + ri + ((mi & 1) << 3);
#pragma unroll
        for (int d2 = 0; d2 < NDT / 2; ++d2) {
          const int ch = 2 * d2 + (mi >> 1);
          uint32_t b[4];
          ldsm_x4_trans(vbase + (uint32_t)((ch >> 3) * rph * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)), b);
          Mma<WT>::run(o[2 * d2], pa, b[0], b[1]);
          Mma<WT>::run(o[2 * d2 + 1], pa, b[2], b[3]);
        }
      }
    }
  };

  for (int blk = 0; blk < at.nblocks; ++blk) {
    int lo;
    (void)attn_box_pos(at, blk, &lo);
    const uint64_t tw = mark ? globaltimer_ns() : 0ull;
    const uint8_t* kp = page_wait(S, c, pages, ring);
    Ring rv = ring;
    if (++rv.slot == S.n_pages) { rv.slot = 0; rv.ph ^= 1u; }
    const uint8_t* vp = page_wait(S, c, pages, rv);
    if (mark) page_wait_ns += globaltimer_ns() - tw;
    block(smem_addr(kp), smem_addr(vp), at.pb, at.pb / 128, lo, at.pb);
    page_release(S, c, ring);  // K page
    page_release(S, c, ring);  // V page
  }
  if (at.has_new) block(smem_addr(mini), smem_addr(mini + MINI), 16, 1, 0, at.n_new);
  if (mark) {
    c->tmark[1] = globaltimer_ns();
    c->tmark[4] = page_wait_ns;
  }
  // this warp's partial: head gq's sum over its lane group, output columns 8d + 2cq (+1)
  lrun += __shfl_xor_sync(0xffffffffu, lrun, 1);
  lrun += __shfl_xor_sync(0xffffffffu, lrun, 2);
  constexpr int RW = HD + kPartExtra;
  if (gq < G) {
    float* dst = scratch + (warp * G + gq) * RW;
#pragma unroll
    for (int d = 0; d < NDT; ++d)
      *reinterpret_cast<float2*>(dst + 8 * d + 2 * cq) = make_float2(o[d][0] + o[d][2], o[d][1] + o[d][3]);
    if (cq == 0) {
      dst[HD] = mrun;
      dst[HD + 1] = lrun;
    }
  }
  consumer_sync();
  attn_combine_warps<HD, G>(S, act, at, l, scratch);
}

// the tensor-core instance's attention unit (one call site): the tensor-core op for units of
// at least half a page (attn_use_mma), else the CUDA-core op, per head size and group
template <typename WT, int SYNC>
__device__ __noinline__ void op_attn_any(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c,
                                         uint8_t* pages, float* xbuf, float* scratch, Ring& ring, float* act) {
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const int G = S.Hq / S.Hkv;
  if (S.attn_mma && attn_use_mma(S, A, in)) {
    if (S.hd == 128 && G == 2)
      op_attn_tc<WT, SYNC, 128, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
    else if (S.hd == 128 && G == 4)
      op_attn_tc<WT, SYNC, 128, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
    else if (S.hd == 128 && G == 1)
      op_attn_tc<WT, SYNC, 128, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
    else if (S.hd == 64 && G == 2)
      op_attn_tc<WT, SYNC, 64, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
    else if (S.hd == 64 && G == 4)
      op_attn_tc<WT, SYNC, 64, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
    else
      op_attn_tc<WT, SYNC, 64, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
  } else if (S.hd == 64 && G == 2)
    op_attn<WT, SYNC, 64, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
  else if (S.hd == 128 && G == 2)
    op_attn<WT, SYNC, 128, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
  else if (S.hd == 128 && G == 4)
    op_attn<WT, SYNC, 128, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
  else if (S.hd == 64 && G == 4)
    op_attn<WT, SYNC, 64, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
  else if (S.hd == 128 && G == 1)
    op_attn<WT, SYNC, 128, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
  else
    op_attn<WT, SYNC, 64, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
}

// log-sum-exp merge of the S split partials of one (sequence, kv head) (§8.2 ATTN_REDUCE).
// The (b, j) block of partials is contiguous and made of 16-byte rows: staged into the x
// buffer with vector loads when it fits (the caller has acquired the partials, or polls
// them), else read from global memory eight splits deep.
template <typename WT, int SYNC, bool TC>
__device__ __noinline__ void op_attn_reduce(const DevState& S_arg, const StepArgs& A_arg, const Instr& in_arg, SmemCtl* c,
                                            float* xbuf, float* scratch, float* act) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  const int tid = threadIdx.x;
  const int b = in.a[0], j = in.a[1], l = in.layer;
  if (b >= A.B) return;  // uniform over the CTA
  const int HD = S.hd, G = S.Hq / S.Hkv, RW = HD + kPartExtra;
  const int NS = active_splits(S, A, b);  // splits s < NS wrote partials this step
  const float* part = act_ptr(S, act, ACT_PART, l) + ((size_t)b * S.Hkv + j) * S.S * G * RW;
  float* out = act_ptr(S, act, ACT_O, l) + (size_t)b * S.Hq * HD + (size_t)j * G * HD;
  // the tensor-core GEMV takes O-proj's input in fragment form as well (columns j G HD + t)
  uint16_t* fo = (TC && S.tc && A.B >= 3) ? reinterpret_cast<uint16_t*>(act_ptr(S, act, ACT_OF, l)) : nullptr;
  const int MT = A.B > 8 ? 2 : 1, col0 = j * G * HD;
  const int n4 = NS * G * RW / 4;
  const bool staged = n4 * 16 <= S.xbuf_bytes;
  if (staged) {
    float4* x4 = reinterpret_cast<float4*>(xbuf);
    stage_vec<SYNC, 8>(S, reinterpret_cast<const float4*>(part), n4, c, [&](int i, const float4& v) { x4[i] = v; });
    consumer_sync();
  }
  // per (head, split) weight exp2(m_s - M) / sum_s' exp2(m_s' - M) l_s', one warp per head;
  // a lane keeps its own splits' entries, so only the CTA barrier orders them for the readers
  const int warp = tid >> 5, lane = tid & 31;
  for (int g = warp; g < G; g += kConsumerWarps) {
    float* wg = scratch + g * NS;
    float M = -CUDART_INF_F;
    for (int s = lane; s < NS; s += 32) {
      const int o = (s * G + g) * RW + HD;
      const float ms = staged ? xbuf[o] : load_act<SYNC>(part + o, S, c);
      wg[s] = ms;
      M = fmaxf(M, ms);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float den = 0.f;
    for (int s = lane; s < NS; s += 32) {
      const int o = (s * G + g) * RW + HD + 1;
      const float w = wg[s] == -CUDART_INF_F ? 0.f : exp2f(wg[s] - M);
      wg[s] = w;
      den = fmaf(w, staged ? xbuf[o] : load_act<SYNC>(part + o, S, c), den);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
    const float inv = 1.0f / den;
    for (int s = lane; s < NS; s += 32) wg[s] *= inv;
  }
  consumer_sync();
  if (staged) {
    for (int t = tid; t < G * HD; t += kConsumerThreads) {
      const int g = t / HD, e = t - g * HD;
      const float* wg = scratch + g * NS;
      const float* pe = xbuf + g * RW + e;
      float r0 = 0.f, r1 = 0.f;
      int s = 0;
#pragma unroll 4
      for (; s + 1 < NS; s += 2) {
        r0 = fmaf(wg[s], pe[s * G * RW], r0);
        r1 = fmaf(wg[s + 1], pe[(s + 1) * G * RW], r1);
      }
      if (s < NS) r0 = fmaf(wg[s], pe[s * G * RW], r0);
      out[t] = r0 + r1;
      if (fo) put_frag<WT>(fo, b, col0 + t, MT, r0 + r1);
    }
    return;
  }
  constexpr int U = 8;  // splits whose partial outputs are in flight together
  for (int t = tid; t < G * HD; t += kConsumerThreads) {
    const int g = t / HD, e = t - g * HD;
    const float* wg = scratch + g * NS;
    float acc = 0.f;
    for (int s0 = 0; s0 < NS; s0 += U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = min(s0 + u, NS - 1);  // clamped: always a valid address
        const float* p = part + (size_t)(s * G + g) * RW + e;
        v[u] = (SYNC == SYNC_COUNTER) ? __ldcg(p) : ld_poll_f32(p);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = s0 + u;
        if (s < NS) {
          float ov = v[u];
          if (SYNC == SYNC_SENTINEL && isnan(ov)) ov = poll_slow(part + (size_t)(s * G + g) * RW + e, S, c);
          acc = fmaf(wg[s], ov, acc);
        }
      }
    }
    out[t] = acc;
    if (fo) put_frag<WT>(fo, b, col0 + t, MT, acc);
  }
}

template <typename WT, bool TC>
__device__ __noinline__ void op_embed(const DevState& S, const StepArgs& A, const Instr& in, float* act) {
  float* h0 = act_ptr(S, act, ACT_H, 0);
  // the tensor-core GEMV (batches of 3..16) takes layer 0's QKV input in fragment form
  uint16_t* fo = (TC && S.tc && A.B >= 3) ? reinterpret_cast<uint16_t*>(act_ptr(S, act, ACT_HF, 0)) : nullptr;
  const int MT = A.B > 8 ? 2 : 1;
  const uint16_t* gn = iptr(in, kP2);
  float ssp[kMaxBatch];
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) ssp[b] = 0.f;
  const bool dev = (A.flags & SF_TOK_FROM_DEVICE) != 0;
  const int e1 = min(in.a[1], A.B * S.d);
  for (int e = in.a[0] + threadIdx.x; e < e1; e += kConsumerThreads) {
    const int b = e / S.d, k = e - b * S.d;
    int tok = dev ? (int)ld_relaxed_u32(reinterpret_cast<const uint32_t*>(&S.ctl->tok[b])) : A.tok[b];
    if (tok < 0 || tok >= S.V) {  // only a failed previous step can leave this behind
      set_err(S, 5u /*MK_ERR_STATE*/, -8, tok);
      tok = 0;
    }
    const float y = Unpack<WT>::one(S.embed[(size_t)tok * S.d + k]);
    h0[(size_t)b * S.d + k] = y;
    if (fo) {
      put_frag<WT>(fo, b, k, MT, y * Unpack<WT>::one(gn[k]));
#pragma unroll
      for (int bb = 0; bb < kMaxBatch; ++bb)
        if (bb == b) ssp[bb] += y * y;
    }
  }
  if (fo) put_ssq_slot<kMaxBatch>(smem_ctl(), ssp, act_ptr(S, act, ACT_SSH, 0));
}

// ---------------------------------------------------------------- self-test opcodes
__device__ void op_test_pages(const DevState& S_arg, const Instr& in_arg, SmemCtl* c, uint8_t* pages, float* scratch,
                              Ring& ring_io) {
  const Instr& in = smem_ctl()->cur[threadIdx.x >> 5];
  const DevState& S = smem_ctl()->S;
  c = smem_ctl();
  pages = smem_pages();
  scratch = smem_scratch(S);
  RingCopy ring_copy(ring_io);
  Ring& ring = ring_copy.r;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long* ws = reinterpret_cast<unsigned long long*>(scratch);
  const int words = S.page_bytes / 8, per_warp = words / kConsumerWarps;
  for (int k = 0; k < in.a[1]; ++k) {
    const uint64_t* pg = reinterpret_cast<const uint64_t*>(page_wait(S, c, pages, ring));
    unsigned long long sum = 0;
    for (int i = lane; i < per_warp; i += 32) sum += pg[warp * per_warp + i];
    page_release(S, c, ring);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) ws[warp] = sum;
    consumer_sync();
    if (tid == 0) {
      unsigned long long t = 0;
      for (int w = 0; w < kConsumerWarps; ++w) t += ws[w];
      S.test_buf[in.a[2] + k] = (int64_t)t;
    }
    consumer_sync();
  }
}

// ---------------------------------------------------------------- compute warps: loop
// Thread 0 takes the next unit its loader claimed from the attention pool (bounded wait).
__device__ __noinline__ bool pool_take(const DevState& S_arg, SmemCtl* c) {
  const DevState& S = smem_ctl()->S;
  c = smem_ctl();
  const int s = c->pool_slot;
  const uint32_t ph = c->pool_ph;
  if (!mbar_try_wait(&c->pool_full[s], ph)) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_wait_hint(&c->pool_full[s], ph, 2000u)) {
      if (c->abort) return false;
      if (globaltimer_ns() - t0 > (uint64_t)S.timeout_ns) {
        set_err(S, 4u, -11, s);
        c->abort = 1;
        return false;
      }
    }
  }
  c->pool_unit = c->pool_fifo[s];
  mbar_arrive(&c->pool_empty[s]);
  if (++c->pool_slot == kPoolSlots) {
    c->pool_slot = 0;
    c->pool_ph ^= 1u;
  }
  return true;
}

template <typename WT, int SYNC, bool MS, bool TC, bool AM>
__device__ void consumer(const DevState& S_arg, const StepArgs& A_arg, SmemCtl* c, uint8_t* pages, float* xbuf,
                         float* scratch) {
  const DevState& S = smem_ctl()->S;
  const StepArgs& A = smem_ctl()->args;
  c = smem_ctl();
  pages = smem_pages();
  xbuf = smem_xbuf(S);
  scratch = smem_scratch(S);
  const int tid = threadIdx.x, cta = blockIdx.x;
  const bool nosync = (A.flags & SF_NO_SYNC) != 0;
  const bool TRACE = (A.flags & SF_TRACE) != 0;
  Ring ring{0, 0u};
  const int end = A.q_start[cta + 1];
  // A multi-step launch runs the queue once per step.  Step st > 0 starts when the step
  // before has published its tokens (its last CTA's last instruction is done): then the
  // arguments advance one position, the token comes from the device, and the buffers that
  // step used are prepared for the step after this one.
  // (the step index lives in shared memory, zeroed in the kernel prologue: nothing extra
  // stays in registers across the op calls of a step)
  for (;;) {
  if (MS && c->ms_step > 0) {
    bool bad = false;
    if (tid == 0 && !wait_seq(&S.ctl->tok_seq, A.step + 1u, -9)) {
      c->abort = 1;
      bad = true;
    }
    if (consumer_sync_or(bad || c->abort)) break;
    if (tid == 0) {
      StepArgs& M = smem_ctl()->args;
      M.step += 1u;
      M.epoch += 1u;
      for (int b = 0; b < M.B; ++b) {
        M.pos[b] += 1;
        M.p0[b] += 1;
      }
      M.flags |= SF_TOK_FROM_DEVICE;
      if (M.tok_hist) M.tok_hist += M.B;
    }
    if (tid < kMaxBatch) c->best[tid] = 0ull;
    consumer_sync();
    if ((A.flags & SF_RESET_ARGMAX) && cta == 0 && tid < kMaxBatch)
      S.argkeys[((A.step + 1u) & 1u) * kMaxBatch + tid] = 0ull;
    if (SYNC == SYNC_SENTINEL && !nosync)
      nan_fill(S.act + (int64_t)((A.step + 1u) & 1u) * S.act_floats, S.act_floats, tid, kConsumerThreads);
  }
  // the step's parity of the activation arena, the batch padded for the GEMV, the GQA
  // group: fixed for a one-step launch; re-read per instruction when steps advance
  const int par0 = (SYNC == SYNC_SENTINEL && !nosync) ? (int)(A.step & 1u) : 0;
  float* act0 = S.act + (int64_t)par0 * S.act_floats;
  const int nb0 = A.B <= 1 ? 1 : A.B <= 2 ? 2 : A.B <= 4 ? 4 : A.B <= 8 ? 8 : 16;
  const int G0 = S.Hq / S.Hkv;
  if (MS) {
    if (tid == 0) {
      c->step_act = act0;
      c->step_nb = nb0;
      c->step_G = G0;
    }
    consumer_sync();
  }
  for (int pc = A.q_start[cta]; pc < end; ++pc) {
    Instr in = load_instr(A.instr + pc);
    if (in.op == OP_END) break;
    if (in.op == OP_ATTN_POOL) {
      // dynamic attention: the next unit this CTA's loader claimed from the layer's pool,
      // run below as an ATTENTION instruction; the loop comes back here until the loader
      // reports the pool empty
      bool bad = false;
      if (tid == 0 && !pool_take(S, c)) bad = true;
      if (consumer_sync_or(bad || c->abort)) break;
      const int u = c->pool_unit;
      if (u < 0) continue;
      in = load_instr(A.instr + in.a[0] + u);
      --pc;
    }
    // a split unit past this step's active count has nothing to compute: skipped without a
    // barrier (the decision is uniform over the CTA); with counters it still signals (its
    // waiters count every unit), except under the fused merge, which counts active splits
    // (with the tensor-core GEMV's batches: the rest of the run as well, see attn_run_skip;
    // batches 1..2 have runs of one or two units, and their instance keeps the simpler loop)
    if (in.op == OP_ATTN && !attn_unit_active(S, A, in)) {
      const int skip = TC ? attn_run_skip(S, A, in) : 0;
      if (SYNC == SYNC_COUNTER && in.a[4] < 0 && !nosync && tid == 0 && in.signal_ctr >= 0)
        red_release_add_u32(&S.counters[in.signal_ctr], 1u + (uint32_t)skip);
      if (TC) pc += skip;
      continue;
    }
    if ((tid & 31) == 0) c->cur[tid >> 5] = in;  // the ops read their warp's shared copy
    if (tid == 0 && in.op != OP_LMHEAD) c->lm_staged = 0;  // any other op may overwrite the x buffer
    __syncwarp();
    uint64_t t_fetch = 0, t_ready = 0;
    if (TRACE) {
      t_fetch = globaltimer_ns();
      if (tid == 0) c->tmark[0] = c->tmark[1] = c->tmark[2] = c->tmark[3] = c->tmark[4] = c->tmark[5] = 0ull;
    }
    // ---- wait for the dependency (counter mode; sentinel mode polls the data itself)
    const bool use_ctr = (SYNC == SYNC_COUNTER || in.op >= OP_T_NOP) && !nosync;
    if (use_ctr && in.wait_ctr >= 0) {
      bool bad = false;
      if (tid == 0 && !wait_counter(S, in.wait_ctr, (A.epoch + 1u) * in.wait_n, pc)) {
        c->abort = 1;
        bad = true;
      }
      if (consumer_sync_or(bad || c->abort)) break;
    }
    if (TRACE) t_ready = globaltimer_ns();
    // ---- execute
    float* act = MS ? c->step_act : act0;
    const int nb = MS ? c->step_nb : nb0;
    const int G = MS ? c->step_G : G0;
    switch (in.op) {
      case OP_EMBED:
        op_embed<WT, TC>(S, A, in, act);
        break;
      case OP_QKV:
      case OP_OPROJ:
      case OP_UPGATE:
      case OP_DOWN:
      case OP_LMHEAD:
        if (TC && nb >= 4) {  // batches of 3..16: tensor cores (every context for max_batch >= 3 is set up for them)
          switch (nb) {
            case 4: op_gemv_tc<WT, SYNC, 4>(S, A, in, c, pages, xbuf, scratch, ring, act); break;
            case 8: op_gemv_tc<WT, SYNC, 8>(S, A, in, c, pages, xbuf, scratch, ring, act); break;
            default: op_gemv_tc<WT, SYNC, 16>(S, A, in, c, pages, xbuf, scratch, ring, act); break;
          }
          break;
        }
        if (nb == 1)
          op_gemv<WT, SYNC, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else
          op_gemv<WT, SYNC, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
        break;
      case OP_ATTN:
        if (AM) {
          op_attn_any<WT, SYNC>(S, A, in, c, pages, xbuf, scratch, ring, act);
        } else if (S.hd == 64 && G == 2)
          op_attn<WT, SYNC, 64, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else if (S.hd == 128 && G == 2)
          op_attn<WT, SYNC, 128, 2>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else if (S.hd == 128 && G == 4)
          op_attn<WT, SYNC, 128, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else if (S.hd == 64 && G == 4)
          op_attn<WT, SYNC, 64, 4>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else if (S.hd == 128 && G == 1)
          op_attn<WT, SYNC, 128, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
        else
          op_attn<WT, SYNC, 64, 1>(S, A, in, c, pages, xbuf, scratch, ring, act);
        break;
      case OP_ATTN_REDUCE:
        op_attn_reduce<WT, SYNC, TC>(S, A, in, c, xbuf, scratch, act);
        break;
      case OP_T_ORDER:
      case OP_T_PRODUCE:
        if (tid == 0) {
          if (in.op == OP_T_ORDER) {
            const int64_t n = S.test_buf[(int64_t)cta * 64];  // this CTA's own count (zeroed by the host)
            S.test_buf[(int64_t)cta * 64 + 1 + n] = in.a[1];
            S.test_buf[(int64_t)cta * 64] = n + 1;
          } else {
            S.test_buf[in.a[0]] = in.a[1];
          }
        }
        break;
      case OP_T_CONSUME:
        if (tid == 0) S.test_buf[in.a[2]] = __ldcg(reinterpret_cast<const long long*>(S.test_buf + in.a[0])) + 1;
        break;
      case OP_T_PAGES:
        op_test_pages(S, in, c, pages, scratch, ring);
        break;
      default:
        break;
    }
    // ---- signal
    if (consumer_sync_or(c->abort)) break;
    bool signal = true;
    if (in.op == OP_ATTN && in.a[4] >= 0) {
      // fused merge: count this split's arrival (acq_rel: publishes this CTA's partial,
      // and for the last arriver makes every other split's partial visible); the CTA
      // that brings the count to the step's active split count merges the splits, sets
      // the count back to zero for the next step (ordered before the step's end by this
      // CTA's later releases), then signals the O-proj counter
      bool last = false;
      if (tid == 0) {
        if (TRACE) c->tmark[2] = globaltimer_ns();
        const uint32_t ns = (uint32_t)active_splits(S, A, in.a[0]);
        const uint32_t old = atom_acq_rel_add_u32(&S.counters[in.a[4]], 1u);
        last = old + 1u == ns;
        if (last) st_relaxed_u32(&S.counters[in.a[4]], 0u);
      }
      if (consumer_sync_or(last)) {
        op_attn_reduce<WT, SYNC, TC>(S, A, in, c, xbuf, scratch, act);
        if (consumer_sync_or(c->abort)) break;
        if (TRACE && tid == 0) c->tmark[3] = globaltimer_ns();
      } else {
        signal = false;
      }
    }
    if (in.op == OP_LMHEAD && (in.flags & F_LAST_LM)) {
      // this CTA's share of the vocabulary is done: publish its best key, then the last
      // CTA to finish turns the winning keys into tokens
      const uint32_t kp = A.step & 1u;
      if (tid < A.B) atomicMax(&S.argkeys[kp * kMaxBatch + tid], c->best[tid]);
      consumer_sync();
      if (tid == 0) {
        const uint32_t n_lm = (uint32_t)in.a[2];
        const uint32_t old = atom_acq_rel_add_u32(&S.counters[in.signal_ctr], 1u);
        if (old + 1u == (A.epoch + 1u) * n_lm) {
          for (int b = 0; b < A.B; ++b) {
            const uint64_t key = ld_relaxed_u64(&S.argkeys[kp * kMaxBatch + b]);
            const int32_t tok = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
            S.ctl->tok[b] = tok;
            if (A.tok_hist) A.tok_hist[b] = tok;
            if (A.mail_seq) S.mail->tok[b] = tok;
          }
          if (A.mail_seq) {  // the host thread waits on this word instead of copying Ctl back
            S.mail->err = ld_relaxed_u32(&S.ctl->err.code);
            S.mail->nan_seen = ld_relaxed_u32(&S.ctl->nan_seen);
            st_release_sys_u32(&S.mail->seq, A.mail_seq);
          }
          if (MS) st_release_u32(&S.ctl->tok_seq, A.step + 1u);  // after the tokens: the next step waits on it
        }
      }
    } else if (tid == 0 && use_ctr && signal && in.signal_ctr >= 0) {
      red_release_add_u32(&S.counters[in.signal_ctr], 1u);
    }
    if (TRACE && tid == 0) {
      const uint64_t t_end = globaltimer_ns();
      const uint32_t idx = atomicAdd(&S.ctl->trace_n, 1u);
      if ((int)idx < S.trace_cap) {
        TraceRec rec;
        rec.cta = cta;
        rec.pc = pc;
        rec.op = in.op;
        rec.layer = in.layer;
        rec.t_fetch = t_fetch;
        rec.t_ready = t_ready;
        for (int k = 0; k < 6; ++k) rec.t_mark[k] = c->tmark[k];
        rec.t_end = t_end;
        S.trace[idx] = rec;
      }
    }
  }
  if (!MS) break;
  if (consumer_sync_or(c->abort)) break;
  if (tid == 0) c->ms_step += 1;
  consumer_sync();
  if (c->ms_step >= A.n_steps) break;
  }  // steps
}

}  // namespace

// ---------------------------------------------------------------- the kernel
// WT weight/KV dtype, SYNC counter or sentinel dependencies, MS several steps per launch,
// TC with the tensor-core GEMV (geometries for 3..16 rows), AM with the tensor-core
// attention.  Three variants are built: both (batches of 3 and more), AM alone (batches of
// 1..2 with a long KV capacity) and neither (short batch-1..2 contexts): each op's code
// that a context never runs stays out of its instance, whose instruction footprint and
// register allocation measured faster at batch 1.
template <typename WT, int SYNC, bool MS, bool TC, bool AM>
__global__ void __launch_bounds__(kThreads, 1) mk_step_kernel(const __grid_constant__ DevState S,
                                                              const __grid_constant__ StepArgs A) {
  SmemCtl* c = smem_ctl();
  const int tid = threadIdx.x;
  // programmatic dependent launch: let the next grid be scheduled as soon as SMs free up
  if (A.flags & SF_PDL) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the state and the step's arguments into the control block (shared-space reads from here on)
  {
    constexpr int ws = (int)(sizeof(DevState) / 4), wa = (int)(sizeof(StepArgs) / 4);
    const uint32_t* fs = reinterpret_cast<const uint32_t*>(&S);
    const uint32_t* fa = reinterpret_cast<const uint32_t*>(A.dyn != nullptr ? A.dyn : &A);
    for (int i = tid; i < ws; i += kThreads) reinterpret_cast<uint32_t*>(&c->S)[i] = fs[i];
    for (int i = tid; i < wa; i += kThreads) reinterpret_cast<uint32_t*>(&c->args)[i] = fa[i];
    __syncthreads();
    if (tid == 0 && A.dyn != nullptr) {  // graph launches: their own queues and flags
      c->args.instr = A.instr;
      c->args.q_start = A.q_start;
      c->args.flags |= A.flags;
      c->args.dyn = nullptr;
    }
    if (MS) {
      __syncthreads();
      if (tid == 0) c->largs = c->args;
    }
  }
  uint8_t* pages = smem_pages();
  float* xbuf = smem_xbuf(S);
  float* scratch = smem_scratch(S);
  // the tensor-core pages are 128-byte swizzled copies, whose destination must sit on a
  // 1024-byte boundary: refuse to run (an error, not a faulting copy) if it does not
  if (((TC && S.tc) || (AM && S.attn_mma)) && (smem_addr(pages) & 1023u)) {
    if (tid == 0 && blockIdx.x == 0) set_err(S, 5u /*MK_ERR_STATE*/, -11, (int)(smem_addr(pages) & 1023u));
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < S.n_pages; ++i) {
      mbar_init(&c->full[i], 1);
      mbar_init(&c->empty[i], kConsumerWarps);
      c->last_issue_phase[i] = -1;
    }
    for (int i = 0; i < kPoolSlots; ++i) {
      mbar_init(&c->pool_full[i], 1);
      mbar_init(&c->pool_empty[i], 1);
    }
    c->pool_slot = 0;
    c->pool_ph = 0;
    c->lm_staged = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->xfull[i], 1);
      c->xph[i] = 0;
    }
    c->abort = 0;
    c->ms_step = 0;
    mbar_fence_init();
  }
  if (tid < kMaxBatch) c->best[tid] = 0ull;
  __syncthreads();
  const StepArgs& AA = c->args;
  // per-step housekeeping: the other parity's argmax keys (and, with NaN sentinels, the
  // other parity's activations) are reset for the next step; nothing reads them now
  if ((AA.flags & SF_RESET_ARGMAX) && blockIdx.x == 0 && tid < kMaxBatch)
    S.argkeys[((AA.step + 1u) & 1u) * kMaxBatch + tid] = 0ull;
  if (SYNC == SYNC_SENTINEL && !(AA.flags & SF_NO_SYNC))
    nan_fill(S.act + (int64_t)((AA.step + 1u) & 1u) * S.act_floats, S.act_floats, tid, kThreads);
  __syncthreads();
  if (tid >= kConsumerThreads) {  // the loader streams weights without waiting for the previous grid
    const int w = tid >> 5;
    if (w == kLoaderWarp && (tid & 31) == 0) producer<MS, TC, AM>(S, AA, c, pages);
    return;
  }
  if (AA.flags & SF_PDL) asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous grid's outputs
  consumer<WT, SYNC, MS, TC, AM>(S, AA, c, pages, xbuf, scratch);
  if (c->abort && tid == 0 && !global_err(S)) set_err(S, 4u, -7, -1);
}

}  // namespace mk
