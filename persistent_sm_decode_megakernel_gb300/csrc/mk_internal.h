// Internal layout shared by the host runtime and the device code (plain old data only).
//
// Instruction format follows "8 · Écrire son megakernel", §8.2 (opcode, counter to wait,
// expected value, counter to signal, integer arguments): here the expected value is the
// number of signals the counter receives per decode step, and the device compares
// against (epoch + 1) * that number, so counters never need resetting between steps.
#pragma once
#include <stdint.h>
#include <vector_types.h>  // float2

namespace mk {

constexpr int kMaxBatch = 16;
constexpr int kConsumerWarps = 8;                 // compute warps per CTA
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + the loader (TMA) warp
constexpr int kLoaderWarp = kConsumerWarps;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kMaxPages = 16;

enum Op : uint8_t {
  OP_END = 0,
  OP_EMBED = 1,        // h0 = E[tok] (fp32)
  OP_QKV = 2,          // RMSNorm + q/k/v rows + RoPE; k,v into the cache   (§8.2 RMSNORM_QKV_ROPE)
  OP_ATTN = 3,         // split-KV partial attention                       (§8.2 ATTENTION)
  OP_ATTN_REDUCE = 4,  // log-sum-exp merge of the splits                  (§8.2 ATTN_REDUCE)
  OP_OPROJ = 5,        // h_mid = h + W_o o                                (§8.2 O_PROJ)
  OP_UPGATE = 6,       // RMSNorm + a = silu(W_g x) * (W_u x)              (§8.2 MLP_UP_GATE)
  OP_DOWN = 7,         // h_out = h_mid + W_d a                            (§8.2 MLP_DOWN)
  OP_LMHEAD = 8,       // final RMSNorm + logits + argmax                  (§8.2 LM_HEAD)
  OP_ATTN_POOL = 9,    // claim ATTENTION units of a layer from a shared pool until it is empty
  // build-ladder self-test opcodes (§8.6 steps 1-4)
  OP_T_NOP = 16,
  OP_T_ORDER = 17,
  OP_T_PRODUCE = 18,
  OP_T_CONSUME = 19,
  OP_T_PAGES = 20,
};

constexpr int kNumPhaseOps = 8;  // EMBED..LMHEAD, for the multi-launch phase tables

enum : uint8_t {
  F_LAST_LM = 1,
  F_MERGE_IN = 2,  // OPROJ: merge the KV-split partials while staging the input
};

// where a schedule merges the KV-split partials
enum MergeMode { MERGE_OP = 0, MERGE_LAST_ARRIVER = 1, MERGE_IN_OPROJ = 2 };

// 64-byte instruction
struct Instr {
  uint8_t op;
  uint8_t flags;
  uint16_t layer;
  int32_t wait_ctr;     // -1: none
  uint32_t wait_n;      // signals per step on wait_ctr
  int32_t signal_ctr;   // -1: none
  int32_t a[12];        // op arguments (see the builder)
};
static_assert(sizeof(Instr) == 64, "instruction is 64 bytes");

// Argument layout (the host writes absolute device pointers into the instruction so that
// neither role has to chase per-layer pointer tables on the critical path):
//   EMBED   a0 e0, a1 e1 (flattened [B, d] range), p2 layer 0's attention gain
//   QKV     a0 matrix (0 q, 1 k, 2 v), a1 head, a2 first pair i0, a3 pairs n,
//           p2 gain, p3 cache of this layer (k or v), p4 rows i0.., p5 rows hd/2+i0..
//   ATTN    a0 b, a1 kv head j, a2 split s, a3 splits S, a4 arrival counter (-1: the
//           merge is a separate ATTN_REDUCE), a5 units of the same layer that follow in
//           this queue (split order), p4 keys of (b, j) at t = 0, p5 values
//   REDUCE  a0 b, a1 j
//   OPROJ / DOWN   a0 row0, a1 rows, p4 first row (OPROJ with F_MERGE_IN: its input is
//           merged from the split partials while it is staged), p2 the RMSNorm gain of the
//           output's next consumer (OPROJ: the MLP gain; DOWN: the next layer's attention
//           gain, or the final gain after the last layer)
//   UPGATE  a0 row0, a1 rows, p2 gain, p4 gate rows, p5 up rows
//   LMHEAD  a0 row0, a1 rows, a2 CTAs with LM rows, p2 final gain, p4 first row
//   POOL    a0 index of the layer's first ATTENTION unit in the instruction array (the pools
//           follow the queues), a1 units, a2 claim counter, a3 CTAs (a step claims a1 + a3
//           times: every CTA's last claim comes back empty)
// With the tensor-core GEMV (batches of 3..16), p4 / p5 of the GEMV ops hold the tensor maps
// of the row segments instead of the row pointers.
// pK = the 64-bit value in a[2K], a[2K+1]
constexpr int kP2 = 4, kP3 = 6, kP4 = 8, kP5 = 10;
inline void set_ptr(Instr& in, int at, const void* p) {
  const uint64_t v = reinterpret_cast<uint64_t>(p);
  in.a[at] = (int32_t)(uint32_t)(v & 0xFFFFFFFFu);
  in.a[at + 1] = (int32_t)(uint32_t)(v >> 32);
}

struct ErrWord {
  uint32_t code;        // mk_status, 0 = none
  int32_t cta;
  int32_t pc;
  int32_t ctr;
};

// small block read back by the host after every step (one device-to-host copy)
struct Ctl {
  ErrWord err;
  int32_t tok[kMaxBatch];       // greedy token of the last completed step (device feed)
  uint32_t trace_n;
  uint32_t nan_seen;
  uint32_t tok_seq;             // step number + 1 of the last step whose tokens are in tok
  uint32_t pad;
};

// Mapped host memory the last LM-head CTA fills for a host-token step (mk_decode_step
// without logits): the tokens, the sticky error code and the NaN flag, then seq with a
// system-scope release, so that the host thread waiting on seq needs no copy or sync.
struct HostMail {
  uint32_t seq;
  uint32_t err;
  uint32_t nan_seen;
  uint32_t pad;
  int32_t tok[kMaxBatch];
};

struct TraceRec {
  int32_t cta, pc, op, layer;
  uint64_t t_fetch, t_ready, t_mark[6], t_end;
};

// fp32 activations [rows][width] per layer; with the tensor-core GEMV also the inputs of
// its ops in fragment form (ACT_HF: RMSNorm gain x h for the next QKV or the LM head,
// ACT_HMF: gain x h_mid for UP/GATE, ACT_AF: a for DOWN, ACT_OF: o for O-proj), written by
// their producers as
// 16-bit hi/lo halves in the order the mma fragments take them (see frag_index), and the
// sums of squares of h and h_mid for the RMSNorms, one slot of kMaxBatch floats per
// producing CTA (ACT_SSH, ACT_SSM: [kMaxSsqSlots][kMaxBatch])
enum ActKind {
  ACT_H = 0, ACT_HMID, ACT_Q, ACT_KVN, ACT_PART, ACT_O, ACT_A, ACT_HF, ACT_HMF, ACT_AF, ACT_OF, ACT_SSH, ACT_SSM,
  ACT_NUM
};
constexpr int kMaxSsqSlots = 256;  // the tensor-core GEMV runs on at most this many CTAs

struct DevState {
  // model
  int L, d, Hq, Hkv, hd, F, V, dtype, max_batch, max_ctx, S;
  float eps;
  // slice widths of the row-major GEMVs (elements), one per weight family
  int ws_qkv, ws_o, ws_up, ws_down, ws_lm;
  // weights; per-layer device arrays of device pointers
  const uint16_t* embed;
  const uint16_t* final_norm;
  const uint16_t* lm_head;
  const uint16_t* const* attn_norm;
  const uint16_t* const* wq;
  const uint16_t* const* wk;
  const uint16_t* const* wv;
  const uint16_t* const* wo;
  const uint16_t* const* mlp_norm;
  const uint16_t* const* w_gate;
  const uint16_t* const* w_up;
  const uint16_t* const* w_down;
  uint16_t* const* kcache;
  uint16_t* const* vcache;
  const float2* rope;          // [max_ctx][hd/2] (cos, sin), computed in double on the host
  int rope_by_seq;             // 1: rope holds one row per sequence (row b = position pos[b])
  // activations: two parity sets of act_floats each (sentinel mode alternates them)
  float* act;
  int64_t act_floats;
  int64_t act_off[ACT_NUM];    // offset of layer 0 of each kind
  int64_t act_stride[ACT_NUM]; // per-layer stride of each kind
  unsigned long long* argkeys; // [2][kMaxBatch]
  uint32_t* counters;
  int n_counters;
  Ctl* ctl;
  HostMail* mail;              // device address of the context's mapped host mailbox
  TraceRec* trace;
  int trace_cap;
  // execution
  int n_cta;
  int page_bytes, n_pages;
  int page_stride;             // bytes between ring slots (>= page_bytes)
  int tc;                      // batches of 3..16 use the tensor-core GEMV
  int attn_mma;                // split-KV units of at least half a page use tensor cores
  int xbuf_bytes, scratch_bytes;
  int smem_bytes;              // dynamic shared memory of a launch with this state (host use)
  int sync_mode;
  int64_t timeout_ns;
  int backoff_max_ns;
  int split_min_positions;     // a KV split of a step covers at least this many positions
  int inflight_pages;          // loader: page copies in flight at most (0: up to the pool size)
  // self-test buffers
  int64_t* test_buf;
  int64_t test_len;
};

enum StepFlags : int {
  SF_TOK_FROM_DEVICE = 1,  // embed the token chosen by the previous step (device feed)
  SF_NO_SYNC = 2,          // multi-launch: stream order replaces waits and signals
  SF_TRACE = 4,
  SF_RESET_ARGMAX = 8,     // this launch resets the other parity's argmax keys
  SF_PDL = 16,             // a programmatic dependent launch: compute warps wait for the
                           // previous grid; the loader streams weights before that
};

struct StepArgs {
  const Instr* instr;
  const int32_t* q_start;      // [n_cta + 1] queue offsets of this launch
  uint32_t epoch;              // counter epoch of this schedule (targets = (epoch+1) * n)
  uint32_t step;               // global step number (parity of argmax keys / sentinel sets)
  int B;
  int flags;
  int32_t tok[kMaxBatch];
  int32_t pos[kMaxBatch];
  // Row b of the step is position pos[b] of cache sequence seq[b]; positions below p0[b]
  // are in the cache from earlier launches, positions p0[b]..pos[b] are this launch's rows
  // b - (pos[b] - p0[b]) .. b (a prompt chunk: consecutive rows, consecutive positions).
  // A decode step has seq[b] = b and p0[b] = pos[b].
  int32_t seq[kMaxBatch];
  int32_t p0[kMaxBatch];
  float* logits;               // [B][V] or null
  int32_t* tok_hist;           // device [B] copy of this step's tokens, or null
  int n_steps;                 // greedy steps this launch runs back to back (0 or 1: one)
  uint32_t mail_seq;           // non-zero: post the tokens to the host mailbox with this seq
  // non-null: the per-step fields (epoch .. tok_hist; flags OR-ed) are read from this device
  // copy at kernel start -- the launches of a CUDA graph keep fixed parameters
  const StepArgs* dyn;
};

// Tensor-core GEMV (batches of 3..16): a page holds kTcRows weight rows of kTcKw columns
// (one window of the input), landed by one tensor-map copy as kTcKw / 64 column chunks of
// [kTcRows rows][128 bytes] with the 128-byte swizzle (16-byte granule g of row r stored at
// g ^ (r % 8)), so that the 8 rows an mma fragment reads sit in different banks.
constexpr int kTcKw = 1024;
constexpr int kTcRows = 16;
constexpr int kTcChunkCols = 64;                          // columns per 128-byte chunk row
constexpr int kTcChunkBytes = kTcRows * 128;              // one column chunk of a page
constexpr int kTcPageBytes = kTcRows * kTcKw * 2;         // 32768
constexpr int kTcPartialFloats = 2 * kConsumerWarps * kTcRows * kMaxBatch;  // double-buffered warp partials

// above this many positions per KV split a step uses all of the schedule's splits
constexpr int kSplitLongPositions = 2048;

// a split's partial attention record per head: hd weighted value sums, the running max,
// the exp-sum, two pad floats (16-byte rows, so records move as float4)
constexpr int kPartExtra = 4;
constexpr int kTmapBytes = 128;  // one tensor map (CUtensorMap) in device memory
constexpr int kKvInflight = 4;    // page copies in flight at least, for the tensor-core attention's K / V boxes

// shared-memory layout sizes (bytes)
constexpr int kCtlSmem = 4096;   // barriers, flags, small broadcast values

}  // namespace mk
