/*
 * mk.h -- C ABI of the persistent single-launch decode megakernel for GB300 (sm_103a).
 *
 * One decode step of a Llama-style decoder runs as ONE launch of a persistent kernel:
 * one CTA per SM (exactly one wave, "8 · Écrire son megakernel", §8.3), each CTA walking
 * its own instruction queue (§8.2: RMSNORM_QKV_ROPE, ATTENTION, ATTN_REDUCE, O_PROJ,
 * MLP_UP_GATE, MLP_DOWN, LM_HEAD), ops gated by dependency counters (§8.5) or by NaN
 * sentinels ("7 · AMD et le monokernel", §7.3), weights streamed into a shared-memory page
 * pool by TMA bulk copies from a producer warp so the HBM stream never stops (§7.5, §8.4).
 *
 * Conventions for every function below
 *   - Return value: mk_status; MK_OK (0) on success.  No C++ exception crosses the ABI.
 *     The text of the last failure on the calling thread is returned by mk_last_error().
 *   - "device" pointers are CUDA device addresses on the device that was current when
 *     mk_create was called; "host" pointers are ordinary CPU memory.
 *   - Ownership: weights, KV cache and optional logits buffers belong to the caller, who
 *     keeps them alive (and unmodified, for weights) until mk_destroy.  The context owns
 *     its instruction queues, counters, activation buffers and trace buffer.
 *   - All device work is enqueued on the stream given to mk_create.  A context is not
 *     thread-safe: one host thread at a time.
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MK_OK = 0,
  MK_ERR_INVALID = 1,    /* bad argument, descriptor, pointer alignment or schedule      */
  MK_ERR_OCCUPANCY = 2,  /* fewer than one resident CTA per SM (§8.3: would deadlock)    */
  MK_ERR_CUDA = 3,       /* a CUDA runtime call failed                                   */
  MK_ERR_TIMEOUT = 4,    /* a device-side wait ran past its limit; the step was abandoned */
  MK_ERR_STATE = 5,      /* context unusable until mk_reset (after a timeout)            */
  MK_ERR_NAN = 6         /* a logit was NaN; the returned token is meaningless           */
} mk_status;

typedef enum { MK_F16 = 0, MK_BF16 = 1 } mk_dtype;
typedef enum { MK_SYNC_COUNTER = 0, MK_SYNC_SENTINEL = 1 } mk_sync_mode;
/* MK_EXEC_GRAPH: the multi-launch control captured once per batch size into a CUDA graph
 * whose launches are programmatic dependent launches (each grid's loader streams its
 * weights while the previous grid drains; its compute warps wait for that grid), with the
 * per-step arguments in device memory. */
typedef enum { MK_EXEC_PERSISTENT = 0, MK_EXEC_MULTILAUNCH = 1, MK_EXEC_GRAPH = 2 } mk_exec_mode;

typedef struct mk_ctx mk_ctx;

/* Shape of the decoder (the pages never define the layer; see the reading in the oracle):
 * RMSNorm(eps) -> q,k,v projections -> rotate-half RoPE(theta) -> causal GQA attention
 * (query head i reads kv head i / (n_heads / n_kv_heads)) -> O projection + residual ->
 * RMSNorm -> SwiGLU MLP + residual; final RMSNorm; untied LM head; greedy argmax. */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  int dtype;              /* mk_dtype of weights AND KV cache                            */
  float rms_eps, rope_theta;
  int max_batch;          /* 1..16 sequences per step; from 3 on, steps of 3..16 sequences
                             run the tensor-core GEMV (mma.sync, weights landed by tensor-map
                             copies), which needs d_model, ffn_dim and n_heads*head_dim to be
                             multiples of 64                                              */
  int max_ctx;            /* KV-cache capacity in positions, at most 4194304 (2^22); from
                             8192 on, batch-1..2 contexts run the tensor-core attention
                             (mk_options.attn_tensor_cores)                               */
} mk_model_desc;

/* Weights: device pointers, row-major, nn.Linear convention [out, in], 16-byte aligned.
 * Model-level: embed [vocab, d], final_norm [d], lm_head [vocab, d].
 * Per layer (host arrays of n_layers device pointers): attn_norm [d], wq [n_heads*hd, d],
 * wk, wv [n_kv_heads*hd, d], wo [d, n_heads*hd], mlp_norm [d], w_gate, w_up [ffn, d],
 * w_down [d, ffn].  The host arrays are read during mk_create only. */
typedef struct {
  const void *embed, *final_norm, *lm_head;
  const void *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
  const void *const *mlp_norm, *const *w_gate, *const *w_up, *const *w_down;
} mk_weights;

/* KV cache: host arrays of n_layers device pointers, each [max_batch, n_kv_heads,
 * max_ctx, head_dim] in the model dtype.  Position t of sequence b, kv head j, lives at
 * ((b * n_kv_heads + j) * max_ctx + t) * head_dim.  The kernel writes the new token's
 * rotated key and its value at the step's position and reads positions below it. */
typedef struct {
  void *const *k_cache;
  void *const *v_cache;
} mk_kv;

/* Options; a zero-initialised struct selects the defaults. */
typedef struct {
  int sync_mode;          /* mk_sync_mode: counters (§8.5) or NaN sentinels (§7.3).
                             Measured on the 2b model: sentinels are faster at batches 1..2,
                             counters from batch 4 on (their dependency wait lets the
                             tensor-core GEMV's inputs land by one bulk copy per op)       */
  int exec_mode;          /* mk_exec_mode: one persistent launch, or the multi-launch control */
  int page_bytes;         /* shared-memory page size (default 32768; power of two, 4K..32K) */
  int n_pages;            /* pages in the pool (default: as many as fit)                  */
  int kv_splits;          /* split-KV partitions per (sequence, kv head); 0 = one wave's worth */
  int trace;              /* 1: record the per-instruction journal (§8.7)                  */
  double wait_timeout_s;  /* limit of every device-side wait (default 2.0 s)              */
  int backoff_max_ns;     /* cap of the exponential __nanosleep backoff (§8.5; default 256) */
  int max_ctas;           /* test hook: use at most this many CTAs (0 = one per SM)        */
  int fault_drop_signal;  /* test hook: k > 0 removes the k-th counter signal from the
                             schedule and skips the host-side validator, so that the
                             device wait must time out (fault injection on the host)     */
  int split_min_positions; /* a step uses as many KV splits (up to kv_splits) as give each
                              at least this many positions (0: default 16)               */
  int attn_merge;         /* where the KV-split partials are merged (§8.2 ATTN_REDUCE):
                             0 auto, 1 a separate step (the ATTN_REDUCE op with sentinels,
                             the last-arriving split with counters), 2 inside the O-proj
                             input staging of every O-proj unit (no extra dependency hop;
                             auto picks it when the partials of a step are small), 3 the
                             last-arriving split (an atomic arrival count) in either
                             synchronisation mode                                        */
  int inflight_pages;     /* at most this many page copies of a CTA in flight at once
                             (0: default 2; < 0: the pool size).  Landed pages still
                             fill the whole pool; fewer copies queued in the memory
                             system shorten the waits of the loads and stores that
                             carry the dependencies between ops                          */
  int attn_pool;          /* 1: dynamic work queue of the split-KV attention units ("8 ·
                             Écrire son megakernel", §8.8, dynamic queue): each layer's
                             units sit in a shared pool and every CTA's loader claims them
                             one at a time (an atomic claim counter) as its ring frees,
                             instead of a fixed share dealt to its queue; persistent
                             control only (0: fixed shares, the default)                 */
  int attn_tensor_cores;  /* tensor-core attention: a split-KV unit of at least half a page
                             of cached positions (64 at head_dim 128, 128 at 64) runs q K^T
                             and P V on mma.sync (q and P as hi/lo 16-bit halves, fp32
                             accumulators), its K / V pages landed by tensor-map copies;
                             needs 32 KB pages.  0 (default): in contexts of max_batch >= 3
                             and in those of max_ctx >= 8192 (a batch-1..2 context then
                             runs the kernel variant with this code, which measured ~3.7 %
                             slower at short positions than the one without); 1: in every
                             context; -1: never (CUDA cores only)                         */
} mk_options;

typedef struct {
  int n_sm;               /* multiprocessors on the device                                 */
  int blocks_per_sm;      /* cudaOccupancyMaxActiveBlocksPerMultiprocessor result          */
  int n_ctas;             /* grid size = one wave                                          */
  int threads_per_cta;
  int smem_bytes;         /* dynamic shared memory per CTA                                 */
  int page_bytes, n_pages;
  int kv_splits;
  int n_instructions;     /* total over all queues                                         */
  int n_counters;
  int launches_per_step;  /* 1 for the persistent kernel, ~6 per layer + 2 for multi-launch */
  long long weight_bytes_per_step;  /* streamed weight bytes of one decode step            */
  int kernel_variant;     /* the step kernel's variant: 0 without tensor-core code, 1 with
                             the tensor-core attention, 2 with the tensor-core GEMV and
                             attention (max_batch >= 3)                                  */
} mk_info_t;

/* One journal record per executed instruction (§8.7), times from %globaltimer (ns). */
typedef struct {
  int32_t cta, pc, op, layer;
  uint64_t t_fetch;       /* instruction fetched                                           */
  uint64_t t_ready;       /* dependency satisfied                                          */
  uint64_t t_mark[6];     /* op-internal marks, 0 when unused.  GEMV: [0] inputs staged,
                             [1] last weight page consumed, [2] and [4] DURATIONS: ns compute
                             warp 0 spent waiting for pages to land, and from each page's
                             arrival to its release, [3] outputs written.  ATTENTION: [0] q
                             staged, [1] KV pages consumed, [2] split partial written,
                             [3] merge done.  GEMV [5]: SM clock cycles compute thread 0
                             spent in the epilogue                                       */
  uint64_t t_end;         /* outputs written (before the signal)                           */
} mk_trace_rec;

/* Build the context: validates the descriptor and pointers, sizes the persistent grid
 * (cudaFuncSetAttribute + cudaOccupancyMaxActiveBlocksPerMultiprocessor, §8.3; refuses
 * with MK_ERR_OCCUPANCY when fewer than one CTA fits), builds the per-CTA instruction
 * queues and counter wiring, checks them with the static validator (deadlock freedom,
 * every read ordered after its writer, every output written exactly once), uploads
 * them, and precomputes the RoPE table.  `stream` is a cudaStream_t (NULL = legacy). */
mk_status mk_create(const mk_model_desc *desc, const mk_weights *weights, const mk_kv *kv,
                    const mk_options *opts, void *stream, mk_ctx **out);

/* Prompt pass ("7 · AMD et le monokernel", §7.1: the monokernel runs prefill, decode and
 * sampling without leaving the persistent kernel).  tokens host [B, P] row-major at
 * positions 0..P-1 of each sequence.  Fills KV positions 0..P-1 and returns the greedy
 * next token of each sequence in next_tok (host [B]); logits (device [B, vocab] fp32, or
 * NULL) receives the last position's logits.  Runs the decode step once per position
 * (teacher forcing).  Synchronous; MK_ERR_INVALID for a bad argument (nothing enqueued),
 * a device error as for mk_decode_step. */
mk_status mk_prefill(mk_ctx *ctx, const int32_t *tokens, int B, int P,
                     int32_t *next_tok, float *logits);

/* The hot path: one decode step, ONE kernel launch ("8 · Écrire son megakernel", §8.2: every
 * CTA walks its instruction queue -- fetch, wait for the dependency, execute, signal; §8.3:
 * the grid is one wave, sized by the occupancy query).  in_tok host [B] sits at position
 * pos host [B] (the cache holds 0..pos[b]-1); out_tok host [B] receives the argmax
 * token (lowest index among ties); logits device [B, vocab] fp32 or NULL.  Returns once
 * out_tok holds the tokens: with logits NULL (persistent control) the last LM-head CTA
 * posts them to a mapped host mailbox and the calling thread waits on that word (no copy,
 * no stream synchronisation; the kernel's last instructions may still be finishing, and
 * the next call queues behind them); otherwise, or after a device error, through one
 * small device-to-host copy and a stream synchronisation. */
mk_status mk_decode_step(mk_ctx *ctx, const int32_t *in_tok, const int32_t *pos, int B,
                         int32_t *out_tok, float *logits);

/* n_steps greedy decode steps without host round trips: step s embeds the token chosen
 * by step s-1 on the device.  With persistent control (MK_EXEC_PERSISTENT) all n_steps
 * run in ONE launch: the kernel walks its queues once per step, each step starting when
 * the step before has published its tokens (every CTA waits on that word; the loader
 * streams the next step's weights meanwhile and waits only before KV-cache blocks).  The
 * other controls enqueue one step (or one graph) after another.  in_tok host [B] at
 * positions pos0 host [B], or in_tok NULL to continue from the token the previous step
 * chose on the device; out_tok device [n_steps, B] int32 (or NULL) receives every step's
 * token.  Requires pos0[b] + n_steps <= max_ctx.  Asynchronous: returns after enqueueing;
 * call mk_synchronize for the status (a device wait that runs out ends the launch with
 * MK_ERR_TIMEOUT, as for one step). */
mk_status mk_decode_steps(mk_ctx *ctx, const int32_t *in_tok, const int32_t *pos0, int B,
                          int n_steps, int32_t *out_tok_dev);

/* Waits for the context's stream and reports a device-side error of enqueued steps. */
mk_status mk_synchronize(mk_ctx *ctx);

/* Clears counters, epoch and the error word after MK_ERR_TIMEOUT / MK_ERR_STATE. */
mk_status mk_reset(mk_ctx *ctx);

/* Releases everything the context owns: the queues, counters, activation buffers and
 * journal that mk_create allocated beside the launch it sized ("8 · Écrire son
 * megakernel", §8.3, the launcher and the global state it hands the kernel).  Never the
 * caller's weights, KV cache or logits.  Waits for the context's stream first.  NULL is a
 * no-op; always MK_OK. */
mk_status mk_destroy(mk_ctx *ctx);

mk_status mk_info(const mk_ctx *ctx, mk_info_t *info);

/* Copies up to max_records journal records of the last step (trace option) to host
 * memory; *n_records receives the number recorded. */
mk_status mk_get_trace(mk_ctx *ctx, mk_trace_rec *records, int max_records, int *n_records);

/* Debug/parity read of an activation vector of the last step, fp32, to host memory.
 * which: 0 h_in of layer (h after the embedding for layer 0; layer = n_layers gives the
 * final h), 1 h_mid (after attention), 2 q (rotated), 3 attention output o, 4 MLP
 * activation silu(gate)*up.  dst host [max_batch, width]; bytes must equal that size. */
mk_status mk_read_activation(mk_ctx *ctx, int which, int layer, float *dst, size_t bytes);

/* Host-only planning (no GPU needed): builds and validates the schedule for n_ctas
 * queues and reports its statistics in info (n_instructions, n_counters, kv_splits,
 * weight bytes).  Used to test the builder and validator on a CPU-only machine. */
mk_status mk_plan(const mk_model_desc *desc, const mk_options *opts, int n_ctas,
                  mk_info_t *info);

/* Build-ladder self tests of the persistent machinery ("8 · Écrire son megakernel",
 * §8.6, steps 1-4) on the current device:
 *   kind 1: a persistent kernel with one trivial instruction per CTA terminates;
 *   kind 2: dispatch of two opcodes keeps queue order;
 *   kind 3: counters between dependent instructions on different CTAs;
 *   kind 4: page pool: many TMA pages through a small pool, checksummed, none leaked.
 * result host [n] (n >= 4): [0] = 1 on pass, [1] CTAs used, [2..] kind-specific. */
mk_status mk_selftest(int kind, int64_t *result, int n);

/* Grid-barrier latency microbenchmark (§7.3 measurement): a one-wave kernel doing
 * n_barriers all-CTA barriers, with atomic counters (mode 0) or NaN sentinels (mode 1).
 * *us_per_barrier receives the mean latency in microseconds. */
mk_status mk_barrier_bench(int mode, int n_barriers, double *us_per_barrier);

/* SM -> die map ("7 · AMD et le monokernel", §7.4: die/chiplet locality; CUDA exposes no
 * such map, so it is measured).  A one-wave probe (one CTA per SM of the current device)
 * times cross-SM round trips from the SM that CTA 0 lands on to every other SM through
 * one shared 128-byte line, one pair at a time (reps >= 4 round trips each, the first two
 * discarded), and splits the SMs in two groups by those times (mk_two_groups).  die_of_sm host [max_sm] receives, indexed
 * by SM id, 0 for the reference SM's group and 1 for the other; rtt_cycles host [max_sm]
 * (or NULL) the mean round trip in SM cycles (0 for the reference SM); *n_sm the SM count.
 * MK_ERR_INVALID if max_sm is below the SM count, MK_ERR_TIMEOUT if a probe wait ran out
 * (each is bounded at 2 s). */
mk_status mk_die_map(int reps, int max_sm, int *die_of_sm, float *rtt_cycles, int *n_sm);

/* L2 line latency from two SMs (the address -> die interleave, "7 · AMD et le monokernel",
 * §7.4).  Allocates a zeroed device buffer of buf_bytes (freed before returning) and, for
 * each byte offset offsets host [n] (4-byte aligned, inside the buffer), times from the SM
 * with id sm_a and from sm_b a chain of reps >= 2 dependent L2-only loads of that line; lat_a,
 * lat_b host [n] receive the mean SM clock cycles per load (NaN if no CTA ran on that SM).
 * The line's home die is the one whose SM sees the shorter time.  MK_ERR_INVALID for bad
 * arguments (nothing launched). */
mk_status mk_line_latency(long long buf_bytes, const int64_t *offsets, int n, int sm_a, int sm_b, int reps,
                          float *lat_a, float *lat_b);

/* Two-means split of n >= 2 values (host only): group host [n] receives 0 for values at
 * or below the threshold, 1 above; *threshold (or NULL) the midpoint between the two
 * group means after convergence.  All values equal: every value in group 0. */
mk_status mk_two_groups(const float *x, int n, int *group, float *threshold);

/* One decode step that allocates no device memory, for callers that cannot call
 * cudaMalloc (code running inside an allocator or under a host framework that owns every
 * device allocation).  The pages have no counterpart to this entry point.  Same inputs
 * and outputs as mk_decode_step, passed directly (no context): desc, weights and kv as
 * for mk_create; in_tok, pos, out_tok host [B]; logits device [B, vocab] or NULL; work is
 * enqueued on `stream` (a cudaStream_t).
 * Every other buffer the step needs (queues, counters, the activations of B sequences,
 * one RoPE row per sequence) lives in one 16 MiB device array built into the library,
 * which each GPU that loads it holds until exit; models and batches that need more are
 * refused with MK_ERR_INVALID (the need depends on the model and B, not on positions).
 * The first call on a device (with that device current) looks the array up with
 * cudaGetSymbolAddress.  Every call is synchronous -- it waits for its step and copies
 * the status back -- so it cannot be used inside a stream capture.  All calls share the
 * array and keep its last contents; each call clears what must start at zero, and a call
 * with the same descriptor, pointers and B as the previous one on that device reuses the
 * schedule already in the array.  Calls whose GPU work overlaps race on the array and
 * must be serialised by the caller. */
mk_status mk_decode_step_noalloc(const mk_model_desc *desc, const mk_weights *weights, const mk_kv *kv,
                                 const int32_t *in_tok, const int32_t *pos, int B, int32_t *out_tok,
                                 float *logits, void *stream);

/* HBM page-stream microbenchmark: the megakernel's loader / compute-warp structure with
 * nothing else (P1 §7.5 continuous weight streaming, P2 §8.4 pages).  One CTA per SM
 * streams total_bytes / #SM of contiguous device memory through n_pages TMA pages of
 * page_bytes; mode 0: pages are released unread, mode 1: each compute warp first runs
 * the fp16 GEMV slice product on its eighth; hint bit 0: L2 evict-first policy; hint bit 1:
 * every CTA streams the same total_bytes / #SM (the access pattern of a GEMV input that
 * all SMs read; *gbps then counts the bytes delivered to the SMs).  *gbps gets the best of
 * three timed runs.  Allocates total_bytes of device memory for the run (hint bit 1:
 * total_bytes / #SM). */
mk_status mk_stream_bench(int page_bytes, int n_pages, int mode, int hint, long long total_bytes, double *gbps);

const char *mk_last_error(void);
const char *mk_status_string(mk_status s);

#ifdef __cplusplus
}
#endif
#endif /* MK_H_ */
