// Host runtime behind the C ABI of include/mk.h: context set-up, one-wave launch sizing
// ("8 · Écrire son megakernel", §8.3), schedule upload, the decode-step launches, and
// the build-ladder self tests (§8.6).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"
#include "mk_kernels.h"
#include "mk_plan.h"

using namespace mk;

namespace {

thread_local std::string g_last_error;

mk_status fail(mk_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

#define MK_CUDA(call)                                                                           \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess) {                                                                    \
      return fail(MK_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));            \
    }                                                                                           \
  } while (0)

struct DevBuf {
  void* p = nullptr;
  ~DevBuf() {
    if (p) cudaFree(p);
  }
};

// one schedule per batch size: queues, per-phase queues and its own counters/epoch
struct Sched {
  Plan plan;
  int n_instr = 0;
  DevBuf instr, qstart, counters;
  DevBuf tmaps;                     // tensor maps of the tensor-core pages
  std::vector<DevBuf> ph_instr, ph_qstart;
  uint32_t epoch = 0;
  DevBuf dyn;                       // MK_EXEC_GRAPH: the step's arguments in device memory
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t gexec = nullptr;
  const TraceRec* graph_trace = nullptr;  // the journal buffer the captured launches write
  ~Sched() {
    if (gexec) cudaGraphExecDestroy(gexec);
    if (graph) cudaGraphDestroy(graph);
  }
};

}  // namespace

namespace mk {
// lets the other translation units of the library report through mk_last_error
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace mk

// Prompt chunks (mk_prefill): up to kMaxBatch rows per launch -- consecutive positions of
// each prompt -- run through the same kernel with the tensor-core geometry, schedules of
// their own and an activation arena of kMaxBatch rows (kept apart from the decode arena, so
// that a decode step's NaN refill does not grow with the chunk size).
struct PrefillState {
  bool ready = false;
  ModelShape m{};     // the model with max_batch = kMaxBatch (schedules of up to 16 rows)
  Geometry geo{};
  DevState st{};      // the context's state with this geometry and the chunk arena
  DevBuf act, logits; // arena [2 parities]; logits of the last chunk's rows [kMaxBatch][V]
  std::map<int, std::unique_ptr<Sched>> scheds;
};

struct mk_ctx {
  ModelShape m{};
  mk_options opts{};
  Geometry geo{};
  cudaStream_t stream = nullptr;
  int device = 0;
  int n_sm = 0, bpsm = 0, n_cta = 0;
  const void* kernel = nullptr;     // one step per launch
  const void* kernel_ms = nullptr;  // several steps per launch (mk_decode_steps)
  // the same with the tensor-core GEMV (geometries for 3..16 rows: max_batch >= 3 and the
  // prompt chunks); contexts of max_batch <= 2 decode with the instances without it
  const void* kernel_tc = nullptr;
  const void* kernel_tc_ms = nullptr;
  DevState st{};  // template, counters patched per schedule
  ModelPtrs ptrs;  // device addresses written into every instruction
  DevBuf ptr_tables, rope, act, argkeys, ctl, trace;
  int trace_cap = 0;
  Ctl* host_ctl = nullptr;  // pinned
  HostMail* mail = nullptr;  // pinned, mapped into the device's address space
  uint32_t mail_seq = 0;
  std::map<int, std::unique_ptr<Sched>> scheds;
  uint32_t step = 0;
  bool broken = false;
  int last_B = 1;
  PrefillState pf;
  const void* last_arena = nullptr;  // activation arena of the last launch (NaN sentinels)
  ~mk_ctx() {
    if (host_ctl) cudaFreeHost(host_ctl);
    if (mail) cudaFreeHost(mail);
  }
};

namespace {

mk_status upload(DevBuf& b, const void* src, size_t bytes) {
  MK_CUDA(cudaMalloc(&b.p, std::max<size_t>(bytes, 16)));
  if (src && bytes) MK_CUDA(cudaMemcpy(b.p, src, bytes, cudaMemcpyHostToDevice));
  return MK_OK;
}

// the queues back to back, then the attention pools (their claim loops' a0 becomes an
// index into the uploaded array)
mk_status upload_queues(const std::vector<std::vector<Instr>>& qs, DevBuf& ibuf, DevBuf& qbuf, int* n_out,
                        const std::vector<Instr>* pool = nullptr) {
  std::vector<Instr> flat;
  std::vector<int32_t> qs_off;
  for (const auto& q : qs) {
    qs_off.push_back((int32_t)flat.size());
    flat.insert(flat.end(), q.begin(), q.end());
  }
  qs_off.push_back((int32_t)flat.size());
  if (pool && !pool->empty()) {
    const int32_t base = (int32_t)flat.size();
    for (auto& in : flat)
      if (in.op == OP_ATTN_POOL) in.a[0] += base;
    flat.insert(flat.end(), pool->begin(), pool->end());
  }
  if (n_out) *n_out = (int)flat.size();
  mk_status s = upload(ibuf, flat.data(), flat.size() * sizeof(Instr));
  if (s) return s;
  return upload(qbuf, qs_off.data(), qs_off.size() * sizeof(int32_t));
}

mk_status get_sched_in(mk_ctx* ctx, const ModelShape& m, const Geometry& geo,
                       std::map<int, std::unique_ptr<Sched>>& scheds, int B, Sched** out) {
  auto it = scheds.find(B);
  if (it != scheds.end()) {
    *out = it->second.get();
    return MK_OK;
  }
  auto sc = std::make_unique<Sched>();
  // small batches merge the KV splits inside the O-proj staging; otherwise counter mode
  // merges them in the last-arriving split and sentinel mode keeps the separate
  // ATTN_REDUCE op (it has no atomics to elect a last arriver)
  const int merge = choose_merge(m, geo, B, ctx->opts.sync_mode == MK_SYNC_COUNTER, ctx->opts.attn_merge);
  const bool pool = ctx->opts.attn_pool == 1 && ctx->opts.exec_mode == MK_EXEC_PERSISTENT;
  std::string e = build_plan(m, geo, ctx->n_cta, B, ctx->opts.fault_drop_signal, merge, &sc->plan, pool);
  if (!e.empty()) return fail(MK_ERR_INVALID, "schedule: " + e);
  bake_pointers(m, ctx->ptrs, &sc->plan);
  if (ctx->opts.fault_drop_signal <= 0) {
    e = validate_plan(m, geo, sc->plan);
    if (!e.empty()) return fail(MK_ERR_INVALID, "schedule rejected by the validator: " + e);
  }
  int nb = 1;
  while (nb < B) nb <<= 1;
  if (use_tc(geo, nb) || geo.attn_mma) {
    std::vector<TmapImage> maps;
    if (use_tc(geo, nb)) {
      e = build_tc_maps(m, geo, &sc->plan, &maps);
      if (!e.empty()) return fail(MK_ERR_CUDA, "tensor maps: " + e);
    }
    e = build_kv_maps(m, geo, ctx->m.max_batch, &sc->plan, &maps);
    if (!e.empty()) return fail(MK_ERR_CUDA, "tensor maps: " + e);
    mk_status s = upload(sc->tmaps, maps.data(), maps.size() * sizeof(TmapImage));
    if (s) return s;
    const uintptr_t dev = reinterpret_cast<uintptr_t>(sc->tmaps.p);
    const bool gm = use_tc(geo, nb);
    for (auto& q : sc->plan.queues) place_tc_maps(q, dev, gm);
    for (auto& ph : sc->plan.phase_queues)
      for (auto& q : ph) place_tc_maps(q, dev, gm);
    place_tc_maps(sc->plan.pool, dev, gm);
  }
  mk_status s = upload_queues(sc->plan.queues, sc->instr, sc->qstart, &sc->n_instr, &sc->plan.pool);
  if (s) return s;
  MK_CUDA(cudaMalloc(&sc->counters.p, sizeof(uint32_t) * std::max(1, sc->plan.n_counters)));
  MK_CUDA(cudaMemset(sc->counters.p, 0, sizeof(uint32_t) * std::max(1, sc->plan.n_counters)));
  if (ctx->opts.exec_mode != MK_EXEC_PERSISTENT) {
    const size_t np = sc->plan.phase_queues.size();
    sc->ph_instr.resize(np);
    sc->ph_qstart.resize(np);
    for (size_t k = 0; k < np; ++k) {
      s = upload_queues(sc->plan.phase_queues[k], sc->ph_instr[k], sc->ph_qstart[k], nullptr);
      if (s) return s;
    }
  }
  if (ctx->opts.trace) {
    const int need = sc->n_instr + 64;
    if (need > ctx->trace_cap) {
      if (ctx->trace.p) cudaFree(ctx->trace.p);
      ctx->trace.p = nullptr;
      MK_CUDA(cudaMalloc(&ctx->trace.p, sizeof(TraceRec) * need));
      ctx->trace_cap = need;
      ctx->st.trace = reinterpret_cast<TraceRec*>(ctx->trace.p);
      ctx->st.trace_cap = need;
    }
  }
  *out = sc.get();
  scheds[B] = std::move(sc);
  return MK_OK;
}

mk_status get_sched(mk_ctx* ctx, int B, Sched** out) { return get_sched_in(ctx, ctx->m, ctx->geo, ctx->scheds, B, out); }

mk_status launch(mk_ctx* ctx, const void* fn, const DevState& S, const StepArgs& A, bool cooperative,
                 bool programmatic = false, cudaStream_t stream = nullptr, bool own_stream = false) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(ctx->n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S.smem_bytes;
  cfg.stream = own_stream ? stream : ctx->stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 2 : 1;
  void* args[2] = {const_cast<DevState*>(&S), const_cast<StepArgs*>(&A)};
  MK_CUDA(cudaLaunchKernelExC(&cfg, fn, args));
  return MK_OK;
}

// MK_EXEC_GRAPH: the per-op launches captured once (on a private stream) into a graph with
// programmatic dependencies between consecutive launches; each step copies its arguments
// to device memory and launches the graph.
mk_status run_graph(mk_ctx* ctx, Sched* sc, const DevState& S, const StepArgs& A, const void* fn) {
  if (sc->gexec && sc->graph_trace != ctx->st.trace) {  // the journal buffer moved: capture again
    cudaGraphExecDestroy(sc->gexec);
    cudaGraphDestroy(sc->graph);
    sc->gexec = nullptr;
    sc->graph = nullptr;
  }
  if (!sc->dyn.p) MK_CUDA(cudaMalloc(&sc->dyn.p, sizeof(StepArgs)));
  if (!sc->gexec) {
    cudaStream_t cs;
    MK_CUDA(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    mk_status st = MK_OK;
    if (e == cudaSuccess) {
      for (size_t k = 0; k < sc->ph_instr.size() && st == MK_OK; ++k) {
        StepArgs Ak{};
        Ak.instr = reinterpret_cast<const Instr*>(sc->ph_instr[k].p);
        Ak.q_start = reinterpret_cast<const int32_t*>(sc->ph_qstart[k].p);
        Ak.flags = SF_NO_SYNC | (k == 0 ? SF_RESET_ARGMAX : SF_PDL);
        Ak.dyn = reinterpret_cast<const StepArgs*>(sc->dyn.p);
        st = launch(ctx, fn, S, Ak, false, k > 0, cs, true);
      }
      cudaGraph_t g = nullptr;
      const cudaError_t e2 = cudaStreamEndCapture(cs, &g);
      if (st == MK_OK && e2 != cudaSuccess) e = e2;
      if (st == MK_OK && e == cudaSuccess) {
        sc->graph = g;
        e = cudaGraphInstantiate(&sc->gexec, g, 0);
      } else if (g) {
        cudaGraphDestroy(g);
      }
    }
    cudaStreamDestroy(cs);
    if (st) return st;
    if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(e));
    sc->graph_trace = ctx->st.trace;
  }
  StepArgs D = A;  // the per-step fields; the launches keep their own queues and flags
  D.instr = nullptr;
  D.q_start = nullptr;
  D.dyn = nullptr;
  D.flags = A.flags & (SF_TOK_FROM_DEVICE | SF_TRACE);
  MK_CUDA(cudaMemcpyAsync(sc->dyn.p, &D, sizeof(D), cudaMemcpyHostToDevice, ctx->stream));
  MK_CUDA(cudaGraphLaunch(sc->gexec, ctx->stream));
  return MK_OK;
}

// enqueue one decode step (one launch, or the multi-launch control's per-op launches); with
// persistent control, n_steps > 1 greedy steps in the one launch (tok_hist then [n_steps][B])
mk_status enqueue_step(mk_ctx* ctx, Sched* sc, int B, const int32_t* tok, const int32_t* pos, bool tok_from_dev,
                       float* logits, int32_t* tok_hist, int n_steps = 1, uint32_t mail_seq = 0,
                       const DevState* base = nullptr, const int32_t* seq = nullptr, const int32_t* p0 = nullptr) {
  DevState S = base ? *base : ctx->st;
  S.trace = ctx->st.trace;
  S.trace_cap = ctx->st.trace_cap;
  // NaN sentinels: a launch expects its arena's current parity to hold sentinels, which the
  // launch before it on the same arena left behind; after a switch of arenas, refill both
  if (ctx->opts.sync_mode == MK_SYNC_SENTINEL && ctx->last_arena != S.act) {
    if (ctx->last_arena) MK_CUDA(cudaMemsetAsync(S.act, 0xFF, sizeof(float) * 2 * S.act_floats, ctx->stream));
    ctx->last_arena = S.act;
  }
  S.counters = reinterpret_cast<uint32_t*>(sc->counters.p);
  S.n_counters = sc->plan.n_counters;
  StepArgs A{};
  A.epoch = sc->epoch;
  A.step = ctx->step;
  A.B = B;
  A.flags = SF_RESET_ARGMAX | (tok_from_dev ? SF_TOK_FROM_DEVICE : 0) | (ctx->opts.trace ? SF_TRACE : 0);
  for (int b = 0; b < B; ++b) {
    A.tok[b] = tok ? tok[b] : 0;
    A.pos[b] = pos[b];
    A.seq[b] = seq ? seq[b] : b;
    A.p0[b] = p0 ? p0[b] : pos[b];
    // the kernel reads this launch's positions p0..pos of row b from rows b - (pos - p0) .. b:
    // they must exist and hold that sequence's consecutive positions
    const int n_new = A.pos[b] - A.p0[b] + 1;
    if (n_new < 1 || n_new > b + 1 || A.seq[b] < 0 || A.seq[b] >= ctx->m.max_batch)
      return fail(MK_ERR_INVALID, "step rows: bad sequence or first new position");
    for (int i = 1; i < n_new; ++i)
      if (A.seq[b - i] != A.seq[b] || A.pos[b - i] != A.pos[b] - i)
        return fail(MK_ERR_INVALID, "step rows: a chunk's rows must be consecutive positions of one sequence");
  }
  A.logits = logits;
  A.tok_hist = tok_hist;
  A.n_steps = n_steps;
  A.mail_seq = mail_seq;
  if (n_steps > 1 && ctx->opts.exec_mode != MK_EXEC_PERSISTENT)
    return fail(MK_ERR_INVALID, "several steps in one launch need persistent control");
  const void* fn = S.tc ? (n_steps > 1 ? ctx->kernel_tc_ms : ctx->kernel_tc) : (n_steps > 1 ? ctx->kernel_ms : ctx->kernel);
  if (ctx->opts.trace) MK_CUDA(cudaMemsetAsync(&reinterpret_cast<Ctl*>(ctx->ctl.p)->trace_n, 0, 4, ctx->stream));
  mk_status s;
  if (ctx->opts.exec_mode == MK_EXEC_GRAPH) {
    s = run_graph(ctx, sc, S, A, fn);
    if (s) return s;
  } else if (ctx->opts.exec_mode == MK_EXEC_MULTILAUNCH) {
    const size_t np = sc->ph_instr.size();
    for (size_t k = 0; k < np; ++k) {
      StepArgs Ak = A;
      Ak.flags |= SF_NO_SYNC;
      if (k) Ak.flags &= ~SF_RESET_ARGMAX;
      Ak.instr = reinterpret_cast<const Instr*>(sc->ph_instr[k].p);
      Ak.q_start = reinterpret_cast<const int32_t*>(sc->ph_qstart[k].p);
      s = launch(ctx, fn, S, Ak, false);
      if (s) return s;
    }
  } else {
    A.instr = reinterpret_cast<const Instr*>(sc->instr.p);
    A.q_start = reinterpret_cast<const int32_t*>(sc->qstart.p);
    s = launch(ctx, fn, S, A, true);
    if (s) return s;
  }
  sc->epoch += (uint32_t)n_steps;
  ctx->step += (uint32_t)n_steps;
  ctx->last_B = B;
  return MK_OK;
}

mk_status read_status(mk_ctx* ctx) {
  MK_CUDA(cudaMemcpyAsync(ctx->host_ctl, ctx->ctl.p, sizeof(Ctl), cudaMemcpyDeviceToHost, ctx->stream));
  MK_CUDA(cudaStreamSynchronize(ctx->stream));
  const ErrWord& e = ctx->host_ctl->err;
  if (e.code) {
    ctx->broken = true;
    char buf[200];
    snprintf(buf, sizeof buf, "device error %u at cta %d pc %d counter %d", e.code, e.cta, e.pc, e.ctr);
    return fail((mk_status)e.code, buf);
  }
  if (ctx->host_ctl->nan_seen) return fail(MK_ERR_NAN, "a logit was NaN");
  return MK_OK;
}

// The prompt-chunk state, allocated at the first chunked mk_prefill: the context's device
// state with the chunk geometry, an arena of kMaxBatch rows (NaN-filled) and the logits of
// the last chunk's rows.
mk_status ensure_prefill(mk_ctx* ctx) {
  PrefillState& pf = ctx->pf;
  if (pf.ready) return MK_OK;
  const Geometry& g = pf.geo;
  DevState S = ctx->st;
  S.S = g.S;
  S.ws_qkv = g.ws_qkv; S.ws_o = g.ws_o; S.ws_up = g.ws_up; S.ws_down = g.ws_down; S.ws_lm = g.ws_lm;
  S.page_bytes = g.page_bytes;
  S.n_pages = g.n_pages;
  S.page_stride = g.page_stride;
  S.tc = g.tc;
  S.attn_mma = g.attn_mma;
  S.xbuf_bytes = g.xbuf_bytes;
  S.scratch_bytes = g.scratch_bytes;
  S.smem_bytes = g.smem_bytes;
  S.max_batch = kMaxBatch;
  arena_layout(pf.m, g, kMaxBatch, &S);
  MK_CUDA(cudaMalloc(&pf.act.p, sizeof(float) * 2 * S.act_floats));
  MK_CUDA(cudaMemset(pf.act.p, 0xFF, sizeof(float) * 2 * S.act_floats));  // all NaN
  S.act = reinterpret_cast<float*>(pf.act.p);
  MK_CUDA(cudaMalloc(&pf.logits.p, sizeof(float) * (size_t)kMaxBatch * ctx->m.V));
  pf.st = S;
  pf.ready = true;
  return MK_OK;
}

mk_status check_step_args(mk_ctx* ctx, const int32_t* tok, const int32_t* pos, int B) {
  if (ctx->broken) return fail(MK_ERR_STATE, "context needs mk_reset after a device error");
  if (B < 1 || B > ctx->m.max_batch) return fail(MK_ERR_INVALID, "B out of range");
  if (!pos) return fail(MK_ERR_INVALID, "pos is NULL");
  for (int b = 0; b < B; ++b) {
    if (tok && (tok[b] < 0 || tok[b] >= ctx->m.V)) return fail(MK_ERR_INVALID, "token id out of range");
    if (pos[b] < 0 || pos[b] >= ctx->m.max_ctx) return fail(MK_ERR_INVALID, "position out of range");
  }
  return MK_OK;
}

}  // namespace

extern "C" {

const char* mk_last_error(void) { return g_last_error.c_str(); }

const char* mk_status_string(mk_status s) {
  switch (s) {
    case MK_OK: return "MK_OK";
    case MK_ERR_INVALID: return "MK_ERR_INVALID";
    case MK_ERR_OCCUPANCY: return "MK_ERR_OCCUPANCY";
    case MK_ERR_CUDA: return "MK_ERR_CUDA";
    case MK_ERR_TIMEOUT: return "MK_ERR_TIMEOUT";
    case MK_ERR_STATE: return "MK_ERR_STATE";
    case MK_ERR_NAN: return "MK_ERR_NAN";
  }
  return "MK_ERR_UNKNOWN";
}

mk_status mk_plan(const mk_model_desc* desc, const mk_options* opts, int n_ctas, mk_info_t* info) {
  std::string e = check_desc(desc);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  if (n_ctas < 1 || !info) return fail(MK_ERR_INVALID, "n_ctas must be positive and info non-NULL");
  mk_options o{};
  if (opts) o = *opts;
  if (o.attn_merge < 0 || o.attn_merge > 3) return fail(MK_ERR_INVALID, "attn_merge must be 0..3");
  if (o.attn_tensor_cores < -1 || o.attn_tensor_cores > 1) return fail(MK_ERR_INVALID, "attn_tensor_cores must be -1, 0 or 1");
  const ModelShape m = shape_of(desc);
  Geometry g;
  e = make_geometry(m, n_ctas, o.page_bytes, o.n_pages, o.kv_splits, 232448, &g, o.attn_tensor_cores);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  Plan p;
  e = build_plan(m, g, n_ctas, m.max_batch, o.fault_drop_signal,
                 choose_merge(m, g, m.max_batch, o.sync_mode == MK_SYNC_COUNTER, o.attn_merge), &p,
                 o.attn_pool == 1 && o.exec_mode == MK_EXEC_PERSISTENT);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  e = validate_plan(m, g, p);
  if (!e.empty()) return fail(MK_ERR_INVALID, "schedule rejected by the validator: " + e);
  std::memset(info, 0, sizeof *info);
  info->n_ctas = n_ctas;
  info->threads_per_cta = kThreads;
  info->smem_bytes = g.smem_bytes;
  info->kernel_variant = g.instance();
  info->page_bytes = g.page_bytes;
  info->n_pages = g.n_pages;
  info->kv_splits = g.S;
  for (const auto& q : p.queues) info->n_instructions += (int)q.size();
  info->n_instructions += (int)p.pool.size();
  info->n_counters = p.n_counters;
  info->launches_per_step = o.exec_mode != MK_EXEC_PERSISTENT ? (int)p.phase_queues.size() : 1;
  info->weight_bytes_per_step = p.weight_bytes;
  return MK_OK;
}

mk_status mk_create(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv, const mk_options* opts,
                    void* stream, mk_ctx** out) {
  if (!out) return fail(MK_ERR_INVALID, "out is NULL");
  *out = nullptr;
  std::string e = check_desc(desc);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  e = check_model_pointers(desc, w, kv);  // present and 16-byte aligned (bulk copies need it)
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  const ModelShape m = shape_of(desc);
  const void* const* tabs[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};

  auto ctx = std::make_unique<mk_ctx>();
  ctx->m = m;
  if (opts) ctx->opts = *opts;
  mk_options& o = ctx->opts;
  if (o.wait_timeout_s <= 0) o.wait_timeout_s = 2.0;
  if (o.backoff_max_ns <= 0) o.backoff_max_ns = 256;
  if (o.sync_mode != MK_SYNC_COUNTER && o.sync_mode != MK_SYNC_SENTINEL) return fail(MK_ERR_INVALID, "sync_mode");
  if (o.exec_mode != MK_EXEC_PERSISTENT && o.exec_mode != MK_EXEC_MULTILAUNCH && o.exec_mode != MK_EXEC_GRAPH)
    return fail(MK_ERR_INVALID, "exec_mode");
  if (o.attn_merge < 0 || o.attn_merge > 3) return fail(MK_ERR_INVALID, "attn_merge must be 0..3");
  if (o.attn_pool < 0 || o.attn_pool > 1) return fail(MK_ERR_INVALID, "attn_pool must be 0 or 1");
  if (o.attn_tensor_cores < -1 || o.attn_tensor_cores > 1) return fail(MK_ERR_INVALID, "attn_tensor_cores must be -1, 0 or 1");
  ctx->stream = reinterpret_cast<cudaStream_t>(stream);
  MK_CUDA(cudaGetDevice(&ctx->device));
  MK_CUDA(cudaDeviceGetAttribute(&ctx->n_sm, cudaDevAttrMultiProcessorCount, ctx->device));
  int smem_optin = 0;
  MK_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device));
  int n_cta_guess = ctx->n_sm;
  if (o.max_ctas > 0) n_cta_guess = std::min(n_cta_guess, o.max_ctas);
  e = make_geometry(m, n_cta_guess, o.page_bytes, o.n_pages, o.kv_splits, smem_optin, &ctx->geo, o.attn_tensor_cores);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  // one wave (§8.3): opt in to the shared memory, ask how many CTAs fit, launch exactly that
  ctx->kernel_tc = step_kernel_entry(m.dtype, o.sync_mode, false, 2);
  ctx->kernel_tc_ms = step_kernel_entry(m.dtype, o.sync_mode, true, 2);
  ctx->kernel = step_kernel_entry(m.dtype, o.sync_mode, false, ctx->geo.instance());
  ctx->kernel_ms = step_kernel_entry(m.dtype, o.sync_mode, true, ctx->geo.instance());
  for (const void* fn : {ctx->kernel, ctx->kernel_ms, ctx->kernel_tc, ctx->kernel_tc_ms})
    // the attribute is per function (shared by every context in the process): the device's
    // limit, so that no context's launch is refused after another context sets a lower one
    MK_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin));
  MK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctx->bpsm, ctx->kernel, kThreads, ctx->geo.smem_bytes));
  if (ctx->bpsm < 1) return fail(MK_ERR_OCCUPANCY, "the kernel does not fit on an SM (blocks per SM < 1)");
  ctx->n_cta = ctx->n_sm * ctx->bpsm;
  if (o.max_ctas > 0) ctx->n_cta = std::min(ctx->n_cta, o.max_ctas);
  if (ctx->n_cta != n_cta_guess) {
    e = make_geometry(m, ctx->n_cta, o.page_bytes, o.n_pages, o.kv_splits, smem_optin, &ctx->geo, o.attn_tensor_cores);
    if (!e.empty()) return fail(MK_ERR_INVALID, e);
  }
  const Geometry& g = ctx->geo;
  {  // prompt chunks: the tensor-core geometry of kMaxBatch rows, if it fits the same wave
    PrefillState& pf = ctx->pf;
    pf.m = m;
    pf.m.max_batch = kMaxBatch;
    if (o.exec_mode == MK_EXEC_PERSISTENT &&
        make_geometry(pf.m, ctx->n_cta, o.page_bytes, o.n_pages, o.kv_splits, smem_optin, &pf.geo,
                      o.attn_tensor_cores).empty()) {
      int bp = 0;
      MK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bp, ctx->kernel_tc, kThreads, pf.geo.smem_bytes));
      if (bp < ctx->bpsm) pf.geo.smem_bytes = 0;  // chunks would not run in one wave: per-position prefill
    } else {
      pf.geo.smem_bytes = 0;
    }
  }

  // device state
  DevState& S = ctx->st;
  S.L = m.L; S.d = m.d; S.Hq = m.Hq; S.Hkv = m.Hkv; S.hd = m.hd; S.F = m.F; S.V = m.V;
  S.dtype = m.dtype; S.max_batch = m.max_batch; S.max_ctx = m.max_ctx; S.S = g.S; S.eps = m.eps;
  S.ws_qkv = g.ws_qkv; S.ws_o = g.ws_o; S.ws_up = g.ws_up; S.ws_down = g.ws_down; S.ws_lm = g.ws_lm;
  S.embed = static_cast<const uint16_t*>(w->embed);
  S.final_norm = static_cast<const uint16_t*>(w->final_norm);
  S.lm_head = static_cast<const uint16_t*>(w->lm_head);
  {
    std::vector<const void*> tab;
    for (auto t : tabs)
      for (int l = 0; l < m.L; ++l) tab.push_back(t[l]);
    for (int l = 0; l < m.L; ++l) tab.push_back(kv->k_cache[l]);
    for (int l = 0; l < m.L; ++l) tab.push_back(kv->v_cache[l]);
    mk_status s = upload(ctx->ptr_tables, tab.data(), tab.size() * sizeof(void*));
    if (s) return s;
    auto base = reinterpret_cast<const uint16_t* const*>(ctx->ptr_tables.p);
    S.attn_norm = base + 0 * m.L; S.wq = base + 1 * m.L; S.wk = base + 2 * m.L; S.wv = base + 3 * m.L;
    S.wo = base + 4 * m.L; S.mlp_norm = base + 5 * m.L; S.w_gate = base + 6 * m.L; S.w_up = base + 7 * m.L;
    S.w_down = base + 8 * m.L;
    auto mbase = reinterpret_cast<uint16_t* const*>(ctx->ptr_tables.p);
    S.kcache = mbase + 9 * m.L;
    S.vcache = mbase + 10 * m.L;
  }
  {  // RoPE table: angle pos * theta^(-2i/hd), evaluated in double, stored as fp32
    const int half = m.hd / 2;
    std::vector<float> tab((size_t)m.max_ctx * half * 2);
    for (int i = 0; i < half; ++i) {
      const double f = std::pow((double)m.theta, -2.0 * i / m.hd);
      for (int t = 0; t < m.max_ctx; ++t) {
        const double a = (double)t * f;
        tab[((size_t)t * half + i) * 2] = (float)std::cos(a);
        tab[((size_t)t * half + i) * 2 + 1] = (float)std::sin(a);
      }
    }
    mk_status s = upload(ctx->rope, tab.data(), tab.size() * sizeof(float));
    if (s) return s;
    S.rope = reinterpret_cast<const float2*>(ctx->rope.p);
  }
  {  // activation arena: two parity sets
    arena_layout(m, g, m.max_batch, &S);
    MK_CUDA(cudaMalloc(&ctx->act.p, sizeof(float) * 2 * S.act_floats));
    MK_CUDA(cudaMemset(ctx->act.p, 0xFF, sizeof(float) * 2 * S.act_floats));  // all NaN
    S.act = reinterpret_cast<float*>(ctx->act.p);
  }
  MK_CUDA(cudaMalloc(&ctx->argkeys.p, sizeof(unsigned long long) * 2 * kMaxBatch));
  MK_CUDA(cudaMemset(ctx->argkeys.p, 0, sizeof(unsigned long long) * 2 * kMaxBatch));
  S.argkeys = reinterpret_cast<unsigned long long*>(ctx->argkeys.p);
  MK_CUDA(cudaMalloc(&ctx->ctl.p, sizeof(Ctl)));
  MK_CUDA(cudaMemset(ctx->ctl.p, 0, sizeof(Ctl)));
  S.ctl = reinterpret_cast<Ctl*>(ctx->ctl.p);
  MK_CUDA(cudaMallocHost(reinterpret_cast<void**>(&ctx->host_ctl), sizeof(Ctl)));
  MK_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&ctx->mail), sizeof(HostMail), cudaHostAllocMapped));
  memset(ctx->mail, 0, sizeof(HostMail));
  {
    void* dp = nullptr;
    MK_CUDA(cudaHostGetDevicePointer(&dp, ctx->mail, 0));
    S.mail = reinterpret_cast<HostMail*>(dp);
  }
  S.n_cta = ctx->n_cta;
  S.page_bytes = g.page_bytes;
  S.n_pages = g.n_pages;
  S.page_stride = g.page_stride;
  S.tc = g.tc;
  S.attn_mma = g.attn_mma;
  S.xbuf_bytes = g.xbuf_bytes;
  S.scratch_bytes = g.scratch_bytes;
  S.smem_bytes = g.smem_bytes;
  S.sync_mode = o.sync_mode;
  S.timeout_ns = (int64_t)(o.wait_timeout_s * 1e9);
  S.backoff_max_ns = o.backoff_max_ns;
  S.split_min_positions = o.split_min_positions > 0 ? o.split_min_positions : 16;
  S.inflight_pages = o.inflight_pages < 0 ? 0 : (o.inflight_pages == 0 ? 2 : o.inflight_pages);
  ModelPtrs& mp = ctx->ptrs;
  mp.final_norm = w->final_norm;
  mp.lm_head = w->lm_head;
  std::vector<const void*>* dst[11] = {&mp.attn_norm, &mp.wq, &mp.wk, &mp.wv, &mp.wo, &mp.mlp_norm,
                                       &mp.w_gate, &mp.w_up, &mp.w_down, &mp.kcache, &mp.vcache};
  for (int k = 0; k < 9; ++k) dst[k]->assign(tabs[k], tabs[k] + m.L);
  mp.kcache.assign(kv->k_cache, kv->k_cache + m.L);
  mp.vcache.assign(kv->v_cache, kv->v_cache + m.L);
  // the schedule for the largest batch is built (and validated) now; others on first use
  Sched* sc = nullptr;
  mk_status s = get_sched(ctx.get(), m.max_batch, &sc);
  if (s) return s;
  MK_CUDA(cudaDeviceSynchronize());
  *out = ctx.release();
  return MK_OK;
}

mk_status mk_destroy(mk_ctx* ctx) {
  if (!ctx) return MK_OK;
  cudaStreamSynchronize(ctx->stream);
  delete ctx;
  return MK_OK;
}

mk_status mk_info(const mk_ctx* ctx, mk_info_t* info) {
  if (!ctx || !info) return fail(MK_ERR_INVALID, "NULL argument");
  std::memset(info, 0, sizeof *info);
  info->n_sm = ctx->n_sm;
  info->blocks_per_sm = ctx->bpsm;
  info->n_ctas = ctx->n_cta;
  info->threads_per_cta = kThreads;
  info->smem_bytes = ctx->geo.smem_bytes;
  info->kernel_variant = ctx->geo.instance();
  info->page_bytes = ctx->geo.page_bytes;
  info->n_pages = ctx->geo.n_pages;
  info->kv_splits = ctx->geo.S;
  auto it = ctx->scheds.find(ctx->last_B);
  if (it == ctx->scheds.end()) it = ctx->scheds.begin();
  if (it != ctx->scheds.end()) {
    info->n_instructions = it->second->n_instr;
    info->n_counters = it->second->plan.n_counters;
    info->launches_per_step =
        ctx->opts.exec_mode != MK_EXEC_PERSISTENT ? (int)it->second->plan.phase_queues.size() : 1;
    info->weight_bytes_per_step = it->second->plan.weight_bytes;
  }
  return MK_OK;
}

mk_status mk_decode_step(mk_ctx* ctx, const int32_t* in_tok, const int32_t* pos, int B, int32_t* out_tok,
                         float* logits) {
  if (!ctx) return fail(MK_ERR_INVALID, "ctx is NULL");
  if (!in_tok || !out_tok) return fail(MK_ERR_INVALID, "in_tok/out_tok NULL");
  mk_status s = check_step_args(ctx, in_tok, pos, B);
  if (s) return s;
  Sched* sc = nullptr;
  s = get_sched(ctx, B, &sc);
  if (s) return s;
  // Without logits to hand back, the step posts its tokens to the mapped mailbox and the
  // host waits on that word alone: no device-to-host copy, no stream synchronisation (the
  // kernel's tail still runs; the next launch queues behind it).  Any error, or a kernel
  // that ends without posting, takes the synchronous path through the control block.
  const bool mail = logits == nullptr && ctx->opts.exec_mode == MK_EXEC_PERSISTENT;
  const uint32_t seq = mail ? ++ctx->mail_seq : 0u;
  if (mail && seq == 0u) return fail(MK_ERR_STATE, "mailbox sequence wrapped");
  s = enqueue_step(ctx, sc, B, in_tok, pos, false, logits, nullptr, 1, seq);
  if (s) return s;
  if (mail) {
    const volatile uint32_t* w = &ctx->mail->seq;
    for (uint32_t k = 1;; ++k) {
      if (*w == seq) break;
      if ((k & 255u) == 0u && cudaStreamQuery(ctx->stream) != cudaErrorNotReady) break;
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    if (*w == seq && ctx->mail->err == 0u) {
      for (int b = 0; b < B; ++b) out_tok[b] = ctx->mail->tok[b];
      if (ctx->mail->nan_seen) return fail(MK_ERR_NAN, "a logit was NaN");
      return MK_OK;
    }
  }
  s = read_status(ctx);
  if (s && s != MK_ERR_NAN) return s;
  for (int b = 0; b < B; ++b) out_tok[b] = ctx->host_ctl->tok[b];
  return s;
}

mk_status mk_decode_steps(mk_ctx* ctx, const int32_t* in_tok, const int32_t* pos0, int B, int n_steps,
                          int32_t* out_tok_dev) {
  if (!ctx) return fail(MK_ERR_INVALID, "ctx is NULL");
  if (n_steps < 1) return fail(MK_ERR_INVALID, "n_steps < 1");
  if (!in_tok && ctx->step == 0) return fail(MK_ERR_INVALID, "in_tok NULL before any step chose a token");
  mk_status s = check_step_args(ctx, in_tok, pos0, B);
  if (s) return s;
  for (int b = 0; b < B; ++b)
    if ((long long)pos0[b] + n_steps > ctx->m.max_ctx) return fail(MK_ERR_INVALID, "positions exceed max_ctx");
  Sched* sc = nullptr;
  s = get_sched(ctx, B, &sc);
  if (s) return s;
  if (ctx->opts.exec_mode == MK_EXEC_PERSISTENT)  // all the steps in one launch
    return enqueue_step(ctx, sc, B, in_tok, pos0, !in_tok, nullptr, out_tok_dev, n_steps);
  int32_t pos[kMaxBatch];
  for (int k = 0; k < n_steps; ++k) {
    for (int b = 0; b < B; ++b) pos[b] = pos0[b] + k;
    s = enqueue_step(ctx, sc, B, k == 0 ? in_tok : nullptr, pos, k > 0 || !in_tok, nullptr,
                     out_tok_dev ? out_tok_dev + (size_t)k * B : nullptr);
    if (s) return s;
  }
  return MK_OK;
}

mk_status mk_synchronize(mk_ctx* ctx) {
  if (!ctx) return fail(MK_ERR_INVALID, "ctx is NULL");
  return read_status(ctx);
}

mk_status mk_prefill(mk_ctx* ctx, const int32_t* tokens, int B, int P, int32_t* next_tok, float* logits) {
  if (!ctx) return fail(MK_ERR_INVALID, "ctx is NULL");
  if (!tokens || !next_tok || P < 1) return fail(MK_ERR_INVALID, "tokens/next_tok NULL or P < 1");
  if (P > ctx->m.max_ctx) return fail(MK_ERR_INVALID, "P exceeds max_ctx");
  if (B < 1 || B > ctx->m.max_batch) return fail(MK_ERR_INVALID, "B out of range");
  for (long long i = 0; i < (long long)B * P; ++i)
    if (tokens[i] < 0 || tokens[i] >= ctx->m.V) return fail(MK_ERR_INVALID, "token id out of range");
  if (ctx->broken) return fail(MK_ERR_STATE, "context needs mk_reset after a device error");
  mk_status s;
  if (ctx->pf.geo.smem_bytes > 0) {
    // Prompt chunks: each launch takes c = kMaxBatch / B consecutive positions of every
    // sequence as rows (row b*n + i = position t0 + i of sequence b), so that the weights
    // stream once per chunk for up to kMaxBatch rows on the tensor-core GEMV; a row
    // attends to the cached positions below t0 and to its chunk's rows up to its own.
    s = ensure_prefill(ctx);
    if (s) return s;
    const int c = std::max(1, kMaxBatch / B);
    int32_t tok[kMaxBatch], pos[kMaxBatch], seq[kMaxBatch], p0[kMaxBatch];
    int n = 0;
    for (int t0 = 0; t0 < P; t0 += c) {
      n = std::min(c, P - t0);
      const int rows = B * n;
      for (int b = 0; b < B; ++b)
        for (int i = 0; i < n; ++i) {
          const int r = b * n + i;
          tok[r] = tokens[(size_t)b * P + t0 + i];
          pos[r] = t0 + i;
          seq[r] = b;
          p0[r] = t0;
        }
      Sched* sc = nullptr;
      s = get_sched_in(ctx, ctx->pf.m, ctx->pf.geo, ctx->pf.scheds, rows, &sc);
      if (s) return s;
      const bool last = t0 + n >= P;
      float* lg = last && logits ? reinterpret_cast<float*>(ctx->pf.logits.p) : nullptr;
      s = enqueue_step(ctx, sc, rows, tok, pos, false, lg, nullptr, 1, 0, &ctx->pf.st, seq, p0);
      if (s) return s;
    }
    // each sequence's last position is row b*n + n-1 of the last chunk
    if (logits)
      for (int b = 0; b < B; ++b)
        MK_CUDA(cudaMemcpyAsync(logits + (size_t)b * ctx->m.V,
                                reinterpret_cast<float*>(ctx->pf.logits.p) + (size_t)(b * n + n - 1) * ctx->m.V,
                                sizeof(float) * ctx->m.V, cudaMemcpyDeviceToDevice, ctx->stream));
    s = read_status(ctx);
    if (s && s != MK_ERR_NAN) return s;
    for (int b = 0; b < B; ++b) next_tok[b] = ctx->host_ctl->tok[b * n + n - 1];
    // the device copy of the chosen tokens (read by steps that embed them on the device)
    MK_CUDA(cudaMemcpy(reinterpret_cast<Ctl*>(ctx->ctl.p)->tok, next_tok, sizeof(int32_t) * B, cudaMemcpyHostToDevice));
    ctx->last_B = B;
    return s;
  }
  Sched* sc = nullptr;
  s = get_sched(ctx, B, &sc);
  if (s) return s;
  int32_t tok[kMaxBatch], pos[kMaxBatch];
  for (int t = 0; t < P; ++t) {  // teacher-forced steps, enqueued back to back
    for (int b = 0; b < B; ++b) {
      tok[b] = tokens[(size_t)b * P + t];
      pos[b] = t;
    }
    s = enqueue_step(ctx, sc, B, tok, pos, false, t == P - 1 ? logits : nullptr, nullptr);
    if (s) return s;
  }
  s = read_status(ctx);
  if (s && s != MK_ERR_NAN) return s;
  for (int b = 0; b < B; ++b) next_tok[b] = ctx->host_ctl->tok[b];
  return s;
}

mk_status mk_reset(mk_ctx* ctx) {
  if (!ctx) return fail(MK_ERR_INVALID, "ctx is NULL");
  MK_CUDA(cudaStreamSynchronize(ctx->stream));
  for (auto& kv : ctx->scheds) {
    MK_CUDA(cudaMemset(kv.second->counters.p, 0, sizeof(uint32_t) * std::max(1, kv.second->plan.n_counters)));
    kv.second->epoch = 0;
  }
  MK_CUDA(cudaMemset(ctx->ctl.p, 0, sizeof(Ctl)));
  MK_CUDA(cudaMemset(ctx->argkeys.p, 0, sizeof(unsigned long long) * 2 * kMaxBatch));
  MK_CUDA(cudaMemset(ctx->act.p, 0xFF, sizeof(float) * 2 * ctx->st.act_floats));
  MK_CUDA(cudaDeviceSynchronize());
  ctx->step = 0;
  ctx->broken = false;
  memset(ctx->mail, 0, sizeof(HostMail));
  ctx->mail_seq = 0;
  return MK_OK;
}

mk_status mk_get_trace(mk_ctx* ctx, mk_trace_rec* recs, int max_records, int* n_records) {
  if (!ctx || !n_records) return fail(MK_ERR_INVALID, "NULL argument");
  *n_records = 0;
  if (!ctx->opts.trace || !ctx->trace.p) return fail(MK_ERR_INVALID, "context created without the trace option");
  MK_CUDA(cudaStreamSynchronize(ctx->stream));
  uint32_t n = 0;
  MK_CUDA(cudaMemcpy(&n, &reinterpret_cast<Ctl*>(ctx->ctl.p)->trace_n, 4, cudaMemcpyDeviceToHost));
  n = std::min<uint32_t>(n, (uint32_t)ctx->trace_cap);
  n = std::min<uint32_t>(n, (uint32_t)std::max(0, max_records));
  if (n && recs) {
    std::vector<TraceRec> tmp(n);
    MK_CUDA(cudaMemcpy(tmp.data(), ctx->trace.p, n * sizeof(TraceRec), cudaMemcpyDeviceToHost));
    for (uint32_t i = 0; i < n; ++i) {
      recs[i].cta = tmp[i].cta;
      recs[i].pc = tmp[i].pc;
      recs[i].op = tmp[i].op;
      recs[i].layer = tmp[i].layer;
      recs[i].t_fetch = tmp[i].t_fetch;
      recs[i].t_ready = tmp[i].t_ready;
      for (int k = 0; k < 6; ++k) recs[i].t_mark[k] = tmp[i].t_mark[k];
      recs[i].t_end = tmp[i].t_end;
    }
  }
  *n_records = (int)n;
  return MK_OK;
}

mk_status mk_read_activation(mk_ctx* ctx, int which, int layer, float* dst, size_t bytes) {
  if (!ctx || !dst) return fail(MK_ERR_INVALID, "NULL argument");
  const ModelShape& m = ctx->m;
  int kind, width, max_layer = m.L - 1;
  switch (which) {
    case 0: kind = ACT_H; width = m.d; max_layer = m.L; break;
    case 1: kind = ACT_HMID; width = m.d; break;
    case 2: kind = ACT_Q; width = m.Hq * m.hd; break;
    case 3: kind = ACT_O; width = m.Hq * m.hd; break;
    case 4: kind = ACT_A; width = m.F; break;
    default: return fail(MK_ERR_INVALID, "which must be 0..4");
  }
  if (layer < 0 || layer > max_layer) return fail(MK_ERR_INVALID, "layer out of range");
  const size_t need = sizeof(float) * (size_t)m.max_batch * width;
  if (bytes != need) return fail(MK_ERR_INVALID, "bytes must equal max_batch * width * 4");
  MK_CUDA(cudaStreamSynchronize(ctx->stream));
  const bool multi = ctx->opts.exec_mode != MK_EXEC_PERSISTENT;
  const int par = (ctx->opts.sync_mode == MK_SYNC_SENTINEL && !multi) ? (int)((ctx->step + 1u) & 1u) : 0;
  const float* src = ctx->st.act + (int64_t)par * ctx->st.act_floats + ctx->st.act_off[kind] +
                     (int64_t)layer * ctx->st.act_stride[kind];
  MK_CUDA(cudaMemcpy(dst, src, need, cudaMemcpyDeviceToHost));
  return MK_OK;
}

// ---------------------------------------------------------------- build-ladder self tests
mk_status mk_selftest(int kind, int64_t* result, int n) {
  if (!result || n < 4 || kind < 1 || kind > 4) return fail(MK_ERR_INVALID, "kind must be 1..4 and n >= 4");
  std::memset(result, 0, sizeof(int64_t) * n);
  int dev = 0, n_sm = 0;
  MK_CUDA(cudaGetDevice(&dev));
  MK_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  const void* fn = step_kernel_entry(MK_F16, MK_SYNC_COUNTER, false, 0);
  const int page = 16384, n_pages = 4;
  const int smem = n_pages * page + 0 + 256 + kCtlSmem;
  MK_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448));
  int bpsm = 0;
  MK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bpsm, fn, kThreads, smem));
  if (bpsm < 1) return fail(MK_ERR_OCCUPANCY, "self-test kernel does not fit");
  const int n_cta = n_sm;  // one CTA per SM: every pair of CTAs co-resident
  std::vector<std::vector<Instr>> qs(n_cta);
  auto I = [](int op, int wc, uint32_t wn, int sc) {
    Instr in{};
    in.op = (uint8_t)op;
    in.wait_ctr = wc;
    in.wait_n = wn;
    in.signal_ctr = sc;
    return in;
  };
  int n_ctr = 1;
  const int chunks = 3 * n_pages + 1;
  const int64_t words_per_page = page / 8;
  int64_t test_len = 0;
  std::vector<int64_t> init;
  switch (kind) {
    case 1:  // terminates
      for (int c = 0; c < n_cta; ++c) qs[c].push_back(I(OP_T_NOP, -1, 0, -1));
      test_len = 64;
      break;
    case 2:  // two opcodes interleaved; the per-CTA log must match queue order
      for (int c = 0; c < n_cta; ++c)
        for (int k = 0; k < 20; ++k) {
          Instr in = I(k % 3 == 2 ? OP_T_PRODUCE : OP_T_ORDER, -1, 0, -1);
          in.a[0] = n_cta * 64 + c * 32 + k;  // PRODUCE target slot
          in.a[1] = c * 1000 + k;
          qs[c].push_back(in);
        }
      test_len = (int64_t)n_cta * 96;
      break;
    case 3: {  // chain through every CTA, then a fan-in to CTA 0
      n_ctr = n_cta + 1;
      const int all = n_cta;
      {
        Instr p = I(OP_T_PRODUCE, -1, 0, 0);
        p.a[0] = 0;
        p.a[1] = 7;
        qs[0].push_back(p);
      }
      for (int c = 1; c < n_cta; ++c) {
        Instr in = I(OP_T_CONSUME, c - 1, 1, c);
        in.a[0] = c - 1;
        in.a[2] = c;
        qs[c].push_back(in);
        qs[c].push_back(I(OP_T_NOP, -1, 0, all));
      }
      Instr fin = I(OP_T_CONSUME, all, (uint32_t)(n_cta - 1), -1);
      fin.a[0] = n_cta - 1;
      fin.a[2] = n_cta;
      qs[0].push_back(fin);
      test_len = n_cta + 8;
      break;
    }
    case 4: {  // more pages than the pool holds, checksummed
      const int64_t res_base = (int64_t)n_cta * chunks * words_per_page;
      for (int c = 0; c < n_cta; ++c) {
        Instr in = I(OP_T_PAGES, -1, 0, -1);
        in.a[0] = c * chunks * (int)words_per_page;
        in.a[1] = chunks;
        in.a[2] = (int)(res_base + (int64_t)c * chunks);
        qs[c].push_back(in);
      }
      test_len = res_base + (int64_t)n_cta * chunks;
      init.resize(test_len, 0);
      uint64_t x = 0x9E3779B97F4A7C15ull;
      for (int64_t i = 0; i < res_base; ++i) {
        x ^= x << 13; x ^= x >> 7; x ^= x << 17;
        init[i] = (int64_t)x;
      }
      break;
    }
  }
  for (auto& q : qs) q.push_back(I(OP_END, -1, 0, -1));
  DevBuf ib, qb, ctr, tb, ctl;
  mk_status s = upload_queues(qs, ib, qb, nullptr);
  if (s) return s;
  MK_CUDA(cudaMalloc(&ctr.p, 4 * n_ctr));
  MK_CUDA(cudaMemset(ctr.p, 0, 4 * n_ctr));
  MK_CUDA(cudaMalloc(&tb.p, 8 * test_len));
  if (!init.empty())
    MK_CUDA(cudaMemcpy(tb.p, init.data(), 8 * test_len, cudaMemcpyHostToDevice));
  else
    MK_CUDA(cudaMemset(tb.p, 0, 8 * test_len));
  MK_CUDA(cudaMalloc(&ctl.p, sizeof(Ctl)));
  MK_CUDA(cudaMemset(ctl.p, 0, sizeof(Ctl)));
  DevState S{};
  S.counters = reinterpret_cast<uint32_t*>(ctr.p);
  S.n_counters = n_ctr;
  S.ctl = reinterpret_cast<Ctl*>(ctl.p);
  S.n_cta = n_cta;
  S.page_bytes = page;
  S.page_stride = page;
  S.n_pages = n_pages;
  S.xbuf_bytes = 0;
  S.scratch_bytes = 256;
  S.timeout_ns = 2000000000LL;
  S.backoff_max_ns = 256;
  S.test_buf = reinterpret_cast<int64_t*>(tb.p);
  S.test_len = test_len;
  S.max_batch = 1;
  S.Hq = S.Hkv = 1;
  S.hd = 64;
  S.d = 8;
  StepArgs A{};
  A.instr = reinterpret_cast<const Instr*>(ib.p);
  A.q_start = reinterpret_cast<const int32_t*>(qb.p);
  A.B = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[2] = {&S, &A};
  MK_CUDA(cudaLaunchKernelExC(&cfg, fn, args));
  MK_CUDA(cudaDeviceSynchronize());
  Ctl hc{};
  MK_CUDA(cudaMemcpy(&hc, ctl.p, sizeof(Ctl), cudaMemcpyDeviceToHost));
  std::vector<int64_t> out(test_len);
  MK_CUDA(cudaMemcpy(out.data(), tb.p, 8 * test_len, cudaMemcpyDeviceToHost));
  result[1] = n_cta;
  result[2] = hc.err.code;
  bool pass = hc.err.code == 0;
  switch (kind) {
    case 2:
      for (int c = 0; c < n_cta && pass; ++c) {
        int k_order = 0;
        for (int k = 0; k < 20; ++k) {
          if (k % 3 == 2) {
            pass &= out[(int64_t)n_cta * 64 + c * 32 + k] == c * 1000 + k;
          } else {
            pass &= out[(int64_t)c * 64 + 1 + k_order] == c * 1000 + k;
            ++k_order;
          }
        }
        pass &= out[(int64_t)c * 64] == k_order;
      }
      break;
    case 3:
      for (int c = 0; c < n_cta && pass; ++c) pass &= out[c] == 7 + c;
      pass &= out[n_cta] == 7 + n_cta;
      result[3] = out[n_cta];
      break;
    case 4: {
      const int64_t res_base = (int64_t)n_cta * chunks * words_per_page;
      int64_t bad = 0;
      for (int c = 0; c < n_cta; ++c)
        for (int k = 0; k < chunks; ++k) {
          uint64_t sum = 0;
          const int64_t base = ((int64_t)c * chunks + k) * words_per_page;
          for (int64_t i = 0; i < words_per_page; ++i) sum += (uint64_t)init[base + i];
          if ((uint64_t)out[res_base + (int64_t)c * chunks + k] != sum) ++bad;
        }
      result[3] = bad;
      pass &= bad == 0;
      break;
    }
    default:
      break;
  }
  result[0] = pass ? 1 : 0;
  return MK_OK;
}

mk_status mk_two_groups(const float* x, int n, int* group, float* threshold) {
  if (!x || !group || n < 2) return fail(MK_ERR_INVALID, "two groups: NULL argument or n < 2");
  double lo = x[0], hi = x[0];
  for (int i = 1; i < n; ++i) {
    lo = std::min(lo, (double)x[i]);
    hi = std::max(hi, (double)x[i]);
  }
  double thr = hi;  // all equal: one group
  if (hi > lo) {
    thr = 0.5 * (lo + hi);
    for (int it = 0; it < 100; ++it) {  // Lloyd's iterations in one dimension
      double s0 = 0, s1 = 0;
      int n0 = 0, n1 = 0;
      for (int i = 0; i < n; ++i) {
        if (x[i] <= thr) { s0 += x[i]; ++n0; } else { s1 += x[i]; ++n1; }
      }
      if (!n0 || !n1) break;
      const double t = 0.5 * (s0 / n0 + s1 / n1);
      if (t == thr) break;
      thr = t;
    }
  }
  for (int i = 0; i < n; ++i) group[i] = x[i] <= thr ? 0 : 1;
  if (threshold) *threshold = (float)thr;
  return MK_OK;
}

mk_status mk_die_map(int reps, int max_sm, int* die_of_sm, float* rtt_cycles, int* n_sm_out) {
  if (!die_of_sm || !n_sm_out || reps < 4) return fail(MK_ERR_INVALID, "die map: NULL argument or reps < 4");
  int dev = 0, n_sm = 0, smem_optin = 0;
  MK_CUDA(cudaGetDevice(&dev));
  MK_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  MK_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  *n_sm_out = n_sm;
  if (max_sm < n_sm) return fail(MK_ERR_INVALID, "die map: max_sm below the SM count");
  // more than half an SM's shared memory per CTA: exactly one CTA per SM
  const int smem = smem_optin / 2 + 1024;
  const void* fn = rtt_kernel_entry();
  MK_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  int bpsm = 0;
  MK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bpsm, fn, 32, smem));
  if (bpsm != 1) return fail(MK_ERR_OCCUPANCY, "die map: the probe does not run one CTA per SM");
  DevBuf words, smid, cyc, bad;
  MK_CUDA(cudaMalloc(&words.p, 256));  // turn word | ping, pong (two 128-byte lines)
  MK_CUDA(cudaMemset(words.p, 0, 256));
  MK_CUDA(cudaMalloc(&smid.p, sizeof(uint32_t) * n_sm));
  MK_CUDA(cudaMalloc(&cyc.p, sizeof(uint64_t) * n_sm));
  MK_CUDA(cudaMalloc(&bad.p, sizeof(uint32_t)));
  MK_CUDA(cudaMemset(bad.p, 0, sizeof(uint32_t)));
  uint32_t* w = reinterpret_cast<uint32_t*>(words.p);
  uint32_t* sp = reinterpret_cast<uint32_t*>(smid.p);
  uint64_t* cp = reinterpret_cast<uint64_t*>(cyc.p);
  uint32_t* bp = reinterpret_cast<uint32_t*>(bad.p);
  int64_t timeout = 2000000000LL;
  void* args[6] = {&w, &reps, &timeout, &sp, &cp, &bp};
  MK_CUDA(cudaLaunchCooperativeKernel(fn, dim3(n_sm), dim3(32), args, smem, nullptr));
  MK_CUDA(cudaDeviceSynchronize());
  std::vector<uint32_t> hs(n_sm);
  std::vector<uint64_t> hc(n_sm);
  uint32_t hb = 0;
  MK_CUDA(cudaMemcpy(hs.data(), smid.p, sizeof(uint32_t) * n_sm, cudaMemcpyDeviceToHost));
  MK_CUDA(cudaMemcpy(hc.data(), cyc.p, sizeof(uint64_t) * n_sm, cudaMemcpyDeviceToHost));
  MK_CUDA(cudaMemcpy(&hb, bad.p, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  if (hb) return fail(MK_ERR_TIMEOUT, "die map: a probe wait ran out");
  std::vector<float> rtt(n_sm);
  for (int i = 0; i < n_sm; ++i) {
    if (hs[i] >= (uint32_t)max_sm) return fail(MK_ERR_STATE, "die map: SM id out of range");
    rtt[i] = (float)hc[i];
  }
  // the reference SM itself: the smallest time measured, so it joins its own group
  float mn = 0.f;
  bool first = true;
  for (int i = 1; i < n_sm; ++i) {
    if (first || rtt[i] < mn) mn = rtt[i];
    first = false;
  }
  std::vector<float> x(rtt);
  x[0] = mn;
  std::vector<int> grp(n_sm);
  mk_status s = mk_two_groups(x.data(), n_sm, grp.data(), nullptr);
  if (s) return s;
  for (int i = 0; i < max_sm; ++i) {
    die_of_sm[i] = -1;
    if (rtt_cycles) rtt_cycles[i] = 0.f;
  }
  for (int i = 0; i < n_sm; ++i) {
    die_of_sm[hs[i]] = grp[i];
    if (rtt_cycles) rtt_cycles[hs[i]] = rtt[i];
  }
  return MK_OK;
}

mk_status mk_line_latency(long long buf_bytes, const int64_t* offsets, int n, int sm_a, int sm_b, int reps,
                          float* lat_a, float* lat_b) {
  if (!offsets || !lat_a || !lat_b || n < 1 || reps < 2 || buf_bytes < 4 || buf_bytes > (1LL << 34))
    return fail(MK_ERR_INVALID, "line latency: NULL argument or bad size");
  for (int i = 0; i < n; ++i)
    if (offsets[i] < 0 || offsets[i] > buf_bytes - 4 || (offsets[i] & 3))
      return fail(MK_ERR_INVALID, "line latency: an offset is outside the buffer or not 4-byte aligned");
  int dev = 0, n_sm = 0, smem_optin = 0;
  MK_CUDA(cudaGetDevice(&dev));
  MK_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  MK_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  if (sm_a < 0 || sm_b < 0 || sm_a >= n_sm || sm_b >= n_sm || sm_a == sm_b)
    return fail(MK_ERR_INVALID, "line latency: sm_a and sm_b must be two different SM ids");
  const int smem = smem_optin / 2 + 1024;  // exactly one CTA per SM, so both SMs run one
  const void* fn = line_lat_kernel_entry();
  MK_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  int bpsm = 0;
  MK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bpsm, fn, 32, smem));
  if (bpsm != 1) return fail(MK_ERR_OCCUPANCY, "line latency: the probe does not run one CTA per SM");
  DevBuf buf, offs, lat;
  MK_CUDA(cudaMalloc(&buf.p, (size_t)buf_bytes));
  MK_CUDA(cudaMemset(buf.p, 0, (size_t)buf_bytes));
  MK_CUDA(cudaMalloc(&offs.p, sizeof(long long) * n));
  MK_CUDA(cudaMemcpy(offs.p, offsets, sizeof(long long) * n, cudaMemcpyHostToDevice));
  MK_CUDA(cudaMalloc(&lat.p, sizeof(float) * 2 * n));
  MK_CUDA(cudaMemset(lat.p, 0xFF, sizeof(float) * 2 * n));  // NaN: not measured
  const uint32_t* bp = reinterpret_cast<const uint32_t*>(buf.p);
  const long long* op = reinterpret_cast<const long long*>(offs.p);
  float* lp = reinterpret_cast<float*>(lat.p);
  void* args[7] = {&bp, &op, &n, &sm_a, &sm_b, &reps, &lp};
  MK_CUDA(cudaLaunchCooperativeKernel(fn, dim3(n_sm), dim3(32), args, smem, nullptr));
  MK_CUDA(cudaDeviceSynchronize());
  MK_CUDA(cudaMemcpy(lat_a, lp, sizeof(float) * n, cudaMemcpyDeviceToHost));
  MK_CUDA(cudaMemcpy(lat_b, lp + n, sizeof(float) * n, cudaMemcpyDeviceToHost));
  return MK_OK;
}

mk_status mk_barrier_bench(int mode, int n_barriers, double* us_per_barrier) {
  if (!us_per_barrier || n_barriers < 1 || (mode != 0 && mode != 1))
    return fail(MK_ERR_INVALID, "mode must be 0/1, n_barriers >= 1");
  int dev = 0, n_sm = 0;
  MK_CUDA(cudaGetDevice(&dev));
  MK_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  DevBuf ctr, slots, out;
  MK_CUDA(cudaMalloc(&ctr.p, 4));
  MK_CUDA(cudaMemset(ctr.p, 0, 4));
  MK_CUDA(cudaMalloc(&slots.p, sizeof(float) * (size_t)n_barriers * n_sm));
  MK_CUDA(cudaMemset(slots.p, 0xFF, sizeof(float) * (size_t)n_barriers * n_sm));
  MK_CUDA(cudaMalloc(&out.p, 16));
  MK_CUDA(cudaMemset(out.p, 0, 16));
  uint32_t* c = reinterpret_cast<uint32_t*>(ctr.p);
  float* sl = reinterpret_cast<float*>(slots.p);
  int64_t timeout = 2000000000LL;
  uint64_t* o = reinterpret_cast<uint64_t*>(out.p);
  void* args[6] = {&c, &sl, &n_barriers, &mode, &timeout, &o};
  MK_CUDA(cudaLaunchCooperativeKernel(barrier_kernel_entry(), dim3(n_sm), dim3(256), args, 0, nullptr));
  MK_CUDA(cudaDeviceSynchronize());
  uint64_t h[2];
  MK_CUDA(cudaMemcpy(h, out.p, 16, cudaMemcpyDeviceToHost));
  if (h[1]) return fail(MK_ERR_TIMEOUT, "barrier benchmark timed out");
  *us_per_barrier = (double)h[0] / 1000.0 / n_barriers;
  return MK_OK;
}

mk_status mk_stream_bench(int page_bytes, int n_pages, int mode, int hint, long long total_bytes, double* gbps) {
  if (!gbps || page_bytes < 1024 || page_bytes > 65536 || (page_bytes & 15) || n_pages < 1 || n_pages > kMaxPages ||
      mode < 0 || mode > 5 || hint < 0 || hint > 3 || total_bytes < (1LL << 20) || (mode >= 2 && page_bytes != 32768))
    return fail(MK_ERR_INVALID, "stream bench: bad arguments");
  int dev = 0, n_sm = 0;
  MK_CUDA(cudaGetDevice(&dev));
  MK_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  const long long per_cta = total_bytes / n_sm / page_bytes * page_bytes;
  const int smem = n_pages * page_bytes + (page_bytes / 16) * 4;
  const void* fn = stream_kernel_entry();
  MK_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  DevBuf src, sink;
  const size_t src_bytes = (size_t)per_cta * ((hint & 2) ? 1 : n_sm);  // bit 1: one region read by all
  MK_CUDA(cudaMalloc(&src.p, src_bytes));
  MK_CUDA(cudaMemset(src.p, 0x3C, src_bytes));
  MK_CUDA(cudaMalloc(&sink.p, sizeof(float) * n_sm * kConsumerWarps));
  const uint8_t* sp = reinterpret_cast<const uint8_t*>(src.p);
  float* sk = reinterpret_cast<float*>(sink.p);
  long long pc = per_cta;
  void* args[7] = {&sp, &pc, &page_bytes, &n_pages, &mode, &hint, &sk};
  cudaEvent_t e0, e1;
  MK_CUDA(cudaEventCreate(&e0));
  MK_CUDA(cudaEventCreate(&e1));
  float best = 1e30f;
  for (int it = 0; it < 4; ++it) {
    MK_CUDA(cudaEventRecord(e0, nullptr));
    MK_CUDA(cudaLaunchKernel(fn, dim3(n_sm), dim3(kThreads), args, smem, nullptr));
    MK_CUDA(cudaEventRecord(e1, nullptr));
    MK_CUDA(cudaEventSynchronize(e1));
    float ms = 0.f;
    MK_CUDA(cudaEventElapsedTime(&ms, e0, e1));
    if (it > 0) best = std::min(best, ms);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  std::vector<float> hs(n_sm * kConsumerWarps);
  MK_CUDA(cudaMemcpy(hs.data(), sink.p, hs.size() * 4, cudaMemcpyDeviceToHost));
  for (float v : hs)
    if (std::isnan(v)) return fail(MK_ERR_TIMEOUT, "stream bench: a wait ran out");
  *gbps = (double)per_cta * n_sm / (best * 1e-3) / 1e9;
  return MK_OK;
}

}  // extern "C"
