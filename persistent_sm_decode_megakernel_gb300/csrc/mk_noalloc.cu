// mk_decode_step_noalloc: one decode step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside an allocator that must not
// re-enter it, plugins whose host process owns every device allocation and forbids
// their own, or a process whose memory is fully pre-reserved by another framework's
// caching allocator.  mk_create needs device memory for its queues, counters and
// activation buffers, so those callers get this entry point instead: every buffer the
// step needs beyond the caller's own inputs and outputs lives in one file-scope device
// array of kScratchBytes, which each GPU that loads the library holds until the process
// exits.  The step kernel is the same persistent kernel mk_decode_step launches (counter
// synchronisation, the same schedule builder); only where its scratch lives differs.
//
// Rules of use:
//   * The first call on a device (with that device current) looks up the array's device
//     address with cudaGetSymbolAddress.  Every call is synchronous: it waits for its
//     step and reads the status back with a device-to-host copy, so it cannot be
//     enqueued inside a stream capture.
//   * All calls share the one array and leave their contents in it; every call clears
//     what must start at zero (counters, error word, argmax keys).  Calls whose GPU work
//     overlaps (two streams, two host threads) race on the array: serialise them.
//   * The array holds the schedule, the counters, the activations of B sequences and one
//     RoPE row per sequence: its size depends on the model and the batch, not on the
//     positions.  Models whose needs exceed kScratchBytes are refused with MK_ERR_INVALID
//     and a message giving both sizes.
//   * The schedule of the last call on a device stays in the array: a call with the same
//     descriptor, weight and cache pointers and batch reuses it (no rebuild, no upload).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"
#include "mk_kernels.h"
#include "mk_plan.h"

namespace mk {
void set_last_error(const std::string& msg);  // defined beside mk_last_error
}

namespace {

constexpr size_t kScratchBytes = 16u << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the device symbol: its
// device address comes from cudaGetSymbolAddress below, never from taking its address.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// What the array of a device holds after a successful call: the schedule of `key`.
struct Prepared {
  bool valid = false;
  std::vector<uintptr_t> key;
  mk::DevState S{};
  int n_cta = 0, smem = 0, n_counters = 0;
  size_t o_ctl = 0, o_keys = 0, o_ctr = 0, o_rope = 0, o_q = 0, o_ins = 0;
};

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};
Prepared g_prep[kMaxDevices];

mk_status fail(mk_status s, const std::string& m) {
  mk::set_last_error(m);
  return s;
}

#define NA_CUDA(call)                                                                    \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) return fail(MK_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

mk_status scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(MK_ERR_INVALID, "device index out of range");
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return fail(MK_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    g_scratch_dev[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_dev[dev]);
  return MK_OK;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// everything the schedule and the device state of a call depend on
std::vector<uintptr_t> key_of(const mk_model_desc& d, const mk_weights* w, const mk_kv* kv, int B, int n_sm,
                              int smem_optin) {
  std::vector<uintptr_t> k;
  const int iv[] = {d.n_layers, d.d_model, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn_dim, d.vocab, d.dtype,
                    d.max_batch, d.max_ctx, B, n_sm, smem_optin};
  for (int v : iv) k.push_back((uintptr_t)(uint32_t)v);
  uint32_t fb[2];
  std::memcpy(&fb[0], &d.rms_eps, 4);
  std::memcpy(&fb[1], &d.rope_theta, 4);
  k.push_back(fb[0]);
  k.push_back(fb[1]);
  k.push_back((uintptr_t)w->embed);
  k.push_back((uintptr_t)w->final_norm);
  k.push_back((uintptr_t)w->lm_head);
  const void* const* tabs[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
  for (auto t : tabs)
    for (int l = 0; l < d.n_layers; ++l) k.push_back((uintptr_t)t[l]);
  for (int l = 0; l < d.n_layers; ++l) {
    k.push_back((uintptr_t)kv->k_cache[l]);
    k.push_back((uintptr_t)kv->v_cache[l]);
  }
  return k;
}

// Builds, validates and uploads the schedule of one call into the array (stream-ordered),
// and fills P with the device state that points into it.
mk_status prepare(const mk_model_desc& d, const mk_weights* w, const mk_kv* kv, int B, int n_sm, int smem_optin,
                  unsigned char* base, cudaStream_t s, Prepared* P) {
  using namespace mk;
  const ModelShape m = shape_of(&d);
  const int L = m.L;
  Geometry g;
  std::string e = make_geometry(m, n_sm, 0, 0, 0, smem_optin, &g);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  const void* fn = step_kernel_entry(m.dtype, MK_SYNC_COUNTER, false, g.instance());
  NA_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin));
  int bpsm = 0;
  NA_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bpsm, fn, kThreads, g.smem_bytes));
  if (bpsm < 1) return fail(MK_ERR_OCCUPANCY, "the kernel does not fit on an SM");
  const int n_cta = n_sm * bpsm;  // one wave, as for mk_create
  if (n_cta != n_sm) {
    e = make_geometry(m, n_cta, 0, 0, 0, smem_optin, &g);
    if (!e.empty()) return fail(MK_ERR_INVALID, e);
  }
  Plan plan;
  e = build_plan(m, g, n_cta, B, 0, choose_merge(m, g, B, true, 0), &plan);
  if (!e.empty()) return fail(MK_ERR_INVALID, "schedule: " + e);
  ModelPtrs mp;
  mp.final_norm = w->final_norm;
  mp.lm_head = w->lm_head;
  const void* const* tabs[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
  std::vector<const void*>* dst[9] = {&mp.attn_norm, &mp.wq, &mp.wk, &mp.wv, &mp.wo,
                                      &mp.mlp_norm, &mp.w_gate, &mp.w_up, &mp.w_down};
  for (int k = 0; k < 9; ++k) dst[k]->assign(tabs[k], tabs[k] + L);
  mp.kcache.assign(kv->k_cache, kv->k_cache + L);
  mp.vcache.assign(kv->v_cache, kv->v_cache + L);
  bake_pointers(m, mp, &plan);
  e = validate_plan(m, g, plan);
  if (!e.empty()) return fail(MK_ERR_INVALID, "schedule rejected by the validator: " + e);
  int nb = 1;
  while (nb < B) nb <<= 1;
  std::vector<TmapImage> maps;
  if (use_tc(g, nb)) {
    e = build_tc_maps(m, g, &plan, &maps);
    if (!e.empty()) return fail(MK_ERR_CUDA, "tensor maps: " + e);
  }
  e = build_kv_maps(m, g, m.max_batch, &plan, &maps);
  if (!e.empty()) return fail(MK_ERR_CUDA, "tensor maps: " + e);

  // host images of the read-only tables
  std::vector<Instr> flat;
  std::vector<int32_t> qoff;
  for (const auto& q : plan.queues) {
    qoff.push_back((int32_t)flat.size());
    flat.insert(flat.end(), q.begin(), q.end());
  }
  qoff.push_back((int32_t)flat.size());
  std::vector<const void*> ptrs;
  for (auto t : tabs)
    for (int l = 0; l < L; ++l) ptrs.push_back(t[l]);
  for (int l = 0; l < L; ++l) ptrs.push_back(kv->k_cache[l]);
  for (int l = 0; l < L; ++l) ptrs.push_back(kv->v_cache[l]);

  // activation arena (one set: counter synchronisation needs no second parity)
  DevState S{};
  arena_layout(m, g, B, &S);

  // carve the array
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur = up256(cur + bytes);
    return at;
  };
  P->o_ctl = take(sizeof(Ctl));
  P->o_keys = take(sizeof(unsigned long long) * 2 * kMaxBatch);
  P->o_ctr = take(sizeof(uint32_t) * (size_t)plan.n_counters);
  const size_t o_ptr = take(sizeof(void*) * ptrs.size());
  P->o_rope = take(sizeof(float2) * (size_t)kMaxBatch * (m.hd / 2));
  P->o_q = take(sizeof(int32_t) * qoff.size());
  P->o_ins = take(sizeof(Instr) * flat.size());
  const size_t o_maps = take(sizeof(TmapImage) * maps.size());
  const size_t o_act = take(sizeof(float) * (size_t)S.act_floats);
  if (cur > kScratchBytes) {
    char buf[200];
    snprintf(buf, sizeof buf, "this model and batch need %zu bytes of scratch; the no-alloc entry holds %zu", cur,
             kScratchBytes);
    return fail(MK_ERR_INVALID, buf);
  }
  NA_CUDA(cudaMemcpyAsync(base + o_ptr, ptrs.data(), sizeof(void*) * ptrs.size(), cudaMemcpyHostToDevice, s));
  NA_CUDA(cudaMemcpyAsync(base + P->o_q, qoff.data(), sizeof(int32_t) * qoff.size(), cudaMemcpyHostToDevice, s));
  if (!maps.empty()) {
    place_tc_maps(flat, reinterpret_cast<uintptr_t>(base + o_maps), use_tc(g, nb));
    NA_CUDA(cudaMemcpyAsync(base + o_maps, maps.data(), sizeof(TmapImage) * maps.size(), cudaMemcpyHostToDevice, s));
  }
  NA_CUDA(cudaMemcpyAsync(base + P->o_ins, flat.data(), sizeof(Instr) * flat.size(), cudaMemcpyHostToDevice, s));
  // the pageable copies above return once their source is consumed: the host vectors may go

  S.L = L; S.d = m.d; S.Hq = m.Hq; S.Hkv = m.Hkv; S.hd = m.hd; S.F = m.F; S.V = m.V; S.dtype = m.dtype;
  S.max_batch = B;  // the arena holds B rows
  S.max_ctx = m.max_ctx; S.S = g.S; S.eps = m.eps;
  S.ws_qkv = g.ws_qkv; S.ws_o = g.ws_o; S.ws_up = g.ws_up; S.ws_down = g.ws_down; S.ws_lm = g.ws_lm;
  S.embed = static_cast<const uint16_t*>(w->embed);
  S.final_norm = static_cast<const uint16_t*>(w->final_norm);
  S.lm_head = static_cast<const uint16_t*>(w->lm_head);
  auto pt = reinterpret_cast<const uint16_t* const*>(base + o_ptr);
  auto mpt = reinterpret_cast<uint16_t* const*>(base + o_ptr);
  S.attn_norm = pt; S.wq = pt + L; S.wk = pt + 2 * L; S.wv = pt + 3 * L; S.wo = pt + 4 * L;
  S.mlp_norm = pt + 5 * L; S.w_gate = pt + 6 * L; S.w_up = pt + 7 * L; S.w_down = pt + 8 * L;
  S.kcache = mpt + 9 * L;
  S.vcache = mpt + 10 * L;
  S.rope = reinterpret_cast<const float2*>(base + P->o_rope);
  S.rope_by_seq = 1;  // row b holds sequence b's position
  S.act = reinterpret_cast<float*>(base + o_act);
  S.argkeys = reinterpret_cast<unsigned long long*>(base + P->o_keys);
  S.counters = reinterpret_cast<uint32_t*>(base + P->o_ctr);
  S.n_counters = plan.n_counters;
  S.ctl = reinterpret_cast<Ctl*>(base + P->o_ctl);
  S.n_cta = n_cta;
  S.page_bytes = g.page_bytes;
  S.n_pages = g.n_pages;
  S.page_stride = g.page_stride;
  S.tc = g.tc;
  S.attn_mma = g.attn_mma;
  S.xbuf_bytes = g.xbuf_bytes;
  S.scratch_bytes = g.scratch_bytes;
  S.smem_bytes = g.smem_bytes;
  S.sync_mode = MK_SYNC_COUNTER;
  S.timeout_ns = 2000000000LL;
  S.backoff_max_ns = 256;
  S.split_min_positions = 16;
  S.inflight_pages = 2;
  P->S = S;
  P->n_cta = n_cta;
  P->smem = g.smem_bytes;
  P->n_counters = plan.n_counters;
  return MK_OK;
}

}  // namespace

extern "C" mk_status mk_decode_step_noalloc(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                                            const int32_t* in_tok, const int32_t* pos, int B, int32_t* out_tok,
                                            float* logits, void* stream) {
  using namespace mk;
  if (!in_tok || !pos || !out_tok) return fail(MK_ERR_INVALID, "NULL argument");
  std::string e = check_desc(desc);  // the same checks as mk_create
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  e = check_model_pointers(desc, w, kv);
  if (!e.empty()) return fail(MK_ERR_INVALID, e);
  const mk_model_desc& d = *desc;
  if (B < 1 || B > d.max_batch) return fail(MK_ERR_INVALID, "B out of range");
  if (d.head_dim != 64 && d.head_dim != 128) return fail(MK_ERR_INVALID, "head_dim must be 64 or 128");
  for (int b = 0; b < B; ++b) {
    if (in_tok[b] < 0 || in_tok[b] >= d.vocab) return fail(MK_ERR_INVALID, "token id out of range");
    if (pos[b] < 0 || pos[b] >= d.max_ctx) return fail(MK_ERR_INVALID, "position out of range");
  }
  int dev = 0, n_sm = 0, smem_optin = 0;
  NA_CUDA(cudaGetDevice(&dev));
  NA_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  NA_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lk(g_mu);
  unsigned char* base = nullptr;
  mk_status st = scratch_address(dev, &base);
  if (st) return st;
  Prepared& P = g_prep[dev];
  std::vector<uintptr_t> key = key_of(d, w, kv, B, n_sm, smem_optin);
  if (!P.valid || P.key != key) {
    P.valid = false;  // the array's schedule is about to change
    st = prepare(d, w, kv, B, n_sm, smem_optin, base, s, &P);
    if (st) return st;
    P.key = std::move(key);
  }
  const int half = d.head_dim / 2;
  float2 rope[kMaxBatch * 64];  // one RoPE row per sequence: angle pos[b] * theta^(-2i/hd), in double
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < half; ++i) {
      const double a = (double)pos[b] * std::pow((double)d.rope_theta, -2.0 * i / d.head_dim);
      rope[b * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  // this call's inputs (the array still holds the previous call's contents)
  NA_CUDA(cudaMemsetAsync(base + P.o_ctl, 0, sizeof(Ctl), s));
  NA_CUDA(cudaMemsetAsync(base + P.o_keys, 0, sizeof(unsigned long long) * 2 * kMaxBatch, s));
  NA_CUDA(cudaMemsetAsync(base + P.o_ctr, 0, sizeof(uint32_t) * (size_t)P.n_counters, s));
  NA_CUDA(cudaMemcpyAsync(base + P.o_rope, rope, sizeof(float2) * (size_t)B * half, cudaMemcpyHostToDevice, s));

  StepArgs A{};
  A.instr = reinterpret_cast<const Instr*>(base + P.o_ins);
  A.q_start = reinterpret_cast<const int32_t*>(base + P.o_q);
  A.epoch = 0;
  A.step = 0;
  A.B = B;
  A.flags = SF_RESET_ARGMAX;
  for (int b = 0; b < B; ++b) {
    A.tok[b] = in_tok[b];
    A.pos[b] = pos[b];
    A.seq[b] = b;       // row b is sequence b
    A.p0[b] = pos[b];   // one new position per row
  }
  A.logits = logits;
  A.tok_hist = nullptr;
  DevState S = P.S;
  const void* fn = step_kernel_entry(d.dtype, MK_SYNC_COUNTER, false, S.tc ? 2 : (S.attn_mma ? 1 : 0));
  NA_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(P.n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[2] = {&S, &A};
  NA_CUDA(cudaLaunchKernelExC(&cfg, fn, args));
  Ctl hc;
  NA_CUDA(cudaMemcpyAsync(&hc, base + P.o_ctl, sizeof(Ctl), cudaMemcpyDeviceToHost, s));
  NA_CUDA(cudaStreamSynchronize(s));
  P.valid = true;
  if (hc.err.code) {
    char buf[160];
    snprintf(buf, sizeof buf, "device error %u at cta %d pc %d counter %d", hc.err.code, hc.err.cta, hc.err.pc,
             hc.err.ctr);
    return fail((mk_status)hc.err.code, buf);
  }
  for (int b = 0; b < B; ++b) out_tok[b] = hc.tok[b];
  if (hc.nan_seen) return fail(MK_ERR_NAN, "a logit was NaN");
  return MK_OK;
}
