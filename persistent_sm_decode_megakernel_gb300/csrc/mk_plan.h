// Host-side schedule: per-CTA instruction queues, counter wiring, tile geometry, and the
// static validator that certifies a schedule before it is ever launched
// ("8 · Écrire son megakernel", §8.7, static verification: no deadlock, no race).
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"

namespace mk {

struct ModelShape {
  int L, d, Hq, Hkv, hd, F, V, dtype, max_batch, max_ctx;
  float eps, theta;
};

// tile and shared-memory geometry shared by every schedule of a context
struct Geometry {
  int page_bytes = 16384;
  int n_pages = 0;
  int nb_max = 1;        // batch padded to a power of two (register tiles)
  int xbuf_bytes = 0;
  int scratch_bytes = 0;
  int smem_bytes = 0;
  int ws_qkv = 0, ws_o = 0, ws_up = 0, ws_down = 0, ws_lm = 0;
  int S = 1;             // kv splits per (sequence, kv head)
  int tc = 0;            // max_batch >= 3: batches of 3..16 run the tensor-core GEMV
  int page_stride = 0;   // bytes between ring slots
  int attn_mma = 0;      // split-KV units of at least half a page run on tensor cores
  // the kernel instance: 2 with the tensor-core GEMV and attention, 1 with the tensor-core
  // attention alone, 0 with neither
  int instance() const { return tc ? 2 : (attn_mma ? 1 : 0); }
};
// a GEMV of batch nb uses the tensor-core path
inline bool use_tc(const Geometry& g, int nb) { return g.tc && nb >= 4; }

struct Plan {
  int n_cta = 0;
  int B = 1;
  std::vector<std::vector<Instr>> queues;  // per CTA, END-terminated
  std::vector<uint32_t> signals;          // per counter: signals per step
  int n_counters = 0;
  // multi-launch control: phases in dependency order; per phase the compacted queues
  std::vector<std::vector<std::vector<Instr>>> phase_queues;
  int64_t weight_bytes = 0;               // streamed weight bytes per step
  int merge = MERGE_OP;                   // MergeMode of the KV-split partials
  // dynamic attention (attn_pool): each layer's ATTENTION units, in claim order (split-major),
  // layer after layer; the queues hold one OP_ATTN_POOL per layer whose a0 indexes this array
  std::vector<Instr> pool;
};

// device addresses the host writes into the instructions (see the layout in mk_internal.h)
struct ModelPtrs {
  const void* final_norm = nullptr;
  const void* lm_head = nullptr;
  std::vector<const void*> attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down, kcache, vcache;
};

// The checks every entry point that takes a model descriptor applies (mk_create, mk_plan and
// the allocation-free step): "" when the descriptor is usable, else the reason.
std::string check_desc(const mk_model_desc* d);
// weights and KV tables: every pointer present and 16-byte aligned (bulk copies need it)
std::string check_model_pointers(const mk_model_desc* d, const mk_weights* w, const mk_kv* kv);
ModelShape shape_of(const mk_model_desc* d);

// activation arena of `rows` rows: fills S->act_off, act_stride and act_floats (one parity)
void arena_layout(const ModelShape& m, const Geometry& g, int rows, DevState* S);

// returns "" on success, else a message
// KV capacity from which batch-1..2 contexts take the tensor-core attention (and the kernel
// variant with it: at short positions that variant measured ~3.7 % slower than the one without)
constexpr int kAttnMmaMinCtx = 8192;
// attn_tc: the tensor-core attention -- 0 where it pays (contexts of max_batch >= 3 or of
// KV capacity >= kAttnMmaMinCtx), 1 in every context, -1 never (mk_options.attn_tensor_cores)
std::string make_geometry(const ModelShape& m, int n_cta, int page_bytes, int n_pages_req, int kv_splits,
                          int smem_limit, Geometry* g, int attn_tc = 0);
// attn_pool: ATTENTION units claimed at run time from a per-layer pool instead of dealt to
// the CTAs' queues (persistent control only: the multi-launch phases keep static units)
std::string build_plan(const ModelShape& m, const Geometry& g, int n_cta, int B, int drop_signal, int merge,
                       Plan* p, bool attn_pool = false);
// the merge a schedule of batch B uses: `requested` 1 or 2 (mk_options.attn_merge), or 0 =
// in the O-proj staging while one step's partials stay under kMergeInBytes, else the
// separate step of the sync mode
constexpr long long kMergeInBytes = 24 * 1024;
int choose_merge(const ModelShape& m, const Geometry& g, int B, bool counters, int requested);
void bake_pointers(const ModelShape& m, const ModelPtrs& w, Plan* p);

// Tensor-core schedules land each weight page with one tensor-map copy.  build_tc_maps
// encodes one map per weight segment of every GEMV instruction (segments with the same
// rows share one) and leaves the map's index + 1 in the instruction's p4 / p5 (0: none);
// place_tc_maps then turns the indices into the device addresses of the uploaded maps.
// Call after bake_pointers (the maps are made from the baked row pointers).
struct TmapImage {
  alignas(64) unsigned char bytes[128];
};
std::string build_tc_maps(const ModelShape& m, const Geometry& g, Plan* p, std::vector<TmapImage>* maps);
// The tensor-core attention's K and V pages: per layer one map of the key cache and, right
// after it, one of the value cache, over [64-element half rows, positions, halves, cache
// sequences x kv heads] (128-byte swizzled boxes of a page's positions); each ATTENTION
// instruction (queued or pooled) gets the key map's index + 1 in p3.  cache_batch: the
// caches' sequence extent.  Appends to maps.
std::string build_kv_maps(const ModelShape& m, const Geometry& g, int cache_batch, Plan* p,
                          std::vector<TmapImage>* maps);
// gemv_maps: build_tc_maps ran (else the GEMV instructions keep their row pointers)
void place_tc_maps(std::vector<Instr>& q, uintptr_t maps_dev, bool gemv_maps);
std::string validate_plan(const ModelShape& m, const Geometry& g, const Plan& p);

}  // namespace mk
