// Schedule builder and static validator (host only, no CUDA).
//
// The builder turns one decode step into per-CTA instruction queues (§8.2 "liste plate,
// par SM"): every op of every layer is cut into units balanced over all CTAs by streamed
// bytes, each CTA's queue lists its units in layer order, and each op's units signal one
// counter that the next op's units wait for in full.
//
// The validator certifies a schedule before it is uploaded (§8.7, static verification):
// it simulates the queues with counter semantics (every queue must run to its end: no
// deadlock), checks that every counter's per-step signal count equals what each waiter
// expects, that every buffer an instruction reads was fully written by instructions that
// happen before it (no race), that every output element is written exactly once, and
// that no instruction exceeds the shared-memory scratch it is given.
#include "mk_plan.h"

#include <algorithm>
#include <cstdio>
#include <numeric>

namespace mk {

static int pow2_at_least(int b) {
  int n = 1;
  while (n < b) n <<= 1;
  return n;
}

// largest divisor of K that is a multiple of 8 elements (16 bytes) and at most max_ws
static int slice_width(int K, int max_ws) {
  int best = 0;
  for (int w = 8; w <= std::min(K, max_ws); w += 8)
    if (K % w == 0) best = w;
  return best;
}

static std::string fmt(const char* f, long long a = 0, long long b = 0, long long c = 0) {
  char buf[256];
  snprintf(buf, sizeof buf, f, a, b, c);
  return buf;
}

std::string check_desc(const mk_model_desc* d) {
  if (!d) return "desc is NULL";
  if (d->n_layers < 1 || d->d_model < 8 || d->n_heads < 1 || d->n_kv_heads < 1 || d->head_dim < 8 ||
      d->ffn_dim < 8 || d->vocab < 2)
    return "descriptor dimensions must be positive";
  if (d->n_heads % d->n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (d->dtype != MK_F16 && d->dtype != MK_BF16) return "dtype must be MK_F16 or MK_BF16";
  if (d->max_batch < 1 || d->max_batch > kMaxBatch) return "max_batch must be in [1, 16]";
  if (d->max_ctx < 1 || d->max_ctx > (1 << 22)) return "max_ctx must be in [1, 4194304]";
  if (!(d->rms_eps > 0.f) || !(d->rope_theta > 0.f)) return "rms_eps and rope_theta must be positive";
  if (d->d_model % 8 || d->ffn_dim % 8) return "d_model and ffn_dim must be multiples of 8";
  return "";
}

static bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

std::string check_model_pointers(const mk_model_desc* d, const mk_weights* w, const mk_kv* kv) {
  if (!w || !kv) return "weights or kv is NULL";
  if (!aligned16(w->embed) || !aligned16(w->final_norm) || !aligned16(w->lm_head))
    return "embed/final_norm/lm_head must be non-NULL and 16-byte aligned";
  const void* const* tabs[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
  for (auto t : tabs) {
    if (!t) return "a per-layer weight table is NULL";
    for (int l = 0; l < d->n_layers; ++l)
      if (!aligned16(t[l])) return "per-layer weight pointers must be 16-byte aligned";
  }
  if (!kv->k_cache || !kv->v_cache) return "kv tables are NULL";
  for (int l = 0; l < d->n_layers; ++l)
    if (!aligned16(kv->k_cache[l]) || !aligned16(kv->v_cache[l]))
      return "KV-cache pointers must be non-NULL and 16-byte aligned";
  return "";
}

ModelShape shape_of(const mk_model_desc* d) {
  ModelShape m;
  m.L = d->n_layers;
  m.d = d->d_model;
  m.Hq = d->n_heads;
  m.Hkv = d->n_kv_heads;
  m.hd = d->head_dim;
  m.F = d->ffn_dim;
  m.V = d->vocab;
  m.dtype = d->dtype;
  m.max_batch = d->max_batch;
  m.max_ctx = d->max_ctx;
  m.eps = d->rms_eps;
  m.theta = d->rope_theta;
  return m;
}

std::string make_geometry(const ModelShape& m, int n_cta, int page_bytes, int n_pages_req, int kv_splits,
                          int smem_limit, Geometry* g, int attn_tc) {
  *g = Geometry();
  const int G = m.Hq / m.Hkv;
  if (m.hd != 64 && m.hd != 128) return "head_dim must be 64 or 128";
  if (G != 1 && G != 2 && G != 4) return "n_heads / n_kv_heads must be 1, 2 or 4";
  g->page_bytes = page_bytes > 0 ? page_bytes : 32768;
  if ((g->page_bytes & (g->page_bytes - 1)) || g->page_bytes < 4096 || g->page_bytes > 32768)
    return "page_bytes must be a power of two in [4096, 32768]";
  if (g->page_bytes < 64 * m.hd) return fmt("page_bytes must be at least 64 * head_dim = %lld", 64LL * m.hd);
  g->nb_max = pow2_at_least(m.max_batch);
  g->tc = m.max_batch >= 3 ? 1 : 0;  // batches of 3..16 run the tensor-core GEMV
  // tensor-core attention (a K or V page is one box of page_bytes / (2 hd) positions) in the
  // instance with the tensor-core code: contexts of batches of 3 and more, or of long
  // capacity (there its units grow long enough to pay; short ones keep the instance without
  // it, whose smaller code measured faster at batch 1)
  const bool want = attn_tc > 0 || (attn_tc == 0 && (g->tc || m.max_ctx >= kAttnMmaMinCtx));
  g->attn_mma = g->page_bytes == 32768 && want ? 1 : 0;
  g->page_stride = g->page_bytes;
  if (g->tc) {
    if (g->page_bytes != 32768) return "batches of 3 and more need 32 KB pages";
    if (m.d % kTcChunkCols || m.F % kTcChunkCols || (m.Hq * m.hd) % kTcChunkCols)
      return "batches of 3 and more need d_model, ffn_dim and n_heads*head_dim to be multiples of 64";
    g->page_stride = kTcPageBytes;
  }
  const int max_ws = g->page_bytes / (2 * kConsumerWarps);
  g->ws_qkv = slice_width(m.d, max_ws);
  g->ws_up = g->ws_qkv;
  g->ws_lm = g->ws_qkv;
  g->ws_o = slice_width(m.Hq * m.hd, max_ws);
  g->ws_down = slice_width(m.F, max_ws);
  if (!g->ws_qkv || !g->ws_o || !g->ws_down) return "d_model, n_heads*head_dim and ffn_dim must be multiples of 8";
  const int kmax = std::max(m.d, std::max(m.Hq * m.hd, m.F));
  // x buffer: a batch of GEMV inputs, or q of one GQA group plus the new key/value; with
  // the tensor-core path, batches of 1..2 inputs or one window of 16 sequences' hi/lo halves
  // (a prompt chunk's attention stages q and up to kMaxBatch new key/value rows: tc only)
  const int xfloats = g->tc ? std::max(std::max(2 * kmax, kMaxBatch * std::min(kTcKw, kmax)), (G + kMaxBatch) * m.hd)
                            : std::max(g->nb_max * kmax, (G + 1) * m.hd);
  g->xbuf_bytes = ((xfloats * 4 + 127) / 128) * 128;
  // the tensor-core attention's query fragments and two 16-row pages of new keys / values
  const int attn_x = (m.hd / 16) * 32 * 16 + 2 * (m.hd / 64) * 16 * 128;
  if (g->attn_mma) g->xbuf_bytes = std::max(g->xbuf_bytes, ((attn_x + 127) / 128) * 128);
  if (kv_splits > 0) {
    g->S = kv_splits;
  } else {
    g->S = n_cta / std::gcd(n_cta, m.Hkv);
    if (g->S > 64) g->S = std::max(1, n_cta / m.Hkv);
  }
  if (g->S < 1 || g->S > 256) return "kv_splits out of range [1, 256]";
  int scratch = g->tc ? kTcPartialFloats * 4 + 8192 : 16384;
  scratch = std::max(scratch, kConsumerWarps * G * (m.hd + kPartExtra) * 4);
  scratch = std::max(scratch, g->S * G * 2 * 4);
  g->scratch_bytes = ((scratch + 127) / 128) * 128;
  const int avail = smem_limit - g->xbuf_bytes - g->scratch_bytes - kCtlSmem;
  int np = avail > 0 ? avail / g->page_stride : 0;
  np = std::min(np, kMaxPages);
  if (n_pages_req > 0) np = std::min(np, n_pages_req);
  if (np < 2)
    return fmt("shared memory too small: x buffer %lld B + scratch %lld B leave %lld pages (max_batch too large)",
               g->xbuf_bytes, g->scratch_bytes, np);
  g->n_pages = np;
  g->smem_bytes = np * g->page_stride + g->xbuf_bytes + g->scratch_bytes + kCtlSmem;
  return "";
}

void arena_layout(const ModelShape& m, const Geometry& g, int rows, DevState* S) {
  const int G = m.Hq / m.Hkv;
  const long long R = rows;
  long long sizes[ACT_NUM], layers[ACT_NUM];
  sizes[ACT_H] = R * m.d; layers[ACT_H] = m.L + 1;
  sizes[ACT_HMID] = R * m.d; layers[ACT_HMID] = m.L;
  sizes[ACT_Q] = R * m.Hq * m.hd; layers[ACT_Q] = m.L;
  sizes[ACT_KVN] = R * 2 * m.Hkv * m.hd; layers[ACT_KVN] = m.L;
  sizes[ACT_PART] = R * m.Hkv * (long long)g.S * G * (m.hd + kPartExtra); layers[ACT_PART] = m.L;
  sizes[ACT_O] = R * m.Hq * m.hd; layers[ACT_O] = m.L;
  sizes[ACT_A] = R * m.F; layers[ACT_A] = m.L;
  // fragment forms: the tensor-core GEMV's batch tile (8 or 16 sequences) x width, as
  // hi/lo 16-bit halves (one float's worth per element)
  const long long FR = g.tc ? (rows > 8 ? 16 : 8) : 0;
  sizes[ACT_HF] = FR * m.d; layers[ACT_HF] = m.L + 1;
  sizes[ACT_HMF] = FR * m.d; layers[ACT_HMF] = m.L;
  sizes[ACT_AF] = FR * m.F; layers[ACT_AF] = m.L;
  sizes[ACT_OF] = FR * m.Hq * m.hd; layers[ACT_OF] = m.L;
  const long long SS = g.tc ? (long long)kMaxSsqSlots * kMaxBatch : 0;
  sizes[ACT_SSH] = SS; layers[ACT_SSH] = m.L + 1;
  sizes[ACT_SSM] = SS; layers[ACT_SSM] = m.L;
  long long off = 0;
  for (int k = 0; k < ACT_NUM; ++k) {
    const long long stride = (sizes[k] + 31) / 32 * 32;
    S->act_off[k] = off;
    S->act_stride[k] = stride;
    off += stride * layers[k];
  }
  S->act_floats = (off + 31) / 32 * 32;
}

static inline int split_lo(long long total, int parts, int i) { return (int)(total * i / parts); }

static Instr mk_instr(int op, int layer, int wait_ctr, uint32_t wait_n, int signal_ctr) {
  Instr in{};
  in.op = (uint8_t)op;
  in.layer = (uint16_t)layer;
  in.wait_ctr = wait_ctr;
  in.wait_n = wait_n;
  in.signal_ctr = signal_ctr;
  return in;
}

int choose_merge(const ModelShape& m, const Geometry& g, int B, bool counters, int requested) {
  const int G = m.Hq / m.Hkv;
  const long long part_bytes = 4LL * B * m.Hkv * g.S * G * (m.hd + kPartExtra);
  const long long weight_floats = 3LL * B * m.Hkv * g.S * G;  // (max, sum) pairs + merge weights
  const bool fits = part_bytes <= kMergeInBytes && weight_floats * 4 <= g.scratch_bytes;
  const bool tc = use_tc(g, pow2_at_least(B));  // the tensor-core GEMV stages its own input layout
  if (requested == 3) return MERGE_LAST_ARRIVER;
  if (!tc && (requested == 2 || (requested == 0 && fits))) return MERGE_IN_OPROJ;
  return counters ? MERGE_LAST_ARRIVER : MERGE_OP;
}

std::string build_plan(const ModelShape& m, const Geometry& g, int n_cta, int B, int drop_signal, int merge,
                       Plan* p, bool attn_pool) {
  if (B < 1 || B > m.max_batch) return "batch out of range";
  *p = Plan();
  p->merge = merge;
  const bool fuse_reduce = merge == MERGE_LAST_ARRIVER;
  p->n_cta = n_cta;
  p->B = B;
  p->queues.assign(n_cta, {});
  const int nb = pow2_at_least(B);
  const int scratch_floats = g.scratch_bytes / 4;
  const int half = m.hd / 2;
  const int G = m.Hq / m.Hkv;
  auto rows_cap = [&](int K, int ws, int segs) {  // rows per GEMV instruction (rowpart scratch)
    if (use_tc(g, nb)) return std::max(1, (scratch_floats - kTcPartialFloats) / (nb * segs));
    const int spr = K / ws;
    return std::max(1, scratch_floats / (spr * nb * segs));
  };
  auto new_ctr = [&]() {
    p->signals.push_back(0);
    return (int)p->signals.size() - 1;
  };
  // pending instructions: collected first, then the wait counts are filled in
  struct Pending {
    int cta;
    Instr in;
  };
  std::vector<Pending> all;
  auto emit = [&](int cta, const Instr& in) {
    all.push_back({cta, in});
    if (in.signal_ctr >= 0) p->signals[in.signal_ctr]++;
  };

  // EMBED
  const int c_emb = new_ctr();
  for (int c = 0; c < n_cta; ++c) {
    const int e0 = split_lo((long long)B * m.d, n_cta, c), e1 = split_lo((long long)B * m.d, n_cta, c + 1);
    if (e1 <= e0) continue;
    Instr in = mk_instr(OP_EMBED, 0, -1, 0, c_emb);
    in.a[0] = e0;
    in.a[1] = e1;
    emit(c, in);
  }
  int prev = c_emb;
  for (int l = 0; l < m.L; ++l) {
    // RMSNORM_QKV_ROPE: rotate-half pairs (i, i + hd/2) stay in one instruction
    const int c_qkv = new_ctr();
    {
      const int heads = m.Hq + 2 * m.Hkv;
      const long long pairs = (long long)heads * half;
      const int cap = std::max(1, rows_cap(m.d, g.ws_qkv, 1) / 2);
      auto emit_qkv = [&](int c, int hh, int i0, int n) {
        Instr in = mk_instr(OP_QKV, l, prev, 0, c_qkv);
        in.a[0] = hh < m.Hq ? 0 : (hh < m.Hq + m.Hkv ? 1 : 2);
        in.a[1] = hh < m.Hq ? hh : (hh < m.Hq + m.Hkv ? hh - m.Hq : hh - m.Hq - m.Hkv);
        in.a[2] = i0;
        in.a[3] = n;
        emit(c, in);
      };
      if (n_cta >= heads) {
        // each head to its own group of CTAs: every CTA gets exactly one instruction (a
        // pair range crossing a head would cost a second one, with its own staging)
        for (int hh = 0; hh < heads; ++hh) {
          const int c0 = split_lo(n_cta, heads, hh), c1 = split_lo(n_cta, heads, hh + 1);
          for (int c = c0; c < c1; ++c) {
            int i0 = split_lo(half, c1 - c0, c - c0);
            const int i1 = split_lo(half, c1 - c0, c - c0 + 1);
            while (i0 < i1) {
              const int n = std::min(i1 - i0, cap);
              emit_qkv(c, hh, i0, n);
              i0 += n;
            }
          }
        }
      } else {
        for (int c = 0; c < n_cta; ++c) {
          long long p0 = split_lo(pairs, n_cta, c);
          const long long p1 = split_lo(pairs, n_cta, c + 1);
          while (p0 < p1) {
            const int hh = (int)(p0 / half);
            const long long seg_end = std::min<long long>(p1, (long long)(hh + 1) * half);
            const int n = (int)std::min<long long>(seg_end - p0, cap);
            emit_qkv(c, hh, (int)(p0 % half), n);
            p0 += n;
          }
        }
      }
    }
    // ATTENTION: B * Hkv * S split units, dealt round-robin with the split index varying
    // slowest, so that the units of the splits a step actually uses (s below its active
    // count, which shrinks with the batch and the context) land on distinct CTAs.  Fused:
    // each unit counts its arrival on the (b, j) counter; the last of the S merges the
    // splits and signals c_red (one signal per (b, j) and step).  Merged in the O-proj
    // staging: every unit signals c_att, which the O-proj units wait for.
    const int c_att = new_ctr();
    const int c_red = new_ctr();
    {
      const int nbj = B * m.Hkv, nu = nbj * g.S;
      std::vector<int> arr;
      if (fuse_reduce)
        for (int k = 0; k < nbj; ++k) arr.push_back(new_ctr());
      const int pool0 = (int)p->pool.size();
      for (int u = 0; u < nu; ++u) {
        const int bj = u % nbj, sp = u / nbj;
        Instr in = mk_instr(OP_ATTN, l, c_qkv, 0, fuse_reduce ? c_red : c_att);
        in.a[0] = bj / m.Hkv;
        in.a[1] = bj % m.Hkv;
        in.a[2] = sp;
        in.a[3] = g.S;
        in.a[4] = fuse_reduce ? arr[bj] : -1;
        if (attn_pool) {
          p->pool.push_back(in);  // claimed at run time; its signal is counted below
          p->signals[in.signal_ctr]++;
        } else {
          emit(u % n_cta, in);
        }
      }
      if (attn_pool) {  // one claim loop per CTA and layer
        const int c_claim = new_ctr();
        for (int c = 0; c < n_cta; ++c) {
          Instr in = mk_instr(OP_ATTN_POOL, l, c_qkv, 0, -1);
          in.a[0] = pool0;
          in.a[1] = nu;
          in.a[2] = c_claim;
          in.a[3] = n_cta;
          emit(c, in);
        }
      }
      if (fuse_reduce) {
        p->signals[c_red] = (uint32_t)(B * m.Hkv);
        for (int k : arr) p->signals[k] = (uint32_t)g.S;  // arrivals (never waited on)
      }
    }
    // ATTN_REDUCE: one unit per (sequence, kv head), spread over the CTAs
    if (merge == MERGE_OP) {
      const int nu = B * m.Hkv;
      for (int u = 0; u < nu; ++u) {
        Instr in = mk_instr(OP_ATTN_REDUCE, l, c_att, 0, c_red);
        in.a[0] = u / m.Hkv;
        in.a[1] = u % m.Hkv;
        emit((int)((long long)u * n_cta / nu), in);
      }
    }
    // O_PROJ, MLP_UP_GATE, MLP_DOWN: row ranges
    auto rows_op = [&](int op, int rows, int K, int ws, int segs, int wait, int sig, uint8_t flags) {
      const int cap = rows_cap(K, ws, segs);
      for (int c = 0; c < n_cta; ++c) {
        int r0 = split_lo(rows, n_cta, c);
        const int r1 = split_lo(rows, n_cta, c + 1);
        while (r0 < r1) {
          const int n = std::min(r1 - r0, cap);
          Instr in = mk_instr(op, l, wait, 0, sig);
          in.flags = flags;
          in.a[0] = r0;
          in.a[1] = n;
          emit(c, in);
          r0 += n;
        }
      }
    };
    const int c_o = new_ctr();
    if (merge == MERGE_IN_OPROJ)
      rows_op(OP_OPROJ, m.d, m.Hq * m.hd, g.ws_o, 1, c_att, c_o, F_MERGE_IN);
    else
      rows_op(OP_OPROJ, m.d, m.Hq * m.hd, g.ws_o, 1, c_red, c_o, 0);
    const int c_ug = new_ctr();
    rows_op(OP_UPGATE, m.F, m.d, g.ws_up, 2, c_o, c_ug, 0);
    const int c_dn = new_ctr();
    rows_op(OP_DOWN, m.d, m.F, g.ws_down, 1, c_ug, c_dn, 0);
    prev = c_dn;
  }
  // LM_HEAD: vocabulary rows; the last chunk of each CTA publishes its argmax
  {
    const int c_lm = new_ctr();
    const int cap = rows_cap(m.d, g.ws_lm, 1);
    int n_lm = 0;
    for (int c = 0; c < n_cta; ++c)
      if (split_lo(m.V, n_cta, c + 1) > split_lo(m.V, n_cta, c)) ++n_lm;
    for (int c = 0; c < n_cta; ++c) {
      int r0 = split_lo(m.V, n_cta, c);
      const int r1 = split_lo(m.V, n_cta, c + 1);
      while (r0 < r1) {
        const int n = std::min(r1 - r0, cap);
        const bool last = r0 + n == r1;
        Instr in = mk_instr(OP_LMHEAD, m.L, prev, 0, last ? c_lm : -1);
        in.a[0] = r0;
        in.a[1] = n;
        if (last) {
          in.flags = F_LAST_LM;
          in.a[2] = n_lm;
        }
        emit(c, in);
        r0 += n;
      }
    }
  }
  p->n_counters = (int)p->signals.size();
  // wait counts = every signal of the awaited counter in one step
  for (auto& pe : all)
    if (pe.in.wait_ctr >= 0) pe.in.wait_n = p->signals[pe.in.wait_ctr];
  for (auto& in : p->pool)
    if (in.wait_ctr >= 0) in.wait_n = p->signals[in.wait_ctr];
  int sig_seen = 0;
  for (auto& pe : all) {
    // fault injection: the k-th signal is removed, its waiters keep expecting it
    const bool fused = pe.in.op == OP_ATTN && pe.in.a[4] >= 0;  // signals only if last: not a fixed signal
    if (drop_signal > 0 && pe.in.signal_ctr >= 0 && !(pe.in.flags & F_LAST_LM) && !fused &&
        ++sig_seen == drop_signal)
      pe.in.signal_ctr = -1;
    p->queues[pe.cta].push_back(pe.in);
  }
  for (auto& q : p->queues) q.push_back(mk_instr(OP_END, 0, -1, 0, -1));
  // a CTA's split-KV units of one layer sit together, in split order: each carries how many
  // units of the same run follow it (a5), so that a CTA meeting a split past every
  // sequence's active count skips the rest of the run in one step
  for (auto& q : p->queues)
    for (size_t i = 0; i < q.size(); ++i)
      if (q[i].op == OP_ATTN) {
        int n = 0;
        while (i + 1 + n < q.size() && q[i + 1 + n].op == OP_ATTN && q[i + 1 + n].layer == q[i].layer) ++n;
        q[i].a[5] = n;
      }
  // the tensor-core GEMV's RMSNorm inputs carry one sum-of-squares slot per CTA, written by
  // that CTA's EMBED, O-proj or DOWN instruction: each CTA must hold exactly one of each
  // (per layer)
  if (use_tc(g, nb)) {
    if (n_cta > kMaxSsqSlots) return fmt("the tensor-core GEMV runs on at most %lld CTAs", (long long)kMaxSsqSlots);
    for (int c = 0; c < n_cta; ++c) {
      std::vector<int> n_o(m.L, 0), n_dn(m.L, 0);
      int n_emb = 0;
      for (const auto& in : p->queues[c]) {
        if (in.op == OP_EMBED) ++n_emb;
        if (in.op == OP_OPROJ) ++n_o[in.layer];
        if (in.op == OP_DOWN) ++n_dn[in.layer];
      }
      bool ok = n_emb == 1;
      for (int l = 0; l < m.L; ++l) ok = ok && n_o[l] == 1 && n_dn[l] == 1;
      if (!ok)
        return fmt("cta %lld: the tensor-core GEMV needs one EMBED, O-proj and DOWN instruction per CTA and layer "
                   "(d_model too small for the CTA count?)",
                   (long long)c);
    }
  }

  // multi-launch control: one launch per (op, layer) in dependency order
  auto phase_of = [&](const Instr& in) -> int {
    if (in.op == OP_EMBED) return 0;
    if (in.op == OP_LMHEAD) return 1 + 6 * m.L;
    if (in.op == OP_ATTN_POOL) return 1 + 6 * in.layer + (OP_ATTN - OP_QKV);
    return 1 + 6 * in.layer + (in.op - OP_QKV);
  };
  const int n_phase = 2 + 6 * m.L;
  std::vector<std::vector<std::vector<Instr>>> phases(n_phase, std::vector<std::vector<Instr>>(n_cta));
  std::vector<int> used(n_phase, 0);
  for (int c = 0; c < n_cta; ++c)
    for (const auto& in : p->queues[c])
      if (in.op != OP_END) {
        phases[phase_of(in)][c].push_back(in);
        used[phase_of(in)] = 1;
      }
  for (int k = 0; k < n_phase; ++k) {  // phases with no work (the fused merge) launch nothing
    if (!used[k]) continue;
    for (auto& q : phases[k]) q.push_back(mk_instr(OP_END, 0, -1, 0, -1));
    p->phase_queues.push_back(std::move(phases[k]));
  }

  // streamed weight bytes of one step
  long long per_layer = (long long)(m.Hq + 2 * m.Hkv) * m.hd * m.d + (long long)m.d * m.Hq * m.hd +
                        3LL * m.d * m.F + 2LL * m.d;
  p->weight_bytes = 2 * ((long long)m.L * per_layer + (long long)m.V * m.d + m.d);
  (void)G;
  return "";
}

void bake_pointers(const ModelShape& m, const ModelPtrs& w, Plan* p) {
  auto at = [](const void* base, size_t elems) {
    return static_cast<const void*>(static_cast<const uint16_t*>(base) + elems);
  };
  auto bake = [&](Instr& in) {
    const int l = in.layer;
    switch (in.op) {
      case OP_QKV: {
        const int mat = in.a[0], head = in.a[1], i0 = in.a[2];
        const void* W = mat == 0 ? w.wq[l] : (mat == 1 ? w.wk[l] : w.wv[l]);
        const size_t ra = (size_t)head * m.hd + i0;
        set_ptr(in, kP2, w.attn_norm[l]);
        set_ptr(in, kP3, mat == 0 ? nullptr : (mat == 1 ? w.kcache[l] : w.vcache[l]));
        set_ptr(in, kP4, at(W, ra * m.d));
        set_ptr(in, kP5, at(W, (ra + m.hd / 2) * m.d));
        break;
      }
      case OP_ATTN: {
        const size_t base = ((size_t)in.a[0] * m.Hkv + in.a[1]) * m.max_ctx * m.hd;
        set_ptr(in, kP4, at(w.kcache[l], base));
        set_ptr(in, kP5, at(w.vcache[l], base));
        break;
      }
      case OP_OPROJ:
        set_ptr(in, kP2, w.mlp_norm[l]);  // the gain of h_mid's consumer (fragment form)
        set_ptr(in, kP4, at(w.wo[l], (size_t)in.a[0] * m.Hq * m.hd));
        break;
      case OP_EMBED: set_ptr(in, kP2, w.attn_norm[0]); break;
      case OP_UPGATE:
        set_ptr(in, kP2, w.mlp_norm[l]);
        set_ptr(in, kP4, at(w.w_gate[l], (size_t)in.a[0] * m.d));
        set_ptr(in, kP5, at(w.w_up[l], (size_t)in.a[0] * m.d));
        break;
      case OP_DOWN:
        set_ptr(in, kP2, l + 1 < m.L ? w.attn_norm[l + 1] : w.final_norm);  // the gain of h's next consumer
        set_ptr(in, kP4, at(w.w_down[l], (size_t)in.a[0] * m.F));
        break;
      case OP_LMHEAD:
        set_ptr(in, kP2, w.final_norm);
        set_ptr(in, kP4, at(w.lm_head, (size_t)in.a[0] * m.d));
        break;
      default: break;
    }
  };
  for (auto& q : p->queues)
    for (auto& in : q) bake(in);
  for (auto& in : p->pool) bake(in);
  for (auto& ph : p->phase_queues)
    for (auto& q : ph)
      for (auto& in : q) bake(in);
}

// ---------------------------------------------------------------- validator
namespace {
struct Bits {
  std::vector<uint64_t> w;
  explicit Bits(int n = 0) : w((n + 63) / 64, 0) {}
  void set(int i) { w[i >> 6] |= 1ull << (i & 63); }
  bool has(int i) const { return (w[i >> 6] >> (i & 63)) & 1; }
  void merge(const Bits& o) {
    for (size_t i = 0; i < w.size(); ++i) w[i] |= o.w[i];
  }
};
}  // namespace

std::string validate_plan(const ModelShape& m, const Geometry& g, const Plan& p) {
  const int n_cta = p.n_cta, B = p.B, half = m.hd / 2;
  const int nb = pow2_at_least(B);
  const int scratch_floats = g.scratch_bytes / 4;
  const int n_group = 2 + 6 * m.L;
  auto group_of = [&](const Instr& in) -> int {
    if (in.op == OP_EMBED) return 0;
    if (in.op == OP_LMHEAD) return 1 + 6 * m.L;
    if (in.op == OP_ATTN_POOL) return 1 + 6 * in.layer + (OP_ATTN - OP_QKV);
    return 1 + 6 * in.layer + (in.op - OP_QKV);
  };
  if ((int)p.queues.size() != n_cta) return "queue count != CTA count";
  // Attention pools: the units of a layer may run on any CTA, each exactly once, after its
  // claim loop's dependency.  For the checks below each pool is run whole by the first CTA
  // that reaches one of its claim loops (one admissible interleaving; a unit waits on
  // nothing but the QKV counter every claim loop also waits on, so any other assignment
  // is ordered the same way).
  std::vector<int> pool_layer(p.pool.size(), -1);
  for (int c = 0; c < n_cta; ++c)
    for (const auto& in : p.queues[c])
      if (in.op == OP_ATTN_POOL) {
        if (in.a[0] < 0 || in.a[1] < 1 || (size_t)in.a[0] + in.a[1] > p.pool.size() || in.a[3] != n_cta ||
            in.a[2] < 0 || in.a[2] >= p.n_counters)
          return fmt("cta %lld: bad attention pool arguments", c);
        for (int u = in.a[0]; u < in.a[0] + in.a[1]; ++u) {
          const Instr& un = p.pool[u];
          if (un.op != OP_ATTN || un.layer != in.layer || un.wait_ctr != in.wait_ctr)
            return "attention pool unit does not match its claim loop";
          if (pool_layer[u] >= 0 && pool_layer[u] != in.layer) return "attention pool ranges overlap";
          pool_layer[u] = in.layer;
        }
      }
  for (size_t u = 0; u < p.pool.size(); ++u)
    if (pool_layer[u] < 0) return "attention pool unit without a claim loop";

  // -- structure, argument ranges, scratch limits, signal counts
  std::vector<uint32_t> sig(p.n_counters, 0);
  std::vector<int> group_units(n_group, 0);
  for (int c = 0; c <= n_cta; ++c) {  // c == n_cta: the pooled units
    std::vector<Instr> pooled;
    if (c == n_cta) {
      pooled = p.pool;
      pooled.push_back(mk_instr(OP_END, 0, -1, 0, -1));
    }
    const auto& q = c < n_cta ? p.queues[c] : pooled;
    if (q.empty() || q.back().op != OP_END) return fmt("queue %lld does not end with OP_END", c);
    for (size_t k = 0; k + 1 < q.size(); ++k) {
      const Instr& in = q[k];
      if (in.op == OP_ATTN_POOL) {
        if (in.wait_ctr >= p.n_counters || in.signal_ctr != -1) return "bad attention pool counters";
        continue;
      }
      if (in.op < OP_EMBED || in.op > OP_LMHEAD) return fmt("cta %lld pc %lld: bad opcode %lld", c, k, in.op);
      if (in.op != OP_LMHEAD && in.layer >= m.L) return "layer out of range";
      if (in.signal_ctr >= p.n_counters || in.wait_ctr >= p.n_counters) return "counter index out of range";
      const bool fused = in.op == OP_ATTN && in.a[4] >= 0;
      if (fused && (p.merge != MERGE_LAST_ARRIVER || in.a[4] >= p.n_counters)) return "bad arrival counter";
      // a fused split signals only when it is the last of its (b, j): once per (b, j)
      if (in.signal_ctr >= 0 && (!fused || in.a[2] == 0)) sig[in.signal_ctr]++;
      group_units[group_of(in)]++;
      int rows = 0, K = 0, ws = 1;
      switch (in.op) {
        case OP_QKV: {
          const int H = in.a[0] == 0 ? m.Hq : m.Hkv;
          if (in.a[0] < 0 || in.a[0] > 2 || in.a[1] < 0 || in.a[1] >= H || in.a[2] < 0 || in.a[3] < 1 ||
              in.a[2] + in.a[3] > half)
            return fmt("cta %lld pc %lld: QKV arguments out of range", c, k);
          rows = 2 * in.a[3];
          K = m.d;
          ws = g.ws_qkv;
          break;
        }
        case OP_ATTN:
          if (in.a[0] < 0 || in.a[0] >= B || in.a[1] < 0 || in.a[1] >= m.Hkv || in.a[3] != g.S || in.a[2] < 0 ||
              in.a[2] >= g.S)
            return fmt("cta %lld pc %lld: ATTENTION arguments out of range", c, k);
          break;
        case OP_ATTN_REDUCE:
          if (in.a[0] < 0 || in.a[0] >= B || in.a[1] < 0 || in.a[1] >= m.Hkv) return "REDUCE arguments out of range";
          break;
        case OP_OPROJ:
          rows = in.a[1];
          K = m.Hq * m.hd;
          ws = g.ws_o;
          if (((in.flags & F_MERGE_IN) != 0) != (p.merge == MERGE_IN_OPROJ)) return "O-proj merge flag mismatch";
          if ((in.flags & F_MERGE_IN) && 3LL * B * m.Hkv * g.S * (m.Hq / m.Hkv) > scratch_floats)
            return "split-merge weights exceed the scratch";
          break;
        case OP_UPGATE: rows = 2 * in.a[1]; K = m.d; ws = g.ws_up; break;
        case OP_DOWN: rows = in.a[1]; K = m.F; ws = g.ws_down; break;
        case OP_LMHEAD: rows = in.a[1]; K = m.d; ws = g.ws_lm; break;
        default: break;
      }
      if (K) {
        if (rows < 1) return "empty GEMV instruction";
        const long long need = use_tc(g, nb) ? (long long)rows * nb + kTcPartialFloats : (long long)rows * (K / ws) * nb;
        if (need > scratch_floats)
          return fmt("cta %lld pc %lld: GEMV row partials exceed the scratch (%lld floats)", c, k, scratch_floats);
      }
    }
  }
  for (int c = 0; c <= n_cta; ++c)
    for (const auto& in : c < n_cta ? p.queues[c] : p.pool) {
      if (in.wait_ctr >= 0 && in.wait_n != sig[in.wait_ctr])
        return fmt("counter %lld: waiters expect %lld signals, the schedule gives %lld", in.wait_ctr, in.wait_n,
                   sig[in.wait_ctr]);
      if ((in.flags & F_LAST_LM) && (uint32_t)in.a[2] != sig[in.signal_ctr]) return "LM arrival count mismatch";
    }

  // -- simulation with counter semantics: every queue must reach OP_END
  std::vector<size_t> pc(n_cta, 0);
  std::vector<uint32_t> cnt(p.n_counters, 0);
  // happens-before summary per executed instruction: groups fully done before it
  std::vector<std::vector<Bits>> done(n_cta);
  for (int c = 0; c < n_cta; ++c) done[c].assign(p.queues[c].size(), Bits(n_group));
  std::vector<std::vector<Bits>> signalers(p.n_counters);  // what each signal carries
  std::vector<int> ctr_group(p.n_counters, -1);
  std::vector<uint32_t> arrivals(p.n_counters, 0);
  std::vector<char> pool_run(p.pool.size() + 1, 0);
  std::vector<Bits> arrived(p.n_counters, Bits(n_group));
  {
    // a counter "covers" a group when exactly that group's units signal it
    std::vector<int> sig_group(p.n_counters, -2);
    for (int c = 0; c <= n_cta; ++c)
      for (const auto& in : c < n_cta ? p.queues[c] : p.pool)
        if (in.signal_ctr >= 0 && !(in.flags & F_LAST_LM) && !(in.op == OP_ATTN && in.a[4] >= 0)) {
          const int gr = group_of(in);
          int& sg = sig_group[in.signal_ctr];
          sg = (sg == -2 || sg == gr) ? gr : -1;
        }
    for (int k = 0; k < p.n_counters; ++k)
      if (sig_group[k] >= 0 && (int)sig[k] == group_units[sig_group[k]]) ctr_group[k] = sig_group[k];
    // fused merge: its counter completes when every split of every (b, j) has arrived
    for (int c = 0; c <= n_cta; ++c)
      for (const auto& in : c < n_cta ? p.queues[c] : p.pool)
        if (in.op == OP_ATTN && in.a[4] >= 0 && in.signal_ctr >= 0) ctr_group[in.signal_ctr] = group_of(in);
  }
  // required inputs (group ids) of each instruction
  auto required = [&](const Instr& in, int* req) -> int {
    const int l = in.layer;
    const int h_writer = l == 0 ? 0 : 1 + 6 * (l - 1) + 5;
    switch (in.op) {
      case OP_QKV: req[0] = h_writer; return 1;
      case OP_ATTN:
      case OP_ATTN_POOL: req[0] = 1 + 6 * l + 0; return 1;
      case OP_ATTN_REDUCE: req[0] = 1 + 6 * l + 1; return 1;
      case OP_OPROJ: req[0] = 1 + 6 * l + (p.merge == MERGE_OP ? 2 : 1); req[1] = h_writer; return 2;
      case OP_UPGATE: req[0] = 1 + 6 * l + 3; return 1;
      case OP_DOWN: req[0] = 1 + 6 * l + 4; req[1] = 1 + 6 * l + 3; return 2;
      case OP_LMHEAD: req[0] = 1 + 6 * (m.L - 1) + 5; return 1;
      default: return 0;
    }
  };
  bool progress = true;
  while (progress) {
    progress = false;
    for (int c = 0; c < n_cta; ++c) {
      const auto& q = p.queues[c];
      while (pc[c] < q.size() && q[pc[c]].op != OP_END) {
        const Instr& in = q[pc[c]];
        if (in.wait_ctr >= 0 && cnt[in.wait_ctr] < in.wait_n) break;
        Bits f(n_group);
        if (pc[c] > 0) f = done[c][pc[c] - 1];
        if (in.wait_ctr >= 0) {
          for (const Bits& sb : signalers[in.wait_ctr]) f.merge(sb);
          if (ctr_group[in.wait_ctr] >= 0) f.set(ctr_group[in.wait_ctr]);
        }
        int req[2];
        const int nr = required(in, req);
        for (int r = 0; r < nr; ++r)
          if (!f.has(req[r]))
            return fmt("race: cta %lld pc %lld reads data of op group %lld not ordered before it", c, pc[c], req[r]);
        done[c][pc[c]] = f;
        auto run_unit = [&](const Instr& un) {
          if (un.op == OP_ATTN && un.a[4] >= 0) {  // arrival; the S-th one merges and signals
            const int a = un.a[4];
            arrived[a].merge(f);
            if (++arrivals[a] == (uint32_t)un.a[3]) {
              arrivals[a] = 0;
              if (un.signal_ctr >= 0) {
                cnt[un.signal_ctr]++;
                signalers[un.signal_ctr].push_back(arrived[a]);
              }
              arrived[a] = Bits(n_group);
            }
          } else if (un.signal_ctr >= 0) {
            cnt[un.signal_ctr]++;
            signalers[un.signal_ctr].push_back(f);
          }
        };
        if (in.op == OP_ATTN_POOL) {
          if (!pool_run[in.a[0]]) {  // the first claim loop of the layer runs every unit
            pool_run[in.a[0]] = 1;
            for (int u = in.a[0]; u < in.a[0] + in.a[1]; ++u) run_unit(p.pool[u]);
          }
        } else {
          run_unit(in);
        }
        pc[c]++;
        progress = true;
      }
    }
  }
  for (int c = 0; c < n_cta; ++c)
    if (p.queues[c][pc[c]].op != OP_END)
      return fmt("deadlock: cta %lld blocks at pc %lld waiting on counter %lld", c, pc[c], p.queues[c][pc[c]].wait_ctr);

  // -- coverage: every output element written exactly once
  std::vector<int> emb((size_t)B * m.d, 0), lm(m.V, 0);
  std::vector<std::vector<int>> qkv(m.L, std::vector<int>((size_t)(m.Hq + 2 * m.Hkv) * half, 0));
  std::vector<std::vector<int>> att(m.L, std::vector<int>((size_t)B * m.Hkv * g.S, 0));
  std::vector<std::vector<int>> red(m.L, std::vector<int>((size_t)B * m.Hkv, 0));
  std::vector<std::vector<int>> orow(m.L, std::vector<int>(m.d, 0)), urow(m.L, std::vector<int>(m.F, 0)),
      drow(m.L, std::vector<int>(m.d, 0));
  auto mark = [&](std::vector<int>& v, long long a, long long n) -> bool {
    if (a < 0 || a + n > (long long)v.size()) return false;
    for (long long i = a; i < a + n; ++i) v[i]++;
    return true;
  };
  for (int c = 0; c <= n_cta; ++c)
    for (const auto& in : c < n_cta ? p.queues[c] : p.pool) {
      bool ok = true;
      const int l = in.layer;
      switch (in.op) {
        case OP_EMBED: ok = mark(emb, in.a[0], in.a[1] - in.a[0]); break;
        case OP_QKV: {
          const int hh = in.a[0] == 0 ? in.a[1] : (in.a[0] == 1 ? m.Hq + in.a[1] : m.Hq + m.Hkv + in.a[1]);
          ok = mark(qkv[l], (long long)hh * half + in.a[2], in.a[3]);
          break;
        }
        case OP_ATTN: ok = mark(att[l], ((long long)in.a[0] * m.Hkv + in.a[1]) * g.S + in.a[2], 1); break;
        case OP_ATTN_REDUCE: ok = mark(red[l], (long long)in.a[0] * m.Hkv + in.a[1], 1); break;
        case OP_OPROJ: ok = mark(orow[l], in.a[0], in.a[1]); break;
        case OP_UPGATE: ok = mark(urow[l], in.a[0], in.a[1]); break;
        case OP_DOWN: ok = mark(drow[l], in.a[0], in.a[1]); break;
        case OP_LMHEAD: ok = mark(lm, in.a[0], in.a[1]); break;
        default: break;
      }
      if (!ok) return fmt("cta %lld: output range out of bounds (op %lld)", c, in.op);
    }
  auto once = [](const std::vector<int>& v) {
    return std::all_of(v.begin(), v.end(), [](int x) { return x == 1; });
  };
  if (!once(emb) || !once(lm)) return "embedding or LM-head rows not covered exactly once";
  for (int l = 0; l < m.L; ++l)
    if (!once(qkv[l]) || !once(att[l]) || (p.merge == MERGE_OP && !once(red[l])) || !once(orow[l]) || !once(urow[l]) ||
        !once(drow[l]))
      return fmt("layer %lld: an op's outputs are not covered exactly once", l);
  return "";
}

}  // namespace mk
