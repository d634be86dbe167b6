// Tensor maps of the tensor-core GEMV pages ("8 · Écrire son megakernel", §8.4: the loader
// streams weight pages into shared memory).  A page is kTcRows rows of one kTcKw-column
// window of a weight segment; one 3D tensor-map copy lands it as kTcKw / 64 column chunks of
// [kTcRows rows][128 bytes], 128-byte swizzled:
//   dim 0: 64 columns (128 contiguous bytes), dim 1: rows (stride K * 2 bytes),
//   dim 2: 64-column chunks (stride 128 bytes); box {64, kTcRows, kTcKw / 64}.
// Rows past the segment and chunks past K are outside the map: the copy fills them with
// zeros and reads nothing there, so a page never touches another instruction's rows.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <tuple>
#include <utility>

#include "mk_plan.h"

namespace mk {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder(std::string* err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
    *err = std::string("cuTensorMapEncodeTiled not available: ") + cudaGetErrorString(e);
    return nullptr;
  }
  fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  return fn;
}

bool is_gemv(int op) { return op == OP_QKV || op == OP_OPROJ || op == OP_UPGATE || op == OP_DOWN || op == OP_LMHEAD; }

uint64_t get_u64(const Instr& in, int at) { return (uint64_t)(uint32_t)in.a[at] | ((uint64_t)(uint32_t)in.a[at + 1] << 32); }
void put_u64(Instr& in, int at, uint64_t v) {
  in.a[at] = (int32_t)(uint32_t)(v & 0xFFFFFFFFu);
  in.a[at + 1] = (int32_t)(uint32_t)(v >> 32);
}

// rows of the instruction's two segments and the row length K (as the kernel's make_gemv)
void segments(const ModelShape& m, const Instr& in, int* r0, int* r1, int* K) {
  *r1 = 0;
  switch (in.op) {
    case OP_QKV: *r0 = *r1 = in.a[3]; *K = m.d; break;
    case OP_OPROJ: *r0 = in.a[1]; *K = m.Hq * m.hd; break;
    case OP_UPGATE: *r0 = *r1 = in.a[1]; *K = m.d; break;
    case OP_DOWN: *r0 = in.a[1]; *K = m.F; break;
    default: *r0 = in.a[1]; *K = m.d; break;  // OP_LMHEAD
  }
}

}  // namespace

std::string build_tc_maps(const ModelShape& m, const Geometry& g, Plan* p, std::vector<TmapImage>* maps) {
  maps->clear();
  std::string err;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder(&err);
  if (!enc) return err;
  std::map<std::tuple<uint64_t, int, int>, uint64_t> seen;  // (rows pointer, rows, K) -> index + 1
  auto map_of = [&](uint64_t rows_ptr, int rows, int K, std::string* e) -> uint64_t {
    if (rows <= 0) return 0;
    const auto key = std::make_tuple(rows_ptr, rows, K);
    auto it = seen.find(key);
    if (it != seen.end()) return it->second;
    CUtensorMap tm;
    const cuuint64_t dims[3] = {(cuuint64_t)kTcChunkCols, (cuuint64_t)rows, (cuuint64_t)(K / kTcChunkCols)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    const cuuint32_t box[3] = {(cuuint32_t)kTcChunkCols, (cuuint32_t)kTcRows, (cuuint32_t)(kTcKw / kTcChunkCols)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, reinterpret_cast<void*>(rows_ptr), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *e = "cuTensorMapEncodeTiled failed with " + std::to_string((int)r);
      return 0;
    }
    TmapImage img;
    static_assert(sizeof(CUtensorMap) == sizeof(TmapImage) && sizeof(TmapImage) == kTmapBytes, "tensor map image size");
    std::memcpy(img.bytes, &tm, sizeof tm);
    maps->push_back(img);
    seen[key] = maps->size();
    return maps->size();
  };
  auto fix = [&](std::vector<Instr>& q) {
    for (auto& in : q) {
      if (!is_gemv(in.op) || !err.empty()) continue;
      int r0, r1, K;
      segments(m, in, &r0, &r1, &K);
      if (K % kTcChunkCols) {
        err = "tensor-core pages need rows that are a multiple of 64 columns";
        return;
      }
      const uint64_t i0 = map_of(get_u64(in, kP4), r0, K, &err);
      const uint64_t i1 = map_of(get_u64(in, kP5), r1, K, &err);
      put_u64(in, kP4, i0);
      put_u64(in, kP5, i1);
    }
  };
  (void)g;
  for (auto& q : p->queues) fix(q);
  for (auto& ph : p->phase_queues)
    for (auto& q : ph) fix(q);
  return err;
}

std::string build_kv_maps(const ModelShape& m, const Geometry& g, int cache_batch, Plan* p,
                          std::vector<TmapImage>* maps) {
  std::string err;
  if (!g.attn_mma) return err;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder(&err);
  if (!enc) return err;
  const int esz = 2, halves = m.hd / 64, pb = g.page_bytes / (m.hd * esz);
  const uint64_t per_seq_head = (uint64_t)m.max_ctx * m.hd * esz;  // bytes of one (sequence, kv head)
  std::map<std::pair<uint64_t, uint64_t>, uint64_t> seen;         // (key base, value base) -> index + 1
  auto encode = [&](uint64_t base, TmapImage* img) {
    CUtensorMap tm;
    // dim 0: 64 elements of a row (128 bytes), dim 1: positions, dim 2: the row's 64-element
    // halves, dim 3: cache sequence x kv head; a box is one page: [half][position][128 B]
    const cuuint64_t dims[4] = {64, (cuuint64_t)m.max_ctx, (cuuint64_t)halves, (cuuint64_t)cache_batch * m.Hkv};
    const cuuint64_t strides[3] = {(cuuint64_t)m.hd * esz, 128, per_seq_head};
    const cuuint32_t box[4] = {64, (cuuint32_t)pb, (cuuint32_t)halves, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, reinterpret_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      err = "cuTensorMapEncodeTiled (KV cache) failed with " + std::to_string((int)r);
      return false;
    }
    std::memcpy(img->bytes, &tm, sizeof tm);
    return true;
  };
  auto fix = [&](std::vector<Instr>& q) {
    for (auto& in : q) {
      if (in.op != OP_ATTN || !err.empty()) continue;
      // the baked pointers address (b, j) at t = 0: back to the layer's cache base
      const uint64_t off = ((uint64_t)in.a[0] * m.Hkv + in.a[1]) * per_seq_head;
      const uint64_t kb = get_u64(in, kP4) - off, vb = get_u64(in, kP5) - off;
      const auto key = std::make_pair(kb, vb);
      auto it = seen.find(key);
      uint64_t idx;
      if (it != seen.end()) {
        idx = it->second;
      } else {
        TmapImage ik, iv;
        if (!encode(kb, &ik) || !encode(vb, &iv)) return;
        maps->push_back(ik);
        maps->push_back(iv);
        idx = maps->size() - 1;  // the key map's index + 1
        seen[key] = idx;
      }
      put_u64(in, kP3, idx);
    }
  };
  for (auto& q : p->queues) fix(q);
  for (auto& ph : p->phase_queues)
    for (auto& q : ph) fix(q);
  fix(p->pool);
  return err;
}

void place_tc_maps(std::vector<Instr>& q, uintptr_t maps_dev, bool gemv_maps) {
  static const int gemv_slots[2] = {kP4, kP5}, attn_slots[1] = {kP3};
  for (auto& in : q) {
    const bool gemv = is_gemv(in.op);
    if (gemv ? !gemv_maps : in.op != OP_ATTN) continue;  // without GEMV maps p4 / p5 are row pointers
    const int* slots = gemv ? gemv_slots : attn_slots;
    const int n = gemv ? 2 : 1;
    for (int k = 0; k < n; ++k) {
      const uint64_t v = get_u64(in, slots[k]);
      put_u64(in, slots[k], v ? (uint64_t)maps_dev + (v - 1) * sizeof(TmapImage) : 0);
    }
  }
}

}  // namespace mk
