// pt_api.cu -- the extern "C" entry points declared in include/pt.h:
// argument validation, error reporting, dispatch to the kernels, and the
// TMA tensor-map helper.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "pt.h"
#include "pt_internal.h"

namespace pt {

namespace {
thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
const char* g_err_ptr() { return g_err; }
uint64_t launches() { return g_launches.load(std::memory_order_relaxed); }

namespace {
struct ProfPair {
  cudaEvent_t first, second;
  int dev;
};
struct ProfRecord {
  std::vector<ProfPair> pairs;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::map<std::string, ProfRecord> g_prof;
// Timing events are recycled, per device: creating two per scope costs the
// host more than the launches they bracket.
constexpr int kProfDev = 64;
std::vector<cudaEvent_t> g_ev_free[kProfDev];

// Caller holds g_prof_mu.
bool take_event(int dev, cudaEvent_t* e) {
  if (dev < 0 || dev >= kProfDev) return false;
  if (!g_ev_free[dev].empty()) {
    *e = g_ev_free[dev].back();
    g_ev_free[dev].pop_back();
    return true;
  }
  return cudaEventCreate(e) == cudaSuccess;
}
}  // namespace

ProfScope::ProfScope(cudaStream_t s, const char* n) : stream(s), name(n), end_event(nullptr) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaEvent_t a, b;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!take_event(dev, &a)) return;
  if (!take_event(dev, &b)) {
    g_ev_free[dev].push_back(a);
    return;
  }
  cudaEventRecord(a, s);
  end_event = b;
  g_prof[name].pairs.push_back(ProfPair{a, b, dev});
}

ProfScope::~ProfScope() {
  if (end_event) cudaEventRecord(static_cast<cudaEvent_t>(end_event), stream);
}

encode_tiled_fn get_encode_tiled() {
  static encode_tiled_fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<encode_tiled_fn>(p);
  });
  return fn;
}

bool make_tmap_thd(CUtensorMap* map, const void* base, int T, int H, int D, int rows) {
  encode_tiled_fn enc = get_encode_tiled();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is unavailable from the driver");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for T=%d H=%d D=%d", (int)r, T, H, D);
    return false;
  }
  return true;
}

bool make_tmap_acc32(CUtensorMap* map, float* base, int rows, int H) {
  encode_tiled_fn enc = get_encode_tiled();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is unavailable from the driver");
    return false;
  }
  cuuint64_t dims[3] = {64, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {64 * 4, (cuuint64_t)H * 64 * 4};
  cuuint32_t box[3] = {32, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for the fp32 accumulator, rows=%d H=%d", (int)r, rows, H);
    return false;
  }
  return true;
}

int num_sms(int device) {
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 148;
  if (!cache[device]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
    cache[device] = n > 0 ? n : 148;
  }
  return cache[device];
}

}  // namespace pt

using pt::set_error;

namespace {

pt_status as_status(int rc) {
  switch (rc) {
    case 0: return PT_OK;
    case 1: return PT_ERR_INVALID_ARG;
    case 2: return PT_ERR_UNSUPPORTED;
    case 4: return PT_ERR_TIMEOUT;
    case 5: return PT_ERR_NOMEM;
    default: return PT_ERR_CUDA;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of the attention calls.
pt_status check_attn(const char* who, pt_dtype dtype, int T, int Hq, int Hkv, int D, const pt_blockmap* bm,
                     std::initializer_list<const void*> ptrs) {
  if (!bm) {
    set_error("%s: block map is NULL", who);
    return PT_ERR_INVALID_ARG;
  }
  if (T != bm->T) {
    set_error("%s: T = %d but the block map was built for T = %d", who, T, bm->T);
    return PT_ERR_INVALID_ARG;
  }
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) {
    set_error("%s: Hq = %d must be a positive multiple of Hkv = %d", who, Hq, Hkv);
    return PT_ERR_INVALID_ARG;
  }
  if (D <= 0 || D > 512) {
    set_error("%s: head_dim %d outside 1..512", who, D);
    return D <= 0 ? PT_ERR_INVALID_ARG : PT_ERR_UNSUPPORTED;
  }
  if (dtype != PT_BF16 && dtype != PT_F32) {
    set_error("%s: unknown dtype %d", who, (int)dtype);
    return PT_ERR_INVALID_ARG;
  }
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != bm->device) {
    set_error("%s: block map lives on device %d, current device is %d", who, bm->device, dev);
    return PT_ERR_INVALID_ARG;
  }
  if (T == 0) return PT_OK;
  for (const void* p : ptrs) {
    if (!p) {
      set_error("%s: a tensor pointer is NULL", who);
      return PT_ERR_INVALID_ARG;
    }
    if (!aligned16(p)) {
      set_error("%s: tensor pointers must be 16-byte aligned", who);
      return PT_ERR_INVALID_ARG;
    }
  }
  return PT_OK;
}

// bf16 head dims with a tensor-core forward on 128 x 128 maps (the backward
// has its own list: pt::bwd_tc_supported).
bool use_tensor_cores(pt_dtype dtype, int D, const pt_blockmap* bm) {
  return dtype == PT_BF16 && (D == 64 || D == 128 || D == 256 || D == 512) && bm->BM == 128 && bm->BN == 128;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Partial-sum slots the backward may use to split long kv-major columns
// across SMs: enough for a few chunks per SM, never more than the columns.
size_t partial_slots(int T, int Hq) {
  const size_t cols = ((size_t)T + 127) / 128 * (size_t)Hq;
  return std::min<size_t>(256, 2 * cols);
}

}  // namespace

extern "C" {

pt_status pt_build_blockmap_tree(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr,
                                 const int32_t* path_nodes, int32_t n_samples, int32_t block_m, int32_t block_n,
                                 cudaStream_t stream, pt_blockmap** out) {
  if (!out) {
    set_error("pt_build_blockmap_tree: out is NULL");
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  return as_status(pt::build_tree(node_lengths, n_nodes, path_ptr, path_nodes, n_samples, block_m, block_n, stream,
                                  out));
}

pt_status pt_build_blockmap_seg(const int32_t* group_id, const int32_t* suffix_id, int32_t T, int32_t block_m,
                                int32_t block_n, cudaStream_t stream, pt_blockmap** out) {
  if (!out) {
    set_error("pt_build_blockmap_seg: out is NULL");
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  return as_status(pt::build_seg(group_id, suffix_id, T, block_m, block_n, stream, out));
}

pt_status pt_build_blockmap_draft(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                                  const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                                  const int32_t* anchor_doc, int32_t block_m, int32_t block_n, cudaStream_t stream,
                                  pt_blockmap** out) {
  if (!out) {
    set_error("pt_build_blockmap_draft: NULL out");
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  return as_status(pt::build_draft(ctx_len, n_blocks, block_size, anchors, block_keep, causal, window, ctx_doc,
                                   anchor_doc, block_m, block_n, stream, out));
}

pt_status pt_blockmap_dense(const pt_blockmap* src, cudaStream_t stream, pt_blockmap** out) {
  if (!src || !out) {
    set_error("pt_blockmap_dense: NULL argument");
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  return as_status(pt::build_dense(src, stream, out));
}

pt_status pt_blockmap_info(const pt_blockmap* bm, int32_t* T, int32_t* block_m, int32_t* block_n, int32_t* nq,
                           int32_t* nk, int64_t* nnz, int64_t* n_full) {
  if (!bm) {
    set_error("pt_blockmap_info: NULL map");
    return PT_ERR_INVALID_ARG;
  }
  if (nnz || n_full)  // list sizes: may wait for the build on the device
    if (int rc = pt::ensure_counts(bm)) return as_status(rc);
  if (T) *T = bm->T;
  if (block_m) *block_m = bm->BM;
  if (block_n) *block_n = bm->BN;
  if (nq) *nq = bm->nq;
  if (nk) *nk = bm->nk;
  if (nnz) *nnz = bm->nnz;
  if (n_full) *n_full = bm->n_full;
  return PT_OK;
}

pt_status pt_blockmap_export(const pt_blockmap* bm, int32_t* q_ptr, int32_t* kv_idx, uint8_t* kind, int32_t* k_ptr,
                             int32_t* q_idx, uint8_t* kindT) {
  if (!bm) {
    set_error("pt_blockmap_export: NULL map");
    return PT_ERR_INVALID_ARG;
  }
  if (int rc = pt::ensure_counts(bm)) return as_status(rc);
  struct Item {
    void* dst;
    const void* src;
    size_t bytes;
  } items[] = {
      {q_ptr, bm->q_ptr, sizeof(int32_t) * (bm->nq + 1)}, {kv_idx, bm->kv_idx, sizeof(int32_t) * bm->nnz},
      {kind, bm->kind, (size_t)bm->nnz},                  {k_ptr, bm->k_ptr, sizeof(int32_t) * (bm->nk + 1)},
      {q_idx, bm->q_idx, sizeof(int32_t) * bm->nnz},      {kindT, bm->kindT, (size_t)bm->nnz},
  };
  for (const Item& it : items) {
    if (!it.dst || it.bytes == 0) continue;
    cudaError_t e = cudaMemcpy(it.dst, it.src, it.bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      set_error("pt_blockmap_export: %s", cudaGetErrorString(e));
      return PT_ERR_CUDA;
    }
  }
  return PT_OK;
}

pt_status pt_blockmap_export_masks(const pt_blockmap* bm, int32_t* pidx, int32_t* pidxT, uint32_t* mask_rows,
                                   uint32_t* mask_cols) {
  if (!bm) {
    set_error("pt_blockmap_export_masks: NULL map");
    return PT_ERR_INVALID_ARG;
  }
  if (int rc = pt::ensure_counts(bm)) return as_status(rc);
  if (bm->n_partial > 0 && (!bm->mask_rows || !bm->mask_cols)) {
    set_error("pt_blockmap_export_masks: this map has no tile masks (tile sizes other than 128 x 128)");
    return PT_ERR_UNSUPPORTED;
  }
  struct Item {
    void* dst;
    const void* src;
    size_t bytes;
  } items[] = {
      {pidx, bm->pidx, sizeof(int32_t) * bm->nnz},
      {pidxT, bm->pidxT, sizeof(int32_t) * bm->nnz},
      {mask_rows, bm->mask_rows, sizeof(uint32_t) * 512 * bm->n_partial},
      {mask_cols, bm->mask_cols, sizeof(uint32_t) * 512 * bm->n_partial},
  };
  for (const Item& it : items) {
    if (!it.dst || it.bytes == 0 || !it.src) continue;
    cudaError_t e = cudaMemcpy(it.dst, it.src, it.bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      set_error("pt_blockmap_export_masks: %s", cudaGetErrorString(e));
      return PT_ERR_CUDA;
    }
  }
  return PT_OK;
}

void pt_blockmap_free(pt_blockmap* bm) { pt::free_map(bm); }

pt_status pt_attn_fwd(const void* Q, const void* K, const void* V, pt_dtype dtype, int32_t T, int32_t Hq,
                      int32_t Hkv, int32_t D, float scale, const pt_blockmap* bm, void* O, float* LSE,
                      cudaStream_t stream) {
  pt_status st = check_attn("pt_attn_fwd", dtype, T, Hq, Hkv, D, bm, {Q, K, V, O, LSE});
  if (st != PT_OK || T == 0) return st;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)D);
  if (dtype == PT_BF16) {
    if (use_tensor_cores(dtype, D, bm))
      return as_status(pt::fwd_tc(Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, stream));
    if (D % 8 != 0) {
      set_error("pt_attn_fwd: bf16 needs head_dim %% 8 == 0 (got %d)", D);
      return PT_ERR_UNSUPPORTED;
    }
    return as_status(pt::fwd_simt(true, Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, stream));
  }
  return as_status(pt::fwd_simt(false, Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, stream));
}

size_t pt_bwd_workspace_bytes(int32_t T, int32_t Hq, int32_t D) {
  if (T <= 0 || Hq <= 0 || D <= 0) return 256;
  const size_t tpad = ((size_t)T + 127) / 128 * 128;
  // head_dim 64: an fp32 dQ accumulator first, for the one-pass backward
  const size_t dq_acc = D == 64 ? round256(sizeof(float) * tpad * Hq * D) : 0;
  return 2 * round256(sizeof(float) * tpad * Hq) + dq_acc +
         round256(partial_slots(T, Hq) * 128 * 2 * sizeof(float) * D);
}

pt_status pt_attn_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                      pt_dtype dtype, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, float scale,
                      const pt_blockmap* bm, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  pt_status st = check_attn("pt_attn_bwd", dtype, T, Hq, Hkv, D, bm, {dO, Q, K, V, O, LSE, dQ, dK, dV});
  if (st != PT_OK || T == 0) return st;
  // the two row statistics are required; partial-sum room beyond them is optional
  const size_t need = 2 * round256(sizeof(float) * (((size_t)T + 127) / 128 * 128) * Hq);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
    set_error("pt_attn_bwd: workspace must be 256-byte aligned and hold at least %zu bytes (got %zu; %zu advised)",
              need, workspace_bytes, pt_bwd_workspace_bytes(T, Hq, D));
    return PT_ERR_INVALID_ARG;
  }
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)D);
  const size_t tpad = ((size_t)T + 127) / 128 * 128;
  const size_t stats = round256(sizeof(float) * tpad * Hq);
  float* delta = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + stats);
  float* partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * stats);
  const size_t partial_bytes = workspace_bytes - 2 * stats;
  if (dtype == PT_BF16) {
    if (use_tensor_cores(dtype, D, bm) && pt::bwd_tc_supported(D))
      return as_status(pt::bwd_tc(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, lse2, partial,
                                  partial_bytes, true, stream));
    if (D % 8 != 0) {
      set_error("pt_attn_bwd: bf16 needs head_dim %% 8 == 0 (got %d)", D);
      return PT_ERR_UNSUPPORTED;
    }
    return as_status(pt::bwd_simt(true, dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, stream));
  }
  return as_status(pt::bwd_simt(false, dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, stream));
}

pt_status pt_sync_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    set_error("pt_sync_status: %s", cudaGetErrorString(e));
    return PT_ERR_CUDA;
  }
  int worst = 0;
  int codes[] = {pt::take_status_blockmap(stream), pt::take_status_fwd(stream), pt::take_status_bwd(stream),
                 pt::take_status_simt(stream), pt::take_status_fold(stream)};
  for (int c : codes) {
    if (c < 0) {
      set_error("pt_sync_status: could not read the device status word");
      return PT_ERR_CUDA;
    }
    if (c && !worst) worst = c;
  }
  if (worst == PT_STATUS_TIMEOUT) {
    set_error("a bounded in-kernel wait ran out");
    return PT_ERR_TIMEOUT;
  }
  if (worst == PT_STATUS_INVALID) {
    set_error("a device-side check of a block map's lists or labels failed (a listed tile that keeps nothing, "
              "kept pairs missing from the lists, or more partial tiles than the lists' bound)");
    return PT_ERR_INVALID_ARG;
  }
  if (worst) {
    set_error("device status %d", worst);
    return PT_ERR_CUDA;
  }
  return PT_OK;
}

const char* pt_last_error(void) { return pt::g_err_ptr(); }

uint64_t pt_launch_count(void) { return pt::launches(); }

pt_status pt_debug_wait_timeout(cudaStream_t stream) { return as_status(pt::wait_timeout_probe(stream)); }

pt_status pt_blockmap_prepare_bwd(const pt_blockmap* bm, int32_t Hq, int32_t Hkv, int32_t D, cudaStream_t stream) {
  if (!bm || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) {
    set_error("pt_blockmap_prepare_bwd: bad map or head layout (Hq=%d, Hkv=%d, D=%d)", Hq, Hkv, D);
    return PT_ERR_INVALID_ARG;
  }
  if (D > 512) {
    set_error("pt_blockmap_prepare_bwd: head_dim %d outside 1..512", D);
    return PT_ERR_UNSUPPORTED;
  }
  return as_status(pt::prepare_bwd_noalloc(bm, Hq, Hkv, D, stream));
}

void pt_debug_drop_listed_tile(int32_t n) { pt::debug_drop_listed_tiles(n); }

pt_status pt_debug_pool_usage(int32_t device, uint64_t* used_bytes, uint64_t* reserved_bytes) {
  if (!used_bytes || !reserved_bytes || device < 0) {
    set_error("pt_debug_pool_usage: bad arguments");
    return PT_ERR_INVALID_ARG;
  }
  return as_status(pt::pool_usage(device, used_bytes, reserved_bytes));
}

pt_status pt_debug_tree_lists(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr,
                              const int32_t* path_nodes, int32_t n_samples, int32_t block_m, int32_t block_n,
                              int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx, int64_t cap, int64_t* nnz) {
  if (!q_ptr || !nnz || cap < 0 || (cap > 0 && !kv_idx)) {
    set_error("pt_debug_tree_lists: bad output arguments");
    return PT_ERR_INVALID_ARG;
  }
  if (pt::debug_tree_lists(node_lengths, n_nodes, path_ptr, path_nodes, n_samples, block_m, block_n, q_ptr, q_ptr_len,
                           kv_idx, cap, nnz))
    return PT_ERR_INVALID_ARG;
  return PT_OK;
}

pt_status pt_debug_draft_lists(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                               const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                               const int32_t* anchor_doc, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx,
                               int64_t cap, int64_t* nnz, int64_t* kept_pairs) {
  if (!q_ptr || !nnz || !kept_pairs || cap < 0 || (cap > 0 && !kv_idx)) {
    set_error("pt_debug_draft_lists: bad output arguments");
    return PT_ERR_INVALID_ARG;
  }
  const int rc = pt::debug_draft_lists(ctx_len, n_blocks, block_size, anchors, block_keep, causal, window, ctx_doc,
                                       anchor_doc, q_ptr, q_ptr_len, kv_idx, cap, nnz, kept_pairs);
  return rc == 0 ? PT_OK : (rc == 2 ? PT_ERR_UNSUPPORTED : PT_ERR_INVALID_ARG);
}

pt_status pt_debug_pack_dq(const int32_t* row_steps, int32_t nq, int32_t Hq, int32_t ctas, int32_t* items,
                           int64_t cap_items, int32_t* cta_rec, int32_t* n_items, int32_t* grid, int32_t* n_empty) {
  if (nq < 0 || (nq > 0 && !row_steps) || Hq < 1 || ctas < 1 || cap_items < 0 || (cap_items > 0 && !items) ||
      !cta_rec || !n_items || !grid || !n_empty) {
    set_error("pt_debug_pack_dq: bad arguments");
    return PT_ERR_INVALID_ARG;
  }
  for (int32_t t = 0; t < nq; ++t)
    if (row_steps[t] < 0) {
      set_error("pt_debug_pack_dq: negative row length at %d", t);
      return PT_ERR_INVALID_ARG;
    }
  if (pt::debug_pack_dq(row_steps, nq, Hq, ctas, items, cap_items, cta_rec, n_items, grid, n_empty))
    return PT_ERR_INVALID_ARG;
  return PT_OK;
}

pt_status pt_debug_pack_dkdv(const int32_t* col_steps, int32_t nk, int32_t g, int32_t Hkv, int32_t max_slots,
                             int32_t ctas, int32_t exact_fill, int32_t* items, int64_t cap_items, int32_t* cta_ptr,
                             int32_t* n_items, int32_t* n_slots, int32_t* grid) {
  if (nk < 0 || (nk > 0 && !col_steps) || g < 1 || Hkv < 1 || ctas < 1 || cap_items < 0 ||
      (cap_items > 0 && !items) || !cta_ptr || !n_items || !n_slots || !grid) {
    set_error("pt_debug_pack_dkdv: bad arguments");
    return PT_ERR_INVALID_ARG;
  }
  for (int32_t j = 0; j < nk; ++j)
    if (col_steps[j] < 0) {
      set_error("pt_debug_pack_dkdv: negative column length at %d", j);
      return PT_ERR_INVALID_ARG;
    }
  if (pt::debug_pack_dkdv(col_steps, nk, g, Hkv, max_slots, ctas, exact_fill != 0, items, cap_items, cta_ptr, n_items,
                          n_slots, grid))
    return PT_ERR_INVALID_ARG;
  return PT_OK;
}

pt_status pt_debug_exp2(const float* x, float* y, int64_t n, int32_t method, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y)) || (method != 0 && method != 1)) {
    set_error("pt_debug_exp2: bad arguments (n=%lld, method=%d)", (long long)n, method);
    return PT_ERR_INVALID_ARG;
  }
  return as_status(pt::exp2_probe(x, y, n, method, stream));
}

void pt_profile_enable(int on) {
  if (on) {  // stock the current device's event pool before the scopes need it
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(pt::g_prof_mu);
    if (dev >= 0 && dev < pt::kProfDev)
      while (pt::g_ev_free[dev].size() < 1024) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) break;
        pt::g_ev_free[dev].push_back(e);
      }
  }
  pt::g_prof_on.store(on != 0);
}

pt_status pt_profile_read(const char* kernel, int64_t* launches, double* total_ms) {
  if (!kernel) {
    set_error("pt_profile_read: NULL kernel name");
    return PT_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(pt::g_prof_mu);
  int64_t n = 0;
  double ms = 0.0;
  auto it = pt::g_prof.find(kernel);
  if (it != pt::g_prof.end()) {
    for (auto& pr : it->second.pairs) {
      if (cudaEventSynchronize(pr.second) != cudaSuccess) {
        set_error("pt_profile_read: event failed");
        return PT_ERR_CUDA;
      }
      float t = 0.f;
      cudaEventElapsedTime(&t, pr.first, pr.second);
      ms += t;
      ++n;
    }
  }
  if (launches) *launches = n;
  if (total_ms) *total_ms = ms;
  return PT_OK;
}

void pt_profile_reset(void) {
  std::lock_guard<std::mutex> lk(pt::g_prof_mu);
  for (auto& kv : pt::g_prof)
    for (auto& pr : kv.second.pairs) {
      // an event back to its device's pool once its record has completed
      cudaEventSynchronize(pr.second);
      if (pr.dev >= 0 && pr.dev < pt::kProfDev) {
        pt::g_ev_free[pr.dev].push_back(pr.first);
        pt::g_ev_free[pr.dev].push_back(pr.second);
      } else {
        cudaEventDestroy(pr.first);
        cudaEventDestroy(pr.second);
      }
    }
  pt::g_prof.clear();
}

}  // extern "C"
