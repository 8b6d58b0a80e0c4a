// pt_internal.h -- definitions shared by the library's translation units
// (host and device).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define PT_STATUS_OK 0
#define PT_STATUS_INVALID 1
#define PT_STATUS_TIMEOUT 4

// Kinds of a (q tile, kv block) pair in the block map.
#define PT_KIND_EMPTY 0
#define PT_KIND_FULL 1
#define PT_KIND_PARTIAL 2

// Per-token tree coordinates.  A node's Euler-tour interval [tin, tout)
// contains exactly the intervals of its descendants, so "node(kv) is an
// ancestor-or-self of node(q)" is tin(kv) <= tin(q) < tout(kv).  Padding
// tokens past T carry (INT32_MAX, 0): they keep nothing and nothing keeps them.
struct pt_tok {
  int32_t tin;
  int32_t tout;
};

// Work lists of the kv-major backward kernel for one head layout.
struct pt_dkdv_lists {
  pt_dkdv_lists* next;
  int g, hkv, max_slots, sms;  // the key: group size, kv heads, partial-sum slots allowed, SM count,
  bool exact_fill;             // and the packing (columns cut at each CTA's share, or longest first)
  int n_items, n_splits, n_slots, grid;
  void* mem;     // one pool allocation: items | splits | CTA index
  void* items;   // DkdvItem[n_items] (device), grouped by the CTA that runs them
  void* splits;  // int4[n_splits]: kv block, kv head, first slot, slot count (device)
  void* cta;     // int[grid + 1]: CTA b runs items [cta[b], cta[b + 1])
};

// Work lists of the q-major (dQ) kernels for one head count.
struct pt_dq_lists {
  pt_dq_lists* next;
  int hq, sms;  // the key
  int grid, n_items, n_empty;
  void* mem;     // one pool allocation: items | CTA records
  void* items;   // int4[n_items]: q tile, head, first list entry, kv blocks; grouped by CTA
  void* cta;     // int4[grid]: first item, end item, kv blocks of the CTA
  int* h_empty;  // [n_empty] q tiles without any kv block (their dQ rows are zero), ascending
};

struct pt_blockmap {
  int device;
  cudaStream_t stream;  // the build stream; memory is returned to the pool in its order
  void* mem_fixed;      // one pool allocation for the arrays sized before classification
  void* mem_lists;      // one pool allocation for the lists and masks
  int32_t T, BM, BN, nq, nk;
  int32_t n_nodes;
  int32_t tpad;  // entries of tok: max(nq*BM, nk*BN)
  int64_t nnz, n_full;
  bool dense;
  pt_tok* tok;          // [tpad]
  int32_t* node_of;     // [T]
  int32_t* node_start;  // [n_nodes]
  int32_t* node_end;    // [n_nodes]
  int32_t* parent;      // [n_nodes], -1 for roots
  // q-major list
  int32_t* q_ptr;   // [nq + 1]
  int32_t* kv_idx;  // [nnz]
  uint8_t* kind;    // [nnz]
  // kv-major transpose
  int32_t* k_ptr;   // [nk + 1]
  int32_t* q_idx;   // [nnz]
  uint8_t* kindT;   // [nnz]
  // longest-first processing orders
  int32_t* q_order;  // [nq] q tiles, most kv blocks first
  int32_t* k_order;  // [nk] kv blocks, most q tiles first
  // keep bitmasks of the partial tiles (128 x 128 maps only)
  int64_t n_partial;
  int32_t* pidx;        // [nnz] mask slot of each q-major entry, -1 when full
  int32_t* pidxT;       // [nnz] mask slot of each kv-major entry, -1 when full
  uint32_t* mask_rows;  // [n_partial][128 q rows][4 words]: bit c = keep(row, kv column c)
  uint32_t* mask_cols;  // [n_partial][128 kv columns][4 words]: bit r = keep(q row r, column)
  // host copies of the list lengths (one allocation: 4 counters | rows | columns),
  // valid once counts_ready.  A build that does not wait for the device leaves
  // them in pinned staging behind counts_ev; pt::ensure_counts fills them in
  // (and nnz, n_full, n_partial) on first use.
  int* h_counts;
  int* h_row_cnt;  // [nq]
  int* h_col_cnt;  // [nk]
  bool counts_ready;
  void* counts_host;  // pinned staging (until counts_ready)
  void* counts_dev;   // the staging's device address
  size_t counts_cap;
  void* counts_ev;    // cudaEvent_t recorded after the copy to counts_host
  // tree maps: the row and column list lengths derived on the host from the
  // node intervals ([nq] rows | [nk] columns), usable before the device's
  // arrive; ensure_counts checks them against the device's
  int* h_rc_pred;
  bool lists_on_host;  // the host built the lists; only the full-tile count comes from the device
  int64_t nnz_cap;    // list entries allocated (>= nnz)
  int64_t p_cap;      // mask slots allocated (>= n_partial)
  // Which rule the map encodes: tree/segment labels (tok, node tables) or
  // draft blocks (pt_build_blockmap_draft: the per-block ranges below).
  int producer;
  int32_t d_ctx, d_bs, d_nb, d_causal, d_window;
  void* d_blk;  // int4[d_nb] (device): kept context [x, y) before any window, anchor z, keep flag w
  // backward work lists, one entry per head layout asked for (built on first
  // use, kept until the map is freed, so no call evicts lists another stream
  // may still be reading)
  struct pt_dkdv_lists* dkdv_lists;
  struct pt_dq_lists* dq_lists;
};

// Work item of the kv-major backward kernel: steps [x0, x1) of the (kv block,
// kv head) column; slot >= 0 means the item is one chunk of a split column and
// writes fp32 partial sums to that slot instead of the outputs.
struct DkdvItem {
  int jb, hk, x0, x1, slot, pad0, pad1, pad2;
};

namespace pt {

// Thread-local error message setter (pt_api.cu).
void set_error(const char* fmt, ...);

// Launch counter (pt_api.cu).
void count_launch(int n = 1);

// Optional per-kernel timing (pt_api.cu).  While enabled with
// pt_profile_enable(1), every kernel launch site brackets its launch with a
// pair of CUDA events on the launching stream; pt_profile_read() sums them.
// Disabled (the default), a scope costs one branch.
struct ProfScope {
  ProfScope(cudaStream_t s, const char* name);
  ~ProfScope();
  cudaStream_t stream;
  const char* name;
  void* end_event;
};

constexpr int PT_PRODUCER_TREE = 0, PT_PRODUCER_DRAFT = 1;

// Draft-block map builder (pt_blockmap.cu).  Returns a PT_* status code.
int build_draft(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                const int32_t* anchor_doc, int32_t BM, int32_t BN, cudaStream_t s, pt_blockmap** out);

// Host list lengths of a map: waits for the build's copy if it has not
// arrived yet.  Returns a PT_* status code (pt_blockmap.cu).
int ensure_counts(const pt_blockmap* bm);

// Row and column list lengths of a map (host arrays of nq and nk): the
// host-derived ones of a tree map while the device's are still in flight,
// else the device's (waiting for them if needed).  Returns a PT_* status code.
int rowcol_counts(const pt_blockmap* bm, const int** row, const int** col);

// True when the map could have partial tiles but carries no masks.
inline bool masks_missing(const pt_blockmap* bm) {
  return !bm->mask_rows && (bm->counts_ready ? bm->n_partial > 0 : bm->p_cap > 0);
}

// Stream-ordered device memory from the library's private pool, and pinned
// staging for small host-to-device uploads (pt_blockmap.cu).
int pool_alloc(void** p, size_t bytes, int dev, cudaStream_t s);
void pool_free(void* p, cudaStream_t s);
// Test hook: the next n tree builds with host-built lists each drop one tile.
void debug_drop_listed_tiles(int n);
// Bytes of the pool on `dev` handed out now and held from the device.
int pool_usage(int dev, uint64_t* used, uint64_t* reserved);
int upload(void* dst, const void* src, size_t bytes, int dev, cudaStream_t s);

// Device status word of each translation unit: read and clear.
int take_status_blockmap(cudaStream_t s);
int take_status_fwd(cudaStream_t s);
int take_status_bwd(cudaStream_t s);
int take_status_simt(cudaStream_t s);
int take_status_fold(cudaStream_t s);

// Block-map builders (pt_blockmap.cu).  Return a PT_* status code.
int build_tree(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
               int32_t n_samples, int32_t BM, int32_t BN, cudaStream_t s, pt_blockmap** out);
int build_seg(const int32_t* group_id, const int32_t* suffix_id, int32_t T, int32_t BM, int32_t BN,
              cudaStream_t s, pt_blockmap** out);
int build_dense(const pt_blockmap* src, cudaStream_t s, pt_blockmap** out);
void free_map(pt_blockmap* bm);

// Tensor-core bf16 kernels (pt_fwd_tc.cu, pt_bwd_tc.cu).
int fwd_tc(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
           const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s);
// allow_build: whether the call may build the map's work lists (from the
// library's pool) when they do not match the head layout yet.
int bwd_tc(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
           int Hq, int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
           float* lse2, float* partial, size_t partial_bytes, bool allow_build, cudaStream_t s);
// Builds the work lists the allocation-free backward needs for a head layout.
int prepare_bwd_noalloc(const pt_blockmap* bm, int Hq, int Hkv, int D, cudaStream_t s);
// Host-only: the q-major lists a tree map's build derives on the host
// (pt_debug_tree_lists).
int debug_tree_lists(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
                     int32_t n_samples, int32_t BM, int32_t BN, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx,
                     int64_t cap, int64_t* nnz);
// Host-only: the lists and kept-pair count a draft-block map's build derives
// on the host (pt_debug_draft_lists).
int debug_draft_lists(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                      const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                      const int32_t* anchor_doc, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx, int64_t cap,
                      int64_t* nnz, int64_t* kept_pairs);
// Host-only: the backward's q-major packing for given row lengths
// (pt_debug_pack_dq).
int debug_pack_dq(const int* row_cnt, int nq, int Hq, int ctas, int32_t* items, long long cap_items, int32_t* cta_rec,
                  int32_t* n_items, int32_t* grid, int32_t* n_empty);
// Host-only: the backward's kv-major packing for given column lengths
// (pt_debug_pack_dkdv).
int debug_pack_dkdv(const int* col_cnt, int nk, int g, int Hkv, int max_slots, int ctas, bool exact_fill, int32_t* items,
                    long long cap_items, int32_t* cta_ptr, int32_t* n_items, int32_t* n_slots, int32_t* grid);
bool bwd_tc_supported(int D);
int wait_timeout_probe(cudaStream_t s);
int exp2_probe(const float* x, float* y, long long n, int method, cudaStream_t s);

// CUDA-core kernels (pt_simt.cu), fp32 or bf16 storage with fp32 math.
int fwd_simt(bool bf16, const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
             const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s);
int bwd_simt(bool bf16, const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             int T, int Hq, int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV,
             float* delta, cudaStream_t s);

// Driver entry point for tensor-map encoding (pt_api.cu).
typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
encode_tiled_fn get_encode_tiled();

// A [T, H, D] bf16 tensor as a 3-D TMA map with boxes of 64 (d) x 1 (head) x
// rows (tokens), 128-byte swizzle.  Returns false (and sets the error) on failure.
bool make_tmap_thd(CUtensorMap* map, const void* base, int T, int H, int D, int rows);
// fp32 [rows][H][64], boxes of 32 columns x 1 head x 128 rows, 128-byte swizzle
bool make_tmap_acc32(CUtensorMap* map, float* base, int rows, int H);

int num_sms(int device);

// Launch with programmatic stream serialization: the kernel may begin while
// the preceding kernel in the stream drains (its CTAs start on the SMs that
// kernel has left) and must call pdl_wait() before touching global memory.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace pt
