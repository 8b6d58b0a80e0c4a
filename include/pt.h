/*
 * pt.h -- C ABI of libpt: exact softmax attention over a prefix-tree token
 * layout, forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * The method.  Many sequences that share prefixes are stored once, flat: a
 * prefix tree whose nodes each own a contiguous run of tokens, every ancestor
 * laid out before its descendants.  A token attends to every token of its
 * ancestor nodes and causally to the tokens of its own node; nothing crosses
 * sibling branches, groups or packed documents.  In the GRPO case one prompt
 * of P tokens is followed by G completions, and each completion sees the
 * whole prompt and itself causally ("cp=1 shared-prefix prefix-tree attention
 * for rollouts", PR description; "prefix_grouper_kernel.py", module
 * docstring and _make_mask_mod).  The result is identical to dense masked
 * attention, but tiles whose pairs are all masked are never visited, so the
 * cost is proportional to the kept pairs, O(P + G*R) per group rather than
 * O(T^2) ("prefix_grouper_kernel.py", module docstring).
 *
 * Conventions shared by every call:
 *  - Device pointers are raw CUDA device addresses on the current device,
 *    16-byte aligned, densely packed (no strides).  Host pointers are plain
 *    host memory.  The caller owns every buffer it passes in.
 *  - Tensors are token-major: Q, dO, O, dQ are [T, Hq, D]; K, V, dK, dV are
 *    [T, Hkv, D]; LSE is [Hq, T] fp32 (natural log).  This is the pages'
 *    [1, T, H, D] layout without the batch dimension
 *    ("prefix_grouper_kernel.py", flex_shared_prefix_attention).
 *  - Grouped-query attention: q head h reads kv head h / (Hq / Hkv)
 *    ("prefix_grouper_kernel.py", enable_gqa = n_heads != n_kv).
 *  - Calls are ordered on the given stream.  Nothing is silently ignored or
 *    replaced by a fallback: an argument the library cannot honour returns an
 *    error status before anything is launched ("cp=1 shared-prefix prefix-tree
 *    attention for rollouts": the HF path fails loudly rather than dropping
 *    the mask).  pt_last_error() gives a message for the calling thread.
 *  - Every wait inside a kernel is bounded; a wait that runs out records
 *    PT_ERR_TIMEOUT in a per-device status word, which pt_sync_status()
 *    returns (and clears).
 */
#ifndef PT_H_
#define PT_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PT_OK = 0,
  PT_ERR_INVALID_ARG = 1, /* malformed tree or labels, bad sizes, null pointers */
  PT_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim, dtype, tile) */
  PT_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  PT_ERR_TIMEOUT = 4,     /* a bounded in-kernel wait ran out */
  PT_ERR_NOMEM = 5        /* device or host allocation failed */
} pt_status;

typedef enum { PT_BF16 = 0, PT_F32 = 1 } pt_dtype;

/* Opaque, device-resident block map.  Owned by the library; free it with
 * pt_blockmap_free.  It depends only on the tree and the tile sizes, so one
 * map serves every layer and both passes ("prefix_grouper_kernel.py",
 * get_block_mask: the mask is cached and reused across layers and steps). */
typedef struct pt_blockmap pt_blockmap;

/* ---------------------------------------------------------------------------
 * pt_build_blockmap_tree -- block map from the tree form.
 *
 * Passage: "cp=1 shared-prefix prefix-tree attention for rollouts": the fold
 * emits the tree as (node_lengths, sample_paths) and the mask is built by
 * AttnMaskSpec.prefix_tree.
 *
 * node_lengths [n_nodes] (host): token count of node i (0 allowed).  Node i
 *   occupies tokens [off_i, off_i + node_lengths[i]) with off the exclusive
 *   prefix sum in id order; T = sum of node_lengths.
 * path_ptr [n_samples + 1], path_nodes [path_ptr[n_samples]] (host): CSR list
 *   of root->leaf paths.  Consecutive entries (a, b) of a path make a the
 *   parent of b.
 * block_m, block_n: q-tile rows and kv-block columns.  The tensor-core
 *   kernels need 128 x 128; the fp32 kernels accept any positive size.
 * stream: the build runs on it.  With 128 x 128 tiles the build does not
 *   wait for the device: the lists are allocated at bounds the host computes
 *   from the node lengths (list entries: the causal tile count; partial
 *   tiles: those in a row or column of tiles holding a node boundary, plus
 *   the diagonal) when those take at most 1 GiB, and the exact list sizes
 *   reach the host behind an event, read on first use (pt_blockmap_info's
 *   nnz and n_full, the exports, the backward's work lists).  Otherwise the
 *   build synchronises the stream once before returning.
 * out: receives the new map.
 *
 * With 128 x 128 tiles the host derives the q-major lists from the node
 * intervals and the device classifies the listed tiles.  The device also
 * sums the kept pairs it finds over the listed tiles and compares the sum
 * with the tree's kept-pair count in closed form (each node's causal
 * triangle plus its tokens times its ancestors' tokens): a listed tile that
 * keeps nothing, or a non-empty tile missing from the lists, records a device
 * error that the next pt_sync_status returns as PT_ERR_INVALID_ARG.
 *
 * Errors: PT_ERR_INVALID_ARG when a length is negative, a path is empty or
 * names a node out of range, a parent does not have a smaller id than its
 * child, two paths disagree on a parent, a path does not start at a root, or
 * a node is on no path.  Nothing is launched in that case.
 * ------------------------------------------------------------------------- */
pt_status pt_build_blockmap_tree(const int32_t* node_lengths, int32_t n_nodes,
                                 const int32_t* path_ptr, const int32_t* path_nodes,
                                 int32_t n_samples, int32_t block_m, int32_t block_n,
                                 cudaStream_t stream, pt_blockmap** out);

/* ---------------------------------------------------------------------------
 * pt_build_blockmap_seg -- block map from per-token segment labels.
 *
 * Passage: "prefix_grouper_kernel.py", PrefixSegInfo and
 * build_seg_info_multigroup: per flat token a group id and a suffix id, -1 on
 * the group's shared-prefix tokens, suffix ids unique across groups.
 *
 * group_id [T], suffix_id [T] (device int32).  Each maximal run of equal
 * (group_id, suffix_id) is one tree node.  A run with suffix_id == -1 is its
 * group's prompt and must open the group; completion runs are its children
 * (roots when the group has no prompt).  Every group id and every suffix id
 * forms exactly one contiguous run; ids lie in [0, T) (suffix ids may also be
 * -1).  Errors: PT_ERR_INVALID_ARG for anything else, detected on the device
 * and returned after the build synchronises the stream.
 * ------------------------------------------------------------------------- */
pt_status pt_build_blockmap_seg(const int32_t* group_id, const int32_t* suffix_id, int32_t T,
                                int32_t block_m, int32_t block_n, cudaStream_t stream,
                                pt_blockmap** out);

/* ---------------------------------------------------------------------------
 * pt_build_blockmap_draft -- block map of the draft-block (DFlash) mask.
 *
 * Passages: "support sequence packing in the Domino and JetSpec drafts" (the
 * query side is the draft blocks only, the context is keys; a block's context
 * prefix is restricted to its anchor's document, create_dflash_block_mask's
 * anchor_positions / block_keep_mask / ctx_doc_id / anchor_doc_id) and the
 * DFlash-family drafter PR (the visibility rule _draft_mask_mod: context
 * before the block, a window counted from each query's real position,
 * block-causal under causal in-block attention).
 *
 * Flat layout, T = ctx_len + n_blocks * block_size: the context tokens
 * first, then block b's tokens at [ctx_len + b * block_size, ... + block_size).
 * Block b's token k sits at real position anchors[b] + k.  Keep rule:
 *   - context rows keep nothing (they are keys only);
 *   - block b's token k keeps context key kv iff kv < anchors[b], and
 *     ctx_doc[kv] == anchor_doc[b] when documents are given, and
 *     (anchors[b] + k) - kv < window when window > 0;
 *   - it keeps its own block's token k' always (causal == 0) or iff k' <= k
 *     (causal != 0), and no other block;
 *   - a block with block_keep[b] == 0 keeps nothing (its rows return 0).
 * anchors [n_blocks] (host) in [0, ctx_len]; block_keep [n_blocks] (host) or
 * NULL for all kept; ctx_doc [ctx_len] and anchor_doc [n_blocks] (host),
 * both or neither; each document id must form one contiguous run of the
 * context.  block_m = block_n = 128 (else PT_ERR_UNSUPPORTED): the kernels
 * read the mask from the map's tile bitmasks.  The build synchronises the
 * stream once.  Errors: PT_ERR_INVALID_ARG for negative sizes, block_size < 1,
 * an anchor out of range, a document split into several runs or only one of
 * the two document arrays.
 * ------------------------------------------------------------------------- */
pt_status pt_build_blockmap_draft(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                                  const uint8_t* block_keep, int32_t causal, int32_t window,
                                  const int32_t* ctx_doc, const int32_t* anchor_doc, int32_t block_m,
                                  int32_t block_n, cudaStream_t stream, pt_blockmap** out);

/* ---------------------------------------------------------------------------
 * pt_blockmap_dense -- the same tree with no tile skipping: every one of the
 * nq x nk tiles is marked partial, so the kernels evaluate the mask on every
 * pair of the T x T square.  This is the "dense masked O(T^2)" comparison the
 * block-sparse map is measured against ("support sequence packing ..." and the
 * drafter speed-up PR: the dense [B, 1, Q, KV] mask path it replaces).
 * ------------------------------------------------------------------------- */
pt_status pt_blockmap_dense(const pt_blockmap* src, cudaStream_t stream, pt_blockmap** out);

/* Sizes of a map: T, nq = ceil(T / block_m), nk = ceil(T / block_n), the
 * number of non-empty tiles and how many of them are full.  Any output
 * pointer may be NULL.  Asking for nnz or n_full waits for the build's device
 * work if the list sizes have not reached the host yet; the other sizes never
 * wait. */
pt_status pt_blockmap_info(const pt_blockmap* bm, int32_t* T, int32_t* block_m, int32_t* block_n,
                           int32_t* nq, int32_t* nk, int64_t* nnz, int64_t* n_full);

/* Host copies of the map, for tests: the q-major list (q_ptr [nq+1]; kv_idx
 * and kind [nnz], kv blocks ascending within a q tile; kind 1 = full,
 * 2 = partial) and its kv-major transpose (k_ptr [nk+1]; q_idx and kindT
 * [nnz], q tiles ascending).  Every pointer is host memory sized by
 * pt_blockmap_info; any may be NULL to skip it. */
pt_status pt_blockmap_export(const pt_blockmap* bm, int32_t* q_ptr, int32_t* kv_idx, uint8_t* kind,
                             int32_t* k_ptr, int32_t* q_idx, uint8_t* kindT);

/* Host copies of the keep bitmasks the tensor-core kernels use (128 x 128
 * maps only), for tests.  Every partial tile has a mask slot; pidx [nnz] and
 * pidxT [nnz] give the slot of each q-major and kv-major entry (-1 for full
 * tiles).  mask_rows [n_partial * 128 * 4]: for slot s, q row r of the tile,
 * word w, bit b is keep(q = 128 i + r, kv = 128 j + 32 w + b); mask_cols
 * [n_partial * 128 * 4] holds the transpose (kv column r, bit over q rows).
 * n_partial = nnz - n_full.  Any pointer may be NULL to skip it;
 * PT_ERR_UNSUPPORTED if the map has no masks (tile sizes other than 128). */
pt_status pt_blockmap_export_masks(const pt_blockmap* bm, int32_t* pidx, int32_t* pidxT, uint32_t* mask_rows,
                                   uint32_t* mask_cols);

/* Release a map.  Its device memory comes from a stream-ordered pool private
 * to the library and is returned in the order of the stream the map was built
 * on, so no device synchronisation happens here.  That stream must still
 * exist, and work that uses the map on other streams must be complete (or
 * ordered before this call on the build stream).  NULL is ignored. */
void pt_blockmap_free(pt_blockmap* bm);

/* ---------------------------------------------------------------------------
 * pt_attn_fwd -- O and LSE.
 *
 * Passage: "prefix_grouper_kernel.py", flex_shared_prefix_attention: softmax
 * attention restricted to the kept pairs, scale 1/sqrt(head_dim) by default,
 * identical in value to dense masked attention.
 *
 * Q [T,Hq,D], K/V [T,Hkv,D] (device, dtype).  O [T,Hq,D] (device, dtype);
 * LSE [Hq,T] (device fp32): LSE = m + ln(sum exp(s - m)) over the kept scores
 * s of the row.  scale <= 0 selects 1/sqrt(D).  The map must have been built
 * for the same T.
 * Supported: PT_BF16 with D in {64, 128, 256, 512} and a 128 x 128 map run
 * on tensor cores (at 512 in two passes over the 256-column halves of O, S
 * computed in both: a 128 x 512 fp32 accumulator would fill TMEM); PT_BF16
 * with another D <= 512 that is a multiple of 8 (or another tile size), and
 * PT_F32 with 1 <= D <= 512, run on CUDA cores with fp32 math.  The drafter
 * PR notes that FlexAttention fails beyond head_dim 256 on sm_103.
 * Hq % Hkv == 0.  Anything else returns PT_ERR_UNSUPPORTED or
 * PT_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
pt_status pt_attn_fwd(const void* Q, const void* K, const void* V, pt_dtype dtype, int32_t T,
                      int32_t Hq, int32_t Hkv, int32_t D, float scale, const pt_blockmap* bm,
                      void* O, float* LSE, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pt_attn_bwd -- dQ, dK, dV.
 *
 * Passage: the backward of the same attention ("prefix_grouper_kernel.py":
 * the compiled backward; the drafter speed-up PR: the FlexAttention GQA
 * backward).  With P = exp(s - LSE), Delta = rowsum(dO * O) and
 * dS = P * (dO V^T - Delta): dV = sum P^T dO, dK = scale sum dS^T Q,
 * dQ = scale dS K, with dK and dV summed over the q heads of each kv head.
 *
 * dO, Q, O [T,Hq,D]; K, V [T,Hkv,D]; LSE [Hq,T] fp32 as pt_attn_fwd wrote it
 * (all device).  Outputs dQ [T,Hq,D], dK/dV [T,Hkv,D] (device, dtype).
 * workspace: device scratch of at least pt_bwd_workspace_bytes(T, Hq, D)
 * bytes, 256-byte aligned, owned by the caller; its contents on entry do not
 * matter.  Calls that share one workspace must not overlap on the GPU.  Its
 * size also picks the head_dim-64 backward (see pt_bwd_workspace_bytes): the
 * full size gives the one-pass kernel, whose dQ may differ between runs in
 * its last bits; the two row statistics alone give the two-pass kernels.
 * Supported shapes as for pt_attn_fwd.
 * ------------------------------------------------------------------------- */
pt_status pt_attn_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                      const float* LSE, pt_dtype dtype, int32_t T, int32_t Hq, int32_t Hkv,
                      int32_t D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of scratch pt_attn_bwd needs: two fp32 row statistics of [Hq, Tpad]
 * entries each, Tpad = ceil(T / 128) * 128 -- -Delta = -rowsum(dO * O) and
 * -LSE * log2(e), stored negated -- then, at head_dim 64 only, an fp32 dQ accumulator of
 * Tpad * Hq * 64 floats, then room for fp32 partial sums, 128 x 2D floats
 * per slot, min(256, 2 * ceil(T/128) * Hq) slots, each part rounded up to
 * 256 bytes.  The partial sums let the tensor-core backward split long
 * kv-major columns across SMs; a smaller workspace (at least the two
 * statistics) is accepted and only splits less.
 * At head_dim 64 (bf16, 128 x 128 tiles) a workspace with room for the dQ
 * accumulator after the statistics selects the one-pass backward: dQ is
 * summed in fp32 by asynchronous adds whose order varies, so dQ may differ
 * between runs in its last bits.  A smaller workspace selects the two-pass
 * backward, whose every output element is written once (run-to-run
 * identical), with the rest of the workspace as partial-sum room. */
size_t pt_bwd_workspace_bytes(int32_t T, int32_t Hq, int32_t D);

/* ---------------------------------------------------------------------------
 * pt_attn_bwd_noalloc -- pt_attn_bwd for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a deployment convenience.
 *
 * Who needs it: a program that embeds this library but owns every byte of
 * device memory through its own allocator (a serving process, a training
 * framework's caching allocator) and offers no way to hand out scratch, or a
 * latency-critical caller for which cudaMalloc, which may synchronise the
 * device, is off limits.  The call takes the same inputs and outputs as
 * pt_attn_bwd but no workspace: its scratch (the -Delta and -LSE*log2(e) rows)
 * lives in a fixed array inside the library, and it calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Limit: the array holds pt_bwd_noalloc_max_scratch_bytes() bytes (8 MiB);
 * shapes that need more (2 * Hq * ceil(T/128)*128 fp32 values, each half
 * rounded up to 256 bytes) return PT_ERR_INVALID_ARG with a message, and
 * pt_attn_bwd with a caller workspace must be used instead.  Every GPU that
 * loads the library keeps the array until the process exits.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls on a device share the one array:
 * calls whose kernels overlap on the GPU (different streams, or different host
 * threads) race and give wrong results, so order them.  Each call overwrites
 * the scratch it reads, so no clearing between calls is needed.
 * The tensor-core backward also reads per-map work lists (which kv-major and
 * q-major work items each SM runs).  They are built once per block map and
 * head layout by pt_blockmap_prepare_bwd, which allocates them in the map's
 * own memory; a call whose map has no lists for its layout returns
 * PT_ERR_INVALID_ARG without launching anything.  The lists are kept per
 * (Hq / Hkv, Hkv, the device's SM count) for the kv-major kernel and per
 * (Hq, SM count) for the q-major kernels at head dims 128, 256 and 512;
 * head dims 64 and 128 share the kv-major lists.  pt_attn_bwd with a workspace
 * builds lists of its own (long columns split across SMs) beside these and
 * never replaces or frees them: every layout's lists stay with the map until
 * pt_blockmap_free.  Maps used only with the CUDA-core paths (fp32, tiles
 * other than 128 x 128, head dims other than 64, 128, 256 and 512) need no
 * lists, and preparing them is a no-op.
 * After cudaDeviceReset the library must not be used again in the process:
 * the array's looked-up address, like every map and pool, belongs to the
 * context that the reset destroyed.
 * Shapes, dtypes, layouts and errors are otherwise those of pt_attn_bwd.
 * ------------------------------------------------------------------------- */
pt_status pt_attn_bwd_noalloc(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                              const float* LSE, pt_dtype dtype, int32_t T, int32_t Hq, int32_t Hkv,
                              int32_t D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV,
                              cudaStream_t stream);

/* Capacity in bytes of the built-in scratch array of pt_attn_bwd_noalloc. */
size_t pt_bwd_noalloc_max_scratch_bytes(void);

/* ---------------------------------------------------------------------------
 * pt_hoststep -- forward and backward from host memory, one step per call.
 *
 * Passage: "prefix_grouper_kernel.py", flex_shared_prefix_attention runs on
 * tensors already on the GPU; a training step still moves each batch's
 * inputs in and its gradients out.  This object holds two device copies of
 * Q, K, V, dO, O, LSE, dQ, dK, dV (and one backward workspace) and
 * alternates between them, so one call's uploads and the previous call's
 * downloads overlap the kernels in between.
 *
 * pt_hoststep_create: buffers for one shape (layouts as pt_attn_fwd /
 *   pt_attn_bwd: Q, dO, dQ [T, Hq, D]; K, V, dK, dV [T, Hkv, D]) on the
 *   current device; two non-blocking copy streams of its own.  Errors:
 *   PT_ERR_INVALID_ARG for a bad dtype or sizes, PT_ERR_UNSUPPORTED for a
 *   head_dim the attention calls do not take (above 512, or not a multiple
 *   of 8 for bf16), PT_ERR_NOMEM.
 * pt_hoststep_run: hQ, hK, hV, hdO (host, read) and hdQ, hdK, hdV (host,
 *   written) are the caller's; pinned memory (cudaHostAlloc or registered)
 *   gives the overlap, pageable memory works but each copy then blocks.  The
 *   uploads go on the object's upload stream, the forward and backward on
 *   `stream` (after the uploads; the map must be built for the same T), the
 *   downloads on the object's download stream after the kernels.  Returns
 *   once everything is queued: the host buffers must stay untouched until
 *   pt_hoststep_sync's stream point has been reached.  Errors: as
 *   pt_attn_fwd / pt_attn_bwd, PT_ERR_INVALID_ARG for NULL pointers or a
 *   map of another T.
 * pt_hoststep_sync: makes `stream` wait for every download queued so far
 *   (synchronise the stream, or record an event on it, to wait on the host).
 * pt_hoststep_last_forward: copies the forward outputs of the most recent
 *   pt_hoststep_run, O [T, Hq, D] (dtype) and LSE [Hq, T] (fp32), into host
 *   memory hO and hLSE; waits for that step's kernels first (blocking).  For
 *   tests and inspection: a training step needs only the gradients.  Must be
 *   called before the next pt_hoststep_run reuses that step's buffers.
 *   Errors: PT_ERR_INVALID_ARG for NULL pointers or before any run.
 * pt_hoststep_free: waits for the object's copies and frees it.
 * ------------------------------------------------------------------------- */
typedef struct pt_hoststep pt_hoststep;
pt_status pt_hoststep_create(pt_dtype dtype, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, pt_hoststep** out);
pt_status pt_hoststep_run(pt_hoststep* h, const void* hQ, const void* hK, const void* hV, const void* hdO,
                          float scale, const pt_blockmap* bm, void* hdQ, void* hdK, void* hdV, cudaStream_t stream);
pt_status pt_hoststep_sync(pt_hoststep* h, cudaStream_t stream);
pt_status pt_hoststep_last_forward(pt_hoststep* h, void* hO, float* hLSE);
void pt_hoststep_free(pt_hoststep* h);

/* ---------------------------------------------------------------------------
 * Shared-prefix fold of rollouts, and its inverse.
 *
 * Passage: "cp=1 shared-prefix prefix-tree attention for rollouts", PR
 * description: a group of one prompt and N sampled completions is folded
 * into one deduplicated flat sequence [prompt | c_0 | c_1 | ...] (the prompt
 * is encoded once instead of N times), each completion gets position ids
 * that continue from its prompt, and the tree is handed on as
 * (node_lengths, sample_paths).  The plan takes that same tree, so one
 * description drives the fold, pt_build_blockmap_tree and the unfold; the
 * shared-prefix group is the depth-2 tree [prompt, c_i], multi-turn rollouts
 * are deeper trees.
 *
 * Layouts.  Flat: node i owns tokens [off_i, off_i + node_lengths[i]), off
 * the exclusive prefix sum in id order (the attention calls' layout).
 * Rollouts: n_samples rows of row_len tokens; row s holds the tokens of its
 * path's nodes, root first, at positions 0, 1, ..., then padding.  A token's
 * data is one contiguous row of row_bytes bytes in both layouts (an id, a
 * hidden state, a Q row...), so a flat tensor is [T, row] and a rollout
 * tensor [n_samples, row_len, row], densely packed.
 *
 * pt_fold_plan: validates the tree as pt_build_blockmap_tree does (every
 *   node on some path, one parent per node, parents before children) and
 *   that no path is longer than row_len; builds the per-token and per-entry
 *   maps on the device (stream-ordered, library-owned memory).  Host arrays
 *   as pt_build_blockmap_tree.  Errors: PT_ERR_INVALID_ARG (malformed tree,
 *   a path longer than row_len, n_samples * row_len >= 2^31), PT_ERR_NOMEM,
 *   PT_ERR_CUDA.
 * pt_fold: flat[t] = roll[the first sample holding token t][its position]:
 *   the deduplication; the other samples are expected to hold the same
 *   bytes there (pt_fold_mismatches checks).  roll is read, flat written.
 * pt_unfold: roll[s][j] = flat[the token at position j of sample s]; shared
 *   tokens are copied into every row that holds them; padding entries are
 *   zero-filled.
 * pt_unfold_grad: the adjoint of pt_unfold, for the backward pass of a loss
 *   taken on the rollout rows: dflat[t] = sum over every copy of t of
 *   droll[s][j] (padding ignored).  Elements are dtype (bf16 or fp32),
 *   width per token; sums are taken in fp32 in sample order (deterministic)
 *   and rounded once to dtype (round to nearest even).
 * pt_fold_positions: pos[t] = the position of token t in the rows that hold
 *   it (int64 [T], the RoPE position ids): a completion's positions continue
 *   from its prompt's.
 * pt_fold_mismatches: *count (device, one unsigned 64-bit counter, zeroed by
 *   the call) = the number of rollout entries whose bytes differ from the
 *   entry pt_fold keeps for their token; 0 when the rollouts really share
 *   their prefixes.
 * Device buffers are the caller's; any alignment works (the kernels move the
 * widest unit that row_bytes and the base addresses allow).  Every call is
 * ordered on `stream` and returns PT_ERR_INVALID_ARG for a NULL plan or
 * buffer, a non-positive row_bytes or width, or a plan of another device.
 * pt_foldplan_free returns the plan's memory in its build stream's order.
 * ------------------------------------------------------------------------- */
typedef struct pt_foldplan pt_foldplan;
pt_status pt_fold_plan(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr,
                       const int32_t* path_nodes, int32_t n_samples, int32_t row_len, cudaStream_t stream,
                       pt_foldplan** out);
pt_status pt_foldplan_info(const pt_foldplan* plan, int32_t* T, int32_t* n_samples, int32_t* row_len);
void pt_foldplan_free(pt_foldplan* plan);
pt_status pt_fold(const pt_foldplan* plan, const void* roll, int64_t row_bytes, void* flat, cudaStream_t stream);
pt_status pt_unfold(const pt_foldplan* plan, const void* flat, int64_t row_bytes, void* roll, cudaStream_t stream);
pt_status pt_unfold_grad(const pt_foldplan* plan, const void* droll, pt_dtype dtype, int64_t width, void* dflat,
                         cudaStream_t stream);
pt_status pt_fold_positions(const pt_foldplan* plan, int64_t* pos, cudaStream_t stream);
pt_status pt_fold_mismatches(const pt_foldplan* plan, const void* roll, int64_t row_bytes, unsigned long long* count,
                             cudaStream_t stream);

/* Synchronise the stream, then return and clear the device status word:
 * PT_ERR_TIMEOUT if an in-kernel wait ran out since the last check,
 * PT_ERR_INVALID_ARG if a device-side check of a block map failed (see
 * pt_build_blockmap_tree and pt_build_blockmap_seg), PT_ERR_CUDA if the
 * stream reported an error, else PT_OK. */
pt_status pt_sync_status(cudaStream_t stream);

/* Message for the last failing call on this thread ("" if none). */
const char* pt_last_error(void);

/* Number of kernel launches the library has issued in this process (all
 * devices, all entry points).  Used by benchmarks to count launches. */
uint64_t pt_launch_count(void);

/* Failure-path check: launch a one-thread kernel that waits on a barrier
 * nothing will complete, using the same bounded wait as the attention
 * kernels.  The wait gives up after about one second and the kernel returns
 * normally, so the context stays usable; the next pt_sync_status on this
 * stream returns PT_ERR_TIMEOUT.  Meant for tests of error reporting; the
 * pages have no counterpart. */
pt_status pt_debug_wait_timeout(cudaStream_t stream);

/* Builds the work lists pt_attn_bwd_noalloc needs for block map bm and head
 * layout (Hq, Hkv, D): the kv-major items packed onto the SMs (no column is
 * split, since that call has no workspace for partial sums) and, at
 * head_dims 128, 256 and 512, the q-major items of the dQ kernels.
 * Allocates them from the library's stream-ordered pool in the map's
 * ownership (freed with the map) and uploads them on `stream`.  A no-op
 * where the backward runs on the CUDA-core kernels (fp32, tiles other than
 * 128 x 128, head dims other than 64, 128, 256 and 512).  Idempotent; returns PT_ERR_INVALID_ARG for a NULL
 * map or a bad head layout and PT_ERR_UNSUPPORTED for head_dim above 512, as
 * pt_attn_bwd does.  The pages have no counterpart. */
pt_status pt_blockmap_prepare_bwd(const pt_blockmap* bm, int32_t Hq, int32_t Hkv, int32_t D, cudaStream_t stream);

/* Test hook for the device-side check of host-built lists: the next n
 * pt_build_blockmap_tree (128 x 128 tiles) or pt_build_blockmap_draft calls
 * each drop one non-empty
 * tile (the last entry of the longest q-tile list) from the lists the host
 * builds, keeping lengths and offsets consistent, so that only the kept-pair
 * check can notice; n <= 0 cancels.  For tests only: the maps it makes are
 * wrong.  The pages have no counterpart. */
void pt_debug_drop_listed_tile(int32_t n);

/* Bytes of the library's private device memory pool on `device`: handed out
 * now (*used_bytes) and held from the device (*reserved_bytes).  The pool is
 * where block maps, fold plans and backward work lists live.  Meant for tests
 * (for instance, that pt_attn_bwd_noalloc on a prepared map takes nothing
 * from it); the pages have no counterpart.  PT_ERR_INVALID_ARG for NULL
 * outputs or a negative device. */
pt_status pt_debug_pool_usage(int32_t device, uint64_t* used_bytes, uint64_t* reserved_bytes);

/* Host-only check of a tree map's lists (no GPU work): the q-major lists that
 * pt_build_blockmap_tree derives on the host for the tree (node_lengths,
 * path_ptr, path_nodes, as that call takes them) at block_m x block_n tiles,
 * before the device classifies the listed tiles: q_ptr[nq + 1] offsets (nq =
 * ceil(T / block_m), room for q_ptr_len entries) into kv_idx[cap], each q
 * tile's kv blocks ascending, and *nnz the entries.  The same host checks as
 * pt_build_blockmap_tree (PT_ERR_INVALID_ARG for a malformed tree), and
 * PT_ERR_INVALID_ARG for too little room (*nnz is still written).  Meant for
 * tests; the pages have no counterpart. */
pt_status pt_debug_tree_lists(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr,
                              const int32_t* path_nodes, int32_t n_samples, int32_t block_m, int32_t block_n,
                              int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx, int64_t cap, int64_t* nnz);

/* Host-only check of a draft-block map's lists (no GPU work): for the layout
 * pt_build_blockmap_draft takes (same arguments, 128 x 128 tiles), the
 * q-major lists its build derives on the host (q_ptr[nq + 1], nq =
 * ceil(T / 128), room for q_ptr_len entries; kv_idx[cap], each q tile's kv
 * blocks ascending; *nnz entries) and the closed-form count of every kept
 * (q, kv) pair that the device's check compares its sum with (*kept_pairs).
 * The same host checks as pt_build_blockmap_draft; PT_ERR_INVALID_ARG also
 * for too little room (*nnz is still written).  Meant for tests; the pages
 * have no counterpart. */
pt_status pt_debug_draft_lists(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                               const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                               const int32_t* anchor_doc, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx,
                               int64_t cap, int64_t* nnz, int64_t* kept_pairs);

/* Host-only check of the backward's q-major work lists (no GPU work): for a
 * map whose q tile t has row_steps[t] listed kv blocks (nq tiles) and Hq q
 * heads, packs the (q tile, q head) items onto `ctas` CTAs exactly as the
 * dQ kernels at head_dims 128, 256 and 512 get them: longest first onto the
 * least loaded CTA.  Writes, per item in CTA order, 4 int32 (q tile, q head,
 * first list entry, kv blocks) to items[4 * cap_items], per CTA 4 int32
 * (first item, end item, kv blocks, 0) to cta_rec[4 * ctas], and *n_items,
 * *grid and *n_empty (q tiles with no kv block, which get no item).
 * PT_ERR_INVALID_ARG for bad arguments or fewer than *n_items rows of room.
 * Meant for tests; the pages have no counterpart. */
pt_status pt_debug_pack_dq(const int32_t* row_steps, int32_t nq, int32_t Hq, int32_t ctas, int32_t* items,
                           int64_t cap_items, int32_t* cta_rec, int32_t* n_items, int32_t* grid, int32_t* n_empty);

/* Host-only check of the backward's kv-major work lists (no GPU work): for a
 * map whose kv block j has col_steps[j] listed q tiles (nk blocks), g q heads
 * per kv head and Hkv kv heads, packs the items onto `ctas` CTAs exactly as
 * pt_attn_bwd does: with exact_fill (the one-pass head_dim-64 kernel's
 * packing) the columns laid end to end and cut at equal per-CTA budgets when
 * max_slots partial-sum slots suffice, else longest first onto the least
 * loaded CTA, columns longer than about one CTA's share cut into equal
 * chunks (max_slots <= 0: none cut).  A column's steps are its (q head,
 * listed q tile) pairs, g * col_steps[j] of them.  Writes, per item in CTA
 * order, 5 int32 (kv block, kv head, first step, end step, slot or -1 for a
 * whole column) to items[5 * cap_items], cta_ptr[grid + 1] (CTA b runs items
 * [cta_ptr[b], cta_ptr[b + 1]); room for ctas + 1 entries), and *n_items,
 * *n_slots, *grid.  PT_ERR_INVALID_ARG for bad arguments or fewer than
 * *n_items rows of room (the counts are still written).  Meant for tests;
 * the pages have no counterpart. */
pt_status pt_debug_pack_dkdv(const int32_t* col_steps, int32_t nk, int32_t g, int32_t Hkv, int32_t max_slots,
                             int32_t ctas, int32_t exact_fill, int32_t* items, int64_t cap_items, int32_t* cta_ptr,
                             int32_t* n_items, int32_t* n_slots, int32_t* grid);

/* Accuracy check of the kernels' two exp2 paths: y[i] = 2^x[i] for i < n,
 * computed with the MUFU instruction (method 0) or with the FMA-pipe
 * polynomial (method 1: Cody-Waite range reduction and a degree-3 minimax
 * polynomial, max relative error 7.8e-5 on [-125, 0], a value in
 * [0, 2^-124] below -125, including -inf) that the softmax loops use for a
 * fixed share of the columns.
 * x and y are device pointers to n floats, owned by the caller.  Returns
 * PT_ERR_INVALID_ARG for n < 0, NULL pointers with n > 0 or another method.
 * Meant for tests; the pages have no counterpart. */
pt_status pt_debug_exp2(const float* x, float* y, int64_t n, int32_t method, cudaStream_t stream);

/* Optional per-kernel timing, for benchmarks and profiling.  While enabled,
 * each kernel launch is bracketed by two CUDA events on its stream, taken
 * from a per-device pool that enabling stocks with 1024 events; disabled
 * (the default) costs one branch.  pt_profile_read synchronises the recorded
 * events and returns the number of launches and their summed duration for
 * one scope name: "fwd_tc", "fwd_simt", "bwd_prep", "bwd_dkdv",
 * "bwd_dkdv_finalize", "bwd_fused" (the one-pass head_dim-64 backward),
 * "bwd_fused_finalize" (its split columns and dQ), "bwd_dv", "bwd_dk",
 * "bwd_dq", "bwd_simt",
 * "blockmap_classify" (tile classes, list sizes, orders),
 * "blockmap_lists" (lists and masks), and the fold calls' "fold_plan",
 * "fold", "unfold", "unfold_grad", "fold_positions", "fold_mismatches".  pt_profile_reset drops every record
 * (its events go back to the pool once they have completed). */
void pt_profile_enable(int on);
pt_status pt_profile_read(const char* kernel, int64_t* launches, double* total_ms);
void pt_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* PT_H_ */
