// pt_blockmap.cu -- the block map: per-token tree coordinates, the class of
// every (q tile, kv block) pair (empty / full / partial), and the q-major list
// with its kv-major transpose.
//
// "prefix_grouper_kernel.py", get_block_mask / create_block_mask: the mask is
// turned into per-tile lists so that masked-out blocks are never computed;
// fully kept tiles skip the per-element mask.  Here the class of a tile is
// counted exactly from the tree (no per-element evaluation): row q keeps, in
// a kv range [k0, k1), the overlap with each proper ancestor node's tokens plus
// the overlap with [start(node(q)), q].
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <numeric>
#include <unordered_map>
#include <vector>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_blockmap(cudaStream_t s) { return take_status_here(s); }

namespace {

constexpr int kScanBlock = 1024;

#define PT_CU(call)                                                                          \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess) {                                                                 \
      set_error("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return 3;                                                                              \
    }                                                                                        \
  } while (0)

// ---------------------------------------------------------------------------
// scans: exclusive prefix sum of n int32 values into out[0..n] (out[n] = total)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_incl_scan(int v, int* sh) {
  // sh: at least 32 ints
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (blockDim.x >> 5)) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    sh[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += sh[warp - 1];
  __syncthreads();
  return v;
}

__global__ void k_scan_blocks(const int* in, int n, int* out, int* block_sums) {
  __shared__ int sh[32];
  int i = blockIdx.x * kScanBlock + threadIdx.x;
  int v = (i < n) ? in[i] : 0;
  int incl = block_incl_scan(v, sh);
  if (i < n) out[i] = incl - v;
  if (threadIdx.x == kScanBlock - 1) block_sums[blockIdx.x] = incl;
}

// Exclusive scan of block sums in one block (loops over chunks), total at [nb].
__global__ void k_scan_sums(int* sums, int nb) {
  __shared__ int sh[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += kScanBlock) {
    int i = base + threadIdx.x;
    int v = (i < nb) ? sums[i] : 0;
    int incl = block_incl_scan(v, sh);
    int c = carry;
    if (i < nb) sums[i] = c + incl - v;
    __syncthreads();
    if (threadIdx.x == kScanBlock - 1) carry = c + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) sums[nb] = carry;
}

__global__ void k_scan_add(int* out, int n, const int* sums, int nb) {
  int i = blockIdx.x * kScanBlock + threadIdx.x;
  if (i < n) out[i] += sums[blockIdx.x];
  if (i == 0) out[n] = sums[nb];
}

// out has n + 1 entries; tmp has at least nblocks + 1 entries.
int exclusive_scan(const int* in, int n, int* out, int* tmp, cudaStream_t s) {
  int nb = (n + kScanBlock - 1) / kScanBlock;
  if (nb == 0) {
    PT_CU(cudaMemsetAsync(out, 0, sizeof(int), s));
    return 0;
  }
  k_scan_blocks<<<nb, kScanBlock, 0, s>>>(in, n, out, tmp);
  k_scan_sums<<<1, kScanBlock, 0, s>>>(tmp, nb);
  k_scan_add<<<nb, kScanBlock, 0, s>>>(out, n, tmp, nb);
  count_launch(3);
  PT_CU(cudaGetLastError());
  return 0;
}

// ---------------------------------------------------------------------------
// tree form: per-token coordinates from device node tables
// ---------------------------------------------------------------------------
__global__ void k_tree_tokens(int T, int tpad, int n_nodes, const int* node_end, const int* tin, const int* tout,
                              pt_tok* tok, int* node_of) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= tpad) return;
  if (t >= T) {
    tok[t] = pt_tok{INT_MAX, 0};
    return;
  }
  // first node whose end is past t (zero-length nodes are skipped)
  int lo = 0, hi = n_nodes - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (node_end[mid] > t)
      hi = mid;
    else
      lo = mid + 1;
  }
  tok[t] = pt_tok{tin[lo], tout[lo]};
  node_of[t] = lo;
}

// ---------------------------------------------------------------------------
// segment form
// ---------------------------------------------------------------------------
// Run starts plus local checks.  err: bit 0 = id out of range, bit 1 = prompt
// run not opening its group.
__global__ void k_seg_flags(const int* g, const int* sfx, int T, int* flags, int* group_seen, int* suffix_seen,
                            int* err) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int gi = g[t], si = sfx[t];
  if (gi < 0 || gi >= T || si < -1 || si >= T) {
    atomicOr(err, 1);
    flags[t] = 0;
    return;
  }
  bool new_group = (t == 0) || g[t - 1] != gi;
  bool new_run = new_group || sfx[t - 1] != si;
  flags[t] = new_run ? 1 : 0;
  if (new_group) atomicAdd(&group_seen[gi], 1);
  if (new_run && si >= 0) atomicAdd(&suffix_seen[si], 1);
  if (new_run && si == -1 && !new_group) atomicOr(err, 2);
}

__global__ void k_seen_check(const int* group_seen, const int* suffix_seen, int T, int* err) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  if (group_seen[t] > 1) atomicOr(err, 4);   // a group id in two runs
  if (suffix_seen[t] > 1) atomicOr(err, 8);  // a suffix id in two runs
}

// run[t] = inclusive count of run starts up to t, minus one.
__global__ void k_seg_nodes(const int* g, const int* sfx, int T, const int* flags, const int* excl, int* node_of,
                            int* node_start, int* node_end, int* grp_first, int* grp_last) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int r = excl[t] + flags[t] - 1;
  node_of[t] = r;
  if (flags[t]) {
    node_start[r] = t;
    if (r > 0) node_end[r - 1] = t;
  }
  if (t == T - 1) node_end[r] = T;
  int gi = g[t];
  if (t == 0 || g[t - 1] != gi) grp_first[gi] = r;
  if (t == T - 1 || g[t + 1] != gi) grp_last[gi] = r;
  (void)sfx;
}

// Per node: parent, Euler interval.  Node ids are run order; a prompt run
// spans its whole group's runs, a completion run only itself.
__global__ void k_seg_tree(const int* g, const int* sfx, int R, const int* node_start, const int* grp_first,
                           const int* grp_last, int* parent, int* tin, int* tout) {
  int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  int t = node_start[r];
  int gi = g[t], si = sfx[t];
  tin[r] = r;
  if (si == -1) {
    parent[r] = -1;
    tout[r] = grp_last[gi] + 1;
  } else {
    int f = grp_first[gi];
    parent[r] = (sfx[node_start[f]] == -1) ? f : -1;
    tout[r] = r + 1;
  }
}

__global__ void k_seg_tokens(int T, int tpad, const int* node_of, const int* tin, const int* tout, pt_tok* tok) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= tpad) return;
  if (t >= T) {
    tok[t] = pt_tok{INT_MAX, 0};
    return;
  }
  int r = node_of[t];
  tok[t] = pt_tok{tin[r], tout[r]};
}

// ---------------------------------------------------------------------------
// tile classes: one warp per (q tile, kv block)
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long overlap(long long a0, long long a1, long long b0, long long b1) {
  long long lo = a0 > b0 ? a0 : b0, hi = a1 < b1 ? a1 : b1;
  return hi > lo ? hi - lo : 0;
}

__global__ void k_classify(int T, int BM, int BN, int nq, int nk, const int* node_of, const int* node_start,
                           const int* node_end, const int* parent, uint8_t* kinds, int* counters, int* row_cnt,
                           int* col_cnt, int* row_part) {
  pdl_wait();  // launched with programmatic dependent launch
  long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (w >= (long long)nq * nk) return;
  int i = (int)(w / nk), j = (int)(w % nk);
  long long q0 = (long long)i * BM, k0 = (long long)j * BN, k1 = k0 + BN;
  long long qlast = q0 + BM - 1 < T - 1 ? q0 + BM - 1 : T - 1;
  if (k0 > qlast) {  // every kv after every q
    if (lane == 0) kinds[w] = PT_KIND_EMPTY;
    return;
  }
  long long kept = 0;
  for (long long q = q0 + lane; q <= qlast; q += 32) {
    int n = node_of[q];
    kept += overlap(node_start[n], q + 1, k0, k1);
    for (int a = parent[n]; a != -1; a = parent[a]) kept += overlap(node_start[a], node_end[a], k0, k1);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
  if (lane == 0) {
    bool in_range = (q0 + BM <= T) && (k1 <= T);
    uint8_t kd = kept == 0 ? PT_KIND_EMPTY
                           : ((in_range && kept == (long long)BM * BN) ? PT_KIND_FULL : PT_KIND_PARTIAL);
    kinds[w] = kd;
    if (kd != PT_KIND_EMPTY) {
      atomicAdd(&row_cnt[i], 1);
      atomicAdd(&col_cnt[j], 1);
      if (kd == PT_KIND_FULL)
        atomicAdd(&counters[0], 1);
      else
        atomicAdd(&row_part[i], 1);
    }
  }
}

// ---------------------------------------------------------------------------
// draft-block form ("support sequence packing in the Domino and JetSpec
// drafts" and the DFlash-family drafter PR: draft blocks attend to the context
// before their anchor, optionally restricted to the anchor's document and to a
// window counted from each query's real position, and to their own block,
// bidirectionally or causally; context rows are keys only)
// ---------------------------------------------------------------------------
struct DraftParams {
  int S, bs, causal, window;
  const int4* blk;  // per block: kept context [x, y) before any window, anchor z, keep flag w
};

DraftParams draft_params(const pt_blockmap* bm) {
  return DraftParams{bm->d_ctx, bm->d_bs, bm->d_causal, bm->d_window, static_cast<const int4*>(bm->d_blk)};
}

// Kept keys of row q: context [c0, c1) and its own block's [b0, b1) (empty
// ranges for context rows and dropped blocks).
__device__ __forceinline__ void draft_row(const DraftParams& d, int q, int& c0, int& c1, int& b0, int& b1) {
  c0 = c1 = b0 = b1 = 0;
  if (q < d.S) return;
  const int b = (q - d.S) / d.bs, k = (q - d.S) % d.bs;
  const int4 bl = d.blk[b];
  if (!bl.w) return;
  c0 = bl.x;
  c1 = bl.y;
  if (d.window > 0) c0 = max(c0, bl.z + k - d.window + 1);  // real position bl.z + k minus kv < window
  if (c1 < c0) c1 = c0;
  b0 = d.S + b * d.bs;
  b1 = b0 + (d.causal ? k + 1 : d.bs);
}

// Maps whose lists the host built (128 x 128 tiles; trees, and draft maps
// with DRAFT): one launch writes the token table (trees: blocks
// [0, tok_blocks), as k_tree_tokens) and, in the other blocks, copies the
// node tables and the host lists from the packed upload into the map and
// classifies every listed tile (trees: from the ancestor intervals; draft
// maps: from each row's two key ranges), full or partial,
// numbering partial tiles in the order they are found (a mask slot is
// reached only through pidx and pidxT).  Packed upload (ints): counters[4]
// (zero) | node tables[5 * N] | q_ptr[nq + 1] |
// k_ptr[nk + 1] | q_order[nq] | k_order[nk] | kv_idx[nnz] | q_idx[nnz] |
// eT[nnz] (kv-major position of each q-major entry).  counters[0] counts full
// tiles and counters[1] hands out mask slots.  A listed tile that keeps
// nothing would mean the host's lists are wrong: it is recorded as an error
// and kept as a partial tile (its mask is empty, so results stay exact).
template <bool DRAFT>
__global__ void k_tree_listed(int T, int tpad, int N, int* __restrict__ map_tabs, pt_tok* __restrict__ tok,
                              int* __restrict__ node_of, int tok_blocks, int* __restrict__ pk, int nq, int nk, int nnz,
                              int* __restrict__ q_ptr, int* __restrict__ k_ptr, int* __restrict__ q_order,
                              int* __restrict__ k_order, int* __restrict__ kv_idx, int* __restrict__ q_idx,
                              uint8_t* __restrict__ kind, int* __restrict__ pidx, uint8_t* __restrict__ kindT,
                              int* __restrict__ pidxT, int2* __restrict__ slot_tile, long long p_cap,
                              DraftParams d) {
  pdl_wait();  // launched with programmatic dependent launch
  // node tables (start | end | parent | tin | tout) come in the packed upload
  // and are read from there; the list blocks also copy them into the map
  const int* tabs = pk + 4;
  const int* node_start = tabs;
  const int* node_end = tabs + N;
  const int* parent = tabs + 2 * N;
  const int* tin = tabs + 3 * N;
  const int* tout = tabs + 4 * N;
  if ((int)blockIdx.x < tok_blocks) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= tpad) return;
    if (t >= T) {
      tok[t] = pt_tok{INT_MAX, 0};
      return;
    }
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (node_end[mid] > t)
        hi = mid;
      else
        lo = mid + 1;
    }
    tok[t] = pt_tok{tin[lo], tout[lo]};
    node_of[t] = lo;
    return;
  }
  int* counters = pk;
  const int* s_qp = tabs + 5 * N;
  const int* s_kp = s_qp + nq + 1;
  const int* s_qo = s_kp + nk + 1;
  const int* s_ko = s_qo + nq;
  const int* s_kv = s_ko + nk;
  const int* s_qi = s_kv + nnz;
  const int* s_et = s_qi + nnz;
  const long long tid = (long long)(blockIdx.x - tok_blocks) * blockDim.x + threadIdx.x;
  const long long nth = (long long)(gridDim.x - tok_blocks) * blockDim.x;
  // the host lists into the map
  const long long n_small = (long long)5 * N + 2 * nq + 2 * nk + 2 + 2 * (long long)nnz;
  for (long long x = tid; x < n_small; x += nth) {
    long long y = x;
    if (y < 5LL * N) { map_tabs[y] = tabs[y]; continue; }
    y -= 5LL * N;
    if (y < nq + 1) { q_ptr[y] = s_qp[y]; continue; }
    y -= nq + 1;
    if (y < nk + 1) { k_ptr[y] = s_kp[y]; continue; }
    y -= nk + 1;
    if (y < nq) { q_order[y] = s_qo[y]; continue; }
    y -= nq;
    if (y < nk) { k_order[y] = s_ko[y]; continue; }
    y -= nk;
    if (y < nnz) { kv_idx[y] = s_kv[y]; continue; }
    y -= nnz;
    q_idx[y] = s_qi[y];
  }
  // classes of the listed tiles: one warp per entry
  const int lane = threadIdx.x & 31;
  for (long long e = tid >> 5; e < nnz; e += nth >> 5) {
    int lo = 0, hi = nq - 1;  // q tile of the entry: last i with q_ptr[i] <= e
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_qp[mid] <= e)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int i = lo, j = s_kv[e];
    const long long q0 = (long long)i * 128, k0 = (long long)j * 128, k1 = k0 + 128;
    const long long qlast = q0 + 127 < T - 1 ? q0 + 127 : T - 1;
    long long kept = 0;
    for (long long q = q0 + lane; q <= qlast; q += 32) {
      if constexpr (DRAFT) {
        const long long kend = k1 < T ? k1 : T;
        int c0, c1, b0, b1;
        draft_row(d, (int)q, c0, c1, b0, b1);
        kept += overlap(c0, c1, k0, kend) + overlap(b0, b1, k0, kend);
      } else {
        int a = 0, b = N - 1;
        while (a < b) {
          const int mid = (a + b) >> 1;
          if (node_end[mid] > q)
            b = mid;
          else
            a = mid + 1;
        }
        kept += overlap(node_start[a], q + 1, k0, k1);
        for (int u = parent[a]; u != -1; u = parent[u]) kept += overlap(node_start[u], node_end[u], k0, k1);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
    if (lane == 0) {
      const bool in_range = q0 + 128 <= T && k1 <= T;
      const bool full = in_range && kept == 128LL * 128;
      if (kept == 0) record_status(PT_STATUS_INVALID);
      // the kept pairs of every listed tile add up to all kept pairs of the
      // tree only if no non-empty tile is missing from the host's lists
      atomicAdd(reinterpret_cast<unsigned long long*>(counters + 2), (unsigned long long)kept);
      const int et = s_et[e];
      if (full) {
        kind[e] = kindT[et] = PT_KIND_FULL;
        pidx[e] = pidxT[et] = -1;
        atomicAdd(&counters[0], 1);
      } else {
        kind[e] = kindT[et] = PT_KIND_PARTIAL;
        const int slot = atomicAdd(&counters[1], 1);
        if (slot < p_cap) {
          pidx[e] = pidxT[et] = slot;
          slot_tile[slot] = make_int2(i, j);
        } else {  // more partial tiles than the allocation's bound: never written past it
          pidx[e] = pidxT[et] = -1;
          record_status(PT_STATUS_INVALID);
        }
      }
    }
  }
}

// Exclusive scans of up to three small arrays in one block (lengths up to a
// few hundred thousand): out[0..n] with out[n] the total.
__global__ void k_scan3(const int* a, int na, int* oa, const int* b, int nb, int* ob, const int* c, int nc, int* oc) {
  pdl_wait();  // launched with programmatic dependent launch
  __shared__ int sh[32];
  __shared__ int carry;
  const int* in[3] = {a, b, c};
  int* out[3] = {oa, ob, oc};
  const int n[3] = {na, nb, nc};
  for (int k = 0; k < 3; ++k) {
    if (!out[k]) continue;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < n[k]; base += kScanBlock) {
      const int idx = base + threadIdx.x;
      const int v = idx < n[k] ? in[k][idx] : 0;
      const int incl = block_incl_scan(v, sh);
      const int cy = carry;
      if (idx < n[k]) out[k][idx] = cy + incl - v;
      __syncthreads();
      if (threadIdx.x == kScanBlock - 1) carry = cy + incl;
      __syncthreads();
    }
    if (threadIdx.x == 0) out[k][n[k]] = carry;
    __syncthreads();
  }
}

// q-major lists: one warp per q tile compacts its row in kv order, numbering
// partial tiles row-major (slot = partial tiles in earlier rows + rank in row).
__global__ void k_fill_rows(const uint8_t* kinds, int nq, int nk, const int* q_ptr, const int* prow_ptr, int* kv_idx,
                            uint8_t* kd, int* pidx, int2* slot_tile, long long slot_cap) {
  pdl_wait();  // launched with programmatic dependent launch
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= nq) return;
  int pos = q_ptr[w], ppos = prow_ptr[w];
  for (int base = 0; base < nk; base += 32) {
    int x = base + lane;
    uint8_t k = x < nk ? kinds[(long long)w * nk + x] : 0;
    unsigned m = __ballot_sync(0xffffffffu, k != 0);
    unsigned mp = __ballot_sync(0xffffffffu, k == PT_KIND_PARTIAL);
    if (k) {
      const unsigned below = (1u << lane) - 1;
      const int off = __popc(m & below);
      kv_idx[pos + off] = x;
      kd[pos + off] = k;
      if (k == PT_KIND_PARTIAL) {
        const int slot = ppos + __popc(mp & below);
        if (slot < slot_cap) {
          pidx[pos + off] = slot;
          slot_tile[slot] = make_int2(w, x);
        } else {  // more partial tiles than the allocation's bound: never written past it
          pidx[pos + off] = -1;
          record_status(PT_STATUS_INVALID);
        }
      } else {
        pidx[pos + off] = -1;
      }
    }
    pos += __popc(m);
    ppos += __popc(mp);
  }
}

// kv-major lists: one warp per kv block compacts its column in q order; each
// entry's mask slot is found in the q tile's row (binary search by kv block).
__global__ void k_fill_cols(const uint8_t* kinds, int nq, int nk, const int* k_ptr, int* q_idx, uint8_t* kdT,
                            const int* q_ptr, const int* kv_idx, const int* pidx, int* pidxT) {
  pdl_wait();  // launched with programmatic dependent launch
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= nk) return;
  int pos = k_ptr[w];
  for (int base = 0; base < nq; base += 32) {
    int x = base + lane;
    uint8_t k = x < nq ? kinds[(long long)x * nk + w] : 0;
    unsigned m = __ballot_sync(0xffffffffu, k != 0);
    if (k) {
      const int off = __popc(m & ((1u << lane) - 1));
      q_idx[pos + off] = x;
      kdT[pos + off] = k;
      int lo = q_ptr[x], hi = q_ptr[x + 1] - 1;  // row x holds kv block w
      while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (kv_idx[mid] < w)
          lo = mid + 1;
        else
          hi = mid;
      }
      pidxT[pos + off] = pidx[lo];
    }
    pos += __popc(m);
  }
}

// First run start at or after `from` in a 128-bit set of run starts (128 if none).
__device__ __forceinline__ int next_run(const uint32_t* w, int from) {
  if (from >= 128) return 128;
  int i = from >> 5;
  uint32_t m = w[i] & (0xffffffffu << (from & 31));
  while (m == 0) {
    if (++i == 4) return 128;
    m = w[i];
  }
  return (i << 5) + __ffs(m) - 1;
}

// bits[a, b) of a 128-bit mask, 0 <= a < b <= 128
__device__ __forceinline__ void set_bits(uint32_t* bits, int a, int b) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int lo = max(a - 32 * w, 0), hi = min(b - 32 * w, 32);
    if (lo < hi) bits[w] |= (hi == 32 ? 0xffffffffu : ((1u << hi) - 1u)) & (0xffffffffu << lo);
  }
}

// Keep bitmasks of one partial 128 x 128 tile, both orientations:
// mask_rows[slot][r][w] bit b = keep(q = i*128 + r, kv = j*128 + 32w + b),
// mask_cols[slot][c][w] bit b = keep(q = i*128 + 32w + b, kv = j*128 + c).
// Pairs outside [0, T) are never kept.
__device__ __forceinline__ void tile_masks(int T, const pt_tok* tok, const int2* slot_tile, uint32_t* mask_rows,
                                           uint32_t* mask_cols, long long s, pt_tok* tq, pt_tok* tk,
                                           uint32_t* kstart, uint32_t* qstart) {
  const int r = threadIdx.x;
  const int2 ij = slot_tile[s];
  const int q0 = ij.x * 128, k0 = ij.y * 128;
  tq[r] = tok[q0 + r];
  tk[r] = tok[k0 + r];
  __syncthreads();
  // Runs: maximal ranges of tokens with the same (tin, tout), i.e. of one node
  // (padding past T is one more run that sees and is seen by nothing).  Every
  // key of a run passes or fails the ancestor test together, so a row sees a
  // run's keys up to the causal limit: one bit range per run.
  const bool ks = r == 0 || tk[r].tin != tk[r - 1].tin || tk[r].tout != tk[r - 1].tout;
  const bool qs = r == 0 || tq[r].tin != tq[r - 1].tin || tq[r].tout != tq[r - 1].tout;
  const uint32_t kb = __ballot_sync(0xffffffffu, ks), qb = __ballot_sync(0xffffffffu, qs);
  if ((r & 31) == 0) {
    kstart[r >> 5] = kb;
    qstart[r >> 5] = qb;
  }
  __syncthreads();
  const int runs = __popc(kstart[0]) + __popc(kstart[1]) + __popc(kstart[2]) + __popc(kstart[3]) +
                   __popc(qstart[0]) + __popc(qstart[1]) + __popc(qstart[2]) + __popc(qstart[3]);
  uint32_t row[4] = {0, 0, 0, 0}, col[4] = {0, 0, 0, 0};
  const int q = q0 + r, kv = k0 + r;
  const pt_tok mq = tq[r], mk = tk[r];
  if (runs <= 48) {
    if (q < T)
      for (int c = 0; c < 128;) {
        const int c1 = next_run(kstart, c + 1);
        const pt_tok t = tk[c];
        if (k0 + c < T && t.tin <= mq.tin && mq.tin < t.tout) {
          const int hi = min(c1, q - k0 + 1);  // k0 + c' <= q
          if (hi > c) set_bits(row, c, hi);
        }
        c = c1;
      }
    if (kv < T)
      for (int c = 0; c < 128;) {
        const int c1 = next_run(qstart, c + 1);
        const pt_tok u = tq[c];
        if (q0 + c < T && mk.tin <= u.tin && u.tin < mk.tout) {
          const int lo = max(c, kv - q0);  // kv <= q0 + c'
          const int hi = min(c1, T - q0);
          if (lo < hi) set_bits(col, lo, hi);
        }
        c = c1;
      }
  } else {  // many short nodes: pair by pair
    for (int c = 0; c < 128; ++c) {
      const int kvc = k0 + c;
      const pt_tok t = tk[c];
      if (q < T && kvc < T && kvc <= q && t.tin <= mq.tin && mq.tin < t.tout) row[c >> 5] |= 1u << (c & 31);
      const int qc = q0 + c;
      const pt_tok u = tq[c];
      if (qc < T && kv < T && kv <= qc && mk.tin <= u.tin && u.tin < mk.tout) col[c >> 5] |= 1u << (c & 31);
    }
  }
  uint4* mr = reinterpret_cast<uint4*>(mask_rows) + (size_t)s * 128 + r;
  uint4* mc = reinterpret_cast<uint4*>(mask_cols) + (size_t)s * 128 + r;
  *mr = make_uint4(row[0], row[1], row[2], row[3]);
  *mc = make_uint4(col[0], col[1], col[2], col[3]);
}

// All partial tiles, grid-stride: slots 0 .. n_partial - 1, n_partial = n_known
// when that is >= 0, else nnz - n_full read on the device (at most p_cap).
__global__ void k_masks(int T, const pt_tok* tok, const int2* slot_tile, uint32_t* mask_rows, uint32_t* mask_cols,
                        long long n_known, const int* nnz_total, const int* n_full, long long p_cap,
                        int* host_counters = nullptr, long long expect_pairs = -1) {
  pdl_wait();  // launched with programmatic dependent launch
  // host-built lists: the kept pairs the classification found over the listed
  // tiles (n_full[2..3], one 64-bit sum) must be every kept pair of the tree
  if (expect_pairs >= 0 && blockIdx.x == 0 && threadIdx.x == 0 &&
      *reinterpret_cast<const unsigned long long*>(n_full + 2) != (unsigned long long)expect_pairs)
    record_status(PT_STATUS_INVALID);
  __shared__ pt_tok tq[128], tk[128];
  __shared__ uint32_t kstart[4], qstart[4];
  // the full-tile count to the host's mapped staging (host-built lists)
  if (host_counters && blockIdx.x == 0 && threadIdx.x < 4) host_counters[threadIdx.x] = n_full[threadIdx.x];
  const long long n_part = min(n_known >= 0 ? n_known : (long long)(*nnz_total - *n_full), p_cap);
  for (long long s = blockIdx.x; s < n_part; s += gridDim.x) {
    tile_masks(T, tok, slot_tile, mask_rows, mask_cols, s, tq, tk, kstart, qstart);
    __syncthreads();
  }
}

// Tile classes and list sizes for a draft map: one warp per tile, kept pairs
// counted per row from its two ranges (exact).
__global__ void k_draft_classify(int T, int BM, int BN, int nq, int nk, DraftParams d, uint8_t* kinds, int* counters,
                                 int* row_cnt, int* col_cnt, int* row_part) {
  pdl_wait();  // launched with programmatic dependent launch
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)nq * nk) return;
  const int i = (int)(w / nk), j = (int)(w % nk);
  const long long q0 = (long long)i * BM, k0 = (long long)j * BN;
  const long long k1 = k0 + BN < T ? k0 + BN : T;
  const long long qend = q0 + BM < T ? q0 + BM : T;
  long long kept = 0;
  for (long long q = q0 + lane; q < qend; q += 32) {
    int c0, c1, b0, b1;
    draft_row(d, (int)q, c0, c1, b0, b1);
    kept += overlap(c0, c1, k0, k1) + overlap(b0, b1, k0, k1);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
  if (lane == 0) {
    const bool in_range = (q0 + BM <= T) && (k0 + BN <= T);
    const uint8_t kd = kept == 0 ? PT_KIND_EMPTY
                                 : ((in_range && kept == (long long)BM * BN) ? PT_KIND_FULL : PT_KIND_PARTIAL);
    kinds[w] = kd;
    if (kd != PT_KIND_EMPTY) {
      atomicAdd(&row_cnt[i], 1);
      atomicAdd(&col_cnt[j], 1);
      if (kd == PT_KIND_FULL)
        atomicAdd(&counters[0], 1);
      else
        atomicAdd(&row_part[i], 1);
    }
  }
}

// Keep bitmasks of the partial tiles of a draft map (layout as k_masks):
// a row's bits are its two ranges clipped to the tile; the column masks are
// the transpose, one ballot per column over each warp's 32 rows.
__global__ void k_draft_masks(int T, DraftParams d, const int2* slot_tile, uint32_t* mask_rows, uint32_t* mask_cols,
                              long long n_known, const int* nnz_total, const int* n_full, long long p_cap,
                              int* host_counters = nullptr, long long expect_pairs = -1) {
  pdl_wait();  // launched with programmatic dependent launch
  // host-built lists: the kept pairs the classification found over the listed
  // tiles (n_full[2..3], one 64-bit sum) must be every kept pair of the map
  if (expect_pairs >= 0 && blockIdx.x == 0 && threadIdx.x == 0 &&
      *reinterpret_cast<const unsigned long long*>(n_full + 2) != (unsigned long long)expect_pairs)
    record_status(PT_STATUS_INVALID);
  // the full-tile count to the host's mapped staging (host-built lists)
  if (host_counters && blockIdx.x == 0 && threadIdx.x < 4) host_counters[threadIdx.x] = n_full[threadIdx.x];
  const long long n_part = min(n_known >= 0 ? n_known : (long long)(*nnz_total - *n_full), p_cap);
  const int r = threadIdx.x, lane = r & 31, wi = r >> 5;
  for (long long s = blockIdx.x; s < n_part; s += gridDim.x) {
    const int2 ij = slot_tile[s];
    const int q0 = ij.x * 128, k0 = ij.y * 128, q = q0 + r;
    const int kend = min(k0 + 128, T);
    uint32_t row[4] = {0, 0, 0, 0};
    if (q < T) {
      int c0, c1, b0, b1;
      draft_row(d, q, c0, c1, b0, b1);
      int a = max(c0, k0), e = min(c1, kend);
      if (a < e) set_bits(row, a - k0, e - k0);
      a = max(b0, k0);
      e = min(b1, kend);
      if (a < e) set_bits(row, a - k0, e - k0);
    }
    reinterpret_cast<uint4*>(mask_rows)[(size_t)s * 128 + r] = make_uint4(row[0], row[1], row[2], row[3]);
    uint32_t col[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      col[m] = 0;
      for (int t = 0; t < 32; ++t) {
        const uint32_t v = __ballot_sync(0xffffffffu, (row[m] >> t) & 1u);
        if (t == lane) col[m] = v;
      }
    }
    // lane holds kv column 32 m + lane, word wi (q rows 32 wi .. 32 wi + 31)
#pragma unroll
    for (int m = 0; m < 4; ++m) mask_cols[((size_t)s * 128 + 32 * m + lane) * 4 + wi] = col[m];
  }
}

// dense map: every tile partial; slot = row-major tile index
__global__ void k_dense_lists(int nq, int nk, int* q_ptr, int* kv_idx, uint8_t* kind, int* k_ptr, int* q_idx,
                              uint8_t* kindT, int* pidx, int* pidxT, int2* slot_tile) {
  long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long n = (long long)nq * nk;
  if (e < n) {
    kv_idx[e] = (int)(e % nk);
    kind[e] = PT_KIND_PARTIAL;
    pidx[e] = (int)e;
    slot_tile[e] = make_int2((int)(e / nk), (int)(e % nk));
    const int j = (int)(e / nq), i = (int)(e % nq);  // kv-major entry e: column j, row i
    q_idx[e] = i;
    kindT[e] = PT_KIND_PARTIAL;
    pidxT[e] = i * nk + j;
  }
  if (e <= nq) q_ptr[e] = (int)(e * nk);
  if (e <= nk) k_ptr[e] = (int)(e * nq);
}

// Longest-first order on the device: element i goes to position
// #{j : cnt[j] > cnt[i] or (cnt[j] == cnt[i] and j < i)}.  One warp per
// element; warps [0, na) order array a, the rest array b.
__global__ void k_lpt2(const int* a, int na, int* oa, const int* b, int nb, int* ob) {
  pdl_wait();  // launched with programmatic dependent launch
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= na + nb) return;
  const int* cnt = w < na ? a : b;
  int* order = w < na ? oa : ob;
  const int n = w < na ? na : nb;
  const int i = w < na ? w : w - na;
  const int ci = cnt[i];
  int rank = 0;
  for (int j = lane; j < n; j += 32) {
    const int cj = cnt[j];
    rank += (cj > ci) || (cj == ci && j < i);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
  if (lane == 0) order[rank] = i;
}

}  // namespace

constexpr int kMaxDev = 64;

// The small per-map transfers (node tables and work lists in, list sizes
// out) go through the SMs, reading or writing the pinned staging through
// its mapping in the device's address space, not through the copy engines.
// A large copy that another stream has queued on an engine (a training
// step's inputs and gradients) would otherwise hold them, and with them the
// kernels queued behind them on this stream.
// early: the source is host staging that the CPU filled before the launch, so
// each thread reads its first 16 bytes before waiting for the previous kernel
// (the read's round trip to host memory overlaps that kernel's tail); the
// wait still precedes every write.
__global__ void k_stage(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long bytes, int vec,
                        int early) {
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  long long done = 0, i0 = tid;
  if (vec) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const long long n16 = bytes >> 4;
    if (early && tid < n16) {
      const uint4 first = s4[tid];
      pdl_wait();  // launched with programmatic dependent launch
      d4[tid] = first;
      i0 = tid + nth;
    } else {
      pdl_wait();
    }
    for (long long i = i0; i < n16; i += nth) d4[i] = s4[i];
    done = n16 << 4;
  } else {
    pdl_wait();
  }
  for (long long i = done + tid; i < bytes; i += nth) dst[i] = src[i];
}

int stage_copy(const void* src, void* dst, size_t bytes, cudaStream_t s, bool early = false) {
  if (!bytes) return 0;
  const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0) ? 1 : 0;
  const long long units = vec ? (long long)(bytes >> 4) + 1 : (long long)bytes;
  const int grid = (int)std::max(1LL, std::min<long long>((units + 255) / 256, 64));
  launch_pdl(k_stage, dim3(grid), dim3(256), 0, s, static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
             (long long)bytes, vec, early ? 1 : 0);
  count_launch();
  if (cudaGetLastError() != cudaSuccess) {
    set_error("staging copy launch failed");
    return 3;
  }
  return 0;
}

// Test hook: the next n tree or draft builds with host-built lists drop one
// listed tile (pt_debug_drop_listed_tile).
std::atomic<int> g_drop_listed_tiles{0};

// ---------------------------------------------------------------------------
// host side: memory
// ---------------------------------------------------------------------------
// Device memory comes from a private stream-ordered pool per device that
// keeps freed blocks for reuse, so building and freeing maps never
// synchronises the device.

cudaMemPool_t pool_for(int dev) {
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDev] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  if (!pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p;
    if (cudaMemPoolCreate(&p, &props) != cudaSuccess) return nullptr;
    uint64_t keep = UINT64_MAX;
    cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev] = p;
  }
  return pools[dev];
}

int pool_alloc(void** p, size_t bytes, int dev, cudaStream_t s) {
  *p = nullptr;
  cudaMemPool_t pool = pool_for(dev);
  if (!pool) {
    set_error("cannot create a device memory pool on device %d", dev);
    return 3;
  }
  cudaError_t e = cudaMallocFromPoolAsync(p, bytes ? bytes : 256, pool, s);
  if (e != cudaSuccess) {
    *p = nullptr;
    set_error("device allocation of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
    return 5;
  }
  return 0;
}

void pool_free(void* p, cudaStream_t s) {
  if (p) cudaFreeAsync(p, s);
}

void debug_drop_listed_tiles(int n) { g_drop_listed_tiles.store(n > 0 ? n : 0); }

// The test hook at work (pt_debug_drop_listed_tile): the last entry of the
// longest q list leaves the host's lists (row_kv, q-major, with the row
// lengths in pred[0, nq) and the column lengths after them), consistently.
void maybe_drop_listed_tile(std::vector<int>& row_kv, std::vector<int>& pred, int nq) {
  if (row_kv.empty() || g_drop_listed_tiles.load() <= 0 || g_drop_listed_tiles.fetch_sub(1) <= 0) return;
  int i_max = 0;
  for (int i = 1; i < nq; ++i)
    if (pred[(size_t)i] > pred[(size_t)i_max]) i_max = i;
  size_t pos = 0;
  for (int i = 0; i <= i_max; ++i) pos += (size_t)pred[(size_t)i];
  const int j = row_kv[pos - 1];
  row_kv.erase(row_kv.begin() + (long)(pos - 1));
  --pred[(size_t)i_max];
  --pred[(size_t)nq + j];
}

int pool_usage(int dev, uint64_t* used, uint64_t* reserved) {
  *used = *reserved = 0;
  cudaMemPool_t pool = pool_for(dev);
  if (!pool) {
    set_error("cannot create a device memory pool on device %d", dev);
    return 3;
  }
  cuuint64_t u = 0, r = 0;
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &u) != cudaSuccess ||
      cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &r) != cudaSuccess) {
    set_error("cannot read the memory pool's usage on device %d", dev);
    return 3;
  }
  *used = u;
  *reserved = r;
  return 0;
}

// Sub-array layout inside one allocation, 256-byte aligned pieces.
struct Layout {
  size_t off = 0;
  template <class T>
  size_t add(size_t n) {
    size_t o = off;
    off += (n * sizeof(T) + 255) & ~size_t(255);
    return o;
  }
};
template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// Pinned staging for host->device uploads (avoids the stream synchronisation
// a pageable copy implies).  A ring of slots per device: a slot is refilled
// only once the copy that last read it has run, so the host blocks only when
// it is several uploads ahead of the GPU.
// Device-to-host copy that waits for the stream: through a pinned buffer
// per device (a copy to pageable memory is staged by the driver and slower).
int download_sync(void* dst, const void* src, size_t bytes, int dev, cudaStream_t s) {
  struct Buf {
    void* host = nullptr;
    size_t cap = 0;
  };
  static std::mutex mu;
  static Buf bufs[kMaxDev];
  if (dev < 0 || dev >= kMaxDev) return 3;
  std::lock_guard<std::mutex> lk(mu);
  Buf& b = bufs[dev];
  if (b.cap < bytes) {
    if (b.host) cudaFreeHost(b.host);
    b.host = nullptr;
    b.cap = 0;
    size_t cap = bytes < (1u << 16) ? (1u << 16) : bytes;
    if (cudaHostAlloc(&b.host, cap, cudaHostAllocDefault) != cudaSuccess) {
      set_error("pinned download buffer of %zu bytes failed", cap);
      return 5;
    }
    b.cap = cap;
  }
  if (bytes && cudaMemcpyAsync(b.host, src, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    set_error("block map download failed");
    return 3;
  }
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_error("block map build failed: %s", cudaGetErrorString(e));
    return 3;
  }
  std::memcpy(dst, b.host, bytes);
  return 0;
}

// Pinned host buffers, each with an event, reused across builds: a build's
// list lengths are copied into one behind its event, and the map holds the
// slot until the lengths are read on the host.
struct PinnedSlot {
  void* host = nullptr;
  void* dev = nullptr;  // the same memory as the device addresses it
  size_t cap = 0;
  cudaEvent_t ev = nullptr;
};
std::mutex g_pinned_mu;
std::vector<PinnedSlot> g_pinned_free[kMaxDev];

int pinned_acquire(int dev, size_t bytes, PinnedSlot* out) {
  if (dev < 0 || dev >= kMaxDev) return 3;
  {
    std::lock_guard<std::mutex> lk(g_pinned_mu);
    std::vector<PinnedSlot>& fl = g_pinned_free[dev];
    for (size_t i = 0; i < fl.size(); ++i)
      if (fl[i].cap >= bytes) {
        // a slot goes back to the pool with its last copy possibly in flight
        // (a map freed before its sizes were read): take it once that is done
        if (cudaEventQuery(fl[i].ev) == cudaErrorNotReady) {
          if (cudaPeekAtLastError() == cudaErrorNotReady) cudaGetLastError();
          continue;
        }
        *out = fl[i];
        fl[i] = fl.back();
        fl.pop_back();
        return 0;
      }
  }
  PinnedSlot sl;
  sl.cap = bytes < (1u << 16) ? (1u << 16) : bytes;
  if (cudaHostAlloc(&sl.host, sl.cap, cudaHostAllocDefault) != cudaSuccess) {
    set_error("pinned staging allocation of %zu bytes failed", sl.cap);
    return 5;
  }
  if (cudaHostGetDevicePointer(&sl.dev, sl.host, 0) != cudaSuccess) {
    cudaFreeHost(sl.host);
    set_error("pinned staging is not mapped into the device's address space");
    return 3;
  }
  if (cudaEventCreateWithFlags(&sl.ev, cudaEventDisableTiming) != cudaSuccess) {
    cudaFreeHost(sl.host);
    set_error("event creation failed");
    return 3;
  }
  *out = sl;
  return 0;
}

void pinned_release(int dev, const PinnedSlot& sl) {
  if (!sl.host || dev < 0 || dev >= kMaxDev) return;
  std::lock_guard<std::mutex> lk(g_pinned_mu);
  g_pinned_free[dev].push_back(sl);
}

int upload(void* dst, const void* src, size_t bytes, int dev, cudaStream_t s) {
  // enough slots that a slot's previous copy (several steps back) is done
  constexpr int kSlots = 16;
  struct Slot {
    void* host = nullptr;
    void* dev = nullptr;  // the slot's device address
    size_t cap = 0;
    cudaEvent_t done = nullptr;
    bool used = false;
  };
  struct Ring {
    Slot slot[kSlots];
    int next = 0;
  };
  static std::mutex mu;
  static Ring rings[kMaxDev];
  if (bytes == 0) return 0;
  if (dev < 0 || dev >= kMaxDev) return 3;
  std::lock_guard<std::mutex> lk(mu);
  Ring& rg = rings[dev];
  Slot& g = rg.slot[rg.next];
  rg.next = (rg.next + 1) % kSlots;
  if (!g.done && cudaEventCreateWithFlags(&g.done, cudaEventDisableTiming) != cudaSuccess) return 3;
  if (g.used) cudaEventSynchronize(g.done);  // usually long complete
  if (g.cap < bytes) {
    if (g.host) cudaFreeHost(g.host);
    g.host = nullptr;
    g.cap = 0;
    size_t cap = bytes < (1u << 20) ? (1u << 20) : bytes;
    if (cudaHostAlloc(&g.host, cap, cudaHostAllocDefault) != cudaSuccess) {
      set_error("pinned staging allocation of %zu bytes failed", cap);
      return 5;
    }
    if (cudaHostGetDevicePointer(&g.dev, g.host, 0) != cudaSuccess) {
      cudaFreeHost(g.host);
      g.host = nullptr;
      set_error("pinned staging is not mapped into the device's address space");
      return 3;
    }
    g.cap = cap;
  }
  std::memcpy(g.host, src, bytes);
  if (int rc = stage_copy(g.dev, dst, bytes, s, true)) return rc;  // host staging, filled above
  cudaEventRecord(g.done, s);
  g.used = true;
  return 0;
}

namespace {

// The part of a map whose size is known before classification: token
// coordinates, node tables, list pointers and orders.
int new_map(int T, int BM, int BN, int node_cap, cudaStream_t s, pt_blockmap** out) {
  pt_blockmap* bm = new pt_blockmap;
  std::memset(bm, 0, sizeof(*bm));
  cudaGetDevice(&bm->device);
  bm->stream = s;
  bm->T = T;
  bm->BM = BM;
  bm->BN = BN;
  bm->nq = (T + BM - 1) / BM;
  bm->nk = (T + BN - 1) / BN;
  bm->tpad = std::max(bm->nq * BM, bm->nk * BN);
  Layout L;
  // node tables: start | end | parent | tin | tout, node_cap entries each
  // (the tree build uploads all five at once; tin and tout feed the token table)
  size_t o_tok = L.add<pt_tok>(bm->tpad), o_node = L.add<int>(T), o_ns = L.add<int>((size_t)5 * node_cap),
         o_qp = L.add<int>(bm->nq + 1),
         o_kp = L.add<int>(bm->nk + 1), o_qo = L.add<int>(bm->nq), o_ko = L.add<int>(bm->nk);
  int rc = pool_alloc(&bm->mem_fixed, L.off, bm->device, s);
  if (rc) {
    delete bm;
    return rc;
  }
  bm->tok = at<pt_tok>(bm->mem_fixed, o_tok);
  bm->node_of = at<int>(bm->mem_fixed, o_node);
  bm->node_start = at<int>(bm->mem_fixed, o_ns);
  bm->node_end = bm->node_start + node_cap;
  bm->parent = bm->node_end + node_cap;
  bm->q_ptr = at<int>(bm->mem_fixed, o_qp);
  bm->k_ptr = at<int>(bm->mem_fixed, o_kp);
  bm->q_order = at<int>(bm->mem_fixed, o_qo);
  bm->k_order = at<int>(bm->mem_fixed, o_ko);
  *out = bm;
  return 0;
}

// The lists part, once nnz and the number of partial tiles are known.
// `nnz` list entries and `n_part` mask slots: the exact sizes, or bounds when
// the build does not wait for them.
int alloc_lists(pt_blockmap* bm, int64_t nnz, int64_t n_part, cudaStream_t s) {
  const bool masks = bm->BM == 128 && bm->BN == 128 && n_part > 0;
  bm->nnz_cap = nnz;
  bm->p_cap = masks ? n_part : 0;
  Layout L;
  size_t o_kv = L.add<int>(nnz), o_kd = L.add<uint8_t>(nnz), o_pi = L.add<int>(nnz), o_qi = L.add<int>(nnz),
         o_kt = L.add<uint8_t>(nnz), o_pt = L.add<int>(nnz);
  size_t o_mr = masks ? L.add<uint32_t>((size_t)n_part * 512) : 0;
  size_t o_mc = masks ? L.add<uint32_t>((size_t)n_part * 512) : 0;
  int rc = pool_alloc(&bm->mem_lists, L.off, bm->device, s);
  if (rc) return rc;
  bm->kv_idx = at<int>(bm->mem_lists, o_kv);
  bm->kind = at<uint8_t>(bm->mem_lists, o_kd);
  bm->pidx = at<int>(bm->mem_lists, o_pi);
  bm->q_idx = at<int>(bm->mem_lists, o_qi);
  bm->kindT = at<uint8_t>(bm->mem_lists, o_kt);
  bm->pidxT = at<int>(bm->mem_lists, o_pt);
  bm->mask_rows = masks ? at<uint32_t>(bm->mem_lists, o_mr) : nullptr;
  bm->mask_cols = masks ? at<uint32_t>(bm->mem_lists, o_mc) : nullptr;
  return 0;
}

#define PT_LAUNCHED(n)                                                          \
  do {                                                                          \
    count_launch(n);                                                            \
    cudaError_t le_ = cudaGetLastError();                                       \
    if (le_ != cudaSuccess) {                                                   \
      set_error("block map kernel launch failed: %s", cudaGetErrorString(le_)); \
      rc = 3;                                                                   \
      break;                                                                    \
    }                                                                           \
  } while (0)

// Shared tail of the builders: given tok, node_of and node tables on the
// device, classify, count, list, order and mask.  Synchronises the stream
// once (to size the lists); everything after that is asynchronous.
int finish_map(pt_blockmap* bm, cudaStream_t s, int64_t p_bound) {
  const int nq = bm->nq, nk = bm->nk, dev = bm->device;
  const long long ntiles = (long long)nq * nk;
  // Bound on the non-empty tiles: the exact count when the builder derived
  // the list lengths on the host, else the causal bound (q tile i meets kv
  // blocks j with j * BN <= its last row).  With a bound on the partial tiles
  // as well, the lists are allocated at the bounds and nothing waits for the
  // device.
  int64_t nnz_bound = 0;
  if (bm->h_rc_pred) {  // exact list lengths are known on the host
    for (int i = 0; i < nq; ++i) nnz_bound += bm->h_rc_pred[i];
  } else {
    for (int i = 0; i < nq; ++i) {
      const long long qlast = std::min<long long>((long long)(i + 1) * bm->BM, bm->T) - 1;
      nnz_bound += std::min<long long>(nk, qlast / bm->BN + 1);
    }
  }
  const bool tiles128 = bm->BM == 128 && bm->BN == 128;
  const int64_t p_bound_c = std::min<int64_t>(p_bound, nnz_bound);
  const bool lazy = tiles128 && p_bound >= 0 &&
                    nnz_bound * 18 + (int64_t)p_bound_c * 4096 <= ((int64_t)1 << 30);
  void* tmpA = nullptr;
  void* tmpB = nullptr;
  int rc = 0;
  do {
    // counters | row counts | column counts are contiguous so one copy brings
    // them to the host; partial counts per row and their scan stay on the device
    Layout LA;
    const size_t ncnt = (size_t)4 + nq + nk;
    size_t o_kinds = LA.add<uint8_t>((size_t)ntiles), o_cnt = LA.add<int>(ncnt + nq),
           o_pp = LA.add<int>((size_t)nq + 1);
    if ((rc = pool_alloc(&tmpA, LA.off, dev, s))) break;
    uint8_t* kinds = at<uint8_t>(tmpA, o_kinds);
    int* counters = at<int>(tmpA, o_cnt);
    int* row_cnt = counters + 4;
    int* col_cnt = row_cnt + nq;
    int* row_part = col_cnt + nk;
    int* prow_ptr = at<int>(tmpA, o_pp);
    {
      ProfScope ps(s, "blockmap_classify");  // tile classes, list sizes, longest-first orders
      if (cudaMemsetAsync(counters, 0, sizeof(int) * (ncnt + nq), s) != cudaSuccess) {
        rc = 3;
        break;
      }
      if (ntiles > 0) {
        long long threads = ntiles * 32;
        if (bm->producer == PT_PRODUCER_DRAFT)
          launch_pdl(k_draft_classify, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, s, bm->T, bm->BM, bm->BN,
                     nq, nk, draft_params(bm), kinds, counters, row_cnt, col_cnt, row_part);
        else
          launch_pdl(k_classify, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, s, bm->T, bm->BM, bm->BN, nq,
                     nk, bm->node_of, bm->node_start, bm->node_end, bm->parent, kinds, counters, row_cnt, col_cnt,
                     row_part);
        PT_LAUNCHED(1);
      }
      launch_pdl(k_scan3, dim3(1), dim3(kScanBlock), 0, s, row_cnt, nq, bm->q_ptr, col_cnt, nk, bm->k_ptr, row_part, nq,
                 prow_ptr);
      PT_LAUNCHED(1);
      if (ntiles > 0) {
        launch_pdl(k_lpt2, dim3((unsigned)(((long long)(nq + nk) * 32 + 255) / 256)), dim3(256), 0, s, row_cnt, nq,
                   bm->q_order, col_cnt, nk, bm->k_order);
        PT_LAUNCHED(1);
      }
    }
    if (rc) break;
    int64_t nnz_alloc, p_alloc;
    if (lazy) {
      // list sizes to pinned staging behind an event; read on first use
      PinnedSlot sl;
      if ((rc = pinned_acquire(dev, sizeof(int) * ncnt, &sl))) break;
      bm->counts_host = sl.host;
      bm->counts_dev = sl.dev;
      bm->counts_cap = sl.cap;
      bm->counts_ev = sl.ev;
      if (stage_copy(counters, sl.dev, sizeof(int) * ncnt, s) != 0 || cudaEventRecord(sl.ev, s) != cudaSuccess) {
        set_error("block map: copy of the list sizes failed");
        rc = 3;
        break;
      }
      bm->counts_ready = false;
      nnz_alloc = nnz_bound;
      p_alloc = p_bound_c;
    } else {
      // the one synchronisation of the build: list sizes to the host
      bm->h_counts = static_cast<int*>(std::malloc(sizeof(int) * ncnt));
      if (!bm->h_counts) {
        rc = 5;
        break;
      }
      if ((rc = download_sync(bm->h_counts, counters, sizeof(int) * ncnt, dev, s))) break;
      bm->h_row_cnt = bm->h_counts + 4;
      bm->h_col_cnt = bm->h_row_cnt + nq;
      int64_t nnz_h = 0;
      for (int i = 0; i < nq; ++i) nnz_h += bm->h_row_cnt[i];
      bm->nnz = nnz_h;
      bm->n_full = bm->h_counts[0];
      bm->n_partial = bm->nnz - bm->n_full;
      bm->counts_ready = true;
      nnz_alloc = bm->nnz;
      p_alloc = bm->n_partial;
    }
    if ((rc = alloc_lists(bm, nnz_alloc, p_alloc, s))) break;
    if (ntiles > 0 && nnz_alloc > 0) {
      ProfScope ps(s, "blockmap_lists");  // the lists and the partial tiles' masks
      if ((rc = pool_alloc(&tmpB, sizeof(int2) * (size_t)std::max<int64_t>(p_alloc, 1), dev, s))) break;
      int2* slot_tile = static_cast<int2*>(tmpB);
      launch_pdl(k_fill_rows, dim3((nq * 32 + 255) / 256), dim3(256), 0, s, kinds, nq, nk, bm->q_ptr, prow_ptr,
                 bm->kv_idx, bm->kind, bm->pidx, slot_tile, (long long)p_alloc);
      launch_pdl(k_fill_cols, dim3((nk * 32 + 255) / 256), dim3(256), 0, s, kinds, nq, nk, bm->k_ptr, bm->q_idx,
                 bm->kindT, bm->q_ptr, bm->kv_idx, bm->pidx, bm->pidxT);
      PT_LAUNCHED(2);
      if (bm->mask_rows) {
        const long long grid = std::min<long long>(p_alloc, (long long)num_sms(dev) * 16);
        if (bm->producer == PT_PRODUCER_DRAFT)
          launch_pdl(k_draft_masks, dim3((unsigned)grid), dim3(128), 0, s, bm->T, draft_params(bm), slot_tile,
                     bm->mask_rows, bm->mask_cols, -1LL, bm->q_ptr + nq, counters, (long long)bm->p_cap,
                     static_cast<int*>(nullptr), -1LL);
        else
          launch_pdl(k_masks, dim3((unsigned)grid), dim3(128), 0, s, bm->T, bm->tok, slot_tile, bm->mask_rows,
                     bm->mask_cols, -1LL, bm->q_ptr + nq, counters, (long long)bm->p_cap, static_cast<int*>(nullptr),
                     -1LL);
        PT_LAUNCHED(1);
      }
    }
  } while (0);
  pool_free(tmpA, s);
  pool_free(tmpB, s);
  return rc;
}

}  // namespace

// Tail of the tree builder at 128 x 128 tiles when the host built the lists
// (row_kv: kv blocks per q tile, ascending, lengths in bm->h_rc_pred):
// derive the transpose, longest-first orders and each entry's kv-major
// position on the host, upload them in one packed copy with zeroed counters,
// then two launches: tokens plus tile classes, and masks.  Nothing waits for
// the device; the full-tile count reaches the host's staging behind an event.
int finish_map_listed(pt_blockmap* bm, cudaStream_t s, int64_t p_bound, const std::vector<int>& row_kv, int N,
                      const int* tab, long long draft_pairs = -1) {
  // draft maps (draft_pairs: their kept pairs in closed form) have no node
  // tables and no token table; their tiles are classified from draft_row
  const bool draft = bm->producer == PT_PRODUCER_DRAFT;
  const int nq = bm->nq, nk = bm->nk, dev = bm->device;
  const int* rc_row = bm->h_rc_pred;
  const int* rc_col = bm->h_rc_pred + nq;
  const int64_t nnz = (int64_t)row_kv.size();
  const int64_t p_alloc = std::min<int64_t>(p_bound >= 0 ? p_bound : nnz, nnz);
  if (nnz * 18 + p_alloc * 4096 > ((int64_t)1 << 30) || nnz > INT_MAX / 4) {
    // too large to allocate at the bound: the device path, which sizes the lists exactly
    if (draft) return finish_map(bm, s, p_bound);
    if (int rc = upload(bm->node_start, tab, sizeof(int) * (size_t)5 * N, dev, s)) return rc;
    k_tree_tokens<<<(bm->tpad + 255) / 256, 256, 0, s>>>(bm->T, bm->tpad, N, bm->node_end,
                                                         bm->node_start + 3 * (size_t)N,
                                                         bm->node_start + 4 * (size_t)N, bm->tok, bm->node_of);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) {
      set_error("block map kernel launch failed");
      return 3;
    }
    return finish_map(bm, s, p_bound);
  }
  // every kept pair of the tree, in closed form: each node's causal triangle
  // plus its tokens times the tokens of its ancestors
  long long expect_pairs = draft ? draft_pairs : 0;
  if (!draft) {
    const int* start = tab;
    const int* end = tab + N;
    const int* parent = tab + 2 * (size_t)N;
    std::vector<long long> anc(N, 0);  // tokens of the ancestors (parents have smaller ids)
    for (int n = 0; n < N; ++n) {
      const long long len = end[n] - start[n];
      if (parent[n] >= 0) anc[n] = anc[parent[n]] + (end[parent[n]] - start[parent[n]]);
      expect_pairs += len * (len + 1) / 2 + len * anc[n];
    }
  }
  // packed: counters[4] (full tiles, partial tiles, the 64-bit kept-pair sum)
  //   | node tables[5N] | q_ptr | k_ptr | q_order | k_order | kv_idx | q_idx | eT
  const size_t n_pk = 4 + 5 * (size_t)N + (size_t)(nq + 1) + (nk + 1) + nq + nk + 3 * (size_t)nnz;
  std::vector<int> pk(n_pk, 0);
  if (N > 0) std::copy(tab, tab + 5 * (size_t)N, pk.data() + 4);
  int* qp = pk.data() + 4 + 5 * (size_t)N;
  int* kp = qp + nq + 1;
  int* qo = kp + nk + 1;
  int* ko = qo + nq;
  int* kv = ko + nk;
  int* qi = kv + nnz;
  int* et = qi + nnz;
  for (int i = 0; i < nq; ++i) qp[i + 1] = qp[i] + rc_row[i];
  for (int j = 0; j < nk; ++j) kp[j + 1] = kp[j] + rc_col[j];
  std::copy(row_kv.begin(), row_kv.end(), kv);
  {
    std::vector<int> fill(kp, kp + nk);
    for (int i = 0; i < nq; ++i)  // q tiles ascending within each kv block
      for (int e = qp[i]; e < qp[i + 1]; ++e) {
        const int pos = fill[(size_t)kv[e]]++;
        qi[pos] = i;
        et[e] = pos;
      }
  }
  // longest first, ties by index (the device's orders use the same rule)
  for (int i = 0; i < nq; ++i) qo[i] = i;
  for (int j = 0; j < nk; ++j) ko[j] = j;
  std::stable_sort(qo, qo + nq, [&](int a, int b) { return rc_row[a] > rc_row[b]; });
  std::stable_sort(ko, ko + nk, [&](int a, int b) { return rc_col[a] > rc_col[b]; });
  int rc = 0;
  void* tmp = nullptr;
  void* tmpB = nullptr;
  do {
    if ((rc = alloc_lists(bm, nnz, p_alloc, s))) break;
    if ((rc = pool_alloc(&tmp, sizeof(int) * n_pk, dev, s))) break;
    if ((rc = upload(tmp, pk.data(), sizeof(int) * n_pk, dev, s))) break;
    if ((rc = pool_alloc(&tmpB, sizeof(int2) * (size_t)std::max<int64_t>(p_alloc, 1), dev, s))) break;
    int2* slot_tile = static_cast<int2*>(tmpB);
    int* counters = static_cast<int*>(tmp);
    PinnedSlot sl;
    if ((rc = pinned_acquire(dev, sizeof(int) * 4, &sl))) break;
    bm->counts_host = sl.host;
    bm->counts_dev = sl.dev;
    bm->counts_cap = sl.cap;
    bm->counts_ev = sl.ev;
    bm->counts_ready = false;
    bm->lists_on_host = true;
    {
      ProfScope ps(s, "blockmap_classify");  // tokens, the lists into place, tile classes
      const int tok_blocks = draft ? 0 : (bm->tpad + 255) / 256;
      const long long list_work = std::max<long long>((long long)nnz * 32, 5LL * N + 2LL * nq + 2LL * nk + 2 + 2 * nnz);
      const int list_blocks = (int)std::max(1LL, std::min<long long>((list_work + 255) / 256, (long long)num_sms(dev) * 8));
      if (draft)
        launch_pdl(k_tree_listed<true>, dim3(tok_blocks + list_blocks), dim3(256), 0, s, bm->T, bm->tpad, N,
                   bm->node_start, bm->tok, bm->node_of, tok_blocks, counters, nq, nk, (int)nnz, bm->q_ptr, bm->k_ptr,
                   bm->q_order, bm->k_order, bm->kv_idx, bm->q_idx, bm->kind, bm->pidx, bm->kindT, bm->pidxT,
                   slot_tile, (long long)bm->p_cap, draft_params(bm));
      else
        launch_pdl(k_tree_listed<false>, dim3(tok_blocks + list_blocks), dim3(256), 0, s, bm->T, bm->tpad, N,
                   bm->node_start, bm->tok, bm->node_of, tok_blocks, counters, nq, nk, (int)nnz, bm->q_ptr, bm->k_ptr,
                   bm->q_order, bm->k_order, bm->kv_idx, bm->q_idx, bm->kind, bm->pidx, bm->kindT, bm->pidxT,
                   slot_tile, (long long)bm->p_cap, DraftParams{0, 1, 0, 0, nullptr});
      PT_LAUNCHED(1);
    }
    {
      ProfScope ps(s, "blockmap_lists");  // the partial tiles' masks
      const long long grid = std::max<long long>(1, std::min<long long>(p_alloc, (long long)num_sms(dev) * 16));
      if (draft)
        launch_pdl(k_draft_masks, dim3((unsigned)grid), dim3(128), 0, s, bm->T, draft_params(bm), slot_tile,
                   bm->mask_rows, bm->mask_cols, -1LL, bm->q_ptr + nq, counters, (long long)bm->p_cap,
                   static_cast<int*>(sl.dev), expect_pairs);
      else
        launch_pdl(k_masks, dim3((unsigned)grid), dim3(128), 0, s, bm->T, bm->tok, slot_tile, bm->mask_rows,
                   bm->mask_cols, -1LL, bm->q_ptr + nq, counters, (long long)bm->p_cap, static_cast<int*>(sl.dev),
                   expect_pairs);
      PT_LAUNCHED(1);
      if (cudaEventRecord(sl.ev, s) != cudaSuccess) {
        rc = 3;
        break;
      }
    }
  } while (0);
  pool_free(tmp, s);
  pool_free(tmpB, s);
  return rc;
}

std::mutex g_counts_mu;

int ensure_counts(const pt_blockmap* cbm) {
  pt_blockmap* bm = const_cast<pt_blockmap*>(cbm);  // the host copy of the sizes is filled in lazily
  std::lock_guard<std::mutex> lk(g_counts_mu);
  if (bm->counts_ready) return 0;
  cudaEvent_t ev = static_cast<cudaEvent_t>(bm->counts_ev);
  cudaError_t e = cudaEventSynchronize(ev);
  if (e != cudaSuccess) {
    set_error("block map build failed: %s", cudaGetErrorString(e));
    return 3;
  }
  const size_t ncnt = (size_t)4 + bm->nq + bm->nk;
  bm->h_counts = static_cast<int*>(std::malloc(sizeof(int) * ncnt));
  if (!bm->h_counts) return 5;
  if (bm->lists_on_host) {  // the device sent its four counters; the lengths are the host's own
    std::memcpy(bm->h_counts, bm->counts_host, sizeof(int) * 4);
    std::memcpy(bm->h_counts + 4, bm->h_rc_pred, sizeof(int) * (size_t)(bm->nq + bm->nk));
  } else {
    std::memcpy(bm->h_counts, bm->counts_host, sizeof(int) * ncnt);
  }
  PinnedSlot sl;
  sl.host = bm->counts_host;
  sl.dev = bm->counts_dev;
  sl.cap = bm->counts_cap;
  sl.ev = ev;
  pinned_release(bm->device, sl);
  bm->counts_host = nullptr;
  bm->counts_ev = nullptr;
  bm->h_row_cnt = bm->h_counts + 4;
  bm->h_col_cnt = bm->h_row_cnt + bm->nq;
  int64_t nnz = 0;
  for (int i = 0; i < bm->nq; ++i) nnz += bm->h_row_cnt[i];
  bm->nnz = nnz;
  bm->n_full = bm->h_counts[0];
  bm->n_partial = nnz - bm->n_full;
  bm->counts_ready = true;
  if (bm->h_rc_pred) {
    for (int i = 0; i < bm->nq + bm->nk; ++i)
      if (bm->h_rc_pred[i] != bm->h_row_cnt[i]) {
        set_error("block map: the host-derived list length of %s %d is %d, the device's %d", i < bm->nq ? "q tile" : "kv block",
                  i < bm->nq ? i : i - bm->nq, bm->h_rc_pred[i], bm->h_row_cnt[i]);
        return 3;
      }
  }
  if (bm->nnz > bm->nnz_cap || bm->n_partial > bm->p_cap) {
    set_error("block map: %lld list entries and %lld partial tiles exceed the allocation's bounds (%lld, %lld)",
              (long long)bm->nnz, (long long)bm->n_partial, (long long)bm->nnz_cap, (long long)bm->p_cap);
    return 3;
  }
  return 0;
}

int rowcol_counts(const pt_blockmap* bm, const int** row, const int** col) {
  if (bm->h_rc_pred) {  // exact, and identical to the device's (ensure_counts checks)
    *row = bm->h_rc_pred;
    *col = bm->h_rc_pred + bm->nq;
    return 0;
  }
  if (int rc = ensure_counts(bm)) return rc;
  *row = bm->h_row_cnt;
  *col = bm->h_col_cnt;
  return 0;
}

void free_map(pt_blockmap* bm) {
  if (!bm) return;
  pool_free(bm->d_blk, bm->stream);
  if (bm->counts_host) {  // sizes never read: the copy may still be in flight (the pool waits for it)
    PinnedSlot sl;
    sl.host = bm->counts_host;
    sl.dev = bm->counts_dev;
    sl.cap = bm->counts_cap;
    sl.ev = static_cast<cudaEvent_t>(bm->counts_ev);
    pinned_release(bm->device, sl);
  }
  for (pt_dkdv_lists* e = bm->dkdv_lists; e;) {
    pt_dkdv_lists* nx = e->next;
    pool_free(e->mem, bm->stream);
    delete e;
    e = nx;
  }
  for (pt_dq_lists* e = bm->dq_lists; e;) {
    pt_dq_lists* nx = e->next;
    pool_free(e->mem, bm->stream);
    std::free(e->h_empty);
    delete e;
    e = nx;
  }
  std::free(bm->h_rc_pred);
  std::free(bm->h_counts);
  pool_free(bm->mem_lists, bm->stream);
  pool_free(bm->mem_fixed, bm->stream);
  delete bm;
}

// Tree form: validation and the Euler tour on the host (O(nodes)), token
// coordinates and tile classes on the device.
// Checks a tree given as node lengths and sample paths and derives each
// node's parent (-1 for a root) and the token count *T_out.  Returns 1,
// with the error set, for a malformed tree or bad tile sizes.
int parse_tree(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
               int32_t n_samples, int32_t BM, int32_t BN, long long* T_out, std::vector<int>* parent_out) {
  if (n_nodes < 0 || n_samples < 0 || (n_nodes > 0 && !node_lengths) || !path_ptr ||
      (n_samples > 0 && !path_nodes)) {
    set_error("pt_build_blockmap_tree: null array or negative count");
    return 1;
  }
  long long T = 0;
  for (int i = 0; i < n_nodes; ++i) {
    if (node_lengths[i] < 0) {
      set_error("pt_build_blockmap_tree: node %d has negative length %d", i, node_lengths[i]);
      return 1;
    }
    T += node_lengths[i];
  }
  if (T > INT_MAX / 2) {
    set_error("pt_build_blockmap_tree: T = %lld too large", T);
    return 1;
  }
  std::vector<int> parent(n_nodes, -2);
  if (path_ptr[0] != 0) {
    set_error("pt_build_blockmap_tree: path_ptr[0] must be 0");
    return 1;
  }
  for (int sidx = 0; sidx < n_samples; ++sidx) {
    int b = path_ptr[sidx], e = path_ptr[sidx + 1];
    if (e <= b) {
      set_error("pt_build_blockmap_tree: sample path %d is empty", sidx);
      return 1;
    }
    for (int k = b; k < e; ++k) {
      int node = path_nodes[k];
      if (node < 0 || node >= n_nodes) {
        set_error("pt_build_blockmap_tree: path %d names node %d, out of range", sidx, node);
        return 1;
      }
      int want = (k == b) ? -1 : path_nodes[k - 1];
      if (want >= node) {
        set_error("pt_build_blockmap_tree: node %d follows %d on path %d (a parent must have a smaller id)", node,
                  want, sidx);
        return 1;
      }
      if (parent[node] == -2)
        parent[node] = want;
      else if (parent[node] != want) {
        set_error("pt_build_blockmap_tree: node %d has parents %d and %d", node, parent[node], want);
        return 1;
      }
    }
  }
  for (int i = 0; i < n_nodes; ++i)
    if (parent[i] == -2) {
      set_error("pt_build_blockmap_tree: node %d is on no sample path", i);
      return 1;
    }
  if (BM <= 0 || BN <= 0) {
    set_error("pt_build_blockmap_tree: tile sizes must be positive (got %d x %d)", BM, BN);
    return 1;
  }
  *T_out = T;
  *parent_out = std::move(parent);
  return 0;
}

// The q-major lists of a tree map, built on the host, so that nothing
// downstream (the backward's work lists) waits for the device: q tile i
// meets the kv blocks that its rows' kept ranges touch.  The rows of node n
// in the tile keep every token of n's ancestors and n's own tokens up to the
// tile's last row of n (keep = ancestor-or-self and kv <= q; ancestors come
// first).  *row_kv: each q tile's kv blocks, ascending, tile after tile;
// *pred: the list lengths, q tiles then kv blocks.
void tree_host_lists(const int32_t* node_lengths, int N, const std::vector<int>& parent, long long T, int BM, int BN,
                     std::vector<int>* row_kv_out, std::vector<int>* pred_out) {
  std::vector<int> se((size_t)2 * std::max(N, 1));
  int *start = se.data(), *end = start + N;
  {
    long long off = 0;
    for (int i = 0; i < N; ++i) {
      start[i] = (int)off;
      off += node_lengths[i];
      end[i] = (int)off;
    }
  }
  const int nq_h = (int)((T + BM - 1) / BM), nk_h = (int)((T + BN - 1) / BN);
  std::vector<int> pred((size_t)nq_h + nk_h, 0);
  std::vector<int> row_kv;  // the q-major lists themselves, kv blocks ascending per q tile
  {
    std::vector<int> stamp((size_t)std::max(nk_h, 1), -1);
    int n0 = 0;  // nodes are in token order: the first that may reach tile i
    for (int i = 0; i < nq_h; ++i) {
      const long long r_lo = (long long)i * BM, r_hi = std::min<long long>(r_lo + BM, T);
      const size_t row0 = row_kv.size();
      while (n0 < N && end[n0] <= r_lo) ++n0;
      auto mark = [&](long long a, long long b) {  // kv tokens [a, b]
        for (long long j = a / BN; j <= b / BN; ++j)
          if (stamp[(size_t)j] != i) {
            stamp[(size_t)j] = i;
            ++pred[(size_t)i];
            ++pred[(size_t)nq_h + j];
            row_kv.push_back((int)j);
          }
      };
      for (int n = n0; n < N && start[n] < r_hi; ++n) {
        if (end[n] <= r_lo || node_lengths[n] == 0) continue;
        mark(start[n], std::min<long long>(end[n], r_hi) - 1);
        for (int a = parent[n]; a >= 0; a = parent[a])
          if (node_lengths[a] > 0) mark(start[a], end[a] - 1);
      }
      std::sort(row_kv.begin() + (long)row0, row_kv.end());
    }
  }
  *row_kv_out = std::move(row_kv);
  *pred_out = std::move(pred);
}

int debug_tree_lists(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
                     int32_t n_samples, int32_t BM, int32_t BN, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx,
                     int64_t cap, int64_t* nnz) {
  long long T = 0;
  std::vector<int> parent;
  if (parse_tree(node_lengths, n_nodes, path_ptr, path_nodes, n_samples, BM, BN, &T, &parent)) return 1;
  std::vector<int> pred, row_kv;
  tree_host_lists(node_lengths, n_nodes, parent, T, BM, BN, &row_kv, &pred);
  const long long nq = (T + BM - 1) / BM;
  *nnz = (int64_t)row_kv.size();
  if (q_ptr_len < nq + 1 || (int64_t)row_kv.size() > cap) {
    set_error("pt_debug_tree_lists: room for %lld offsets and %lld entries, %lld and %zu needed", (long long)q_ptr_len,
              (long long)cap, nq + 1, row_kv.size());
    return 1;
  }
  q_ptr[0] = 0;
  for (long long t = 0; t < nq; ++t) q_ptr[t + 1] = q_ptr[t] + pred[(size_t)t];
  std::copy(row_kv.begin(), row_kv.end(), kv_idx);
  return 0;
}

int build_tree(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
               int32_t n_samples, int32_t BM, int32_t BN, cudaStream_t s, pt_blockmap** out) {
  long long T = 0;
  std::vector<int> parent;
  if (parse_tree(node_lengths, n_nodes, path_ptr, path_nodes, n_samples, BM, BN, &T, &parent)) return 1;
  // Node tables in one host block: start | end | parent | tin | tout.
  // Euler tour: tin = pre-order index (children in id order), tout = tin + subtree size.
  const int N = n_nodes;
  std::vector<int> tab((size_t)5 * std::max(N, 1));
  int *start = tab.data(), *end = start + N, *par = end + N, *tin = par + N, *tout = tin + N;
  {
    long long off = 0;
    for (int i = 0; i < N; ++i) {
      start[i] = (int)off;
      off += node_lengths[i];
      end[i] = (int)off;
      par[i] = parent[i];
    }
    std::vector<int> subtree(N, 1);
    for (int i = N - 1; i >= 0; --i)
      if (parent[i] >= 0) subtree[parent[i]] += subtree[i];
    std::vector<std::vector<int>> ch(N);
    std::vector<int> roots;
    for (int i = 0; i < N; ++i) (parent[i] < 0 ? roots : ch[parent[i]]).push_back(i);
    int counter = 0;
    std::vector<int> stack(roots.rbegin(), roots.rend());
    while (!stack.empty()) {
      int u = stack.back();
      stack.pop_back();
      tin[u] = counter++;
      tout[u] = tin[u] + subtree[u];
      for (auto it = ch[u].rbegin(); it != ch[u].rend(); ++it) stack.push_back(*it);
    }
  }
  // A partial 128 x 128 tile has its q rows or its kv columns in a 128-token
  // tile that holds a node boundary (or the end of the sequence), or lies on
  // the diagonal: a tile whose rows all belong to one node and whose columns
  // all belong to one node is uniform off the diagonal.  That bounds the
  // partial tiles without waiting for the device.
  int64_t p_bound = -1;
  if (BM == 128 && BN == 128) {
    const long long nt = (T + 127) / 128;
    std::vector<char> split((size_t)nt, 0);
    for (int i = 0; i < N; ++i)
      if (node_lengths[i] > 0 && start[i] % 128 != 0) split[(size_t)(start[i] / 128)] = 1;
    if (T % 128 != 0 && nt > 0) split[(size_t)nt - 1] = 1;
    long long m = 0;
    for (char c : split) m += c;
    p_bound = 2 * m * nt + nt;
  }
  // the q-major lists from the tree, on the host
  const int nq_h = (int)((T + BM - 1) / BM);
  std::vector<int> pred, row_kv;
  tree_host_lists(node_lengths, N, parent, T, BM, BN, &row_kv, &pred);
  if (BM == 128 && BN == 128) maybe_drop_listed_tile(row_kv, pred, nq_h);
  pt_blockmap* bm = nullptr;
  int rc = new_map((int)T, BM, BN, N, s, &bm);
  if (rc) return rc;
  bm->n_nodes = N;
  bm->h_rc_pred = static_cast<int*>(std::malloc(sizeof(int) * std::max<size_t>(pred.size(), 1)));
  if (!bm->h_rc_pred) {
    free_map(bm);
    return 5;
  }
  std::copy(pred.begin(), pred.end(), bm->h_rc_pred);
  do {
    // one upload of start | end | parent | tin | tout into the map's node tables
    const bool listed = BM == 128 && BN == 128 && T > 0;  // tables go with the host lists
    if (N > 0 && !listed && (rc = upload(bm->node_start, tab.data(), sizeof(int) * (size_t)5 * N, bm->device, s)))
      break;
    if (bm->tpad > 0 && !listed) {  // the listed path writes the tokens itself
      const int* d_tin = bm->node_start + 3 * (size_t)N;
      k_tree_tokens<<<(bm->tpad + 255) / 256, 256, 0, s>>>((int)T, bm->tpad, N, bm->node_end, d_tin, d_tin + N,
                                                           bm->tok, bm->node_of);
      PT_LAUNCHED(1);
    }
    rc = listed ? finish_map_listed(bm, s, p_bound, row_kv, N, tab.data()) : finish_map(bm, s, p_bound);
  } while (0);
  if (rc) {
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

int build_seg(const int32_t* group_id, const int32_t* suffix_id, int32_t T, int32_t BM, int32_t BN, cudaStream_t s,
              pt_blockmap** out) {
  if (T < 0 || (T > 0 && (!group_id || !suffix_id))) {
    set_error("pt_build_blockmap_seg: null labels or negative T");
    return 1;
  }
  if (BM <= 0 || BN <= 0) {
    set_error("pt_build_blockmap_seg: tile sizes must be positive (got %d x %d)", BM, BN);
    return 1;
  }
  pt_blockmap* bm = nullptr;
  int rc = new_map(T, BM, BN, std::max(T, 1), s, &bm);
  if (rc) return rc;
  void* tmp = nullptr;
  do {
    Layout L;
    const int Tc = std::max(T, 1);
    size_t o_fl = L.add<int>(Tc), o_ex = L.add<int>((size_t)Tc + 1), o_gs = L.add<int>(Tc), o_ss = L.add<int>(Tc),
           o_gf = L.add<int>(Tc), o_gl = L.add<int>(Tc), o_ti = L.add<int>(Tc), o_to = L.add<int>(Tc),
           o_er = L.add<int>(1), o_st = L.add<int>((size_t)Tc / kScanBlock + 2);
    if ((rc = pool_alloc(&tmp, L.off, bm->device, s))) break;
    int *flags = at<int>(tmp, o_fl), *excl = at<int>(tmp, o_ex), *gseen = at<int>(tmp, o_gs),
        *sseen = at<int>(tmp, o_ss), *gfirst = at<int>(tmp, o_gf), *glast = at<int>(tmp, o_gl),
        *tin = at<int>(tmp, o_ti), *tout = at<int>(tmp, o_to), *err = at<int>(tmp, o_er),
        *stmp = at<int>(tmp, o_st);
    if (cudaMemsetAsync(gseen, 0, sizeof(int) * Tc, s) != cudaSuccess ||
        cudaMemsetAsync(sseen, 0, sizeof(int) * Tc, s) != cudaSuccess ||
        cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) {
      rc = 3;
      break;
    }
    int R = 0, herr = 0;
    if (T > 0) {
      int nb = (T + 255) / 256;
      k_seg_flags<<<nb, 256, 0, s>>>(group_id, suffix_id, T, flags, gseen, sseen, err);
      k_seen_check<<<nb, 256, 0, s>>>(gseen, sseen, T, err);
      PT_LAUNCHED(2);
      if ((rc = exclusive_scan(flags, T, excl, stmp, s))) break;
      if (cudaMemcpyAsync(&R, excl + T, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaMemcpyAsync(&herr, err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamSynchronize(s) != cudaSuccess) {
        set_error("pt_build_blockmap_seg: label pass failed");
        rc = 3;
        break;
      }
      if (herr) {
        set_error("pt_build_blockmap_seg: invalid labels (%s%s%s%s)", (herr & 1) ? "id out of range; " : "",
                  (herr & 2) ? "prompt run does not open its group; " : "",
                  (herr & 4) ? "a group id forms more than one run; " : "",
                  (herr & 8) ? "a suffix id forms more than one run" : "");
        rc = 1;
        break;
      }
      k_seg_nodes<<<nb, 256, 0, s>>>(group_id, suffix_id, T, flags, excl, bm->node_of, bm->node_start, bm->node_end,
                                     gfirst, glast);
      k_seg_tree<<<(R + 255) / 256, 256, 0, s>>>(group_id, suffix_id, R, bm->node_start, gfirst, glast, bm->parent,
                                                 tin, tout);
      PT_LAUNCHED(2);
    }
    bm->n_nodes = R;
    if (bm->tpad > 0) {
      k_seg_tokens<<<(bm->tpad + 255) / 256, 256, 0, s>>>(T, bm->tpad, bm->node_of, tin, tout, bm->tok);
      PT_LAUNCHED(1);
    }
    rc = finish_map(bm, s, -1);
  } while (0);
  pool_free(tmp, s);
  if (rc) {
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

// Checks a draft-block layout and derives each block's context range before
// any window, [x, y), its anchor and keep flag (int4 x, y, z, w); *T_out the
// token count.  Returns 1 (or 2 for tiles other than 128 x 128), with the
// error set, for a bad layout.
int parse_draft(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                const uint8_t* block_keep, int32_t window, const int32_t* ctx_doc, const int32_t* anchor_doc,
                int32_t BM, int32_t BN, long long* T_out, std::vector<int4>* blk_out) {
  if (ctx_len < 0 || n_blocks < 0 || block_size < 1 || window < 0 || (n_blocks > 0 && !anchors)) {
    set_error("pt_build_blockmap_draft: negative length, block size < 1, negative window or null anchors");
    return 1;
  }
  if ((ctx_doc == nullptr) != (anchor_doc == nullptr) || (ctx_doc && ctx_len > 0 && !ctx_doc)) {
    set_error("pt_build_blockmap_draft: ctx_doc and anchor_doc must be given together");
    return 1;
  }
  if (BM != 128 || BN != 128) {
    set_error("pt_build_blockmap_draft: draft maps are built for 128 x 128 tiles only (got %d x %d)", BM, BN);
    return 2;
  }
  const long long T = (long long)ctx_len + (long long)n_blocks * block_size;
  if (T > INT_MAX / 2) {
    set_error("pt_build_blockmap_draft: T = %lld too large", T);
    return 1;
  }
  for (int b = 0; b < n_blocks; ++b)
    if (anchors[b] < 0 || anchors[b] > ctx_len) {
      set_error("pt_build_blockmap_draft: anchor %d of block %d outside [0, %d]", anchors[b], b, ctx_len);
      return 1;
    }
  // documents: each id one contiguous run of the context
  std::unordered_map<int32_t, std::pair<int32_t, int32_t>> runs;
  if (ctx_doc) {
    for (int32_t t = 0; t < ctx_len;) {
      int32_t e = t + 1;
      while (e < ctx_len && ctx_doc[e] == ctx_doc[t]) ++e;
      if (!runs.emplace(ctx_doc[t], std::make_pair(t, e)).second) {
        set_error("pt_build_blockmap_draft: document %d is not one contiguous run of the context", ctx_doc[t]);
        return 1;
      }
      t = e;
    }
  }
  // per block: the context it keeps before any window, [x, y); anchor; keep flag
  std::vector<int4> blk((size_t)std::max(n_blocks, 1));
  for (int b = 0; b < n_blocks; ++b) {
    int lo = 0, hi = anchors[b];
    if (ctx_doc) {
      auto it = runs.find(anchor_doc[b]);
      if (it == runs.end()) {
        lo = hi = 0;
      } else {
        lo = it->second.first;
        hi = std::min(it->second.second, anchors[b]);
        if (lo >= hi) lo = hi = 0;
      }
    }
    blk[b] = make_int4(lo, hi, anchors[b], (!block_keep || block_keep[b]) ? 1 : 0);
  }
  *T_out = T;
  *blk_out = std::move(blk);
  return 0;
}

// The q-major lists of a draft-block map, built on the host as for trees.
// The rows of block b in q tile i are its tokens k0..k1; row k keeps the
// context [x, y) cut by the window to kv >= anchor + k - window + 1 (a range
// that shrinks as k grows, so the rows' union is row k0's), and its own
// block up to k (causal) or all of it.  Context rows keep nothing.  Also
// every kept pair of the map in closed form (*pairs_out): row k of a kept
// block keeps its context range (cut by the window) and k + 1 (causal) or
// all of its block's keys.
void draft_host_lists(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const std::vector<int4>& blk,
                      int32_t causal, int32_t window, long long T, int BM, int BN, std::vector<int>* row_kv_out,
                      std::vector<int>* pred_out, long long* pairs_out) {
  const int nq_h = (int)((T + BM - 1) / BM), nk_h = (int)((T + BN - 1) / BN);
  std::vector<int> pred((size_t)nq_h + nk_h, 0);
  std::vector<int> row_kv;  // the lists themselves: kv blocks of each q tile, ascending
  {
    std::vector<int> stamp((size_t)std::max(nk_h, 1), -1);
    for (int i = 0; i < nq_h; ++i) {
      const long long r_lo = std::max<long long>((long long)i * BM, ctx_len);
      const long long r_hi = std::min<long long>((long long)(i + 1) * BM, T);
      const size_t row0 = row_kv.size();
      auto mark = [&](long long a, long long b) {  // kv tokens [a, b]
        for (long long j = a / BN; j <= b / BN; ++j)
          if (stamp[(size_t)j] != i) {
            stamp[(size_t)j] = i;
            ++pred[(size_t)i];
            ++pred[(size_t)nq_h + j];
            row_kv.push_back((int)j);
          }
      };
      for (long long r = r_lo; r < r_hi;) {
        const int b = (int)((r - ctx_len) / block_size);
        const long long b0 = ctx_len + (long long)b * block_size;
        const long long k0 = r - b0, k1 = std::min<long long>(b0 + block_size, r_hi) - 1 - b0;
        r = b0 + k1 + 1;
        if (!blk[b].w) continue;
        long long x = blk[b].x;
        if (window > 0) x = std::max<long long>(x, (long long)blk[b].z + k0 - window + 1);
        if (x < blk[b].y) mark(x, blk[b].y - 1);
        mark(b0, b0 + (causal ? k1 : block_size - 1));
      }
      std::sort(row_kv.begin() + row0, row_kv.end());
    }
  }
  long long draft_pairs = 0;
  for (int b = 0; b < n_blocks; ++b) {
    if (!blk[b].w) continue;
    for (int k = 0; k < block_size; ++k) {
      long long x = blk[b].x;
      if (window > 0) x = std::max<long long>(x, (long long)blk[b].z + k - window + 1);
      draft_pairs += std::max<long long>(0, blk[b].y - x) + (causal ? k + 1 : block_size);
    }
  }
  *row_kv_out = std::move(row_kv);
  *pred_out = std::move(pred);
  *pairs_out = draft_pairs;
}

int debug_draft_lists(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                      const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                      const int32_t* anchor_doc, int32_t* q_ptr, int64_t q_ptr_len, int32_t* kv_idx, int64_t cap,
                      int64_t* nnz, int64_t* kept_pairs) {
  long long T = 0;
  std::vector<int4> blk;
  if (int rc = parse_draft(ctx_len, n_blocks, block_size, anchors, block_keep, window, ctx_doc, anchor_doc, 128, 128,
                           &T, &blk))
    return rc;
  std::vector<int> row_kv, pred;
  long long pairs = 0;
  draft_host_lists(ctx_len, n_blocks, block_size, blk, causal, window, T, 128, 128, &row_kv, &pred, &pairs);
  const long long nq = (T + 127) / 128;
  *nnz = (int64_t)row_kv.size();
  *kept_pairs = pairs;
  if (q_ptr_len < nq + 1 || (int64_t)row_kv.size() > cap) {
    set_error("pt_debug_draft_lists: room for %lld offsets and %lld entries, %lld and %zu needed",
              (long long)q_ptr_len, (long long)cap, nq + 1, row_kv.size());
    return 1;
  }
  q_ptr[0] = 0;
  for (long long t = 0; t < nq; ++t) q_ptr[t + 1] = q_ptr[t] + pred[(size_t)t];
  std::copy(row_kv.begin(), row_kv.end(), kv_idx);
  return 0;
}

int build_draft(int32_t ctx_len, int32_t n_blocks, int32_t block_size, const int32_t* anchors,
                const uint8_t* block_keep, int32_t causal, int32_t window, const int32_t* ctx_doc,
                const int32_t* anchor_doc, int32_t BM, int32_t BN, cudaStream_t s, pt_blockmap** out) {
  long long T = 0;
  std::vector<int4> blk;
  if (int rc = parse_draft(ctx_len, n_blocks, block_size, anchors, block_keep, window, ctx_doc, anchor_doc, BM, BN,
                           &T, &blk))
    return rc;
  const int nq_h = (int)((T + BM - 1) / BM);
  std::vector<int> pred, row_kv;
  long long draft_pairs = 0;
  // the device's sum of kept pairs over the listed tiles must equal draft_pairs
  draft_host_lists(ctx_len, n_blocks, block_size, blk, causal, window, T, BM, BN, &row_kv, &pred, &draft_pairs);
  maybe_drop_listed_tile(row_kv, pred, nq_h);
  long long nnz_exact = 0;
  for (int i = 0; i < nq_h; ++i) nnz_exact += pred[(size_t)i];
  pt_blockmap* bm = nullptr;
  int rc = new_map((int)T, BM, BN, 0, s, &bm);
  if (rc) return rc;
  bm->h_rc_pred = static_cast<int*>(std::malloc(sizeof(int) * std::max<size_t>(pred.size(), 1)));
  if (!bm->h_rc_pred) {
    free_map(bm);
    return 5;
  }
  std::copy(pred.begin(), pred.end(), bm->h_rc_pred);
  bm->producer = PT_PRODUCER_DRAFT;
  bm->d_ctx = ctx_len;
  bm->d_bs = block_size;
  bm->d_nb = n_blocks;
  bm->d_causal = causal ? 1 : 0;
  bm->d_window = window;
  do {
    if ((rc = pool_alloc(&bm->d_blk, sizeof(int4) * blk.size(), bm->device, s))) break;
    if (n_blocks > 0 && (rc = upload(bm->d_blk, blk.data(), sizeof(int4) * (size_t)n_blocks, bm->device, s))) break;
    rc = finish_map_listed(bm, s, nnz_exact, row_kv, 0, nullptr, draft_pairs);  // every listed tile may be partial
  } while (0);
  if (rc) {
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

int build_dense(const pt_blockmap* src, cudaStream_t s, pt_blockmap** out) {
  pt_blockmap* bm = nullptr;
  int rc = new_map(src->T, src->BM, src->BN, std::max(src->n_nodes, 1), s, &bm);
  if (rc) return rc;
  bm->n_nodes = src->n_nodes;
  bm->dense = true;
  bm->producer = src->producer;
  bm->d_ctx = src->d_ctx;
  bm->d_bs = src->d_bs;
  bm->d_nb = src->d_nb;
  bm->d_causal = src->d_causal;
  bm->d_window = src->d_window;
  const int nq = bm->nq, nk = bm->nk;
  const long long n = (long long)nq * nk;
  void* tmp = nullptr;
  do {
    if (n > INT_MAX / 32) {
      set_error("pt_blockmap_dense: %lld tiles is too many", n);
      rc = 2;
      break;
    }
    if (src->producer == PT_PRODUCER_DRAFT) {
      const size_t bytes = sizeof(int4) * (size_t)std::max(src->d_nb, 1);
      if ((rc = pool_alloc(&bm->d_blk, bytes, bm->device, s))) break;
      if (cudaMemcpyAsync(bm->d_blk, src->d_blk, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
        set_error("pt_blockmap_dense: copy failed");
        rc = 3;
        break;
      }
    }
    if (cudaMemcpyAsync(bm->tok, src->tok, sizeof(pt_tok) * bm->tpad, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        (bm->T &&
         cudaMemcpyAsync(bm->node_of, src->node_of, sizeof(int) * bm->T, cudaMemcpyDeviceToDevice, s) != cudaSuccess) ||
        (bm->n_nodes &&
         (cudaMemcpyAsync(bm->node_start, src->node_start, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) !=
              cudaSuccess ||
          cudaMemcpyAsync(bm->node_end, src->node_end, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) !=
              cudaSuccess ||
          cudaMemcpyAsync(bm->parent, src->parent, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) !=
              cudaSuccess))) {
      set_error("pt_blockmap_dense: copy failed");
      rc = 3;
      break;
    }
    bm->nnz = n;
    bm->n_full = 0;
    bm->n_partial = n;
    bm->h_counts = static_cast<int*>(std::malloc(sizeof(int) * (4 + (size_t)nq + nk)));
    if (!bm->h_counts) {
      rc = 5;
      break;
    }
    bm->h_row_cnt = bm->h_counts + 4;
    bm->h_col_cnt = bm->h_row_cnt + nq;
    for (int i = 0; i < nq; ++i) bm->h_row_cnt[i] = nk;
    for (int j = 0; j < nk; ++j) bm->h_col_cnt[j] = nq;
    bm->counts_ready = true;
    if ((rc = alloc_lists(bm, n, n, s))) break;
    if ((rc = pool_alloc(&tmp, sizeof(int2) * (size_t)std::max<long long>(n, 1), bm->device, s))) break;
    int2* slot_tile = static_cast<int2*>(tmp);
    long long cnt = std::max<long long>(n, std::max(nq, nk) + 1);
    k_dense_lists<<<(unsigned)((cnt + 255) / 256), 256, 0, s>>>(nq, nk, bm->q_ptr, bm->kv_idx, bm->kind, bm->k_ptr,
                                                                bm->q_idx, bm->kindT, bm->pidx, bm->pidxT, slot_tile);
    PT_LAUNCHED(1);
    if (bm->mask_rows && n > 0) {
      const long long grid = std::min<long long>(n, (long long)num_sms(bm->device) * 16);
      if (bm->producer == PT_PRODUCER_DRAFT)
        k_draft_masks<<<(unsigned)grid, 128, 0, s>>>(bm->T, draft_params(bm), slot_tile, bm->mask_rows,
                                                     bm->mask_cols, n, nullptr, nullptr, n);
      else
        k_masks<<<(unsigned)grid, 128, 0, s>>>(bm->T, bm->tok, slot_tile, bm->mask_rows, bm->mask_cols, n, nullptr,
                                               nullptr, n);
      PT_LAUNCHED(1);
    }
    // every row has the same length: natural order
    if (nq > 0 && nk > 0) {
      std::vector<int> idx(std::max(nq, nk));
      std::iota(idx.begin(), idx.end(), 0);
      if ((rc = upload(bm->q_order, idx.data(), sizeof(int) * nq, bm->device, s))) break;
      if ((rc = upload(bm->k_order, idx.data(), sizeof(int) * nk, bm->device, s))) break;
    }
  } while (0);
  pool_free(tmp, s);
  if (rc) {
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

}  // namespace pt
