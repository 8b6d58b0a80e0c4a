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
#include <climits>
#include <cstdio>
#include <cstring>
#include <numeric>
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
                           const int* node_end, const int* parent, uint8_t* kinds) {
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
  }
}

// one warp per row (q tile) or per column (kv block): counts of non-empty and full
__global__ void k_counts(const uint8_t* kinds, int nq, int nk, bool by_col, int* cnt, int* n_full) {
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  int nrows = by_col ? nk : nq, len = by_col ? nq : nk;
  if (w >= nrows) return;
  int c = 0, f = 0;
  for (int x = lane; x < len; x += 32) {
    uint8_t k = by_col ? kinds[(long long)x * nk + w] : kinds[(long long)w * nk + x];
    c += (k != 0);
    f += (k == PT_KIND_FULL);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    c += __shfl_xor_sync(0xffffffffu, c, o);
    f += __shfl_xor_sync(0xffffffffu, f, o);
  }
  if (lane == 0) {
    cnt[w] = c;
    if (!by_col) atomicAdd(n_full, f);
  }
}

// ordered compaction of each row (or column) into its list slot.  For the
// kv-major lists, `q_ptr`/`kv_idx`/`pidx` of the finished q-major list give
// each tile's mask slot (binary search of the kv block in the q tile's row).
__global__ void k_fill(const uint8_t* kinds, int nq, int nk, bool by_col, const int* ptr, int* idx, uint8_t* kd,
                       int* pflag, const int* q_ptr, const int* kv_idx, const int* pidx, int* pidxT) {
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  int nrows = by_col ? nk : nq, len = by_col ? nq : nk;
  if (w >= nrows) return;
  int pos = ptr[w];
  for (int base = 0; base < len; base += 32) {
    int x = base + lane;
    uint8_t k = 0;
    if (x < len) k = by_col ? kinds[(long long)x * nk + w] : kinds[(long long)w * nk + x];
    unsigned m = __ballot_sync(0xffffffffu, k != 0);
    if (k) {
      int off = __popc(m & ((1u << lane) - 1));
      idx[pos + off] = x;
      kd[pos + off] = k;
      if (!by_col) {
        pflag[pos + off] = (k == PT_KIND_PARTIAL);
      } else {
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
    }
    pos += __popc(m);
  }
}

// q-major: mask slot of each partial entry (exclusive scan of partial flags),
// and the (q tile, kv block) of every slot.
__global__ void k_slots(int nq, const int* q_ptr, const int* kv_idx, const uint8_t* kind, const int* pscan,
                        int* pidx, int2* slot_tile) {
  int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= nq) return;
  for (int e = q_ptr[w] + lane; e < q_ptr[w + 1]; e += 32) {
    if (kind[e] == PT_KIND_PARTIAL) {
      int s = pscan[e];
      pidx[e] = s;
      slot_tile[s] = make_int2(w, kv_idx[e]);
    } else {
      pidx[e] = -1;
    }
  }
}

// Keep bitmasks of every partial 128 x 128 tile, both orientations:
// mask_rows[slot][r][w] bit b = keep(q = i*128 + r, kv = j*128 + 32w + b),
// mask_cols[slot][c][w] bit b = keep(q = i*128 + 32w + b, kv = j*128 + c).
// Pairs outside [0, T) are never kept.
__global__ void k_masks(int T, const pt_tok* tok, const int2* slot_tile, uint32_t* mask_rows, uint32_t* mask_cols) {
  __shared__ pt_tok tq[128], tk[128];
  const int s = blockIdx.x, r = threadIdx.x;
  const int2 ij = slot_tile[s];
  const int q0 = ij.x * 128, k0 = ij.y * 128;
  tq[r] = tok[q0 + r];
  tk[r] = tok[k0 + r];
  __syncthreads();
  uint32_t row[4] = {0, 0, 0, 0}, col[4] = {0, 0, 0, 0};
  const int q = q0 + r, kv = k0 + r;
  const pt_tok mq = tq[r], mk = tk[r];
  for (int c = 0; c < 128; ++c) {
    const int kvc = k0 + c;
    const pt_tok t = tk[c];
    if (q < T && kvc < T && kvc <= q && t.tin <= mq.tin && mq.tin < t.tout) row[c >> 5] |= 1u << (c & 31);
    const int qc = q0 + c;
    const pt_tok u = tq[c];
    if (qc < T && kv < T && kv <= qc && mk.tin <= u.tin && u.tin < mk.tout) col[c >> 5] |= 1u << (c & 31);
  }
  uint4* mr = reinterpret_cast<uint4*>(mask_rows) + (size_t)s * 128 + r;
  uint4* mc = reinterpret_cast<uint4*>(mask_cols) + (size_t)s * 128 + r;
  *mr = make_uint4(row[0], row[1], row[2], row[3]);
  *mc = make_uint4(col[0], col[1], col[2], col[3]);
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

template <class T>
int dalloc(T** p, size_t n) {
  if (n == 0) n = 1;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T));
  if (e != cudaSuccess) {
    *p = nullptr;
    set_error("cudaMalloc of %zu bytes failed: %s", n * sizeof(T), cudaGetErrorString(e));
    return 5;
  }
  return 0;
}

#define PT_TRY(x)         \
  do {                    \
    int rc_ = (x);        \
    if (rc_) return rc_;  \
  } while (0)

// Longest-first order: most entries first, ties by index.
void lpt_order(const std::vector<int>& cnt, std::vector<int>& order) {
  order.resize(cnt.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cnt[a] > cnt[b]; });
}

// Shared tail of every builder: given tok, node_of and node tables on the
// device, classify, count, list and order.
int finish_map(pt_blockmap* bm, cudaStream_t s) {
  ProfScope ps(s, "blockmap_classify");
  const int nq = bm->nq, nk = bm->nk;
  const long long ntiles = (long long)nq * nk;
  uint8_t* kinds = nullptr;
  int *row_cnt = nullptr, *col_cnt = nullptr, *counters = nullptr, *tmp = nullptr;
  int rc = 0;
  do {
    if ((rc = dalloc(&kinds, (size_t)ntiles))) break;
    if ((rc = dalloc(&row_cnt, nq))) break;
    if ((rc = dalloc(&col_cnt, nk))) break;
    if ((rc = dalloc(&counters, 4))) break;
    if ((rc = dalloc(&tmp, (size_t)std::max(nq, nk) / kScanBlock + 2))) break;
    if ((rc = dalloc(&bm->q_ptr, nq + 1))) break;
    if ((rc = dalloc(&bm->k_ptr, nk + 1))) break;
    if (cudaMemsetAsync(counters, 0, 4 * sizeof(int), s) != cudaSuccess) { rc = 3; break; }
    if (ntiles > 0) {
      long long threads = ntiles * 32;
      k_classify<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(bm->T, bm->BM, bm->BN, nq, nk, bm->node_of,
                                                                   bm->node_start, bm->node_end, bm->parent, kinds);
      k_counts<<<(nq * 32 + 255) / 256, 256, 0, s>>>(kinds, nq, nk, false, row_cnt, counters);
      k_counts<<<(nk * 32 + 255) / 256, 256, 0, s>>>(kinds, nq, nk, true, col_cnt, counters);
      count_launch(3);
    }
    if ((rc = exclusive_scan(row_cnt, nq, bm->q_ptr, tmp, s))) break;
    if ((rc = exclusive_scan(col_cnt, nk, bm->k_ptr, tmp, s))) break;
    std::vector<int> hq(nq), hk(nk);
    int nnz = 0, nfull = 0;
    if (nq && cudaMemcpyAsync(hq.data(), row_cnt, nq * sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) { rc = 3; break; }
    if (nk && cudaMemcpyAsync(hk.data(), col_cnt, nk * sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) { rc = 3; break; }
    if (cudaMemcpyAsync(&nnz, bm->q_ptr + nq, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) { rc = 3; break; }
    if (cudaMemcpyAsync(&nfull, counters, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) { rc = 3; break; }
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      set_error("block map build failed: %s", cudaGetErrorString(e));
      rc = 3;
      break;
    }
    bm->nnz = nnz;
    bm->n_full = nfull;
    if ((rc = dalloc(&bm->kv_idx, nnz))) break;
    if ((rc = dalloc(&bm->kind, nnz))) break;
    if ((rc = dalloc(&bm->q_idx, nnz))) break;
    if ((rc = dalloc(&bm->kindT, nnz))) break;
    if ((rc = dalloc(&bm->q_order, nq))) break;
    if ((rc = dalloc(&bm->k_order, nk))) break;
    if ((rc = dalloc(&bm->pidx, nnz))) break;
    if ((rc = dalloc(&bm->pidxT, nnz))) break;
    bm->n_partial = nnz - nfull;
    const bool masks = bm->BM == 128 && bm->BN == 128 && bm->n_partial > 0;
    if (masks) {
      if ((rc = dalloc(&bm->mask_rows, (size_t)bm->n_partial * 512))) break;
      if ((rc = dalloc(&bm->mask_cols, (size_t)bm->n_partial * 512))) break;
    }
    if (ntiles > 0 && nnz > 0) {
      int* pflag = nullptr;
      int* pscan = nullptr;
      int* stmp = nullptr;
      int2* slot_tile = nullptr;
      if ((rc = dalloc(&pflag, nnz))) break;
      if ((rc = dalloc(&pscan, (size_t)nnz + 1)) || (rc = dalloc(&stmp, (size_t)nnz / kScanBlock + 2)) ||
          (rc = dalloc(&slot_tile, std::max<int64_t>(bm->n_partial, 1)))) {
        cudaFree(pflag);
        cudaFree(pscan);
        cudaFree(stmp);
        break;
      }
      k_fill<<<(nq * 32 + 255) / 256, 256, 0, s>>>(kinds, nq, nk, false, bm->q_ptr, bm->kv_idx, bm->kind, pflag,
                                                     nullptr, nullptr, nullptr, nullptr);
      count_launch();
      rc = exclusive_scan(pflag, nnz, pscan, stmp, s);
      if (!rc) {
        k_slots<<<(nq * 32 + 255) / 256, 256, 0, s>>>(nq, bm->q_ptr, bm->kv_idx, bm->kind, pscan, bm->pidx,
                                                       slot_tile);
        k_fill<<<(nk * 32 + 255) / 256, 256, 0, s>>>(kinds, nq, nk, true, bm->k_ptr, bm->q_idx, bm->kindT, nullptr,
                                                       bm->q_ptr, bm->kv_idx, bm->pidx, bm->pidxT);
        count_launch(2);
        if (masks) {
          k_masks<<<(unsigned)bm->n_partial, 128, 0, s>>>(bm->T, bm->tok, slot_tile, bm->mask_rows, bm->mask_cols);
          count_launch();
        }
      }
      cudaError_t le = cudaStreamSynchronize(s);
      cudaFree(pflag);
      cudaFree(pscan);
      cudaFree(stmp);
      cudaFree(slot_tile);
      if (rc) break;
      if (le != cudaSuccess) {
        set_error("block map lists failed: %s", cudaGetErrorString(le));
        rc = 3;
        break;
      }
    }
    std::vector<int> oq, ok;
    lpt_order(hq, oq);
    lpt_order(hk, ok);
    if (nq && cudaMemcpyAsync(bm->q_order, oq.data(), nq * sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) { rc = 3; break; }
    if (nk && cudaMemcpyAsync(bm->k_order, ok.data(), nk * sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) { rc = 3; break; }
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      set_error("block map build failed: %s", cudaGetErrorString(e));
      rc = 3;
      break;
    }
  } while (0);
  cudaFree(kinds);
  cudaFree(row_cnt);
  cudaFree(col_cnt);
  cudaFree(counters);
  cudaFree(tmp);
  return rc;
}

pt_blockmap* new_map(int T, int BM, int BN) {
  pt_blockmap* bm = new pt_blockmap;
  std::memset(bm, 0, sizeof(*bm));
  cudaGetDevice(&bm->device);
  bm->T = T;
  bm->BM = BM;
  bm->BN = BN;
  bm->nq = (T + BM - 1) / BM;
  bm->nk = (T + BN - 1) / BN;
  bm->tpad = std::max(bm->nq * BM, bm->nk * BN);
  return bm;
}

}  // namespace

void free_map(pt_blockmap* bm) {
  if (!bm) return;
  void* ptrs[] = {bm->tok, bm->node_of, bm->node_start, bm->node_end, bm->parent, bm->q_ptr, bm->kv_idx,
                  bm->kind, bm->k_ptr, bm->q_idx, bm->kindT, bm->q_order, bm->k_order, bm->pidx, bm->pidxT,
                  bm->mask_rows, bm->mask_cols};
  for (void* p : ptrs) cudaFree(p);
  delete bm;
}

// Tree form: validation and the Euler tour on the host (O(nodes)), token
// coordinates and tile classes on the device.
int build_tree(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr, const int32_t* path_nodes,
               int32_t n_samples, int32_t BM, int32_t BN, cudaStream_t s, pt_blockmap** out) {
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
  // Euler tour: tin = pre-order index, tout = tin + subtree size.
  std::vector<int> start(n_nodes), end(n_nodes), tin(n_nodes), tout(n_nodes), subtree(n_nodes, 1);
  long long off = 0;
  for (int i = 0; i < n_nodes; ++i) {
    start[i] = (int)off;
    off += node_lengths[i];
    end[i] = (int)off;
  }
  for (int i = n_nodes - 1; i >= 0; --i)
    if (parent[i] >= 0) subtree[parent[i]] += subtree[i];
  {
    // children in id order; pre-order numbering
    std::vector<std::vector<int>> ch(n_nodes);
    std::vector<int> roots;
    for (int i = 0; i < n_nodes; ++i) (parent[i] < 0 ? roots : ch[parent[i]]).push_back(i);
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
  if (BM <= 0 || BN <= 0) {
    set_error("pt_build_blockmap_tree: tile sizes must be positive (got %d x %d)", BM, BN);
    return 1;
  }
  pt_blockmap* bm = new_map((int)T, BM, BN);
  bm->n_nodes = n_nodes;
  int* d_tin = nullptr;
  int* d_tout = nullptr;
  int rc = 0;
  do {
    if ((rc = dalloc(&bm->tok, bm->tpad))) break;
    if ((rc = dalloc(&bm->node_of, T))) break;
    if ((rc = dalloc(&bm->node_start, n_nodes))) break;
    if ((rc = dalloc(&bm->node_end, n_nodes))) break;
    if ((rc = dalloc(&bm->parent, n_nodes))) break;
    if ((rc = dalloc(&d_tin, n_nodes))) break;
    if ((rc = dalloc(&d_tout, n_nodes))) break;
    size_t nb = sizeof(int) * n_nodes;
    if (n_nodes &&
        (cudaMemcpyAsync(bm->node_start, start.data(), nb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
         cudaMemcpyAsync(bm->node_end, end.data(), nb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
         cudaMemcpyAsync(bm->parent, parent.data(), nb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
         cudaMemcpyAsync(d_tin, tin.data(), nb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
         cudaMemcpyAsync(d_tout, tout.data(), nb, cudaMemcpyHostToDevice, s) != cudaSuccess)) {
      set_error("pt_build_blockmap_tree: upload failed");
      rc = 3;
      break;
    }
    if (bm->tpad > 0) {
      k_tree_tokens<<<(bm->tpad + 255) / 256, 256, 0, s>>>((int)T, bm->tpad, n_nodes, bm->node_end, d_tin, d_tout,
                                                           bm->tok, bm->node_of);
      count_launch();
    }
    rc = finish_map(bm, s);  // synchronises s
  } while (0);
  cudaFree(d_tin);
  cudaFree(d_tout);
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
  pt_blockmap* bm = new_map(T, BM, BN);
  int *flags = nullptr, *excl = nullptr, *gseen = nullptr, *sseen = nullptr, *err = nullptr, *tmp = nullptr;
  int *gfirst = nullptr, *glast = nullptr, *tin = nullptr, *tout = nullptr;
  int rc = 0;
  do {
    if ((rc = dalloc(&bm->tok, bm->tpad))) break;
    if ((rc = dalloc(&bm->node_of, T))) break;
    if ((rc = dalloc(&bm->node_start, T))) break;
    if ((rc = dalloc(&bm->node_end, T))) break;
    if ((rc = dalloc(&bm->parent, T))) break;
    if ((rc = dalloc(&flags, T))) break;
    if ((rc = dalloc(&excl, (size_t)T + 1))) break;
    if ((rc = dalloc(&gseen, T))) break;
    if ((rc = dalloc(&sseen, T))) break;
    if ((rc = dalloc(&gfirst, T))) break;
    if ((rc = dalloc(&glast, T))) break;
    if ((rc = dalloc(&tin, T))) break;
    if ((rc = dalloc(&tout, T))) break;
    if ((rc = dalloc(&err, 1))) break;
    if ((rc = dalloc(&tmp, (size_t)T / kScanBlock + 2))) break;
    if (cudaMemsetAsync(gseen, 0, sizeof(int) * std::max(T, 1), s) != cudaSuccess ||
        cudaMemsetAsync(sseen, 0, sizeof(int) * std::max(T, 1), s) != cudaSuccess ||
        cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) {
      rc = 3;
      break;
    }
    int R = 0, herr = 0;
    if (T > 0) {
      int nb = (T + 255) / 256;
      k_seg_flags<<<nb, 256, 0, s>>>(group_id, suffix_id, T, flags, gseen, sseen, err);
      k_seen_check<<<nb, 256, 0, s>>>(gseen, sseen, T, err);
      count_launch(2);
      if ((rc = exclusive_scan(flags, T, excl, tmp, s))) break;
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
      count_launch(2);
    }
    bm->n_nodes = R;
    if (bm->tpad > 0) {
      k_seg_tokens<<<(bm->tpad + 255) / 256, 256, 0, s>>>(T, bm->tpad, bm->node_of, tin, tout, bm->tok);
      count_launch();
    }
    rc = finish_map(bm, s);
  } while (0);
  int* tmps[] = {flags, excl, gseen, sseen, err, tmp, gfirst, glast, tin, tout};
  for (int* p : tmps) cudaFree(p);
  if (rc) {
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

int build_dense(const pt_blockmap* src, cudaStream_t s, pt_blockmap** out) {
  pt_blockmap* bm = new_map(src->T, src->BM, src->BN);
  bm->n_nodes = src->n_nodes;
  bm->dense = true;
  const int nq = bm->nq, nk = bm->nk;
  const long long n = (long long)nq * nk;
  int rc = 0;
  do {
    if (n > INT_MAX) {
      set_error("pt_blockmap_dense: %lld tiles is too many", n);
      rc = 2;
      break;
    }
    if ((rc = dalloc(&bm->tok, bm->tpad))) break;
    if ((rc = dalloc(&bm->node_of, bm->T))) break;
    if ((rc = dalloc(&bm->node_start, std::max(1, bm->n_nodes)))) break;
    if ((rc = dalloc(&bm->node_end, std::max(1, bm->n_nodes)))) break;
    if ((rc = dalloc(&bm->parent, std::max(1, bm->n_nodes)))) break;
    if ((rc = dalloc(&bm->q_ptr, nq + 1))) break;
    if ((rc = dalloc(&bm->k_ptr, nk + 1))) break;
    if ((rc = dalloc(&bm->kv_idx, n))) break;
    if ((rc = dalloc(&bm->kind, n))) break;
    if ((rc = dalloc(&bm->q_idx, n))) break;
    if ((rc = dalloc(&bm->kindT, n))) break;
    if ((rc = dalloc(&bm->q_order, nq))) break;
    if ((rc = dalloc(&bm->k_order, nk))) break;
    if (cudaMemcpyAsync(bm->tok, src->tok, sizeof(pt_tok) * bm->tpad, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        (bm->T && cudaMemcpyAsync(bm->node_of, src->node_of, sizeof(int) * bm->T, cudaMemcpyDeviceToDevice, s) != cudaSuccess) ||
        (bm->n_nodes &&
         (cudaMemcpyAsync(bm->node_start, src->node_start, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
          cudaMemcpyAsync(bm->node_end, src->node_end, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
          cudaMemcpyAsync(bm->parent, src->parent, sizeof(int) * bm->n_nodes, cudaMemcpyDeviceToDevice, s) != cudaSuccess))) {
      rc = 3;
      break;
    }
    if ((rc = dalloc(&bm->pidx, n))) break;
    if ((rc = dalloc(&bm->pidxT, n))) break;
    int2* slot_tile = nullptr;
    if ((rc = dalloc(&slot_tile, n))) break;
    const bool masks = bm->BM == 128 && bm->BN == 128 && n > 0;
    if (masks && ((rc = dalloc(&bm->mask_rows, (size_t)n * 512)) || (rc = dalloc(&bm->mask_cols, (size_t)n * 512)))) {
      cudaFree(slot_tile);
      break;
    }
    long long cnt = std::max<long long>(n, std::max(nq, nk) + 1);
    k_dense_lists<<<(unsigned)((cnt + 255) / 256), 256, 0, s>>>(nq, nk, bm->q_ptr, bm->kv_idx, bm->kind, bm->k_ptr,
                                                                bm->q_idx, bm->kindT, bm->pidx, bm->pidxT, slot_tile);
    count_launch();
    if (masks) {
      k_masks<<<(unsigned)n, 128, 0, s>>>(bm->T, bm->tok, slot_tile, bm->mask_rows, bm->mask_cols);
      count_launch();
    }
    bm->n_partial = n;
    if (cudaStreamSynchronize(s) != cudaSuccess) {
      cudaFree(slot_tile);
      rc = 3;
      break;
    }
    cudaFree(slot_tile);
    // every row has the same length: natural order (last tiles first is no better)
    std::vector<int> oq(nq), ok(nk);
    std::iota(oq.begin(), oq.end(), 0);
    std::iota(ok.begin(), ok.end(), 0);
    if ((nq && cudaMemcpyAsync(bm->q_order, oq.data(), nq * sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) ||
        (nk && cudaMemcpyAsync(bm->k_order, ok.data(), nk * sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      rc = 3;
      break;
    }
    bm->nnz = n;
    bm->n_full = 0;
  } while (0);
  if (rc) {
    if (rc == 3) set_error("pt_blockmap_dense: CUDA failure");
    free_map(bm);
    return rc;
  }
  *out = bm;
  return 0;
}

}  // namespace pt
