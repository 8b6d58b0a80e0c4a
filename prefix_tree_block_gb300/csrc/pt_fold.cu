// pt_fold.cu -- the shared-prefix fold of rollouts and its inverse, on the GPU.
//
// "cp=1 shared-prefix prefix-tree attention for rollouts" (PR description):
// a group of one prompt and N sampled completions is stored once, as the flat
// sequence [prompt | c_0 | c_1 | ...], each completion's position ids
// continue from its prompt, and the tree goes on to the mask builder as
// (node_lengths, sample_paths).  The plan here is built from that same tree,
// so one description drives the fold, the block map and the unfold:
//
//   flat layout     node i owns tokens [off_i, off_i + len_i), ids in order;
//   rollout layout  sample s is one row of L tokens: its path's nodes, root
//                   first, then padding;
//   fold            flat token t <- the first sample holding it (dedupe);
//   unfold          every row gets its tokens back, padding zero;
//   unfold_grad     the adjoint of unfold: a flat token receives the sum of
//                   the gradients of its copies (fp32 accumulation, samples
//                   in index order, so the result is deterministic).
//
// Everything is HBM traffic: each kernel moves whole token rows with the
// widest aligned vector, a group of lanes per row sized to the row (one lane
// for a 4-byte id, a full warp for a hidden-state row), grid-stride over the
// rows with a warp-uniform trip count.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "pt.h"
#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {
int take_status_fold(cudaStream_t s) { return take_status_here(s); }
}  // namespace pt

struct pt_foldplan {
  int device;
  cudaStream_t stream;  // the build stream; memory goes back to the pool in its order
  void* mem;            // one pool allocation for every array below
  int32_t T, S, L, n_nodes;
  int4* node;          // [n_nodes] {off, len, position of the first token, first sample}
  int32_t* node_sp;    // [n_nodes + 1] CSR: samples whose path holds the node
  int32_t* node_samp;  // [path entries] sample ids, ascending per node
  int32_t* path_ptr;   // [S + 1]
  int32_t* path_nodes; // [path entries]
  int32_t* tok_node;   // [T] node of each flat token
  int32_t* tok_src;    // [T] rollout entry s*L + j the fold reads
  int32_t* tok_pos;    // [T] position id
  int32_t* roll_src;   // [S*L] flat token of each rollout entry, -1 on padding
  // token classes of the gradient: nodes with one sample through them (their
  // tokens are copied) and nodes shared by several (their tokens are summed);
  // {node, first token index within the class}, nodes in id order
  int32_t n1, nM;
  int64_t T1, TM, copiesM;
  int2* cls1;  // [n1]
  int2* clsM;  // [nM]
  // tasks of the bulk-copy gradient: {node, first token in the node, tokens, 0};
  // a task brings about eight rows: eight tokens of a one-sample node (one
  // contiguous copy), or one token of a shared node with all its copies
  int32_t n_tasks;
  int4* tasks;
};

namespace {

using namespace pt;  // device helpers (mbarriers, bulk copies, bounded waits)
using pt::set_error;

// ---------------------------------------------------------------------------
// plan kernels

__global__ void k_fold_tokens(const int4* __restrict__ node, int n_nodes, int T, int L, int32_t* __restrict__ tok_node,
                              int32_t* __restrict__ tok_src, int32_t* __restrict__ tok_pos) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    // first node whose end is past t (zero-length nodes end where they start)
    int lo = 0, hi = n_nodes - 1;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      int4 m = node[mid];
      if (m.x + m.y > t)
        hi = mid;
      else
        lo = mid + 1;
    }
    int4 n = node[lo];
    int pos = n.z + (t - n.x);
    tok_node[t] = lo;
    tok_pos[t] = pos;
    tok_src[t] = n.w * L + pos;
  }
}

__global__ void k_fold_rows(const int4* __restrict__ node, const int32_t* __restrict__ path_ptr,
                            const int32_t* __restrict__ path_nodes, int S, int L, int32_t* __restrict__ roll_src) {
  long long n_rows = (long long)S * L;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < n_rows;
       r += (long long)gridDim.x * blockDim.x) {
    int s = (int)(r / L), j = (int)(r % L);
    int src = -1, acc = 0;
    for (int k = path_ptr[s]; k < path_ptr[s + 1]; ++k) {
      int4 n = node[path_nodes[k]];
      if (j < acc + n.y) {
        src = n.x + (j - acc);
        break;
      }
      acc += n.y;
    }
    roll_src[r] = src;
  }
}

// ---------------------------------------------------------------------------
// row movers.  G lanes (a power of two <= 32) own one row; a warp holds 32/G
// rows per pass, and every warp runs the same number of passes.

struct RowGrid {
  long long rows;
  int g, lg;  // lanes per row and its log2
};

template <class Fn>
__device__ __forceinline__ void for_rows_in(const RowGrid& rg, int block, int n_blocks, Fn&& fn) {
  const int lane = threadIdx.x & 31;
  const long long warp = (block * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = ((long long)n_blocks * blockDim.x) >> 5;
  const int per_warp = 32 >> rg.lg;
  const int grp = lane >> rg.lg, li = lane & (rg.g - 1);
  for (long long base = warp * per_warp; base < rg.rows; base += n_warps * per_warp) {
    long long row = base + grp;
    fn(row, row < rg.rows, li);
  }
}

template <class Fn>
__device__ __forceinline__ void for_rows(const RowGrid& rg, Fn&& fn) {
  for_rows_in(rg, blockIdx.x, gridDim.x, fn);
}

// dst row <- src row (src == nullptr: zeros), nv vectors of type V per row.
template <class V>
__device__ __forceinline__ void move_row(const V* __restrict__ src, V* __restrict__ dst, int nv, int li, int g) {
  constexpr int kU = 4;  // loads in flight per lane before the stores
  for (int v0 = li; v0 < nv; v0 += kU * g) {
    V x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      int v = v0 + u * g;
      if (v < nv) {
        x[u] = src ? src[v] : V{};
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      int v = v0 + u * g;
      if (v < nv) dst[v] = x[u];
    }
  }
}

template <class V>
__global__ void k_fold(const char* __restrict__ roll, char* __restrict__ flat, const int32_t* __restrict__ tok_src,
                       RowGrid rg, long long row_bytes) {
  const int nv = (int)(row_bytes / (long long)sizeof(V));
  for_rows(rg, [&](long long t, bool ok, int li) {
    if (!ok) return;
    const V* src = reinterpret_cast<const V*>(roll + (long long)tok_src[t] * row_bytes);
    move_row<V>(src, reinterpret_cast<V*>(flat + t * row_bytes), nv, li, rg.g);
  });
}

template <class V>
__global__ void k_unfold(const char* __restrict__ flat, char* __restrict__ roll, const int32_t* __restrict__ roll_src,
                         RowGrid rg, long long row_bytes) {
  const int nv = (int)(row_bytes / (long long)sizeof(V));
  for_rows(rg, [&](long long r, bool ok, int li) {
    if (!ok) return;
    int t = roll_src[r];
    const V* src = t >= 0 ? reinterpret_cast<const V*>(flat + (long long)t * row_bytes) : nullptr;
    move_row<V>(src, reinterpret_cast<V*>(roll + r * row_bytes), nv, li, rg.g);
  });
}

__device__ __forceinline__ bool same(uint4 a, uint4 b) { return a.x == b.x && a.y == b.y && a.z == b.z && a.w == b.w; }
__device__ __forceinline__ bool same(uint2 a, uint2 b) { return a.x == b.x && a.y == b.y; }
template <class V>
__device__ __forceinline__ bool same(V a, V b) {
  return a == b;
}

// Counts rollout entries that differ from the entry the fold keeps for their
// token.  The counter is added to (the host zeroes it first).
template <class V>
__global__ void k_fold_mismatch(const char* __restrict__ roll, const int32_t* __restrict__ roll_src,
                                const int32_t* __restrict__ tok_src, RowGrid rg, long long row_bytes,
                                unsigned long long* __restrict__ count) {
  const int nv = (int)(row_bytes / (long long)sizeof(V));
  unsigned local = 0;
  for_rows(rg, [&](long long r, bool ok, int li) {
    bool diff = false;
    if (ok) {
      int t = roll_src[r];
      long long rep = t >= 0 ? tok_src[t] : r;
      if (rep != r) {
        const V* a = reinterpret_cast<const V*>(roll + r * row_bytes);
        const V* b = reinterpret_cast<const V*>(roll + rep * row_bytes);
        for (int v = li; v < nv; v += rg.g) diff |= !same(a[v], b[v]);
      }
    }
    // OR over the row's lanes; every lane of the warp takes part
    for (int m = 1; m < rg.g; m <<= 1) diff |= __shfl_xor_sync(0xffffffffu, (int)diff, m) != 0;
    if (diff && (threadIdx.x & (rg.g - 1)) == 0) ++local;
  });
  for (int m = 16; m; m >>= 1) local += __shfl_xor_sync(0xffffffffu, local, m);
  if ((threadIdx.x & 31) == 0 && local) atomicAdd(count, (unsigned long long)local);
}

// Elements of one 16-byte (or scalar) load, widened to fp32.
template <class E>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float f(float x) { return x; }
  static __device__ __forceinline__ float out(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 out(float x) { return __float2bfloat16_rn(x); }
};

// Entry of a token class holding class token i: the last entry whose first
// token is <= i.
__device__ __forceinline__ int2 class_entry(const int2* __restrict__ cls, int n, long long i) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cls[mid].y <= i)
      lo = mid;
    else
      hi = mid - 1;
  }
  return cls[lo];
}

// dflat <- the adjoint of unfold, width elements of E per token, K per vector.
// Blocks [0, blocks1) copy the tokens that have a single copy (a group of
// lanes per token row, like the fold); the other blocks sum the shared
// tokens, one thread per (token, vector), the loads of up to kC copies in
// flight together, added in sample order in fp32 from the first copy on and
// rounded once.  The split follows the two classes' bytes.
template <class E, int K>
__global__ void k_unfold_grad(const E* __restrict__ droll, E* __restrict__ dflat, const int4* __restrict__ node,
                              const int32_t* __restrict__ node_sp, const int32_t* __restrict__ node_samp,
                              const int2* __restrict__ cls1, int n1, const int2* __restrict__ clsM, int nM,
                              RowGrid rg1, long long TM, int blocks1, int width, int L) {
  struct alignas(sizeof(E) * K) Vec {
    E e[K];
  };
  constexpr int kC = 8;
  const int nv = width / K;
  const Vec* in = reinterpret_cast<const Vec*>(droll);
  Vec* out = reinterpret_cast<Vec*>(dflat);
  if ((int)blockIdx.x < blocks1) {
    for_rows_in(rg1, blockIdx.x, blocks1, [&](long long i, bool ok, int li) {
      if (!ok) return;
      const int2 ce = class_entry(cls1, n1, i);
      const int4 nd = node[ce.x];
      const long long k = i - ce.y;  // token k of the node
      const long long src = (long long)node_samp[node_sp[ce.x]] * L + nd.z + k;
      move_row<Vec>(in + src * nv, out + (nd.x + k) * nv, nv, li, rg1.g);
    });
    return;
  }
  const long long items = TM * nv;
  const long long stride = (long long)(gridDim.x - blocks1) * blockDim.x;
  for (long long it = (long long)(blockIdx.x - blocks1) * blockDim.x + threadIdx.x; it < items; it += stride) {
    const long long r = it / nv;
    const int v = (int)(it - r * nv);
    const int2 ce = class_entry(clsM, nM, r);
    const int4 nd = node[ce.x];
    const long long k = r - ce.y;
    const long long j = nd.z + k;
    const int c0 = node_sp[ce.x], nc = node_sp[ce.x + 1] - c0;
    float acc[K];
    for (int cb = 0; cb < nc; cb += kC) {
      Vec x[kC];
#pragma unroll
      for (int c = 0; c < kC; ++c)
        if (cb + c < nc) x[c] = in[((long long)node_samp[c0 + cb + c] * L + j) * nv + v];
#pragma unroll
      for (int c = 0; c < kC; ++c)
        if (cb + c < nc)
#pragma unroll
          for (int e = 0; e < K; ++e) {
            const float y = Elem<E>::f(x[c].e[e]);
            acc[e] = cb + c == 0 ? y : acc[e] + y;
          }
    }
    Vec o;
#pragma unroll
    for (int e = 0; e < K; ++e) o.e[e] = Elem<E>::out(acc[e]);
    out[(nd.x + k) * nv + v] = o;
  }
}

// The gradient through bulk copies (rows of at most 2 KB, 16-byte multiples),
// a warp per task.  A task is m tokens of one node, m = 8 / (copies per
// token) rounded down, at least 1: for each copy c of the node, tokens
// k0..k0+m-1 sit in one contiguous run of sample c's rollout row, so one lane
// brings them all in with one bulk copy per copy (one mbarrier), and the
// lanes add the copies in sample order in fp32 (from the first copy on) and
// write the m rows.  A token with more copies than a round holds (m = 1) takes
// several rounds with the sums in registers.  Whole-row bulk copies keep many
// bytes in flight per SM without holding them in registers.
constexpr int kBulkC = 8;         // rows per bulk round
constexpr int kBulkWarps = 4;     // warps per block
constexpr int kBulkMaxRow = 2048; // bytes

template <class E>
__global__ void __launch_bounds__(kBulkWarps * 32) k_unfold_grad_bulk(
    const char* __restrict__ droll, E* __restrict__ dflat, const int4* __restrict__ node,
    const int32_t* __restrict__ node_sp, const int32_t* __restrict__ node_samp, const int4* __restrict__ tasks,
    int n_tasks, int W, int L) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t bars[kBulkWarps];
  __shared__ volatile int abort_flag;
  constexpr int K = 16 / (int)sizeof(E);  // elements per 16-byte vector
  struct alignas(16) Vec {
    E e[K];
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* slot = sm + (size_t)warp * kBulkC * W;
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    mbar_init(&bars[warp], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int nv = W / 16;  // vectors per row, at most 128: four per lane
  const int width = W / (int)sizeof(E);
  uint32_t phase = 0;
  for (int ti = blockIdx.x * kBulkWarps + warp; ti < n_tasks; ti += gridDim.x * kBulkWarps) {
    const int4 tk = tasks[ti];
    const int4 nd = node[tk.x];
    const int m = tk.z;
    const long long j0 = nd.z + tk.y, t0 = nd.x + tk.y;
    const int c0 = node_sp[tk.x], nc = node_sp[tk.x + 1] - c0;
    const int per_round = m > 1 ? nc : kBulkC;  // m > 1: every copy fits in one round
    float acc[4][K];
    for (int cb = 0; cb < nc; cb += per_round) {
      const int n = min(per_round, nc - cb);
      if (lane == 0) {
        mbar_expect_tx(&bars[warp], (uint32_t)(n * m * W));
        for (int c = 0; c < n; ++c)
          bulk_load(slot + (size_t)c * m * W, droll + ((long long)node_samp[c0 + cb + c] * L + j0) * W,
                    (uint32_t)(m * W), &bars[warp]);
      }
      const bool ok = mbar_wait(&bars[warp], phase, &abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {  // copies may still be in flight: let them land, then leave
        mbar_wait_drain(&bars[warp], phase, 20000000LL);
        return;
      }
      phase ^= 1;
      if (m > 1) {  // all copies are here: finish each of the m rows now
        for (int u = 0; u < m; ++u)
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int v = lane + 32 * a;
            if (v >= nv) continue;
            float sum[K];
            for (int c = 0; c < n; ++c) {
              const Vec x = *reinterpret_cast<const Vec*>(slot + ((size_t)c * m + u) * W + v * 16);
#pragma unroll
              for (int e = 0; e < K; ++e) {
                const float y = Elem<E>::f(x.e[e]);
                sum[e] = c == 0 ? y : sum[e] + y;
              }
            }
            Vec o;
#pragma unroll
            for (int e = 0; e < K; ++e) o.e[e] = Elem<E>::out(sum[e]);
            *reinterpret_cast<Vec*>(dflat + (t0 + u) * width + v * K) = o;
          }
      } else {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int v = lane + 32 * a;
          if (v < nv)
            for (int c = 0; c < n; ++c) {
              const Vec x = *reinterpret_cast<const Vec*>(slot + (size_t)c * W + v * 16);
#pragma unroll
              for (int e = 0; e < K; ++e) {
                const float y = Elem<E>::f(x.e[e]);
                acc[a][e] = (cb + c == 0) ? y : acc[a][e] + y;
              }
            }
        }
      }
      __syncwarp();  // every lane has read the slot before it is refilled
    }
    if (m == 1) {
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int v = lane + 32 * a;
        if (v < nv) {
          Vec o;
#pragma unroll
          for (int e = 0; e < K; ++e) o.e[e] = Elem<E>::out(acc[a][e]);
          *reinterpret_cast<Vec*>(dflat + t0 * width + v * K) = o;
        }
      }
    }
  }
}

__global__ void k_fold_positions(const int32_t* __restrict__ tok_pos, int T, int64_t* __restrict__ pos) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) pos[t] = tok_pos[t];
}

// ---------------------------------------------------------------------------
// host helpers

int lanes_for(long long nv) {  // lanes per row: enough for the row, at most a warp
  int g = 1;
  while (g < 32 && g < nv) g <<= 1;
  return g;
}

RowGrid row_grid(long long rows, long long nv) {
  RowGrid rg;
  rg.rows = rows;
  rg.g = lanes_for(nv);
  rg.lg = 0;
  while ((1 << rg.lg) < rg.g) ++rg.lg;
  return rg;
}

// Blocks of 256 threads for whole passes: every warp takes the same number of
// rows, so no pass runs with part of the GPU idle.
template <class F>
int grid_for(const RowGrid& rg, int dev, F kernel) {
  static std::mutex mu;  // resident blocks per SM of each kernel, asked once
  static std::map<const void*, int> occ;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = occ.find(reinterpret_cast<const void*>(kernel));
    if (it != occ.end()) {
      per_sm = it->second;
    } else {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
      occ[reinterpret_cast<const void*>(kernel)] = per_sm;
    }
  }
  const long long per_warp = 32 / rg.g;
  const long long warps = (rg.rows + per_warp - 1) / per_warp;
  const long long cap = (long long)pt::num_sms(dev) * per_sm * 8;
  const long long passes = std::max(1LL, (warps + cap - 1) / cap);
  const long long w = (warps + passes - 1) / passes;
  return (int)std::max(1LL, (w + 7) / 8);
}

// widest unit in {16, 8, 4, 2, 1} that divides the row and both base addresses
int unit_for(long long row_bytes, const void* a, const void* b) {
  for (int u = 16; u > 1; u >>= 1)
    if (row_bytes % u == 0 && reinterpret_cast<uintptr_t>(a) % u == 0 && reinterpret_cast<uintptr_t>(b) % u == 0)
      return u;
  return 1;
}

int check_plan(const pt_foldplan* p, const char* who) {
  if (!p) {
    set_error("%s: plan is NULL", who);
    return PT_ERR_INVALID_ARG;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) {
    set_error("%s: the plan lives on device %d, the current device is %d", who, p->device, dev);
    return PT_ERR_INVALID_ARG;
  }
  return PT_OK;
}

int launch_status(const char* who) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: launch failed: %s", who, cudaGetErrorString(e));
    return PT_ERR_CUDA;
  }
  return PT_OK;
}

// KERNEL<V> for the vector type of a unit of 16, 8, 4, 2 or 1 bytes
#define PT_BY_UNIT(KERNEL, unit, rg, dev, s, ...)                                                  \
  switch (unit) {                                                                                 \
    case 16: KERNEL<uint4><<<grid_for(rg, dev, KERNEL<uint4>), 256, 0, s>>>(__VA_ARGS__); break;       \
    case 8: KERNEL<uint2><<<grid_for(rg, dev, KERNEL<uint2>), 256, 0, s>>>(__VA_ARGS__); break;        \
    case 4: KERNEL<uint32_t><<<grid_for(rg, dev, KERNEL<uint32_t>), 256, 0, s>>>(__VA_ARGS__); break;  \
    case 2: KERNEL<uint16_t><<<grid_for(rg, dev, KERNEL<uint16_t>), 256, 0, s>>>(__VA_ARGS__); break;  \
    default: KERNEL<uint8_t><<<grid_for(rg, dev, KERNEL<uint8_t>), 256, 0, s>>>(__VA_ARGS__); break;   \
  }

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" pt_status pt_fold_plan(const int32_t* node_lengths, int32_t n_nodes, const int32_t* path_ptr,
                                  const int32_t* path_nodes, int32_t n_samples, int32_t row_len, cudaStream_t stream,
                                  pt_foldplan** out) {
  static const char* who = "pt_fold_plan";
  if (!out) {
    set_error("%s: out is NULL", who);
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (n_nodes < 0 || n_samples < 0 || (n_nodes > 0 && !node_lengths) || !path_ptr || (n_samples > 0 && !path_nodes)) {
    set_error("%s: null array or negative count", who);
    return PT_ERR_INVALID_ARG;
  }
  if (row_len < 0 || (long long)n_samples * row_len > INT_MAX) {
    set_error("%s: %d rows of %d tokens is out of range", who, n_samples, row_len);
    return PT_ERR_INVALID_ARG;
  }
  const int N = n_nodes, S = n_samples, L = row_len;
  // node offsets
  std::vector<int> off(N + 1, 0);
  for (int i = 0; i < N; ++i) {
    if (node_lengths[i] < 0) {
      set_error("%s: node %d has negative length %d", who, i, node_lengths[i]);
      return PT_ERR_INVALID_ARG;
    }
    if ((long long)off[i] + node_lengths[i] > INT_MAX / 2) {
      set_error("%s: too many tokens", who);
      return PT_ERR_INVALID_ARG;
    }
    off[i + 1] = off[i] + node_lengths[i];
  }
  const int T = off[N];
  // parents from consecutive path entries; position of each node's first token
  if (path_ptr[0] != 0) {
    set_error("%s: path_ptr[0] must be 0", who);
    return PT_ERR_INVALID_ARG;
  }
  std::vector<int> parent(N, -2), first_sample(N, -1), depth_pos(N, 0), n_through(N, 0);
  for (int s = 0; s < S; ++s) {
    int b = path_ptr[s], e = path_ptr[s + 1];
    if (e <= b) {
      set_error("%s: sample path %d is empty", who, s);
      return PT_ERR_INVALID_ARG;
    }
    long long row = 0;
    for (int k = b; k < e; ++k) {
      int n = path_nodes[k];
      if (n < 0 || n >= N) {
        set_error("%s: path %d names node %d, out of range", who, s, n);
        return PT_ERR_INVALID_ARG;
      }
      int want = k == b ? -1 : path_nodes[k - 1];
      if (want >= n) {
        set_error("%s: node %d follows %d on path %d (a parent must have a smaller id)", who, n, want, s);
        return PT_ERR_INVALID_ARG;
      }
      if (parent[n] == -2) {
        parent[n] = want;
        first_sample[n] = s;
        depth_pos[n] = (int)row;
      } else if (parent[n] != want) {
        set_error("%s: node %d has parents %d and %d", who, n, parent[n], want);
        return PT_ERR_INVALID_ARG;
      }
      ++n_through[n];
      row += node_lengths[n];
    }
    if (row > L) {
      set_error("%s: sample %d has %lld tokens, more than the row length %d", who, s, row, L);
      return PT_ERR_INVALID_ARG;
    }
  }
  for (int i = 0; i < N; ++i)
    if (parent[i] == -2) {
      set_error("%s: node %d is on no sample path", who, i);
      return PT_ERR_INVALID_ARG;
    }
  const int E = S ? path_ptr[S] : 0;
  // host tables: node int4 | node_sp | node_samp | path_ptr | path_nodes
  std::vector<int4> nodes(std::max(N, 1));
  for (int i = 0; i < N; ++i) nodes[i] = make_int4(off[i], node_lengths[i], depth_pos[i], first_sample[i]);
  std::vector<int32_t> sp(N + 1, 0), samp(std::max(E, 1));
  for (int i = 0; i < N; ++i) sp[i + 1] = sp[i] + n_through[i];
  {
    std::vector<int32_t> fill(sp.begin(), sp.end() - 1);
    for (int s = 0; s < S; ++s)  // ascending samples per node
      for (int k = path_ptr[s]; k < path_ptr[s + 1]; ++k) samp[fill[path_nodes[k]]++] = s;
  }
  // tasks of the bulk-copy gradient (nodes with tokens only)
  std::vector<int4> tasks;
  for (int i = 0; i < N; ++i) {
    if (node_lengths[i] == 0) continue;
    const int m = std::max(1, kBulkC / std::max(n_through[i], 1));
    for (int k0 = 0; k0 < node_lengths[i]; k0 += m) tasks.push_back(make_int4(i, k0, std::min(m, node_lengths[i] - k0), 0));
  }
  // token classes of the gradient (nodes with tokens only)
  std::vector<int2> cls1, clsM;
  long long T1 = 0, TM = 0, copiesM = 0;
  for (int i = 0; i < N; ++i) {
    if (node_lengths[i] == 0) continue;
    if (n_through[i] == 1) {
      cls1.push_back(make_int2(i, (int)T1));
      T1 += node_lengths[i];
    } else {
      clsM.push_back(make_int2(i, (int)TM));
      TM += node_lengths[i];
      copiesM += (long long)node_lengths[i] * n_through[i];
    }
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    set_error("%s: no CUDA device", who);
    return PT_ERR_CUDA;
  }
  auto pad = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_node = pad(sizeof(int4) * nodes.size()), b_sp = pad(4 * sp.size()), b_samp = pad(4 * samp.size()),
               b_pp = pad(4 * (size_t)(S + 1)), b_pn = pad(4 * (size_t)std::max(E, 1)), b_tok = pad(4 * (size_t)std::max(T, 1)),
               b_roll = pad(4 * std::max((size_t)S * L, (size_t)1));
  const size_t b_c1 = pad(sizeof(int2) * std::max<size_t>(cls1.size(), 1)),
               b_cM = pad(sizeof(int2) * std::max<size_t>(clsM.size(), 1)),
               b_tk = pad(sizeof(int4) * std::max<size_t>(tasks.size(), 1));
  const size_t tables = b_node + b_sp + b_samp + b_pp + b_pn + b_c1 + b_cM + b_tk;
  const size_t total = tables + 3 * b_tok + b_roll;
  pt_foldplan* p = new pt_foldplan();
  p->device = dev;
  p->stream = stream;
  p->T = T;
  p->S = S;
  p->L = L;
  p->n_nodes = N;
  p->n1 = (int)cls1.size();
  p->nM = (int)clsM.size();
  p->T1 = T1;
  p->TM = TM;
  p->copiesM = copiesM;
  p->n_tasks = (int32_t)tasks.size();
  int rc = pt::pool_alloc(&p->mem, total, dev, stream);
  if (rc) {
    delete p;
    return (pt_status)rc;
  }
  char* base = static_cast<char*>(p->mem);
  size_t o = 0;
  p->node = reinterpret_cast<int4*>(base + o), o += b_node;
  p->node_sp = reinterpret_cast<int32_t*>(base + o), o += b_sp;
  p->node_samp = reinterpret_cast<int32_t*>(base + o), o += b_samp;
  p->path_ptr = reinterpret_cast<int32_t*>(base + o), o += b_pp;
  p->path_nodes = reinterpret_cast<int32_t*>(base + o), o += b_pn;
  p->cls1 = reinterpret_cast<int2*>(base + o), o += b_c1;
  p->clsM = reinterpret_cast<int2*>(base + o), o += b_cM;
  p->tasks = reinterpret_cast<int4*>(base + o), o += b_tk;
  p->tok_node = reinterpret_cast<int32_t*>(base + o), o += b_tok;
  p->tok_src = reinterpret_cast<int32_t*>(base + o), o += b_tok;
  p->tok_pos = reinterpret_cast<int32_t*>(base + o), o += b_tok;
  p->roll_src = reinterpret_cast<int32_t*>(base + o);
  // one packed upload of the tables (their device layout, padding included)
  std::vector<char> host(tables, 0);
  size_t h = 0;
  std::memcpy(host.data() + h, nodes.data(), sizeof(int4) * N), h += b_node;
  std::memcpy(host.data() + h, sp.data(), 4 * sp.size()), h += b_sp;
  std::memcpy(host.data() + h, samp.data(), 4 * (size_t)E), h += b_samp;
  std::memcpy(host.data() + h, path_ptr, 4 * (size_t)(S + 1)), h += b_pp;
  if (E) std::memcpy(host.data() + h, path_nodes, 4 * (size_t)E);
  h += b_pn;
  if (!cls1.empty()) std::memcpy(host.data() + h, cls1.data(), sizeof(int2) * cls1.size());
  h += b_c1;
  if (!clsM.empty()) std::memcpy(host.data() + h, clsM.data(), sizeof(int2) * clsM.size());
  h += b_cM;
  if (!tasks.empty()) std::memcpy(host.data() + h, tasks.data(), sizeof(int4) * tasks.size());
  rc = pt::upload(p->mem, host.data(), tables, dev, stream);
  if (rc) {
    set_error("%s: upload of the plan tables failed", who);
    pt::pool_free(p->mem, stream);
    delete p;
    return PT_ERR_CUDA;
  }
  {
    pt::ProfScope ps(stream, "fold_plan");
    const int cap = pt::num_sms(dev) * 8;
    if (T > 0) {
      k_fold_tokens<<<std::max(1, std::min((T + 255) / 256, cap)), 256, 0, stream>>>(p->node, N, T, L, p->tok_node,
                                                                                      p->tok_src, p->tok_pos);
      pt::count_launch();
    }
    long long rows = (long long)S * L;
    if (rows > 0) {
      k_fold_rows<<<(int)std::max(1LL, std::min((rows + 255) / 256, (long long)cap)), 256, 0, stream>>>(
          p->node, p->path_ptr, p->path_nodes, S, L, p->roll_src);
      pt::count_launch();
    }
  }
  rc = launch_status(who);
  if (rc) {
    pt::pool_free(p->mem, stream);
    delete p;
    return (pt_status)rc;
  }
  *out = p;
  return PT_OK;
}

extern "C" pt_status pt_foldplan_info(const pt_foldplan* p, int32_t* T, int32_t* n_samples, int32_t* row_len) {
  if (!p) {
    set_error("pt_foldplan_info: plan is NULL");
    return PT_ERR_INVALID_ARG;
  }
  if (T) *T = p->T;
  if (n_samples) *n_samples = p->S;
  if (row_len) *row_len = p->L;
  return PT_OK;
}

extern "C" void pt_foldplan_free(pt_foldplan* p) {
  if (!p) return;
  pt::pool_free(p->mem, p->stream);
  delete p;
}

extern "C" pt_status pt_fold(const pt_foldplan* p, const void* roll, int64_t row_bytes, void* flat,
                             cudaStream_t stream) {
  static const char* who = "pt_fold";
  int rc = check_plan(p, who);
  if (rc) return (pt_status)rc;
  if (row_bytes <= 0 || row_bytes > INT_MAX) {
    set_error("%s: row_bytes %lld out of range", who, (long long)row_bytes);
    return PT_ERR_INVALID_ARG;
  }
  if (p->T == 0) return PT_OK;
  if (!roll || !flat) {
    set_error("%s: null buffer", who);
    return PT_ERR_INVALID_ARG;
  }
  const int unit = unit_for(row_bytes, roll, flat);
  RowGrid rg = row_grid(p->T, row_bytes / unit);
  {
    pt::ProfScope ps(stream, "fold");
    PT_BY_UNIT(k_fold, unit, rg, p->device, stream, static_cast<const char*>(roll), static_cast<char*>(flat),
               p->tok_src, rg, (long long)row_bytes);
    pt::count_launch();
  }
  return (pt_status)launch_status(who);
}

extern "C" pt_status pt_unfold(const pt_foldplan* p, const void* flat, int64_t row_bytes, void* roll,
                               cudaStream_t stream) {
  static const char* who = "pt_unfold";
  int rc = check_plan(p, who);
  if (rc) return (pt_status)rc;
  if (row_bytes <= 0 || row_bytes > INT_MAX) {
    set_error("%s: row_bytes %lld out of range", who, (long long)row_bytes);
    return PT_ERR_INVALID_ARG;
  }
  const long long rows = (long long)p->S * p->L;
  if (rows == 0) return PT_OK;
  if (!roll || (!flat && p->T > 0)) {
    set_error("%s: null buffer", who);
    return PT_ERR_INVALID_ARG;
  }
  const int unit = unit_for(row_bytes, flat ? flat : roll, roll);
  RowGrid rg = row_grid(rows, row_bytes / unit);
  {
    pt::ProfScope ps(stream, "unfold");
    PT_BY_UNIT(k_unfold, unit, rg, p->device, stream, static_cast<const char*>(flat),
               static_cast<char*>(roll), p->roll_src, rg, (long long)row_bytes);
    pt::count_launch();
  }
  return (pt_status)launch_status(who);
}

extern "C" pt_status pt_unfold_grad(const pt_foldplan* p, const void* droll, pt_dtype dtype, int64_t width,
                                    void* dflat, cudaStream_t stream) {
  static const char* who = "pt_unfold_grad";
  int rc = check_plan(p, who);
  if (rc) return (pt_status)rc;
  if (dtype != PT_BF16 && dtype != PT_F32) {
    set_error("%s: unknown dtype %d", who, (int)dtype);
    return PT_ERR_INVALID_ARG;
  }
  const int es = dtype == PT_BF16 ? 2 : 4;
  if (width <= 0 || width * es > INT_MAX) {
    set_error("%s: width %lld out of range", who, (long long)width);
    return PT_ERR_INVALID_ARG;
  }
  if (p->T == 0) return PT_OK;
  if (!droll || !dflat) {
    set_error("%s: null buffer", who);
    return PT_ERR_INVALID_ARG;
  }
  const bool vec = unit_for(width * es, droll, dflat) == 16;
  const int K = vec ? 16 / es : 1;
  const long long nv = width / K;
  RowGrid rg1 = row_grid(p->T1, nv);
  // shared tokens by bulk copies when their rows allow it; the rest as below
  const long long W = width * es;
  const bool bulk = vec && W <= kBulkMaxRow && p->n_tasks > 0;
  // one wave of blocks, split between the copied and the summed tokens by bytes
  auto split = [&](auto kernel, int& blocks, int& blocks1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    blocks = pt::num_sms(p->device) * per_sm;
    const double b1 = 2.0 * p->T1, bM = (double)p->copiesM + p->TM;
    blocks1 = (int)(blocks * b1 / std::max(1.0, b1 + bM) + 0.5);
    if (p->T1 > 0) blocks1 = std::max(blocks1, 1);
    if (p->TM > 0) blocks1 = std::min(blocks1, blocks - 1);
    if (p->TM == 0) blocks1 = blocks;
  };
  {
    pt::ProfScope ps(stream, "unfold_grad");
#define PT_GRAD(E, KK, A, B)                                                                                   \
  do {                                                                                                         \
    if (bulk) {                                                                                                \
      const size_t smem = (size_t)kBulkWarps * kBulkC * W;                                                     \
      int per_sm = 0;                                                                                          \
      if (cudaFuncSetAttribute(k_unfold_grad_bulk<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != \
              cudaSuccess ||                                                                                   \
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_unfold_grad_bulk<E>, kBulkWarps * 32, smem) !=  \
              cudaSuccess || per_sm < 1)                                                                       \
        per_sm = 1;                                                                                            \
      const long long need = ((long long)p->n_tasks + kBulkWarps - 1) / kBulkWarps;                              \
      const int gb = (int)std::max(1LL, std::min<long long>(need, (long long)pt::num_sms(p->device) * per_sm)); \
      k_unfold_grad_bulk<E><<<gb, kBulkWarps * 32, smem, stream>>>(static_cast<const char*>(A),               \
                                                                   static_cast<E*>(B), p->node, p->node_sp,    \
                                                                   p->node_samp, p->tasks, p->n_tasks, (int)W, \
                                                                   p->L);                                      \
    } else {                                                                                                   \
      int blocks, blocks1;                                                                                     \
      split(k_unfold_grad<E, KK>, blocks, blocks1);                                                            \
      k_unfold_grad<E, KK><<<blocks, 256, 0, stream>>>(static_cast<const E*>(A), static_cast<E*>(B), p->node,    \
                                                       p->node_sp, p->node_samp, p->cls1, p->n1, p->clsM, p->nM, \
                                                       rg1, p->TM, blocks1, (int)width, p->L);                   \
    }                                                                                                          \
  } while (0)
    if (dtype == PT_BF16) {
      if (vec)
        PT_GRAD(__nv_bfloat16, 8, droll, dflat);
      else
        PT_GRAD(__nv_bfloat16, 1, droll, dflat);
    } else {
      if (vec)
        PT_GRAD(float, 4, droll, dflat);
      else
        PT_GRAD(float, 1, droll, dflat);
    }
#undef PT_GRAD
    pt::count_launch();
  }
  return (pt_status)launch_status(who);
}

extern "C" pt_status pt_fold_positions(const pt_foldplan* p, int64_t* pos, cudaStream_t stream) {
  static const char* who = "pt_fold_positions";
  int rc = check_plan(p, who);
  if (rc) return (pt_status)rc;
  if (p->T == 0) return PT_OK;
  if (!pos) {
    set_error("%s: null buffer", who);
    return PT_ERR_INVALID_ARG;
  }
  {
    pt::ProfScope ps(stream, "fold_positions");
    const int cap = pt::num_sms(p->device) * 8;
    k_fold_positions<<<std::max(1, std::min((p->T + 255) / 256, cap)), 256, 0, stream>>>(p->tok_pos, p->T, pos);
    pt::count_launch();
  }
  return (pt_status)launch_status(who);
}

extern "C" pt_status pt_fold_mismatches(const pt_foldplan* p, const void* roll, int64_t row_bytes,
                                        unsigned long long* count, cudaStream_t stream) {
  static const char* who = "pt_fold_mismatches";
  int rc = check_plan(p, who);
  if (rc) return (pt_status)rc;
  if (row_bytes <= 0 || row_bytes > INT_MAX) {
    set_error("%s: row_bytes %lld out of range", who, (long long)row_bytes);
    return PT_ERR_INVALID_ARG;
  }
  if (!count) {
    set_error("%s: count is NULL", who);
    return PT_ERR_INVALID_ARG;
  }
  if (cudaMemsetAsync(count, 0, sizeof(unsigned long long), stream) != cudaSuccess) {
    set_error("%s: clearing the counter failed", who);
    return PT_ERR_CUDA;
  }
  const long long rows = (long long)p->S * p->L;
  if (rows == 0) return PT_OK;
  if (!roll) {
    set_error("%s: null buffer", who);
    return PT_ERR_INVALID_ARG;
  }
  const int unit = unit_for(row_bytes, roll, roll);
  RowGrid rg = row_grid(rows, row_bytes / unit);
  {
    pt::ProfScope ps(stream, "fold_mismatches");
    PT_BY_UNIT(k_fold_mismatch, unit, rg, p->device, stream, static_cast<const char*>(roll), p->roll_src,
               p->tok_src, rg, (long long)row_bytes, count);
    pt::count_launch();
  }
  return (pt_status)launch_status(who);
}
