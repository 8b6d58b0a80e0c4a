// pt_bwd_tc.cu -- tensor-core backward for bf16: dQ, dK, dV over the kept pairs.
//
// The backward of the block-sparse attention of "prefix_grouper_kernel.py"
// (the compiled FlexAttention backward it pads for) and of the drafter
// speed-up PR's GQA backward: with P = exp(s - LSE), Delta = rowsum(dO * O),
// dS = P * (dO V^T - Delta):  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,
// dK and dV summed over the q heads that share a kv head (native GQA: K and
// V are never repeated).  Empty tiles are skipped; partial tiles use the
// block map's 128 x 128 keep bitmasks.
//
// At head_dim 64, when the caller's workspace holds an fp32 dQ accumulator,
// one kv-major kernel (k_bwd_fused, section 2b) computes dQ, dK and dV in
// one pass, dQ added into the accumulator by TMA reduce-adds (not run-to-run
// bitwise identical), then one finalize launch converts it.  Otherwise,
// three launches on the caller's stream:
//  1. k_bwd_prep  (HBM-bound) -Delta = -rowsum(dO * O) and -LSE * log2(e)
//                 into the workspace, [Hq, Tpad] each, Tpad = ceil(T/128)*128
//                 (negated so that the kernels form s scale_log2 - LSE log2(e)
//                 and dP - Delta with packed f32x2 fma and add); padding rows
//                 get values that make them contribute nothing.
//  2. k_bwd_dkdv  persistent, kv-major: a work item is (kv block, kv head).
//                 K and V stay in shared memory while the q tiles of the
//                 block's column list stream through for every q head of the
//                 group.  Each (q head, q tile) step is split into two halves
//                 of 64 q rows, one per compute warpgroup: S^T = K Q_half^T and
//                 dP^T = V dO_half^T land in that warpgroup's TMEM columns
//                 (kv rows in lanes); it writes P^T and dS^T back over them
//                 as bf16, and dV += P^T dO_half, dK += dS^T Q_half read them
//                 straight from TMEM.  While one warpgroup computes, the
//                 tensor pipe runs the other warpgroup's MMAs.
//  3. k_bwd_dq    persistent, q-major: a work item is (q tile, q head).  Q and
//                 dO stay resident while the kv blocks of the tile's list
//                 stream through; each block is split into two halves of 64
//                 kv columns, one per warpgroup: S = Q K_half^T, dP = dO
//                 V_half^T, dS back into TMEM, then dQ += dS K_half.
// In the three-launch form every output element is written once (no
// atomics), so results are deterministic.  TMEM per CTA: 2 x (64 + 64)
// columns of S/dP plus the accumulators (dV, dK: 2D; dQ: D) -- at most 512.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <cmath>
#include <mutex>
#include <queue>
#include <type_traits>
#include <vector>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_bwd(cudaStream_t s) { return take_status_here(s); }

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
// A block takes 8 tokens x all heads: D/8 threads per (token, head) read
// dO and O in their stored (token-major) order with 16-byte loads; the
// per-row sums go through shared memory so that Delta and LSE2, head-major
// [Hq][Tpad], are written (and LSE read) a 32-byte sector at a time.
constexpr int kPrepTokens = 8;
template <int D>
__global__ void __launch_bounds__(256) k_bwd_prep(const __nv_bfloat16* __restrict__ dO,
                                                  const __nv_bfloat16* __restrict__ O, const float* __restrict__ LSE,
                                                  int T, int Tpad, int Hq, float* __restrict__ ndelta,
                                                  float* __restrict__ nlse2, float4* __restrict__ dq_acc) {
  pdl_wait();  // launched with programmatic dependent launch
  constexpr int VPT = D > 256 ? 2 : 1;  // 16-byte vectors of dO and O per thread (a row stays within a warp)
  constexpr int TPR = D / (8 * VPT);    // threads per (token, head) row
  extern __shared__ float sh_delta[];  // [kPrepTokens][Hq + 1]
  const int q0 = blockIdx.x * kPrepTokens;
  const int sub = threadIdx.x % TPR;
  // rows is a multiple of 32 / TPR, the rows of one warp: a warp's lanes
  // run the same trips, as the shuffles below need
  const int rows = kPrepTokens * Hq;
#pragma unroll 4
  for (int r = threadIdx.x / TPR; r < rows; r += 256 / TPR) {
    const int ql = r / Hq, h = r % Hq, q = q0 + ql;
    float s = 0.f;
    if (q < T) {
#pragma unroll
      for (int vv = 0; vv < VPT; ++vv) {
        const int col = (vv * TPR + sub) * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(dO + ((size_t)q * Hq + h) * D + col);
        const uint4 b = *reinterpret_cast<const uint4*>(O + ((size_t)q * Hq + h) * D + col);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float2 x = __bfloat1622float2(pa[k]), y = __bfloat1622float2(pb[k]);
          s = fmaf(x.x, y.x, s);
          s = fmaf(x.y, y.y, s);
        }
      }
    }
#pragma unroll
    for (int o = TPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, TPR);
    if (sub == 0) sh_delta[ql * (Hq + 1) + h] = s;
  }
  if (dq_acc) {  // the one-pass backward's fp32 dQ accumulator: these tokens' rows start at zero
    float4* z = dq_acc + (size_t)q0 * Hq * (D / 4);
    for (int i = threadIdx.x; i < rows * (D / 4); i += 256) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < rows; i += 256) {
    const int h = i / kPrepTokens, ql = i % kPrepTokens, q = q0 + ql;
    const size_t row = (size_t)h * Tpad + q;  // q < Tpad: Tpad is a multiple of 128
    // both stored negated: the kernels form s scale_log2 - LSE log2(e) and
    // dP - Delta as one packed fma or add per column pair
    ndelta[row] = -sh_delta[ql * (Hq + 1) + h];
    const float l = q < T ? LSE[(size_t)h * T + q] : -INFINITY;
    // rows that keep nothing (padding) get -inf so exp2(s scale_log2 + nlse2) = 0
    nlse2[row] = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
  }
}

// ---------------------------------------------------------------------------
// shared pieces
// ---------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  static constexpr int NP = D / 64;
  static constexpr int PANEL = 128 * 128;  // 128 rows x 128 B
  static constexpr int HALF = 64 * 128;    // rows 64..127 of a panel start here
  static constexpr int TILE = NP * PANEL;
  static constexpr int STAGES = D == 64 ? 4 : 2;
  // TMEM columns: S (or S^T) at 0 and dP (or dP^T) at 128, 128 columns each;
  // warpgroup w reads columns [64w, 64w + 64) of both and writes its packed
  // bf16 results to the first 32 of them.  Accumulators from 256.
  static constexpr int TM_S = 0, TM_DP = 128, TM_ACC0 = 256, TM_ACC1 = 256 + D;
  // With room in TMEM the packed P (or P^T) and dS (or dS^T) go to their own
  // 64-column regions, so the next step's S/dP can be computed while this
  // step's math runs: dQ (one accumulator) always has room; dK/dV only at D = 64.
  // Without that room (dK/dV at D = 128) the kv-major kernel runs each step
  // as S^T, dK of the previous step, dP^T, dV: P^T is computed while the
  // tensor core works through the two middle products.
  static constexpr bool DQ_OVL = true, DKDV_OVL = (D == 64);
  // At head_dim 64 the products come in short chains (S and dP: 4 MMAs, the
  // accumulating products: 8), and the tensor pipe leaves its latency (about
  // 300 cycles) between one thread's chains into different accumulators.
  // There a second MMA warp issues the accumulating products (dV and dK, or
  // dQ) while the first issues S and dP (or S^T and dP^T): the pipe
  // overlaps the two threads' chains.
  static constexpr bool TWO_ISSUERS = (D == 64);
  static constexpr int THREADS = TWO_ISSUERS ? 352 : 320;
  static constexpr int TM_DQ_DS = 256 + D;                    // dq: packed dS
  static constexpr int TM_KV_P = 256 + 2 * D, TM_KV_DS = 320 + 2 * D;  // dkdv: packed P^T, dS^T
};

struct BwdParams {
  const int* ptr;         // k_ptr (dkdv) or q_ptr (dq)
  const int* idx;         // q_idx or kv_idx
  const int* pidx;        // mask slot per entry (-1: full)
  const int* order;       // k_order or q_order
  const uint32_t* masks;  // mask_cols (dkdv) or mask_rows (dq)
  const float* ndelta;    // [Hq, Tpad]: -Delta
  const float* nlse2;     // [Hq, Tpad]: -LSE log2(e) (-inf for rows that keep nothing)
  __nv_bfloat16* out0;    // dK (dkdv) or dQ (dq)
  __nv_bfloat16* out1;    // dV (dkdv)
  const DkdvItem* items;  // dkdv work items, grouped by CTA
  const int* cta_ptr;     // dkdv: CTA b runs items [cta_ptr[b], cta_ptr[b + 1])
  const int4* dq_items;   // pipelined dq: q tile, head, first list entry, kv blocks; grouped by CTA
  const int4* dq_cta;     // pipelined dq: first item, end item, kv blocks of each CTA
  float* partial;         // dkdv: fp32 partial sums of split columns, [slot][128][2D]
  float* dq_acc;          // one-pass kernel: fp32 dQ accumulator, [Tpad][Hq][D]
  int T, Tpad, Hq, Hkv, n_major, n_items;
  float scale, scale_log2;
  int half;  // head_dim 512 passes: which 256-column half of the output
};

// Sum the chunk partials of every split kv-major column, in chunk order, and
// write dV (first D columns of a slot row) and dK (last D) as bf16.
// One 256-thread block's share of that: rows [8 yb, 8 yb + 8) of split
// column sp (kv block, kv head, first slot, slot count); one float4 of the
// 2D columns per thread and row pass.
template <int D>
__device__ __forceinline__ void dkdv_split_rows(const int4 sp, int yb, const float* __restrict__ partial, int T,
                                                int Hkv, __nv_bfloat16* __restrict__ dK,
                                                __nv_bfloat16* __restrict__ dV) {
  constexpr int Q4 = 2 * D / 4;  // float4 per row
  for (int idx = threadIdx.x; idx < 8 * Q4; idx += blockDim.x) {
    const int r = yb * 8 + idx / Q4, c = (idx % Q4) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < sp.w; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(partial + ((size_t)(sp.z + k) * 128 + r) * (2 * D) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int kv = sp.x * 128 + r;
    if (kv >= T) continue;
    __nv_bfloat16* dst = (c < D ? dV : dK) + ((size_t)kv * Hkv + sp.y) * D + (c < D ? c : c - D);
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = pk;
  }
}

template <int D>
__global__ void k_dkdv_finalize(const int4* __restrict__ splits, const float* __restrict__ partial, int T, int Hkv,
                                __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV) {
  pdl_wait();  // launched with programmatic dependent launch
  // block (x, y): split column x, rows [8y, 8y + 8) of its 128
  dkdv_split_rows<D>(splits[blockIdx.x], blockIdx.y, partial, T, Hkv, dK, dV);
}

// Sum the chunk partials of every split kv-major column for one output of
// the head_dim-256 and -512 passes: slot rows of row_floats floats whose
// first W hold this pass's columns; the sums go to columns [col0, col0 + W)
// of the output rows (row stride H * D), as bf16.
template <int W>
__global__ void k_split_finalize(const int4* __restrict__ splits, const float* __restrict__ partial, int row_floats,
                                 int T, int H, int D, int col0, __nv_bfloat16* __restrict__ out) {
  pdl_wait();  // launched with programmatic dependent launch
  const int4 sp = splits[blockIdx.x];  // kv block, kv head, first slot, slot count
  constexpr int Q4 = W / 4;
  for (int idx = threadIdx.x; idx < 8 * Q4; idx += blockDim.x) {
    const int r = blockIdx.y * 8 + idx / Q4, c = (idx % Q4) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < sp.w; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(partial + ((size_t)(sp.z + k) * 128 + r) * row_floats + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int kv = sp.x * 128 + r;
    if (kv >= T) continue;
    __nv_bfloat16* dst = out + ((size_t)kv * H + sp.y) * D + col0 + c;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = pk;
  }
}

// 64 fp32 values (as bits) -> 32 bf16x2 words.
// P = exp2(s scale_log2 - LSE log2(e)) of two columns (s0, s1: raw scores;
// sc2: scale_log2 in both halves; nl2: the two columns' -LSE log2(e))
__device__ __forceinline__ void p_pair(uint32_t s0, uint32_t s1, unsigned long long sc2, unsigned long long nl2,
                                       int c, float& p0, float& p1) {
  float x0, x1;
  f2_unpack(f2_fma(f2_pack(__uint_as_float(s0), __uint_as_float(s1)), sc2, nl2), x0, x1);
  p0 = ex2_mix(x0, c);
  p1 = ex2_mix(x1, c + 1);
}
// dS = P (dP - Delta) of two columns (nd2: the two columns' -Delta)
__device__ __forceinline__ void ds_pair(float p0, float p1, uint32_t d0, uint32_t d1, unsigned long long nd2,
                                        float& ds0, float& ds1) {
  f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(d0), __uint_as_float(d1)), nd2)), ds0, ds1);
}

__device__ __forceinline__ void pack64(const uint32_t* v, uint32_t* out) {
#pragma unroll
  for (int c = 0; c < 32; ++c) out[c] = pack_bf16(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
}

// Store 32 accumulator columns of one row as bf16, times `mul`.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t* v, float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
}

// Barrier block shared by both kernels.
template <int S>
struct BwdBars {
  uint64_t res_full, res_empty;
  uint64_t st_full[S], st_empty[S];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_free, mma_done;
  uint64_t mma_done2;  // the second MMA warp's MMAs are complete (head_dim-64 kernels)
  uint64_t s_free;   // compute warpgroups have loaded S/dP: the MMA may overwrite them
  uint64_t o_written;  // (dq) every compute thread has put its output rows into the staging tile
  uint64_t o_stored;   // (dq) the staging tile's TMA store has read it
  uint64_t ps_free;  // the accumulate MMAs have read the packed P/dS region
  uint64_t dq_full;    // (one-pass kernel) a step's dQ product is in TMEM
  uint64_t dq_free;    // (one-pass kernel) the dQ warpgroup has loaded it
  uint64_t dq_staged;  // (one-pass kernel) the dQ warpgroup has staged it
  uint64_t dq_sfree;   // (one-pass kernel) the reduce-adds have read the staging tile
  uint64_t ps_free2;   // (one-pass kernel) dV/dK and dQ have both read packed P^T and dS^T
  uint64_t mma_done3;  // (one-pass kernel) the dQ MMA warp's MMAs are complete
};

template <int S>
__device__ __forceinline__ void init_bars(BwdBars<S>* b) {
  mbar_init(&b->res_full, 1);
  mbar_init(&b->res_empty, 1);
  for (int s = 0; s < S; ++s) {
    mbar_init(&b->st_full[s], 1);
    mbar_init(&b->st_empty[s], 1);
  }
  for (int w = 0; w < 2; ++w) {
    mbar_init(&b->s_full[w], 1);
    mbar_init(&b->p_full[w], 256);  // both compute warpgroups arrive
  }
  mbar_init(&b->acc_full, 1);
  mbar_init(&b->acc_free, 256);
  mbar_init(&b->mma_done, 1);
  mbar_init(&b->mma_done2, 1);
  mbar_init(&b->s_free, 256);
  mbar_init(&b->o_written, 256);
  mbar_init(&b->o_stored, 1);
  mbar_init(&b->ps_free, 1);
  mbar_init(&b->dq_full, 1);
  mbar_init(&b->dq_free, 128);  // the dQ epilogue warpgroup
  mbar_init(&b->dq_staged, 128);
  mbar_init(&b->dq_sfree, 1);
  mbar_init(&b->ps_free2, 2);  // one commit from each accumulating MMA warp
  mbar_init(&b->mma_done3, 1);
}

// ---------------------------------------------------------------------------
// 2. dK / dV, kv-major
// ---------------------------------------------------------------------------
template <int D>
struct DkdvL {
  using C = BwdCfg<D>;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = C::TILE;
  static constexpr int OFF_ST = 2 * C::TILE;  // stages: Q | dO | lse2 | delta | column masks
  static constexpr int ST_Q = 0, ST_DO = C::TILE, ST_L = 2 * C::TILE, ST_D = ST_L + 512, ST_M = ST_D + 512;
  static constexpr int ST_BYTES = ST_M + 2048;
  static constexpr int OFF_META = OFF_ST + C::STAGES * ST_BYTES;
  static constexpr int OFF_BAR = OFF_META + 64;
  static constexpr int OFF_MISC = OFF_BAR + (int)sizeof(BwdBars<C::STAGES>);
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(C::TM_ACC1 + D <= 512, "TMEM budget");
  static_assert(!C::DKDV_OVL || C::TM_KV_DS + 64 <= 512, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    k_bwd_dkdv(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
               const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = BwdCfg<D>;
  using L = DkdvL<D>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars<S>* B = reinterpret_cast<BwdBars<S>*>(smem + L::OFF_BAR);
  int* meta = reinterpret_cast<int*>(smem + L::OFF_META);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int w_begin = p.cta_ptr[blockIdx.x], w_end = p.cta_ptr[blockIdx.x + 1];

  if (threadIdx.x == 256) {
    init_bars<S>(B);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t sc = 0, it = 0;
      bool ok = true, res_issued = false;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int jb = itm.jb, hk = itm.hk;
        const int e0 = p.ptr[jb], ncol = p.ptr[jb + 1] - e0;
        if (itm.x1 == itm.x0) continue;
        if (it > 0 && !(ok = mbar_wait(&B->res_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(&B->res_full, 2 * C::TILE);
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn) {
          tma_load_3d(smem + L::OFF_K + pn * C::PANEL, &mK, &B->res_full, pn * 64, hk, jb * 128);
          tma_load_3d(smem + L::OFF_V + pn * C::PANEL, &mV, &B->res_full, pn * 64, hk, jb * 128);
        }
        res_issued = true;
        const int n = itm.x1 - itm.x0;
        for (int x = 0; x < n; ++x) {
          const int e = e0 + (itm.x0 + x) % ncol;
          const int h = hk * g + (itm.x0 + x) / ncol, i = p.idx[e], slot = p.pidx[e];
          const uint32_t s = sc % S, u = sc / S;
          if (u > 0 && !(ok = mbar_wait(&B->st_empty[s], (u - 1) & 1, abort_flag))) break;
          uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
          meta[s] = slot;
          mbar_expect_tx(&B->st_full[s], 2 * C::TILE + 1024 + (slot >= 0 ? 2048 : 0));
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn) {
            tma_load_3d(st + L::ST_Q + pn * C::PANEL, &mQ, &B->st_full[s], pn * 64, h, i * 128);
            tma_load_3d(st + L::ST_DO + pn * C::PANEL, &mdO, &B->st_full[s], pn * 64, h, i * 128);
          }
          bulk_load(st + L::ST_L, p.nlse2 + (size_t)h * p.Tpad + i * 128, 512, &B->st_full[s]);
          bulk_load(st + L::ST_D, p.ndelta + (size_t)h * p.Tpad + i * 128, 512, &B->st_full[s]);
          if (slot >= 0) bulk_load(st + L::ST_M, p.masks + (size_t)slot * 512, 2048, &B->st_full[s]);
          ++sc;
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (res_issued) mbar_wait_drain(&B->res_full, it & 1, lim);
        for (uint32_t s = 0; s < S && s < sc; ++s) {
          uint32_t last = sc - 1 - ((sc - 1 - s) % S);
          mbar_wait_drain(&B->st_full[s], (last / S) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint32_t sK = smem_u32(smem + L::OFF_K), sV = smem_u32(smem + L::OFF_V);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int n = itm.x1 - itm.x0;
        if (n == 0) continue;
        
        if (!(ok = mbar_wait(&B->res_full, it & 1, abort_flag))) break;
        tc_fence_after();
        const auto mma_s = [&](uint32_t st) {  // S^T = K Q^T (M = 128 kv, N = 128 q)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_S, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(st + L::ST_Q + off, 16, 1024),
                   IDESC_S, kk > 0);
          }
        };
        const auto mma_dp = [&](uint32_t st) {  // dP^T = V dO^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_DP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(st + L::ST_DO + off, 16, 1024),
                   IDESC_S, kk > 0);
          }
        };
        // dV += P^T dO or dK += dS^T Q (K = 128 q rows), A read from TMEM
        const auto mma_acc = [&](uint32_t acc_col, uint32_t a_col, bool packed_region, uint32_t b_tile, bool first) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acol = packed_region ? kk * 8 : kk * 8 + (kk >= 4 ? 32 : 0);  // in place: halves at 0, 64
            mma_ts(tbase + acc_col, tbase + a_col + acol, sdesc_sw128(b_tile + kk * 2048, C::PANEL, 1024), IDESC_ACC,
                   !first || kk > 0);
          }
        };
        if constexpr (C::DKDV_OVL) {
          // S^T(x) and dP^T(x) once the stage is in and the compute
          // warpgroups have loaded S^T(x-1) and dP^T(x-1); dV and dK are the
          // second MMA warp's
          for (int x = 0; x < n && ok; ++x) {
            const uint32_t y = sc + x, s = y % S;
            uint64_t* bars[2] = {&B->st_full[s], y >= 1 ? &B->s_free : nullptr};
            const uint32_t par[2] = {(y / S) & 1, (y - 1) & 1};
            if (!(ok = mbar_wait_all<2>(bars, par, abort_flag))) break;
            tc_fence_after();
            const uint32_t st = sST + s * L::ST_BYTES;
            mma_s(st);
            mma_dp(st);
            mma_commit(&B->s_full[0]);
            if (x == n - 1) mma_commit(&B->res_empty);
          }
        } else {
          for (int x = 0; x <= n && ok; ++x) {
            const uint32_t y = sc + x, s = y % S;
            const uint32_t st = sST + s * L::ST_BYTES;
            if (x < n) {
              if (!(ok = mbar_wait(&B->st_full[s], (y / S) & 1, abort_flag))) break;
              tc_fence_after();
              mma_s(st);  // P^T(x-1), read by dV(x-1) before, is no longer needed
              mma_commit(&B->s_full[0]);
            }
            if (x >= 1) {
              // dK(x-1) from dS^T packed in place over dP^T(x-1)
              const uint32_t sp = (y - 1) % S;
              if (!(ok = mbar_wait(&B->p_full[1], (y - 1) & 1, abort_flag))) break;
              tc_fence_after();
              mma_acc(C::TM_ACC1, C::TM_DP, false, sST + sp * L::ST_BYTES + L::ST_Q, x == 1);
              mma_commit(&B->st_empty[sp]);
            }
            if (x < n) {
              mma_dp(st);  // after dK(x-1) has read dS^T(x-1)
              mma_commit(&B->s_full[1]);
              if (x == n - 1) mma_commit(&B->res_empty);
              // dV(x) from P^T packed in place over S^T(x)
              if (!(ok = mbar_wait(&B->p_full[0], y & 1, abort_flag))) break;
              if (x == 0 && it > 0 && !(ok = mbar_wait(&B->acc_free, (it - 1) & 1, abort_flag))) break;
              tc_fence_after();
              mma_acc(C::TM_ACC0, C::TM_S, false, st + L::ST_DO, x == 0);
            }
          }
        }
        if (ok && !C::DKDV_OVL) mma_commit(&B->acc_full);  // (OVL: the second MMA warp's)
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done);
      mbar_wait_drain(&B->mma_done, 0, 200000000);
    }
    __syncwarp();
  } else if (C::TWO_ISSUERS && warp == 10) {
    // ------------------------------------------------------------ dV / dK issuer (head_dim 64)
    if (lane == 0) {
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int n = itm.x1 - itm.x0;
        if (n == 0) continue;
        for (int x = 0; x < n && ok; ++x) {
          // dV += P^T dO and dK += dS^T Q of step x, from the packed region,
          // once the compute warpgroups have written it (and, on an item's
          // first step, read the previous item's accumulators)
          const uint32_t y = sc + x, sp = y % S;
          uint64_t* bars[3] = {&B->st_full[sp], &B->p_full[0], (x == 0 && it > 0) ? &B->acc_free : nullptr};
          const uint32_t par[3] = {(y / S) & 1, y & 1, (it - 1) & 1};
          if (!(ok = mbar_wait_all<3>(bars, par, abort_flag))) break;
          tc_fence_after();
          const uint32_t stp = sST + sp * L::ST_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tbase + C::TM_ACC0, tbase + C::TM_KV_P + kk * 8, sdesc_sw128(stp + L::ST_DO + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, x > 0 || kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tbase + C::TM_ACC1, tbase + C::TM_KV_DS + kk * 8, sdesc_sw128(stp + L::ST_Q + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, x > 0 || kk > 0);
          mma_commit(&B->ps_free);
          mma_commit(&B->st_empty[sp]);
        }
        if (ok) mma_commit(&B->acc_full);
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done2);
      mbar_wait_drain(&B->mma_done2, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (kv row per thread)
    const int hw = warp >> 2;  // which 64 q columns of each step this warpgroup takes
    const int r = threadIdx.x & 127;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = tl + C::TM_S + 64 * hw, tP = tl + C::TM_DP + 64 * hw;
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (int w = w_begin; w < w_end && ok; ++w) {
      const DkdvItem itm = p.items[w];
      const int jb = itm.jb, hk = itm.hk;
      const int n = itm.x1 - itm.x0;
      const int kv = jb * 128 + r;
      __nv_bfloat16* orow = (hw ? p.out0 : p.out1) + ((size_t)kv * p.Hkv + hk) * D;  // wg0: dV, wg1: dK
      if (n == 0) {
        if (kv < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        }
        continue;
      }
      
      for (int x = 0; x < n; ++x) {
        const uint32_t y = sc + x, s = y % S;
        ok = mbar_wait(&B->s_full[0], y & 1, abort_flag) && mbar_wait(&B->st_full[s], (y / S) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
        const float4* l2 = reinterpret_cast<const float4*>(st + L::ST_L) + hw * 16;
        const float4* dl = reinterpret_cast<const float4*>(st + L::ST_D) + hw * 16;
        const int slot = meta[s];
        uint2 mk = make_uint2(0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = reinterpret_cast<const uint2*>(st + L::ST_M)[2 * r + hw];
        uint32_t sr[64], pk[32];
        if constexpr (C::DKDV_OVL) {
          uint32_t dr[64];
          tmem_ld32(tS, sr);
          tmem_ld32(tS + 32, sr + 32);
          tmem_ld32(tP, dr);
          tmem_ld32(tP + 32, dr + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&B->s_free);  // S^T and dP^T are in registers: the MMA may reuse them
          uint32_t pk2[32];
          // scalar here: packed pairs made this kernel spill
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 lv = l2[c4], dv = dl[c4];  // -LSE log2(e) and -Delta of the 4 columns
            const float nla[4] = {lv.x, lv.y, lv.z, lv.w}, nda[4] = {dv.x, dv.y, dv.z, dv.w};
            float pv[4], dsv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = c4 * 4 + k;
              const uint32_t word = c < 32 ? mk.x : mk.y;
              const float pr = ex2_mix(fmaf(__uint_as_float(sr[c]), p.scale_log2, nla[k]), c);
              pv[k] = ((word >> (c & 31)) & 1u) ? pr : 0.f;
              dsv[k] = pv[k] * (__uint_as_float(dr[c]) + nda[k]);
            }
            pk[2 * c4] = pack_bf16(pv[0], pv[1]);
            pk[2 * c4 + 1] = pack_bf16(pv[2], pv[3]);
            pk2[2 * c4] = pack_bf16(dsv[0], dsv[1]);
            pk2[2 * c4 + 1] = pack_bf16(dsv[2], dsv[3]);
          }
          // the previous step's accumulate MMAs must be done reading the region
          if (y > 0) {
            ok = mbar_wait(&B->ps_free, (y - 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st32(tl + C::TM_KV_P + 32 * hw, pk);
          tmem_st32(tl + C::TM_KV_DS + 32 * hw, pk2);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&B->p_full[0]);
        } else {
          // P^T first: the MMA runs dK of the previous step and dP^T meanwhile
          tmem_ld32(tS, sr);
          tmem_ld32(tS + 32, sr + 32);
          tmem_ld_wait();
          const unsigned long long sc2 = f2_splat(p.scale_log2);
          const auto pmath = [&](auto masked) {
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
              const float4 nl = l2[c4];  // -LSE log2(e) of the 4 columns
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int c = c4 * 4 + 2 * k2;
                float p0, p1;
                p_pair(sr[c], sr[c + 1], sc2, k2 ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y), c, p0, p1);
                if constexpr (decltype(masked)::value) {
                  const uint32_t word = c < 32 ? mk.x : mk.y;
                  p0 = ((word >> (c & 31)) & 1u) ? p0 : 0.f;
                  p1 = ((word >> ((c + 1) & 31)) & 1u) ? p1 : 0.f;
                }
                sr[c] = __float_as_uint(p0);
                sr[c + 1] = __float_as_uint(p1);
              }
            }
          };
          if (slot >= 0)
            pmath(std::true_type{});
          else
            pmath(std::false_type{});
          pack64(sr, pk);
          tmem_st32(tS, pk);  // in place over this warpgroup's S^T columns
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&B->p_full[0]);
          // then dS^T = P^T (dP^T - Delta)
          ok = mbar_wait(&B->s_full[1], y & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          {
            uint32_t dr[64];
            tmem_ld32(tP, dr);
            tmem_ld32(tP + 32, dr + 32);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
              const float4 nd = dl[c4];  // -Delta of the 4 columns
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int c = c4 * 4 + 2 * k2;
                float d0, d1;
                ds_pair(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), dr[c], dr[c + 1],
                        k2 ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y), d0, d1);
                sr[c] = __float_as_uint(d0);
                sr[c + 1] = __float_as_uint(d1);
              }
            }
          }
          pack64(sr, pk);
          tmem_st32(tP, pk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&B->p_full[1]);
        }
      }
      if (!ok) break;
      ok = mbar_wait(&B->acc_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float mul = hw ? p.scale : 1.f;
      const uint32_t acc = hw ? C::TM_ACC1 : C::TM_ACC0;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + acc + c * 32, v);
        tmem_ld_wait();
        if (itm.slot < 0) {
          if constexpr (D == 128)  // eight rows of 64 contiguous bytes per store instruction
            store_rows32(orow + c * 32, (size_t)p.Hkv * D, kv, p.T, v, mul);
          else if (kv < p.T)  // few items per CTA at head_dim 64: the direct stores are kept
            store_row32(orow + c * 32, v, mul);
        } else {  // one chunk of a split column: fp32 partial sums, summed later in chunk order
          float4* prow = reinterpret_cast<float4*>(p.partial + ((size_t)itm.slot * 128 + r) * (2 * D) + (hw ? D : 0) +
                                                   c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            prow[k] = make_float4(__uint_as_float(v[4 * k]) * mul, __uint_as_float(v[4 * k + 1]) * mul,
                                  __uint_as_float(v[4 * k + 2]) * mul, __uint_as_float(v[4 * k + 3]) * mul);
        }
      }
      tc_fence_before();
      mbar_arrive(&B->acc_free);
      sc += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// 2b. dQ, dK and dV in one kv-major pass (head_dim 64)
// ---------------------------------------------------------------------------
// The kv-major kernel above with the q-major products folded in.  Each
// step's dS^T also goes to shared memory, 128-byte swizzled, one 64-column
// panel per compute warpgroup (kv rows x 64 q columns).  That one tile is
// the K-major A operand of dK += dS^T Q and, read transposed, the MN-major A
// operand of dQ_step = dS K, with K the resident tile.  dQ_step (128 q rows
// x 64 fp32) lands in the TMEM columns that the packed dS^T needs no longer.
// Three MMA warps issue S^T/dP^T, dV/dK and dQ: the tensor pipe overlaps one
// thread's chain into an accumulator with another's, where one thread
// switching between accumulators would leave it idle.  A fourth warpgroup
// loads dQ_step (a q row per thread) into a staging tile (two swizzled
// 128 x 32 fp32 panels), and one of its threads adds the tile into an fp32
// accumulator [Tpad][Hq][64] in the workspace with two tiled TMA reduce-adds
// (a few large operations: the TMA unit takes bulk operations one at a time,
// and one 128-byte operation per thread and step kept it busier than the
// whole step).  The compute warpgroups, whose exponentials and packing bound
// the step, thus do no dQ work.  Registers are moved to them from the other
// two warpgroups (setmaxnreg).  The preprocess kernel zeroes the accumulator
// and k_fused_finalize scales it and writes dQ as bf16.
// Per kept pair the products fall from 14 D flop (S^T, dP^T, dV, dK here;
// S, dP and dQ again in the q-major kernel) to 10 D, and the q-major
// kernel's second exponential pass over every tile goes away.  The price is
// dQ summed in fp32 in an order that varies from run to run.
struct FusedL {
  using C = BwdCfg<64>;
  static constexpr int STAGES = 3;
  static constexpr int OFF_K = 0, OFF_V = C::TILE;
  static constexpr int OFF_ST = 2 * C::TILE;  // stages: Q | dO | lse2 | delta | column masks
  static constexpr int ST_Q = 0, ST_DO = C::TILE, ST_L = 2 * C::TILE, ST_D = ST_L + 512, ST_M = ST_D + 512;
  static constexpr int ST_BYTES = ST_M + 2048;
  // warpgroups: two compute; producer and three MMA warps; dQ epilogue
  static constexpr int THREADS = 512;
  // registers per thread after reallocation; they add up to the launch's
  // 128 per thread (the kernel must be built with exactly 128)
  static constexpr int REG_COMPUTE = 176, REG_CTRL = 72, REG_DQ = 88, REG_LAUNCH = 128;
  static_assert(2 * REG_COMPUTE + REG_CTRL + REG_DQ == 4 * REG_LAUNCH, "register split");
  static constexpr int OFF_DS = OFF_ST + STAGES * ST_BYTES;  // dS^T, two swizzled 64-column panels
  static_assert(OFF_DS % 1024 == 0, "swizzled panel alignment");
  // dQ staging: panel w = fp32 columns [32w, 32w + 32) of the 128 q rows,
  // 128 bytes a row, 128-byte swizzled (the reduce-add's box layout)
  static constexpr int OFF_DQ = OFF_DS + 2 * C::PANEL;
  static constexpr int OFF_META = OFF_DQ + 2 * C::PANEL;
  static constexpr int OFF_BAR = OFF_META + 64;
  static constexpr int OFF_MISC = OFF_BAR + (int)sizeof(BwdBars<STAGES>);
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
  // TMEM columns: S^T, dP^T (128 each), dV, dK, packed P^T, dQ_step (64 each)
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320, TM_P = 384, TM_DQ = 448;
  static_assert(TM_DQ + 64 <= 512, "TMEM budget");
};

__global__ void __launch_bounds__(FusedL::THREADS, 1)
    k_bwd_fused(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const __grid_constant__ CUtensorMap mAcc, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  constexpr int D = 64;
  using C = BwdCfg<D>;
  using L = FusedL;
  constexpr int S = L::STAGES;
  static_assert(C::TWO_ISSUERS, "warp roles");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars<S>* B = reinterpret_cast<BwdBars<S>*>(smem + L::OFF_BAR);
  int* meta = reinterpret_cast<int*>(smem + L::OFF_META);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int w_begin = p.cta_ptr[blockIdx.x], w_end = p.cta_ptr[blockIdx.x + 1];

  if (threadIdx.x == 256) {
    init_bars<S>(B);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
    prefetch_tmap(&mAcc);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp >= 8 && warp < 12) {
  regs_dec<L::REG_CTRL>();  // the whole warpgroup, before its warps take their roles
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t sc = 0, it = 0;
      bool ok = true, res_issued = false;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int jb = itm.jb, hk = itm.hk;
        const int e0 = p.ptr[jb], ncol = p.ptr[jb + 1] - e0;
        if (itm.x1 == itm.x0) continue;
        if (it > 0 && !(ok = mbar_wait(&B->res_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(&B->res_full, 2 * C::TILE);
        tma_load_3d(smem + L::OFF_K, &mK, &B->res_full, 0, hk, jb * 128);
        tma_load_3d(smem + L::OFF_V, &mV, &B->res_full, 0, hk, jb * 128);
        res_issued = true;
        const int n = itm.x1 - itm.x0;
        for (int x = 0; x < n; ++x) {
          const int e = e0 + (itm.x0 + x) % ncol;
          const int h = hk * g + (itm.x0 + x) / ncol, i = p.idx[e], slot = p.pidx[e];
          const uint32_t s = sc % S, u = sc / S;
          if (u > 0 && !(ok = mbar_wait(&B->st_empty[s], (u - 1) & 1, abort_flag))) break;
          uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
          meta[s] = slot;
          mbar_expect_tx(&B->st_full[s], 2 * C::TILE + 1024 + (slot >= 0 ? 2048 : 0));
          tma_load_3d(st + L::ST_Q, &mQ, &B->st_full[s], 0, h, i * 128);
          tma_load_3d(st + L::ST_DO, &mdO, &B->st_full[s], 0, h, i * 128);
          bulk_load(st + L::ST_L, p.nlse2 + (size_t)h * p.Tpad + i * 128, 512, &B->st_full[s]);
          bulk_load(st + L::ST_D, p.ndelta + (size_t)h * p.Tpad + i * 128, 512, &B->st_full[s]);
          if (slot >= 0) bulk_load(st + L::ST_M, p.masks + (size_t)slot * 512, 2048, &B->st_full[s]);
          ++sc;
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (res_issued) mbar_wait_drain(&B->res_full, it & 1, lim);
        for (uint32_t s = 0; s < S && s < sc; ++s) {
          uint32_t last = sc - 1 - ((sc - 1 - s) % S);
          mbar_wait_drain(&B->st_full[s], (last / S) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ S^T / dP^T issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      const uint32_t sK = smem_u32(smem + L::OFF_K), sV = smem_u32(smem + L::OFF_V);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int n = itm.x1 - itm.x0;
        if (n == 0) continue;
        if (!(ok = mbar_wait(&B->res_full, it & 1, abort_flag))) break;
        tc_fence_after();
        // S^T(x) = K Q^T and dP^T(x) = V dO^T once the stage is in and the
        // compute warpgroups have loaded S^T(x-1) and dP^T(x-1)
        for (int x = 0; x < n && ok; ++x) {
          const uint32_t y = sc + x, s = y % S;
          uint64_t* bars[2] = {&B->st_full[s], y >= 1 ? &B->s_free : nullptr};
          const uint32_t par[2] = {(y / S) & 1, (y - 1) & 1};
          if (!(ok = mbar_wait_all<2>(bars, par, abort_flag))) break;
          tc_fence_after();
          const uint32_t st = sST + s * L::ST_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tbase + L::TM_S, sdesc_sw128(sK + kk * 32, 16, 1024), sdesc_sw128(st + L::ST_Q + kk * 32, 16, 1024),
                   IDESC_S, kk > 0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tbase + L::TM_DP, sdesc_sw128(sV + kk * 32, 16, 1024), sdesc_sw128(st + L::ST_DO + kk * 32, 16, 1024),
                   IDESC_S, kk > 0);
          mma_commit(&B->s_full[0]);
        }
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done);
      mbar_wait_drain(&B->mma_done, 0, 200000000);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ dV / dK issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);  // A K-major (or TMEM), B MN-major
      const uint32_t sDS = smem_u32(smem + L::OFF_DS);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int n = itm.x1 - itm.x0;
        if (n == 0) continue;
        for (int x = 0; x < n && ok; ++x) {
          // step x once the compute warpgroups have written packed P^T and
          // dS^T (and, on an item's first step, read the previous item's
          // accumulators)
          const uint32_t y = sc + x, sp = y % S;
          uint64_t* bars[3] = {&B->st_full[sp], &B->p_full[0], (x == 0 && it > 0) ? &B->acc_free : nullptr};
          const uint32_t par[3] = {(y / S) & 1, y & 1, (it - 1) & 1};
          if (!(ok = mbar_wait_all<3>(bars, par, abort_flag))) break;
          tc_fence_after();
          const uint32_t stp = sST + sp * L::ST_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO (A from TMEM; K = 128 q rows)
            mma_ts(tbase + L::TM_DV, tbase + L::TM_P + kk * 8, sdesc_sw128(stp + L::ST_DO + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, x > 0 || kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q (A: the q-column panels of dS^T)
            mma_ss(tbase + L::TM_DK, sdesc_sw128(sDS + (kk >> 2) * C::PANEL + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(stp + L::ST_Q + kk * 2048, C::PANEL, 1024), IDESC_ACC, x > 0 || kk > 0);
          if (x == n - 1) mma_commit(&B->acc_full);
          mma_commit(&B->ps_free2);
          mma_commit(&B->st_empty[sp]);
        }
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done2);
      mbar_wait_drain(&B->mma_done2, 0, 200000000);
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------ dQ issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_DQ = idesc_bf16(128, D, true, true);  // A = dS read transposed (MN-major)
      const uint32_t sK = smem_u32(smem + L::OFF_K), sDS = smem_u32(smem + L::OFF_DS);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; ++w) {
        const DkdvItem itm = p.items[w];
        const int n = itm.x1 - itm.x0;
        if (n == 0) continue;
        if (!(ok = mbar_wait(&B->res_full, it & 1, abort_flag))) break;
        for (int x = 0; x < n && ok; ++x) {
          // dQ_step = dS K (M = 128 q rows, K = 128 kv rows) once dS^T is in
          // shared memory and the dQ warpgroup has loaded the previous step's
          const uint32_t y = sc + x;
          uint64_t* bars[2] = {&B->p_full[0], y > 0 ? &B->dq_free : nullptr};
          const uint32_t par[2] = {y & 1, (y - 1) & 1};
          if (!(ok = mbar_wait_all<2>(bars, par, abort_flag))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tbase + L::TM_DQ, sdesc_sw128(sDS + kk * 2048, C::PANEL, 1024), sdesc_sw128(sK + kk * 2048, C::PANEL, 1024),
                   IDESC_DQ, kk > 0);
          mma_commit(&B->dq_full);
          mma_commit(&B->ps_free2);
          // dQ reads the resident K: the item's tiles are free after its last dQ
          // (S^T and dP^T of that step were complete before its P^T existed)
          if (x == n - 1) mma_commit(&B->res_empty);
        }
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done3);
      mbar_wait_drain(&B->mma_done3, 0, 200000000);
    }
    __syncwarp();
  }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ epilogue (q row per thread)
    regs_dec<L::REG_DQ>();
    const int r = threadIdx.x & 127, r7 = r & 7;
    const bool leader = r == 0;  // issues the reduce-adds
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    uint4* row0 = reinterpret_cast<uint4*>(smem + L::OFF_DQ + r * 128);
    uint4* row1 = reinterpret_cast<uint4*>(smem + L::OFF_DQ + C::PANEL + r * 128);
    uint32_t y = 0;
    bool ok = true;
    for (int w = w_begin; w < w_end && ok; ++w) {
      const DkdvItem itm = p.items[w];
      const int e0 = p.ptr[itm.jb], ncol = p.ptr[itm.jb + 1] - e0;
      for (int x = itm.x0; x < itm.x1; ++x, ++y) {
        // step y's dQ: load it and release the TMEM columns; stage it once the
        // previous tile's reduce-adds have read the staging tile; then add the
        // tile into the accumulator rows of its q tile and head
        ok = mbar_wait(&B->dq_full, y & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[32], u[32];
        tmem_ld32(tl + L::TM_DQ, v);
        tmem_ld32(tl + L::TM_DQ + 32, u);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&B->dq_free);
        if (leader && y > 0) {
          bulk_wait_read0();
          mbar_arrive(&B->dq_sfree);
        }
        ok = y == 0 || mbar_wait(&B->dq_sfree, (y - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 16-byte chunk k of a 128-byte row goes to chunk k ^ (row & 7)
          row0[k ^ r7] = make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
          row1[k ^ r7] = make_uint4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
        }
        fence_proxy_async_smem();  // visible to the TMA
        mbar_arrive(&B->dq_staged);
        if (leader) {
          const int i = p.idx[e0 + x % ncol], h = itm.hk * g + x / ncol;
          ok = mbar_wait(&B->dq_staged, y & 1, abort_flag);
          if (ok) {
            tma_reduce_add_3d(&mAcc, smem + L::OFF_DQ, 0, h, i * 128);
            tma_reduce_add_3d(&mAcc, smem + L::OFF_DQ + C::PANEL, 32, h, i * 128);
            bulk_commit();
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {  // the leader's warp leaves together
          ok = false;
          break;
        }
      }
    }
    if (leader) bulk_wait0();
    if (!ok) *abort_flag = 1;
  } else {
    // ------------------------------------------------------------ compute (kv row per thread)
    regs_inc<L::REG_COMPUTE>();
    const int hw = warp >> 2;  // which 64 q columns of each step this warpgroup takes
    const int r = threadIdx.x & 127;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = tl + L::TM_S + 64 * hw, tP = tl + L::TM_DP + 64 * hw;
    uint4* ds_row = reinterpret_cast<uint4*>(smem + L::OFF_DS + hw * C::PANEL + r * 128);
    const int r7 = r & 7;
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (int w = w_begin; w < w_end && ok; ++w) {
      const DkdvItem itm = p.items[w];
      const int jb = itm.jb, hk = itm.hk;
      const int n = itm.x1 - itm.x0;
      const int kv = jb * 128 + r;
      __nv_bfloat16* orow = (hw ? p.out0 : p.out1) + ((size_t)kv * p.Hkv + hk) * D;  // wg0: dV, wg1: dK
      if (n == 0) {
        if (kv < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        }
        continue;
      }
      for (int x = 0; x < n; ++x) {
        const uint32_t y = sc + x, s = y % S;
        ok = mbar_wait(&B->s_full[0], y & 1, abort_flag) && mbar_wait(&B->st_full[s], (y / S) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
        const float4* l2 = reinterpret_cast<const float4*>(st + L::ST_L) + hw * 16;
        const float4* dl = reinterpret_cast<const float4*>(st + L::ST_D) + hw * 16;
        const int slot = meta[s];
        uint2 mk = make_uint2(0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = reinterpret_cast<const uint2*>(st + L::ST_M)[2 * r + hw];
        uint32_t pk[32], pk2[32];
        {
          uint32_t sr[64], dr[64];
          tmem_ld32(tS, sr);
          tmem_ld32(tS + 32, sr + 32);
          tmem_ld32(tP, dr);
          tmem_ld32(tP + 32, dr + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&B->s_free);  // S^T and dP^T are in registers: the MMA may reuse them
          const unsigned long long sc2 = f2_splat(p.scale_log2);
          // the keep bits only on partial tiles (uniform over the CTA)
          const auto body = [&](auto masked) {
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
              const float4 nl = l2[c4], nd = dl[c4];  // -LSE log2(e) and -Delta of the 4 columns
              float pv[4], dsv[4];
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int c = c4 * 4 + 2 * k2;
                p_pair(sr[c], sr[c + 1], sc2, k2 ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y), c, pv[2 * k2],
                       pv[2 * k2 + 1]);
                if constexpr (decltype(masked)::value) {
                  const uint32_t word = c < 32 ? mk.x : mk.y;
                  pv[2 * k2] = ((word >> (c & 31)) & 1u) ? pv[2 * k2] : 0.f;
                  pv[2 * k2 + 1] = ((word >> ((c + 1) & 31)) & 1u) ? pv[2 * k2 + 1] : 0.f;
                }
                ds_pair(pv[2 * k2], pv[2 * k2 + 1], dr[c], dr[c + 1], k2 ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y),
                        dsv[2 * k2], dsv[2 * k2 + 1]);
              }
              pk[2 * c4] = pack_bf16(pv[0], pv[1]);
              pk[2 * c4 + 1] = pack_bf16(pv[2], pv[3]);
              pk2[2 * c4] = pack_bf16(dsv[0], dsv[1]);
              pk2[2 * c4 + 1] = pack_bf16(dsv[2], dsv[3]);
            }
          };
          if (slot >= 0)
            body(std::true_type{});
          else
            body(std::false_type{});
        }
        // the previous step's dV, dK and dQ products must be done reading
        // packed P^T and the dS^T panels
        if (y > 0) {
          ok = mbar_wait(&B->ps_free2, (y - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st32(tl + L::TM_P + 32 * hw, pk);
#pragma unroll
        for (int c = 0; c < 8; ++c)  // 16-byte chunk c of the row goes to chunk c ^ (row & 7): the 128-byte swizzle
          ds_row[c ^ r7] = make_uint4(pk2[4 * c], pk2[4 * c + 1], pk2[4 * c + 2], pk2[4 * c + 3]);
        fence_proxy_async_smem();  // visible to the tensor core's shared-memory reads
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B->p_full[0]);
      }
      if (!ok) break;
      ok = mbar_wait(&B->acc_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float mul = hw ? p.scale : 1.f;
      const uint32_t acc = hw ? L::TM_DK : L::TM_DV;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + acc + c * 32, v);
        tmem_ld_wait();
        if (itm.slot < 0) {
          if (kv < p.T) store_row32(orow + c * 32, v, mul);
        } else {  // one chunk of a split column: fp32 partial sums, summed later in chunk order
          float4* prow = reinterpret_cast<float4*>(p.partial + ((size_t)itm.slot * 128 + r) * (2 * D) + (hw ? D : 0) +
                                                   c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            prow[k] = make_float4(__uint_as_float(v[4 * k]) * mul, __uint_as_float(v[4 * k + 1]) * mul,
                                  __uint_as_float(v[4 * k + 2]) * mul, __uint_as_float(v[4 * k + 3]) * mul);
        }
      }
      tc_fence_before();
      mbar_arrive(&B->acc_free);
      sc += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}

// After the one-pass kernel, in one launch: blocks [0, 16 n_splits) sum the
// chunk partials of the split kv-major columns into dV and dK (as
// k_dkdv_finalize, block b: column b / 16, rows 8 (b % 16) ..), and the other
// blocks write dQ = scale * the fp32 accumulator as bf16, grid-stride over n8
// runs of 8 values (the rows below T come first in its [Tpad][Hq][D]).
__global__ void __launch_bounds__(256) k_fused_finalize(const int4* __restrict__ splits, int n_splits,
                                                        const float* __restrict__ partial, int T, int Hkv,
                                                        __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV,
                                                        const float4* __restrict__ acc, size_t n8, float scale,
                                                        uint4* __restrict__ dQ) {
  pdl_wait();  // launched with programmatic dependent launch
  const unsigned nsb = 16u * (unsigned)n_splits;
  if (blockIdx.x < nsb) {
    dkdv_split_rows<64>(splits[blockIdx.x >> 4], blockIdx.x & 15, partial, T, Hkv, dK, dV);
    return;
  }
  // two runs per thread and pass: four 16-byte loads in flight
  const size_t stride = (size_t)(gridDim.x - nsb) * blockDim.x;
  for (size_t i = (blockIdx.x - nsb) * (size_t)blockDim.x + threadIdx.x; i < n8; i += 2 * stride) {
    const size_t i2 = i + stride;
    const bool two = i2 < n8;
    const float4 a = __ldcs(acc + 2 * i), b = __ldcs(acc + 2 * i + 1);
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f), d = c;
    if (two) {
      c = __ldcs(acc + 2 * i2);
      d = __ldcs(acc + 2 * i2 + 1);
    }
    dQ[i] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                       pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
    if (two)
      dQ[i2] = make_uint4(pack_bf16(c.x * scale, c.y * scale), pack_bf16(c.z * scale, c.w * scale),
                          pack_bf16(d.x * scale, d.y * scale), pack_bf16(d.z * scale, d.w * scale));
  }
}

// ---------------------------------------------------------------------------
// 3. dQ, q-major
// ---------------------------------------------------------------------------
template <int D>
struct DqL {
  using C = BwdCfg<D>;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = C::TILE;
  static constexpr int OFF_ST = 2 * C::TILE;  // stages: K | V | row masks
  static constexpr int ST_K = 0, ST_V = C::TILE, ST_M = 2 * C::TILE;
  static constexpr int ST_BYTES = ST_M + 2048;
  // dQ tile staged for its TMA store (128-byte swizzled panels, 1024-aligned)
  static constexpr int OFF_OST = OFF_ST + C::STAGES * ST_BYTES;
  static_assert(OFF_OST % 1024 == 0, "staging tile alignment");
  static constexpr int OFF_META = OFF_OST + C::TILE;
  static constexpr int OFF_BAR = OFF_META + 64;
  static constexpr int OFF_MISC = OFF_BAR + (int)sizeof(BwdBars<C::STAGES>);
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(C::TM_ACC0 + D <= 512, "TMEM budget");
  static_assert(C::TM_DQ_DS + 64 <= 512, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    k_bwd_dq(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
             const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
             const __grid_constant__ CUtensorMap mdQ, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = BwdCfg<D>;
  using L = DqL<D>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars<S>* B = reinterpret_cast<BwdBars<S>*>(smem + L::OFF_BAR);
  int* meta = reinterpret_cast<int*>(smem + L::OFF_META);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int n_items = p.n_major * p.Hq;

  if (threadIdx.x == 256) {
    init_bars<S>(B);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
    prefetch_tmap(&mdQ);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t sc = 0, it = 0;
      bool ok = true, res_issued = false;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.order[w / p.Hq], h = w % p.Hq, hk = h / g;
        const int e0 = p.ptr[tile], n = p.ptr[tile + 1] - e0;
        if (n == 0) continue;
        if (it > 0 && !(ok = mbar_wait(&B->res_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(&B->res_full, 2 * C::TILE);
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn) {
          tma_load_3d(smem + L::OFF_Q + pn * C::PANEL, &mQ, &B->res_full, pn * 64, h, tile * 128);
          tma_load_3d(smem + L::OFF_DO + pn * C::PANEL, &mdO, &B->res_full, pn * 64, h, tile * 128);
        }
        res_issued = true;
        for (int x = 0; x < n; ++x) {
          const int j = p.idx[e0 + x], slot = p.pidx[e0 + x];
          const uint32_t s = sc % S, u = sc / S;
          if (u > 0 && !(ok = mbar_wait(&B->st_empty[s], (u - 1) & 1, abort_flag))) break;
          uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
          meta[s] = slot;
          mbar_expect_tx(&B->st_full[s], 2 * C::TILE + (slot >= 0 ? 2048 : 0));
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn) {
            tma_load_3d(st + L::ST_K + pn * C::PANEL, &mK, &B->st_full[s], pn * 64, hk, j * 128);
            tma_load_3d(st + L::ST_V + pn * C::PANEL, &mV, &B->st_full[s], pn * 64, hk, j * 128);
          }
          if (slot >= 0) bulk_load(st + L::ST_M, p.masks + (size_t)slot * 512, 2048, &B->st_full[s]);
          ++sc;
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (res_issued) mbar_wait_drain(&B->res_full, it & 1, lim);
        for (uint32_t s = 0; s < S && s < sc; ++s) {
          uint32_t last = sc - 1 - ((sc - 1 - s) % S);
          mbar_wait_drain(&B->st_full[s], (last / S) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::OFF_Q), sdO = smem_u32(smem + L::OFF_DO);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.order[w / p.Hq];
        const int n = p.ptr[tile + 1] - p.ptr[tile];
        if (n == 0) continue;
        if (!(ok = mbar_wait(&B->res_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int x = 0; x <= n && ok; ++x) {
          const uint32_t s = (sc + x) % S;
          if (x < n) {
            if (!(ok = mbar_wait(&B->st_full[s], ((sc + x) / S) & 1, abort_flag))) break;
            tc_fence_after();
          }
          const uint32_t y = sc + x;  // global block index of this CTA
          if (x < n) {
            // S = Q K^T and dP = dO V^T (M = 128 q, N = 128 kv) as soon as the
            // compute warpgroups have loaded the previous S and dP
            if (y >= 1 && !(ok = mbar_wait(&B->s_free, (y - 1) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t st = sST + s * L::ST_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
              mma_ss(tbase + C::TM_S, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(st + L::ST_K + off, 16, 1024),
                     IDESC_S, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
              mma_ss(tbase + C::TM_DP, sdesc_sw128(sdO + off, 16, 1024), sdesc_sw128(st + L::ST_V + off, 16, 1024),
                     IDESC_S, kk > 0);
            }
            mma_commit(&B->s_full[0]);
            if (x == n - 1) mma_commit(&B->res_empty);
          }
          if (x >= 1 && !C::TWO_ISSUERS) {  // (two issuers: dQ is the second MMA warp's)
            // dQ += dS K for the previous block (K = 128 kv; dS packed in its own region)
            const uint32_t sp = (sc + x - 1) % S;
            if (!(ok = mbar_wait(&B->p_full[0], (y - 1) & 1, abort_flag))) break;
            if (x == 1 && it > 0 && !(ok = mbar_wait(&B->acc_free, (it - 1) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t stp = sST + sp * L::ST_BYTES;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tbase + C::TM_ACC0, tbase + C::TM_DQ_DS + kk * 8,
                     sdesc_sw128(stp + L::ST_K + kk * 2048, C::PANEL, 1024), IDESC_ACC, (x > 1 || kk > 0));
            mma_commit(&B->ps_free);
            mma_commit(&B->st_empty[sp]);
          }
        }
        if (ok && !C::TWO_ISSUERS) mma_commit(&B->acc_full);
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done);
      mbar_wait_drain(&B->mma_done, 0, 200000000);
    }
    __syncwarp();
  } else if (C::TWO_ISSUERS && warp == 10) {
    // ------------------------------------------------------------ dQ issuer (head_dim 64)
    if (lane == 0) {
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.order[w / p.Hq];
        const int n = p.ptr[tile + 1] - p.ptr[tile];
        if (n == 0) continue;
        for (int x = 0; x < n && ok; ++x) {
          // dQ += dS K of block x (K = 128 kv; dS packed in its own region)
          // once the compute warpgroups have written dS (and, on an item's
          // first block, read the previous item's dQ)
          const uint32_t y = sc + x, sp = y % S;
          uint64_t* bars[3] = {&B->st_full[sp], &B->p_full[0], (x == 0 && it > 0) ? &B->acc_free : nullptr};
          const uint32_t par[3] = {(y / S) & 1, y & 1, (it - 1) & 1};
          if (!(ok = mbar_wait_all<3>(bars, par, abort_flag))) break;
          tc_fence_after();
          const uint32_t stp = sST + sp * L::ST_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tbase + C::TM_ACC0, tbase + C::TM_DQ_DS + kk * 8, sdesc_sw128(stp + L::ST_K + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, (x > 0 || kk > 0));
          mma_commit(&B->ps_free);
          mma_commit(&B->st_empty[sp]);
        }
        if (ok) mma_commit(&B->acc_full);
        sc += n;
        ++it;
      }
      mma_commit(&B->mma_done2);
      mbar_wait_drain(&B->mma_done2, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (q row per thread)
    const int hw = warp >> 2;  // which 64 kv columns of each block this warpgroup takes
    const int r = threadIdx.x & 127;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = tl + C::TM_S + 64 * hw, tP = tl + C::TM_DP + 64 * hw;
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const int tile = p.order[w / p.Hq], h = w % p.Hq;
      const int n = p.ptr[tile + 1] - p.ptr[tile];
      const int q = tile * 128 + r;
      __nv_bfloat16* orow = p.out0 + ((size_t)q * p.Hq + h) * D + hw * (D / 2);  // this warpgroup's columns
      if (n == 0) {
        if (q < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D / 16; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        }
        continue;
      }
      const unsigned long long nl2 = f2_splat(p.nlse2[(size_t)h * p.Tpad + q]);  // this row's -LSE log2(e)
      const unsigned long long nd2 = f2_splat(p.ndelta[(size_t)h * p.Tpad + q]);  // and -Delta
      for (int x = 0; x < n; ++x) {
        const uint32_t y = sc + x, s = y % S;
        ok = mbar_wait(&B->s_full[0], y & 1, abort_flag) && mbar_wait(&B->st_full[s], (y / S) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64], dr[64];
        tmem_ld32(tS, sr);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld32(tP, dr);
        tmem_ld32(tP + 32, dr + 32);
        const uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
        const int slot = meta[s];
        uint2 mk = make_uint2(0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = reinterpret_cast<const uint2*>(st + L::ST_M)[2 * r + hw];
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&B->s_free);  // S and dP are in registers: the MMA may reuse them
        const unsigned long long sc2 = f2_splat(p.scale_log2);
        const auto body = [&](auto masked) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float p0, p1, d0, d1;
            p_pair(sr[c], sr[c + 1], sc2, nl2, c, p0, p1);
            if constexpr (decltype(masked)::value) {
              const uint32_t word = c < 32 ? mk.x : mk.y;
              p0 = ((word >> (c & 31)) & 1u) ? p0 : 0.f;
              p1 = ((word >> ((c + 1) & 31)) & 1u) ? p1 : 0.f;
            }
            ds_pair(p0, p1, dr[c], dr[c + 1], nd2, d0, d1);
            dr[c] = __float_as_uint(d0);
            dr[c + 1] = __float_as_uint(d1);
          }
        };
        if (slot >= 0)
          body(std::true_type{});
        else  // full tile: no mask
          body(std::false_type{});
        uint32_t pk[32];
        pack64(dr, pk);
        if (y > 0) {  // the previous dQ MMA must be done reading the dS region
          ok = mbar_wait(&B->ps_free, (y - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st32(tl + C::TM_DQ_DS + 32 * hw, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B->p_full[0]);
      }
      if (!ok) break;
      ok = mbar_wait(&B->acc_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dQ rows into the staging tile (this warpgroup's half of every row),
      // once the previous item's store has read it; then one TMA store
      if (it > 0) {
        ok = mbar_wait(&B->o_stored, (it - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
      uint8_t* ost = smem + L::OFF_OST;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        const int col = hw * (D / 2) + c * 32;  // first of these 32 columns
        tmem_ld32(tl + C::TM_ACC0 + col, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pk[k] = pack_bf16(__uint_as_float(v[2 * k]) * p.scale, __uint_as_float(v[2 * k + 1]) * p.scale);
        uint8_t* prow = ost + (col >> 6) * C::PANEL + r * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (((col & 63) >> 3) + k) ^ (r & 7);
          *reinterpret_cast<uint4*>(prow + chunk * 16) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                                                                    pk[4 * k + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&B->acc_free);
      fence_proxy_async_smem();
      mbar_arrive(&B->o_written);
      if (threadIdx.x == 0) {
        ok = mbar_wait(&B->o_written, it & 1, abort_flag);
        if (ok) {
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn) tma_store_3d(&mdQ, ost + pn * C::PANEL, pn * 64, h, tile * 128);
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&B->o_stored);
        }
      }
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      sc += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
    if (threadIdx.x == 0) bulk_wait0();  // the last dQ store has landed
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// 3b. dQ, q-major, software-pipelined three blocks deep (D = 128)
//
// Each CTA runs a host-built list of (q tile, head) items, packed longest
// first onto the CTAs, as one stream of kv blocks.  One loop iteration of the
// MMA thread issues S(t) = Q K_t^T, dP(t-1) = dO V_{t-1}^T and dQ += dS(t-2)
// K_{t-2}; the last dQ of an item goes before the dP, since the compute
// warpgroups finish an item (its epilogue) before they load the next block's
// S, which that dP waits for.  Each block owns one of three TMEM buffers for
// its life: S lands there, the compute warpgroups load it and release the
// buffer for dP, which lands in the same columns, and they write the packed
// dS over it.  K blocks live in a four-slot ring (read by S and, two
// iterations later, by dQ, so K(t+4) loads while S(t+1)..S(t+3) run) and V
// blocks in a one-slot ring (read by dP only), each filled by its own
// producer warp; an item's Q and dO travel with its first K and V block.
//
// The tensor pipe accepts only a few MMAs ahead of the one executing, and a
// barrier check issued right after a group of MMAs completes only when the
// group has drained; so the MMA thread checks everything a group needs in one
// batch, keeps item boundaries in registers and does as little else as it can
// between groups.  Tile masks are read from global memory, a block ahead.
// ---------------------------------------------------------------------------
template <int D>
struct DqpCfg {
  static constexpr int NP = D / 64;
  static constexpr int PANEL = 128 * 128;  // 128 rows x 128 B
  static constexpr int TILE = NP * PANEL;
  static constexpr int KS = 4, NB = 3;     // K ring slots, TMEM buffers (V ring: one slot)
  static constexpr int THREADS = 352;      // 8 compute warps, K producer, MMA, V producer
  static constexpr int TM_ACC = NB * 128;
  static_assert(TM_ACC + D <= 512, "TMEM budget");
};

template <int D>
struct DqpL {
  using C = DqpCfg<D>;
  static constexpr int OFF_Q = 0, OFF_DO = C::TILE, OFF_K = 2 * C::TILE, OFF_V = OFF_K + C::KS * C::TILE;
  static constexpr int OFF_BAR = OFF_V + C::TILE;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct DqpBars {
  uint64_t k_full[4], k_empty[4], v_full, v_empty, q_empty, do_empty;
  uint64_t s_full[3], s_loaded[3], dp_full[3], p_full[3];
  uint64_t acc_full, acc_free, mma_done;
};

// 64-bit shared-memory descriptor plus a byte offset that keeps the address
// below 256 KB (no carry out of the 14-bit start-address field).
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

template <int D>
__global__ void __launch_bounds__(DqpCfg<D>::THREADS, 1)
    k_bwd_dq_pipe(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                  const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = DqpCfg<D>;
  using L = DqpL<D>;
  static_assert(sizeof(DqpBars) <= 256, "barrier block");
  constexpr uint32_t FIRST = 1, LAST = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqpBars* B = reinterpret_cast<DqpBars*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int4 cta = p.dq_cta[blockIdx.x];  // first item, end item, kv blocks

  if (threadIdx.x == 256) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(&B->k_full[i], 1);
      mbar_init(&B->k_empty[i], 1);
    }
    mbar_init(&B->v_full, 1);
    mbar_init(&B->v_empty, 1);
    mbar_init(&B->q_empty, 1);
    mbar_init(&B->do_empty, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->s_loaded[i], 256);
      mbar_init(&B->dp_full[i], 1);
      mbar_init(&B->p_full[i], 256);
    }
    mbar_init(&B->acc_full, 1);
    mbar_init(&B->acc_free, 256);
    mbar_init(&B->mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    // warp 8: the K ring (and each item's Q); warp 10: the V slot (and dO)
    if (lane == 0) {
      const bool kp = warp == 8;
      uint32_t y = 0;  // blocks whose loads were issued
      bool ok = true;
      for (int k = cta.x; k < cta.y && ok; ++k) {
        const int4 itm = p.dq_items[k];  // q tile, head, first entry, blocks
        const int hk = itm.y / g, ki = k - cta.x;
        for (int x = 0; x < itm.w; ++x) {
          const int j = p.idx[itm.z + x];
          if (kp) {
            const uint32_t sl = y % C::KS;
            if (y >= C::KS && !(ok = mbar_wait(&B->k_empty[sl], (y / C::KS - 1) & 1, abort_flag))) break;
            if (x == 0 && ki > 0 && !(ok = mbar_wait(&B->q_empty, (ki - 1) & 1, abort_flag))) break;
            mbar_expect_tx(&B->k_full[sl], x == 0 ? 2 * C::TILE : C::TILE);
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn) {
              if (x == 0) tma_load_3d(smem + L::OFF_Q + pn * C::PANEL, &mQ, &B->k_full[sl], pn * 64, itm.y, itm.x * 128);
              tma_load_3d(smem + L::OFF_K + sl * C::TILE + pn * C::PANEL, &mK, &B->k_full[sl], pn * 64, hk, j * 128);
            }
          } else {
            if (y >= 1 && !(ok = mbar_wait(&B->v_empty, (y - 1) & 1, abort_flag))) break;
            if (x == 0 && ki > 0 && !(ok = mbar_wait(&B->do_empty, (ki - 1) & 1, abort_flag))) break;
            mbar_expect_tx(&B->v_full, x == 0 ? 2 * C::TILE : C::TILE);
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn) {
              if (x == 0) tma_load_3d(smem + L::OFF_DO + pn * C::PANEL, &mdO, &B->v_full, pn * 64, itm.y, itm.x * 128);
              tma_load_3d(smem + L::OFF_V + pn * C::PANEL, &mV, &B->v_full, pn * 64, hk, j * 128);
            }
          }
          ++y;
        }
      }
      if (!ok) {
        // let every load already issued land before the CTA exits
        const long long lim = 20000000;
        if (kp) {
          for (uint32_t k = 0; k < C::KS && k < y; ++k) {
            const uint32_t last = y - 1 - ((y - 1 - k) % C::KS);
            mbar_wait_drain(&B->k_full[k], (last / C::KS) & 1, lim);
          }
        } else if (y > 0) {
          mbar_wait_drain(&B->v_full, (y - 1) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + L::OFF_Q), 16, 1024);
      const uint64_t dO0 = sdesc_sw128(smem_u32(smem + L::OFF_DO), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + L::OFF_V), 16, 1024);
      const uint64_t dKt0 = sdesc_sw128(smem_u32(smem + L::OFF_K), C::PANEL, 1024);  // K as the MN-major B of dQ
      const uint32_t total = (uint32_t)cta.z;
      // item boundaries of the S stream: [s_beg, s_end), the next item's size prefetched
      int k = cta.x;
      uint32_t s_beg = 0, s_end = total > 0 ? (uint32_t)p.dq_items[k].w : 0;
      int n_next = k + 1 < cta.y ? p.dq_items[k + 1].w : 0;
      uint32_t fp = 0, fq = 0, itq = 0;  // flags of blocks t-1 and t-2; items whose dQ is done
      bool ok = true;
      for (uint32_t t = 0; t < total + 2 && ok; ++t) {
        const bool has_s = t < total, has_dp = t >= 1 && t <= total, has_dq = t >= 2;
        uint32_t fs = 0;
        if (has_s) {
          if (t == s_end) {
            s_beg = s_end;
            s_end += (uint32_t)n_next;
            ++k;
            n_next = k + 1 < cta.y ? p.dq_items[k + 1].w : 0;
          }
          fs = (t == s_beg ? FIRST : 0u) | (t + 1 == s_end ? LAST : 0u);
        }
        const bool dq_first = has_dq && (fq & LAST);
        const bool dp_now = has_dp && !dq_first;
        const uint32_t bs = t % 3, bp = (t + 2) % 3, bq = (t + 1) % 3;  // TMEM buffers of t, t-1, t-2
        {
          uint64_t* const bars[3] = {has_s ? &B->k_full[t % C::KS] : nullptr, dp_now ? &B->v_full : nullptr,
                                     dp_now ? &B->s_loaded[bp] : nullptr};
          const uint32_t par[3] = {(t / C::KS) & 1, (t - 1) & 1, ((t - 1) / 3) & 1};
          if (!(ok = mbar_wait_all(bars, par, abort_flag))) break;
        }
        tc_fence_after();
        if (has_s) {
          const uint64_t db = sdesc_add(dK0, (t % C::KS) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + bs * 128, sdesc_add(dQ0, off), sdesc_add(db, off), IDESC_S, kk > 0);
          }
          mma_commit(&B->s_full[bs]);
          if (fs & LAST) mma_commit(&B->q_empty);
        }
        const auto issue_dp = [&]() {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + bp * 128, sdesc_add(dO0, off), sdesc_add(dV0, off), IDESC_S, kk > 0);
          }
          mma_commit(&B->dp_full[bp]);
          mma_commit(&B->v_empty);
          if (fp & LAST) mma_commit(&B->do_empty);
        };
        if (dp_now) issue_dp();
        if (has_dq) {
          // dQ += dS(t-2) K(t-2) (K = 128 kv rows); warpgroup w's packed dS
          // at buffer columns [64w, 64w + 32)
          const bool first = fq & FIRST;
          {
            uint64_t* const bars[2] = {&B->p_full[bq], first && itq > 0 ? &B->acc_free : nullptr};
            const uint32_t par[2] = {((t - 2) / 3) & 1, (itq - 1) & 1};
            if (!(ok = mbar_wait_all(bars, par, abort_flag))) break;
          }
          tc_fence_after();
          const uint64_t db = sdesc_add(dKt0, ((t - 2) % C::KS) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tbase + C::TM_ACC, tbase + bq * 128 + kk * 8 + (kk >= 4 ? 32 : 0), sdesc_add(db, kk * 2048),
                   IDESC_ACC, !first || kk > 0);
          mma_commit(&B->k_empty[(t - 2) % C::KS]);
          if (fq & LAST) {
            mma_commit(&B->acc_full);
            ++itq;
          }
        }
        if (has_dp && dq_first) {
          uint64_t* const bars[2] = {&B->v_full, &B->s_loaded[bp]};
          const uint32_t par[2] = {(t - 1) & 1, ((t - 1) / 3) & 1};
          if (!(ok = mbar_wait_all(bars, par, abort_flag))) break;
          tc_fence_after();
          issue_dp();
        }
        fq = fp;
        fp = fs;
      }
      mma_commit(&B->mma_done);
      mbar_wait_drain(&B->mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (q row per thread)
    const int hw = warp >> 2;  // which 64 kv columns of each block this warpgroup takes
    const int r = threadIdx.x & 127;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16) + 64 * hw;
    const uint2* masks = reinterpret_cast<const uint2*>(p.masks);
    uint32_t y = 0;
    bool ok = true;
    for (int k = cta.x; k < cta.y && ok; ++k) {
      const int4 itm = p.dq_items[k];  // q tile, head, first entry, blocks
      const int h = itm.y, e0 = itm.z, n = itm.w;
      const int q = itm.x * 128 + r;
      __nv_bfloat16* orow = p.out0 + ((size_t)q * p.Hq + h) * D + hw * (D / 2);  // this warpgroup's columns
      const unsigned long long nl2 = f2_splat(p.nlse2[(size_t)h * p.Tpad + q]);  // this row's -LSE log2(e)
      const unsigned long long nd2 = f2_splat(p.ndelta[(size_t)h * p.Tpad + q]);  // and -Delta
      int slot = p.pidx[e0];
      uint2 mk = slot >= 0 ? masks[(size_t)slot * 256 + 2 * r + hw] : make_uint2(0xffffffffu, 0xffffffffu);
      for (int x = 0; x < n; ++x, ++y) {
        const bool full = slot < 0;  // uniform over the CTA
        // the next block's mask, a block ahead
        uint2 mk_next = make_uint2(0xffffffffu, 0xffffffffu);
        int slot_next = -1;
        if (x + 1 < n) {
          slot_next = p.pidx[e0 + x + 1];
          if (slot_next >= 0) mk_next = masks[(size_t)slot_next * 256 + 2 * r + hw];
        }
        const uint32_t b = y % 3, ph = (y / 3) & 1, col = b * 128;
        ok = mbar_wait(&B->s_full[b], ph, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tl + col, sr);
        tmem_ld32(tl + col + 32, sr + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&B->s_loaded[b]);  // dP may now overwrite S
        const unsigned long long sc2 = f2_splat(p.scale_log2);
        const auto pmath = [&](auto masked) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float p0, p1;
            p_pair(sr[c], sr[c + 1], sc2, nl2, c, p0, p1);
            if constexpr (decltype(masked)::value) {
              const uint32_t word = c < 32 ? mk.x : mk.y;
              p0 = ((word >> (c & 31)) & 1u) ? p0 : 0.f;
              p1 = ((word >> ((c + 1) & 31)) & 1u) ? p1 : 0.f;
            }
            sr[c] = __float_as_uint(p0);
            sr[c + 1] = __float_as_uint(p1);
          }
        };
        if (full)
          pmath(std::false_type{});
        else
          pmath(std::true_type{});
        ok = mbar_wait(&B->dp_full[b], ph, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t pk[32];
        {
          uint32_t dr[64];
          tmem_ld32(tl + col, dr);
          tmem_ld32(tl + col + 32, dr + 32);
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2) {
            float d0, d1;
            ds_pair(__uint_as_float(sr[2 * c2]), __uint_as_float(sr[2 * c2 + 1]), dr[2 * c2], dr[2 * c2 + 1], nd2, d0,
                    d1);
            pk[c2] = pack_bf16(d0, d1);
          }
        }
        tmem_st32(tl + col, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B->p_full[b]);
        mk = mk_next;
        slot = slot_next;
      }
      if (!ok) break;
      ok = mbar_wait(&B->acc_full, (uint32_t)(k - cta.x) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tbase + ((uint32_t)((warp & 3) * 32) << 16) + C::TM_ACC + hw * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(ta + c * 32, v);
        tmem_ld_wait();
        store_rows32(orow + c * 32, (size_t)p.Hq * D, q, p.T, v, p.scale);
      }
      tc_fence_before();
      mbar_arrive(&B->acc_free);
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// 4. head_dim 256: three passes of one half-step kernel
//
// At D = 256 one 128-row tile of Q, K, V or dO takes 64 KB of shared memory
// and one 128 x 256 fp32 accumulator takes 256 TMEM columns, so dK and dV
// cannot both be accumulated in one CTA, nor can all four operand tiles be
// resident.  The backward therefore runs three passes of one kernel:
//   WIDE_DV (kv-major): S^T = K Q^T, P^T, dV += P^T dO;
//   WIDE_DK (kv-major): S^T = K Q^T, dP^T = V dO^T, dS^T, dK += dS^T Q;
//   WIDE_DQ (q-major):  S = Q K^T, dP = dO V^T, dS, dQ += dS K.
// The 128-row A operands (K and V, or Q and dO) stay in shared memory for the
// item; the other side streams in half tiles of 64 rows (N = 64 products), so
// each step of the item is two half-steps.  Half-step y lands in TMEM buffer
// y & 1 (S and dP, 64 columns each) and is worked on by compute warpgroup
// y & 1, which is always the same half of the step.  The operand the
// accumulating product reads ("late": Q or K, or dO for dV) lives in a two-slot
// ring and is released when that product is done; the other ("early") in its
// own ring, released right after S or dP.  Row statistics and tile masks are
// read from global memory: the rings fill the shared memory.
// ---------------------------------------------------------------------------
enum { WIDE_DV = 0, WIDE_DK = 1, WIDE_DQ = 2 };

template <int MODE>
struct WideCfg {
  static constexpr int D = 256, NP = 4;
  static constexpr int RPANEL = 128 * 128;  // resident panel: 128 rows x 128 B
  static constexpr int RTILE = NP * RPANEL;
  static constexpr int HPANEL = 64 * 128;   // half-tile panel: 64 rows x 128 B
  static constexpr int HTILE = NP * HPANEL;
  static constexpr bool HAS_DP = MODE != WIDE_DV;
  static constexpr bool KV_MAJOR = MODE != WIDE_DQ;
  static constexpr int NR = HAS_DP ? 2 : 1;     // resident tiles
  static constexpr int LS = 2;                  // late ring slots
  static constexpr int ES = HAS_DP ? 1 : 2;     // early ring slots
  static constexpr int OFF_R = 0;
  static constexpr int OFF_L = NR * RTILE;
  static constexpr int OFF_E = OFF_L + LS * HTILE;
  // per late slot: the half-step's -LSE log2(e) and -Delta rows (kv-major),
  // copied with its tile, and its mask slot (written by the producer)
  static constexpr int STAT = 512;
  static constexpr int STAT_TX = KV_MAJOR ? (HAS_DP ? 512 : 256) : 0;
  static constexpr int OFF_STAT = OFF_E + ES * HTILE;
  static constexpr int OFF_META = OFF_STAT + LS * STAT;
  static constexpr int OFF_BAR = OFF_META + 16 * LS;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TM_ACC = 256;  // buffers b at 128 b: S at +0, dP at +64
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct WideBars {
  uint64_t r_full, r_empty, l_full[2], l_empty[2], e_full[2], e_empty[2];
  uint64_t s_full[2], p_full[2], acc_full, acc_free, mma_done;
};

template <int MODE>
__global__ void __launch_bounds__(320, 1)
    k_bwd_wide(const __grid_constant__ CUtensorMap mR1, const __grid_constant__ CUtensorMap mR2,
               const __grid_constant__ CUtensorMap mL, const __grid_constant__ CUtensorMap mE, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = WideCfg<MODE>;
  constexpr int D = C::D;
  static_assert(sizeof(WideBars) <= 256, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  WideBars* B = reinterpret_cast<WideBars*>(smem + C::OFF_BAR);
  volatile int* meta = reinterpret_cast<volatile int*>(smem + C::OFF_META);  // [LS][4]: mask slot of the late slot's half-step
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  // items: kv-major from the packed DkdvItem list, q-major from the dq list
  const int i_begin = C::KV_MAJOR ? p.cta_ptr[blockIdx.x] : p.dq_cta[blockIdx.x].x;
  const int i_end = C::KV_MAJOR ? p.cta_ptr[blockIdx.x + 1] : p.dq_cta[blockIdx.x].y;
  // item k -> (major tile, its kv head or q head, steps); step x -> half-step pair
  const auto item = [&](int k, int& major, int& hh, int& n) {
    if (C::KV_MAJOR) {
      const DkdvItem it = p.items[k];
      major = it.jb;
      hh = it.hk;
      n = it.x1 - it.x0;
    } else {
      const int4 it = p.dq_items[k];
      major = it.x;
      hh = it.y;
      n = it.w;
    }
  };
  // step x of item k: streamed tile (q tile or kv block), q head, mask slot
  const auto step = [&](int k, int x, int& minor, int& head, int& slot) {
    if (C::KV_MAJOR) {
      const DkdvItem it = p.items[k];
      const int e0 = p.ptr[it.jb], ncol = p.ptr[it.jb + 1] - e0;
      const int e = e0 + (it.x0 + x) % ncol;
      head = it.hk * g + (it.x0 + x) / ncol;
      minor = p.idx[e];
      slot = p.pidx[e];
    } else {
      const int4 it = p.dq_items[k];
      minor = p.idx[it.z + x];
      head = it.y;
      slot = p.pidx[it.z + x];
    }
  };

  if (threadIdx.x == 256) {
    mbar_init(&B->r_full, 1);
    mbar_init(&B->r_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->l_full[i], 1);
      mbar_init(&B->l_empty[i], 1);
      mbar_init(&B->e_full[i], 1);
      mbar_init(&B->e_empty[i], 1);
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->p_full[i], 128);  // one warpgroup per buffer
    }
    mbar_init(&B->acc_full, 1);
    mbar_init(&B->acc_free, 256);
    mbar_init(&B->mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mR1);
    if (C::HAS_DP) prefetch_tmap(&mR2);
    prefetch_tmap(&mL);
    prefetch_tmap(&mE);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t y = 0, nl = 0, ne = 0, it = 0;  // half-steps, late / early loads, items
      bool ok = true, r_issued = false;
      for (int k = i_begin; k < i_end && ok; ++k) {
        int major, hh, n;
        item(k, major, hh, n);
        if (n == 0) continue;
        r_issued = false;
        if (it > 0 && !(ok = mbar_wait(&B->r_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(&B->r_full, C::NR * C::RTILE);
        // residents: K (and V) of kv block `major` and kv head hh, or Q (and
        // dO) of q tile `major` and q head hh
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn) {
          tma_load_3d(smem + C::OFF_R + pn * C::RPANEL, &mR1, &B->r_full, pn * 64, hh, major * 128);
          if (C::HAS_DP)
            tma_load_3d(smem + C::OFF_R + C::RTILE + pn * C::RPANEL, &mR2, &B->r_full, pn * 64, hh, major * 128);
        }
        r_issued = true;
        for (int x = 0; x < n && ok; ++x) {
          int minor, head, slot;
          step(k, x, minor, head, slot);
          const int hs = C::KV_MAJOR ? head : hh / g;  // head of the streamed tiles
          for (int hf = 0; hf < 2; ++hf, ++y) {
            const int row = minor * 128 + 64 * hf;
            {
              const uint32_t s = y % C::LS;
              if (y >= C::LS && !(ok = mbar_wait(&B->l_empty[s], (y / C::LS - 1) & 1, abort_flag))) break;
              meta[4 * s] = slot;  // made visible by the arrive below
              mbar_expect_tx(&B->l_full[s], C::HTILE + C::STAT_TX);
#pragma unroll
              for (int pn = 0; pn < C::NP; ++pn)
                tma_load_3d(smem + C::OFF_L + s * C::HTILE + pn * C::HPANEL, &mL, &B->l_full[s], pn * 64, hs, row);
              if (C::KV_MAJOR) {  // this half's 64 q rows: row is a multiple of 64, so both copies are aligned
                uint8_t* st = smem + C::OFF_STAT + s * C::STAT;
                bulk_load(st, p.nlse2 + (size_t)head * p.Tpad + row, 256, &B->l_full[s]);
                if (C::HAS_DP) bulk_load(st + 256, p.ndelta + (size_t)head * p.Tpad + row, 256, &B->l_full[s]);
              }
              ++nl;
            }
            {
              const uint32_t s = y % C::ES;
              if (y >= C::ES && !(ok = mbar_wait(&B->e_empty[s], (y / C::ES - 1) & 1, abort_flag))) break;
              mbar_expect_tx(&B->e_full[s], C::HTILE);
#pragma unroll
              for (int pn = 0; pn < C::NP; ++pn)
                tma_load_3d(smem + C::OFF_E + s * C::HTILE + pn * C::HPANEL, &mE, &B->e_full[s], pn * 64, hs, row);
              ++ne;
            }
          }
        }
        if (!ok) break;
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (r_issued) mbar_wait_drain(&B->r_full, it & 1, lim);
        for (uint32_t s = 0; s < C::LS && s < nl; ++s) {
          const uint32_t last = nl - 1 - ((nl - 1 - s) % C::LS);
          mbar_wait_drain(&B->l_full[s], (last / C::LS) & 1, lim);
        }
        for (uint32_t s = 0; s < C::ES && s < ne; ++s) {
          const uint32_t last = ne - 1 - ((ne - 1 - s) % C::ES);
          mbar_wait_drain(&B->e_full[s], (last / C::ES) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 64, false, false);
      constexpr uint32_t IDESC_OUT = idesc_bf16(128, D, false, true);
      const uint32_t sR1 = smem_u32(smem + C::OFF_R), sR2 = sR1 + C::RTILE;
      const uint32_t sL = smem_u32(smem + C::OFF_L), sE = smem_u32(smem + C::OFF_E);
      uint32_t y = 0, it = 0;
      bool ok = true;
      for (int k = i_begin; k < i_end && ok; ++k) {
        int major, hh, n;
        item(k, major, hh, n);
        if (n == 0) continue;
        if (!(ok = mbar_wait(&B->r_full, it & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t n2 = 2 * (uint32_t)n;
        for (uint32_t x = 0; x <= n2 && ok; ++x) {
          const uint32_t yy = y + x;
          if (x < n2) {
            // S (and dP) of half-step yy into buffer yy & 1; the buffer's
            // previous half-step had its accumulate product issued before
            const uint32_t b = yy & 1, ls = yy % C::LS, es = yy % C::ES;
            {
              uint64_t* const bars[2] = {&B->l_full[ls], &B->e_full[es]};
              const uint32_t par[2] = {(yy / C::LS) & 1, (yy / C::ES) & 1};
              if (!(ok = mbar_wait_all(bars, par, abort_flag))) break;
            }
            tc_fence_after();
            // S from the late ring (Q or K), except for dV, where the late
            // ring holds dO and S reads Q from the early ring
            const uint32_t src = C::HAS_DP ? sL + ls * C::HTILE : sE + es * C::HTILE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t offr = (kk >> 2) * C::RPANEL + (kk & 3) * 32, offh = (kk >> 2) * C::HPANEL + (kk & 3) * 32;
              mma_ss(tbase + b * 128, sdesc_sw128(sR1 + offr, 16, 1024), sdesc_sw128(src + offh, 16, 1024), IDESC_S,
                     kk > 0);
            }
            if (C::HAS_DP) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t offr = (kk >> 2) * C::RPANEL + (kk & 3) * 32,
                               offh = (kk >> 2) * C::HPANEL + (kk & 3) * 32;
                mma_ss(tbase + b * 128 + 64, sdesc_sw128(sR2 + offr, 16, 1024),
                       sdesc_sw128(sE + es * C::HTILE + offh, 16, 1024), IDESC_S, kk > 0);
              }
            }
            mma_commit(&B->e_empty[es]);
            mma_commit(&B->s_full[b]);
            if (x == n2 - 1) mma_commit(&B->r_empty);
          }
          if (x >= 1) {
            // accumulate the previous half-step: OUT += X late (K = 64 rows,
            // N = 256), X = P or dS packed over that buffer's first S or dP columns
            const uint32_t yp = yy - 1, bp = yp & 1, lp = yp % C::LS;
            {
              uint64_t* const bars[2] = {&B->p_full[bp], x == 1 && it > 0 ? &B->acc_free : nullptr};
              const uint32_t par[2] = {(yp >> 1) & 1, (it - 1) & 1};
              if (!(ok = mbar_wait_all(bars, par, abort_flag))) break;
            }
            tc_fence_after();
            const uint32_t a = tbase + bp * 128 + (C::HAS_DP ? 64 : 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tbase + C::TM_ACC, a + kk * 8, sdesc_sw128(sL + lp * C::HTILE + kk * 2048, C::HPANEL, 1024),
                     IDESC_OUT, (x > 1 || kk > 0));
            mma_commit(&B->l_empty[lp]);
          }
        }
        if (ok) mma_commit(&B->acc_full);
        y += n2;
        ++it;
      }
      mma_commit(&B->mma_done);
      mbar_wait_drain(&B->mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (major row per thread)
    const int hw = warp >> 2;  // half of every step, and TMEM buffer, of this warpgroup
    const int r = threadIdx.x & 127;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint2* masks = reinterpret_cast<const uint2*>(p.masks);
    uint32_t y = 0, it = 0;
    bool ok = true;
    for (int k = i_begin; k < i_end && ok; ++k) {
      int major, hh, n;
      item(k, major, hh, n);
      const int row = major * 128 + r;  // kv token (kv-major) or q token (q-major)
      __nv_bfloat16* out = MODE == WIDE_DQ ? p.out0 + ((size_t)row * p.Hq + hh) * D + hw * 128
                                           : (MODE == WIDE_DV ? p.out1 : p.out0) + ((size_t)row * p.Hkv + hh) * D +
                                                 hw * 128;  // this warpgroup's 128 columns of the output row
      if (n == 0) {
        if (row < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < 16; ++c) reinterpret_cast<uint4*>(out)[c] = z;
        }
        continue;
      }
      const unsigned long long sc2 = f2_splat(p.scale_log2);
      float l2r = 0.f, dlr = 0.f;  // q-major: this row's -LSE log2(e) and -Delta
      if (!C::KV_MAJOR) {
        l2r = p.nlse2[(size_t)hh * p.Tpad + row];
        dlr = p.ndelta[(size_t)hh * p.Tpad + row];
      }
      for (int x = 0; x < n; ++x) {
        // this warpgroup's half-step yy sits in late slot yy % 2 = hw (y is even)
        const uint32_t yy = y + 2 * x + hw, b = yy & 1;
        ok = mbar_wait(&B->l_full[hw], (yy >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const int slot = meta[4 * hw];
        uint2 mk = make_uint2(0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = masks[(size_t)slot * 256 + 2 * r + hw];  // in flight during the wait for S
        // kv-major: -LSE log2(e) and -Delta of this half's 64 q columns, staged with the slot's tile
        const float4* l4 = reinterpret_cast<const float4*>(smem + C::OFF_STAT + hw * C::STAT);
        const float4* d4 = l4 + 16;
        ok = mbar_wait(&B->s_full[b], (yy >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64], dr[64];
        tmem_ld32(tl + b * 128, sr);
        tmem_ld32(tl + b * 128 + 32, sr + 32);
        if (C::HAS_DP) {
          tmem_ld32(tl + b * 128 + 64, dr);
          tmem_ld32(tl + b * 128 + 96, dr + 32);
        }
        tmem_ld_wait();
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          float la[4], da[4];
          if (C::KV_MAJOR) {
            const float4 lv = l4[c4];
            la[0] = lv.x, la[1] = lv.y, la[2] = lv.z, la[3] = lv.w;
            if (C::HAS_DP) {
              const float4 dv = d4[c4];
              da[0] = dv.x, da[1] = dv.y, da[2] = dv.z, da[3] = dv.w;
            }
          } else {
            la[0] = la[1] = la[2] = la[3] = l2r;
            da[0] = da[1] = da[2] = da[3] = dlr;
          }
          float v[4];
          if constexpr (C::KV_MAJOR) {  // column pairs in packed fp32
#pragma unroll
            for (int j2 = 0; j2 < 2; ++j2) {
              const int c = 4 * c4 + 2 * j2;
              const uint32_t word = c < 32 ? mk.x : mk.y;
              float p0, p1;
              p_pair(sr[c], sr[c + 1], sc2, f2_pack(la[2 * j2], la[2 * j2 + 1]), c, p0, p1);
              p0 = ((word >> (c & 31)) & 1u) ? p0 : 0.f;
              p1 = ((word >> ((c + 1) & 31)) & 1u) ? p1 : 0.f;
              if (C::HAS_DP) {
                ds_pair(p0, p1, dr[c], dr[c + 1], f2_pack(da[2 * j2], da[2 * j2 + 1]), v[2 * j2], v[2 * j2 + 1]);
              } else {
                v[2 * j2] = p0;
                v[2 * j2 + 1] = p1;
              }
            }
          } else {  // scalar: packed pairs made the dQ pass spill
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = 4 * c4 + j;
              const uint32_t word = c < 32 ? mk.x : mk.y;
              float pr = ex2(fmaf(__uint_as_float(sr[c]), p.scale_log2, la[j]));
              pr = ((word >> (c & 31)) & 1u) ? pr : 0.f;
              v[j] = C::HAS_DP ? pr * (__uint_as_float(dr[c]) + da[j]) : pr;
            }
          }
          pk[2 * c4] = pack_bf16(v[0], v[1]);
          pk[2 * c4 + 1] = pack_bf16(v[2], v[3]);
        }
        tmem_st32(tl + b * 128 + (C::HAS_DP ? 64 : 0), pk);  // over the columns just read
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B->p_full[b]);
      }
      if (!ok) break;
      ok = mbar_wait(&B->acc_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float mul = MODE == WIDE_DV ? 1.f : p.scale;
      const int slot = C::KV_MAJOR ? p.items[k].slot : -1;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::TM_ACC + hw * 128 + c * 32, v);
        tmem_ld_wait();
        if (slot < 0) {
          store_rows32(out + c * 32, (size_t)(MODE == WIDE_DQ ? p.Hq : p.Hkv) * D, row, p.T, v, mul);
        } else {  // one chunk of a split column: fp32 partial sums, summed later in chunk order
          float4* prow = reinterpret_cast<float4*>(p.partial + ((size_t)slot * 128 + r) * (2 * D) + hw * 128 + c * 32);
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4)
            prow[k4] = make_float4(__uint_as_float(v[4 * k4]) * mul, __uint_as_float(v[4 * k4 + 1]) * mul,
                                   __uint_as_float(v[4 * k4 + 2]) * mul, __uint_as_float(v[4 * k4 + 3]) * mul);
        }
      }
      tc_fence_before();
      mbar_arrive(&B->acc_free);
      y += 2 * (uint32_t)n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}


// ---------------------------------------------------------------------------
// 5. head_dim 512: six passes of one step kernel
//
// At D = 512 a 128-row tile is 128 KB of shared memory and a 128 x 512 fp32
// accumulator is all of TMEM.  Each output (dV, dK, dQ) is therefore built
// one 256-column half per pass (MODE and p.half), with S (and dP) recomputed
// in every pass:
//   D512_DV (kv-major): S^T = K Q^T, P^T, dV_half += P^T dO_half;
//   D512_DK (kv-major): S^T = K Q^T, dP^T = V dO^T, dS^T, dK_half += dS^T Q_half;
//   D512_DQ (q-major):  S = Q K^T, dP = dO V^T, dS, dQ_half += dS K_half.
// The item's 128-row A operand of S (K, or Q) stays in shared memory; every
// other operand streams through a ring of four 16 KB 64-column panels in the
// order the MMAs consume them: a step's 8 B panels of S, then (with dP) its
// 8 pairs of A and B panels of dP, then the 4 panels of the output half the
// accumulating product reads.  Every group is a multiple of four panels, so
// those 4 panels always sit in slots 0..3 (one N = 256 operand).  TMEM: S at
// 0 and dP at 128 (the packed P or dS is written over the first columns just
// read), the output half at 256.  A step's S is issued after the previous
// step's accumulating product (which reads the packed P or dS over S).
// ---------------------------------------------------------------------------
enum { D512_DV = 0, D512_DK = 1, D512_DQ = 2 };

struct Bwd512Cfg {
  static constexpr int D = 512, NP = 8, PANEL = 128 * 128, RING = 4;
  static constexpr int OFF_R = 0;
  static constexpr int OFF_RING = OFF_R + NP * PANEL;
  static constexpr int OFF_BAR = OFF_RING + RING * PANEL;
  // r_full r_empty ring_full[4] ring_empty[4] s_full p_full acc_full acc_free mma_done
  static constexpr int NBAR = 2 + 2 * RING + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_ACC = 256;
  static constexpr int THREADS = 128 + 64;
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int MODE>
__global__ void __launch_bounds__(Bwd512Cfg::THREADS, 1)
    k_bwd_d512(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mdO, const BwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = Bwd512Cfg;
  constexpr int D = C::D;
  constexpr bool HAS_DP = MODE != D512_DV, KV_MAJOR = MODE != D512_DQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* r_full = bars;
  uint64_t* r_empty = bars + 1;
  uint64_t* ring_full = bars + 2;                // [RING]
  uint64_t* ring_empty = ring_full + C::RING;    // [RING]
  uint64_t* s_full = ring_empty + C::RING;
  uint64_t* p_full = s_full + 1;
  uint64_t* acc_full = p_full + 1;
  uint64_t* acc_free = acc_full + 1;
  uint64_t* mma_done = acc_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int hf = p.half;
  const int i_begin = KV_MAJOR ? p.cta_ptr[blockIdx.x] : p.dq_cta[blockIdx.x].x;
  const int i_end = KV_MAJOR ? p.cta_ptr[blockIdx.x + 1] : p.dq_cta[blockIdx.x].y;
  // item k -> (major tile, its kv head or q head, steps)
  const auto item = [&](int k, int& major, int& hh, int& n) {
    if (KV_MAJOR) {
      const DkdvItem it = p.items[k];
      major = it.jb;
      hh = it.hk;
      n = it.x1 - it.x0;
    } else {
      const int4 it = p.dq_items[k];
      major = it.x;
      hh = it.y;
      n = it.w;
    }
  };
  // step x of item k: streamed tile (q tile or kv block), q head, mask slot
  const auto step = [&](int k, int x, int& minor, int& head, int& slot) {
    if (KV_MAJOR) {
      const DkdvItem it = p.items[k];
      const int e0 = p.ptr[it.jb], ncol = p.ptr[it.jb + 1] - e0;
      const int e = e0 + (it.x0 + x) % ncol;
      head = it.hk * g + (it.x0 + x) / ncol;
      minor = p.idx[e];
      slot = p.pidx[e];
    } else {
      const int4 it = p.dq_items[k];
      minor = p.idx[it.z + x];
      head = it.y;
      slot = p.pidx[it.z + x];
    }
  };

  constexpr int PRODUCER = 4, ISSUER = 5;
  if (threadIdx.x == PRODUCER * 32) {
    mbar_init(r_full, 1);
    mbar_init(r_empty, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(ring_full + s, 1);
      mbar_init(ring_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
    prefetch_tmap(&mdO);
  }
  if (warp == ISSUER) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == PRODUCER) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t c = 0, it = 0;
      bool ok = true, r_issued = false;
      auto ring_load = [&](const CUtensorMap* map, int col, int h, int row) -> bool {
        const uint32_t s = c % C::RING, u = c / C::RING;
        if (u > 0 && !mbar_wait(ring_empty + s, (u - 1) & 1, abort_flag)) return false;
        mbar_expect_tx(ring_full + s, C::PANEL);
        tma_load_3d(smem + C::OFF_RING + s * C::PANEL, map, ring_full + s, col, h, row);
        ++c;
        return true;
      };
      for (int k = i_begin; k < i_end && ok; ++k) {
        int major, hh, n;
        item(k, major, hh, n);
        if (n == 0) continue;
        r_issued = false;
        if (it > 0 && !(ok = mbar_wait(r_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(r_full, C::NP * C::PANEL);
        // the resident A operand of S: K of kv block `major` (kv-major) or Q of q tile `major`
        for (int pn = 0; pn < C::NP; ++pn)
          tma_load_3d(smem + C::OFF_R + pn * C::PANEL, KV_MAJOR ? &mK : &mQ, r_full, pn * 64, hh, major * 128);
        r_issued = true;
        for (int x = 0; x < n && ok; ++x) {
          int minor, head, slot;
          step(k, x, minor, head, slot);
          const int hk = KV_MAJOR ? hh : hh / g;  // kv head of the item
          // S: the B panels (Q of q tile `minor`, or K of kv block `minor`)
          for (int pn = 0; pn < C::NP && ok; ++pn)
            ok = KV_MAJOR ? ring_load(&mQ, pn * 64, head, minor * 128) : ring_load(&mK, pn * 64, hk, minor * 128);
          // dP: A and B panel pairs (V of the kv block and dO of the q tile)
          if (HAS_DP)
            for (int pn = 0; pn < C::NP && ok; ++pn) {
              if (KV_MAJOR)
                ok = ring_load(&mV, pn * 64, hk, major * 128) && ring_load(&mdO, pn * 64, head, minor * 128);
              else
                ok = ring_load(&mdO, pn * 64, hh, major * 128) && ring_load(&mV, pn * 64, hk, minor * 128);
            }
          // the output half's operand: dO (dV), Q (dK) or K (dQ) of the streamed tile
          for (int q4 = 0; q4 < 4 && ok; ++q4) {
            const int col = (4 * hf + q4) * 64;
            ok = MODE == D512_DV ? ring_load(&mdO, col, head, minor * 128)
                                 : (MODE == D512_DK ? ring_load(&mQ, col, head, minor * 128)
                                                    : ring_load(&mK, col, hk, minor * 128));
          }
        }
        if (!ok) break;
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (r_issued) mbar_wait_drain(r_full, it & 1, lim);
        for (uint32_t s = 0; s < C::RING && s < c; ++s) {
          const uint32_t last = c - 1 - ((c - 1 - s) % C::RING);
          mbar_wait_drain(ring_full + s, (last / C::RING) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == ISSUER) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, 256, false, true);
      const uint32_t sR = smem_u32(smem + C::OFF_R), sG = smem_u32(smem + C::OFF_RING);
      uint32_t c = 0, y = 0, it = 0;
      bool ok = true;
      auto wait_panel = [&](uint32_t cc) -> bool {
        return mbar_wait(ring_full + cc % C::RING, (cc / C::RING) & 1, abort_flag);
      };
      for (int k = i_begin; k < i_end && ok; ++k) {
        int major, hh, n;
        item(k, major, hh, n);
        if (n == 0) continue;
        if (!(ok = mbar_wait(r_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int x = 0; x <= n && ok; ++x) {
          if (x >= 1) {
            // the output half += X(x-1) [its 4 panels, slots 0..3], X = P or dS
            // packed over the first columns of S or dP
            const uint32_t yp = y + x - 1;
            if (!(ok = mbar_wait(p_full, yp & 1, abort_flag))) break;
            if (x == 1 && it > 0 && !(ok = mbar_wait(acc_free, (it - 1) & 1, abort_flag))) break;
            for (int q4 = 0; q4 < 4 && ok; ++q4) ok = wait_panel(c + q4);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a = tbase + (HAS_DP ? C::TM_DP : C::TM_S);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tbase + C::TM_ACC, a + kk * 8, sdesc_sw128(sG + (c % C::RING) * C::PANEL + kk * 2048, C::PANEL, 1024),
                     IDESC_ACC, (x > 1 || kk > 0));
            for (int q4 = 0; q4 < 4; ++q4) mma_commit(ring_empty + (c + q4) % C::RING);
            c += 4;
          }
          if (x < n) {
            // S(x) (and dP(x)) over the columns the product above reads (issued
            // after it on this thread, so it reads them first)
            for (int pn = 0; pn < C::NP && ok; ++pn) {
              if (!(ok = wait_panel(c))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(tbase + C::TM_S, sdesc_sw128(sR + pn * C::PANEL + kk * 32, 16, 1024),
                       sdesc_sw128(sG + (c % C::RING) * C::PANEL + kk * 32, 16, 1024), IDESC_S, (pn > 0 || kk > 0));
              mma_commit(ring_empty + c % C::RING);
              ++c;
            }
            if (HAS_DP)
              for (int pn = 0; pn < C::NP && ok; ++pn) {
                if (!(ok = wait_panel(c) && wait_panel(c + 1))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tbase + C::TM_DP, sdesc_sw128(sG + (c % C::RING) * C::PANEL + kk * 32, 16, 1024),
                         sdesc_sw128(sG + ((c + 1) % C::RING) * C::PANEL + kk * 32, 16, 1024), IDESC_S,
                         (pn > 0 || kk > 0));
                mma_commit(ring_empty + c % C::RING);
                mma_commit(ring_empty + (c + 1) % C::RING);
                c += 2;
              }
            if (!ok) break;
            mma_commit(s_full);
            if (x == n - 1) mma_commit(r_empty);
          }
        }
        if (ok) mma_commit(acc_full);
        y += n;
        ++it;
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (major row per thread)
    const int r = threadIdx.x;
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint4* masks = reinterpret_cast<const uint4*>(p.masks);
    uint32_t y = 0, it = 0;
    bool ok = true;
    for (int k = i_begin; k < i_end && ok; ++k) {
      int major, hh, n;
      item(k, major, hh, n);
      const int row = major * 128 + r;  // kv token (kv-major) or q token (q-major)
      __nv_bfloat16* out = MODE == D512_DQ ? p.out0 + ((size_t)row * p.Hq + hh) * D + hf * 256
                                           : (MODE == D512_DV ? p.out1 : p.out0) + ((size_t)row * p.Hkv + hh) * D +
                                                 hf * 256;  // this pass's half of the output row
      const size_t ostride = (size_t)(MODE == D512_DQ ? p.Hq : p.Hkv) * D;
      if (n == 0) {
        if (row < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < 32; ++c) reinterpret_cast<uint4*>(out)[c] = z;
        }
        continue;
      }
      float l2r = 0.f, dlr = 0.f;  // q-major: this row's -LSE log2(e) and -Delta
      if (!KV_MAJOR) {
        l2r = p.nlse2[(size_t)hh * p.Tpad + row];
        dlr = p.ndelta[(size_t)hh * p.Tpad + row];
      }
      for (int x = 0; x < n; ++x) {
        int minor, head, slot;
        step(k, x, minor, head, slot);
        uint4 mk = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = masks[(size_t)slot * 128 + r];
        const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
        // kv-major: -LSE log2(e) and -Delta of the step's 128 q columns (uniform over the warp)
        const float4* l4 = reinterpret_cast<const float4*>(p.nlse2 + (size_t)head * p.Tpad + minor * 128);
        const float4* d4 = reinterpret_cast<const float4*>(p.ndelta + (size_t)head * p.Tpad + minor * 128);
        ok = mbar_wait(s_full, (y + x) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {  // 64 columns at a time
          uint32_t sr[64], dr[64];
          tmem_ld32(tl + C::TM_S + 64 * h2, sr);
          tmem_ld32(tl + C::TM_S + 64 * h2 + 32, sr + 32);
          if (HAS_DP) {
            tmem_ld32(tl + C::TM_DP + 64 * h2, dr);
            tmem_ld32(tl + C::TM_DP + 64 * h2 + 32, dr + 32);
          }
          tmem_ld_wait();
          uint32_t pk[32];
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            float la[4], da[4];
            if (KV_MAJOR) {
              const float4 lv = l4[16 * h2 + c4];
              la[0] = lv.x, la[1] = lv.y, la[2] = lv.z, la[3] = lv.w;
              if (HAS_DP) {
                const float4 dv = d4[16 * h2 + c4];
                da[0] = dv.x, da[1] = dv.y, da[2] = dv.z, da[3] = dv.w;
              }
            } else {
              la[0] = la[1] = la[2] = la[3] = l2r;
              da[0] = da[1] = da[2] = da[3] = dlr;
            }
            float v[4];  // scalar here: packed pairs made the dV pass 17% slower
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = 4 * c4 + j, cc = 64 * h2 + c;  // column within the step
              float pr = ex2(fmaf(__uint_as_float(sr[c]), p.scale_log2, la[j]));
              pr = ((mw[cc >> 5] >> (cc & 31)) & 1u) ? pr : 0.f;
              v[j] = HAS_DP ? pr * (__uint_as_float(dr[c]) + da[j]) : pr;
            }
            pk[2 * c4] = pack_bf16(v[0], v[1]);
            pk[2 * c4 + 1] = pack_bf16(v[2], v[3]);
          }
          // packed over the columns read first (P over S, dS over dP)
          tmem_st32(tl + (HAS_DP ? C::TM_DP : C::TM_S) + 32 * h2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      ok = mbar_wait(acc_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float mul = MODE == D512_DV ? 1.f : p.scale;
      const int slot = KV_MAJOR ? p.items[k].slot : -1;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::TM_ACC + c * 32, v);
        tmem_ld_wait();
        if (slot < 0) {
          store_rows32(out + c * 32, ostride, row, p.T, v, mul);
        } else {  // one chunk of a split column: fp32 partial sums of this half, summed later in chunk order
          float4* prow = reinterpret_cast<float4*>(p.partial + ((size_t)slot * 128 + r) * (2 * D) + c * 32);
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4)
            prow[k4] = make_float4(__uint_as_float(v[4 * k4]) * mul, __uint_as_float(v[4 * k4 + 1]) * mul,
                                   __uint_as_float(v[4 * k4 + 2]) * mul, __uint_as_float(v[4 * k4 + 3]) * mul);
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);
      y += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == ISSUER) tmem_dealloc(tbase, 512);
}
// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <class K>
int reserve_smem(K kernel, int bytes, int dev, int* flags) {
  if (dev >= 0 && dev < 64 && !flags[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("backward kernel: cannot reserve %d bytes of shared memory: %s", bytes, cudaGetErrorString(e));
      return 3;
    }
    flags[dev] = 1;
  }
  return 0;
}

// Work items of the kv-major kernel for one head layout, kept on the map.
// Columns with more steps than about one SM's share are cut into chunks that
// write fp32 partial sums to workspace slots (at most max_slots of them).  The
// items are then packed onto the grid's CTAs longest first, each to the CTA
// with the least work so far (LPT list scheduling), and stored grouped by CTA.
// Every layout asked for gets its own entry, kept until the map is freed: a
// call never frees lists that a kernel of another call may still be reading.
std::mutex g_items_mu;

// Exact-fill packing of the kv-major columns, used when the workspace has
// room for the partial sums it needs: the columns (longest first, then the
// empty ones) are laid end to end and CTA b takes the next steps up to a
// budget of load units (steps, plus about two steps of fixed work per item:
// the resident K/V tile and the epilogue), a column cut at a CTA's budget
// continuing on the next CTA as another chunk.  Every CTA then carries about
// the mean load; longest-first packing of fixed chunks left the most loaded
// CTA 15% above it on the GRPO batch.  No chunk is cut shorter than four
// steps (the budget grows instead).  Returns false (nothing produced) for
// small problems, or when the chunks would need more slots than max_slots.
bool fill_dkdv_items(const int* col_cnt, int nk, int g, int Hkv, int max_slots, int sms, long long total,
                     std::vector<DkdvItem>* packed, std::vector<int4>* splits, std::vector<int>* cta, int* n_slots) {
  constexpr long long kItemCost = 2, kMinChunk = 4;
  if (max_slots <= 0 || sms <= 0 || total < 4LL * sms) return false;
  struct Col {
    long long n;
    int j, hk;
  };
  std::vector<Col> cols;
  cols.reserve((size_t)nk * Hkv);
  for (int j = 0; j < nk; ++j)
    for (int hk = 0; hk < Hkv; ++hk) cols.push_back(Col{(long long)g * col_cnt[j], j, hk});
  std::stable_sort(cols.begin(), cols.end(), [](const Col& a, const Col& b) { return a.n > b.n; });
  const int G = sms;
  long long budget = (total + kItemCost * (long long)cols.size() + G - 1) / G;
  for (int attempt = 0; attempt < 64; ++attempt, budget += std::max(1LL, budget / 64)) {
    std::vector<std::vector<DkdvItem>> bins(G);
    std::vector<long long> load(G, 0);
    std::vector<int4> spl;
    int sl = 0, b = 0;
    bool fits = true;
    for (const Col& c : cols) {
      if (c.n == 0) break;  // the empty columns come last
      long long rem = c.n, x = 0;
      const int first = b;
      int pieces = 0;
      while (rem > 0) {
        if (b >= G) {
          fits = false;
          break;
        }
        const long long room = budget - load[b] - kItemCost;
        if (room <= 0 || (room < rem && room < kMinChunk)) {
          ++b;
          continue;
        }
        const long long take = std::min(rem, room);
        bins[b].push_back(DkdvItem{c.j, c.hk, (int)x, (int)(x + take), -1, 0, 0, 0});
        load[b] += take + kItemCost;
        x += take;
        rem -= take;
        ++pieces;
        if (rem > 0) ++b;
      }
      if (!fits) break;
      if (pieces > 1) {  // a cut column: each chunk writes partial sums to a slot of its own
        int k = 0;
        for (int bb = first; bb <= b && k < pieces; ++bb)
          if (!bins[bb].empty() && bins[bb].back().jb == c.j && bins[bb].back().hk == c.hk)
            bins[bb].back().slot = sl + k++;
        spl.push_back(make_int4(c.j, c.hk, sl, pieces));
        sl += pieces;
        if (sl > max_slots) return false;
      }
    }
    if (!fits) continue;
    // the empty columns (their dK and dV rows are zero) on the least loaded CTAs
    for (const Col& c : cols) {
      if (c.n != 0) continue;
      int bmin = 0;
      for (int bb = 1; bb < G; ++bb)
        if (load[bb] < load[bmin]) bmin = bb;
      bins[bmin].push_back(DkdvItem{c.j, c.hk, 0, 0, -1, 0, 0, 0});
      load[bmin] += kItemCost;
    }
    packed->clear();
    cta->assign(G + 1, 0);
    for (int bb = 0; bb < G; ++bb) {
      for (const DkdvItem& it : bins[bb]) packed->push_back(it);
      (*cta)[bb + 1] = (int)packed->size();
    }
    *splits = std::move(spl);
    *n_slots = sl;
    return true;
  }
  return false;
}

// Packs the kv-major items of a map whose kv blocks have col_cnt[j] q tiles
// listed (nk blocks), for g q heads per kv head and Hkv kv heads, onto `sms`
// CTAs: with exact_fill the columns are cut at equal per-CTA budgets
// (fill_dkdv_items) when max_slots allows, otherwise a column longer than
// about one CTA's share is cut into equal chunks (as few more as max_slots
// needs) and the items are packed longest first onto the least loaded CTA.
// Returns the grid (CTAs that have a list); *n_slots the partial-sum slots.
int pack_dkdv_items(const int* col_cnt, int nk, int g, int Hkv, int max_slots, int sms, bool exact_fill,
                    std::vector<DkdvItem>* packed_out, std::vector<int4>* splits_out, std::vector<int>* cta_out,
                    int* n_slots) {
  long long total = 0;
  for (int j = 0; j < nk; ++j) total += (long long)g * col_cnt[j] * Hkv;
  long long cap = std::max<long long>(4, (total + sms - 1) / std::max(sms, 1));
  auto slots_for = [&](long long c) {
    long long n_slots = 0;
    for (int j = 0; j < nk; ++j) {
      const long long n = (long long)g * col_cnt[j];
      const long long nch = (n + c - 1) / c;
      if (nch > 1) n_slots += nch * Hkv;
    }
    return n_slots;
  };
  if (max_slots <= 0)
    cap = LLONG_MAX / 4;
  else
    while (slots_for(cap) > max_slots) cap *= 2;
  std::vector<DkdvItem> packed;
  std::vector<int4> splits;
  int slot = 0, grid = 0;
  std::vector<int> cta;
  if (exact_fill && fill_dkdv_items(col_cnt, nk, g, Hkv, max_slots, sms, total, &packed, &splits, &cta, &slot)) {
    grid = (int)cta.size() - 1;
  } else {
    std::vector<DkdvItem> items;
    for (int j = 0; j < nk; ++j) {
      const int n = g * col_cnt[j];
      const int nch = n == 0 ? 1 : (int)((n + cap - 1) / cap);
      for (int hk = 0; hk < Hkv; ++hk) {
        if (nch <= 1) {
          items.push_back(DkdvItem{j, hk, 0, n, -1, 0, 0, 0});
        } else {
          splits.push_back(make_int4(j, hk, slot, nch));
          for (int c = 0; c < nch; ++c)
            items.push_back(DkdvItem{j, hk, (int)((long long)c * n / nch), (int)((long long)(c + 1) * n / nch), slot + c,
                                     0, 0, 0});
          slot += nch;
        }
      }
    }
    std::stable_sort(items.begin(), items.end(),
                     [](const DkdvItem& a, const DkdvItem& b) { return (a.x1 - a.x0) > (b.x1 - b.x0); });
    // LPT packing; an item costs its steps plus about two steps of fixed work
    // (the resident K/V tile and the epilogue).
    grid = std::min<int>(sms, std::max<int>((int)items.size(), 1));
    std::vector<std::vector<int>> bins(grid);
    {
      using Load = std::pair<long long, int>;
      std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
      for (int b = 0; b < grid; ++b) heap.push(Load(0, b));
      for (int i = 0; i < (int)items.size(); ++i) {
        Load l = heap.top();
        heap.pop();
        bins[l.second].push_back(i);
        l.first += (items[i].x1 - items[i].x0) + 2;
        heap.push(l);
      }
    }
    cta.assign(grid + 1, 0);
    packed.reserve(items.size());
    for (int b = 0; b < grid; ++b) {
      for (int i : bins[b]) packed.push_back(items[i]);
      cta[b + 1] = (int)packed.size();
    }
  }
  *packed_out = std::move(packed);
  *splits_out = std::move(splits);
  *cta_out = std::move(cta);
  *n_slots = slot;
  return grid;
}

int prepare_dkdv_items(const pt_blockmap* cbm, int g, int Hkv, int max_slots, int sms, bool exact_fill,
                       bool allow_build, cudaStream_t s, const pt_dkdv_lists** out) {
  pt_blockmap* bm = const_cast<pt_blockmap*>(cbm);  // the list cache is the map's only mutable part
  std::lock_guard<std::mutex> lk(g_items_mu);
  for (const pt_dkdv_lists* e = bm->dkdv_lists; e; e = e->next)
    if (e->g == g && e->hkv == Hkv && e->max_slots == max_slots && e->sms == sms && e->exact_fill == exact_fill) {
      *out = e;
      return 0;
    }
  if (!allow_build) {
    set_error("block map's backward work lists are not prepared for this head layout "
              "(call pt_blockmap_prepare_bwd first)");
    return 1;
  }
  const int *row_cnt = nullptr, *col_cnt = nullptr;
  if (int rc = rowcol_counts(bm, &row_cnt, &col_cnt)) return rc;
  const int nk = bm->nk;
  std::vector<DkdvItem> packed;
  std::vector<int4> splits;
  std::vector<int> cta;
  int slot = 0;
  const int grid = pack_dkdv_items(col_cnt, nk, g, Hkv, max_slots, sms, exact_fill, &packed, &splits, &cta, &slot);
  pt_dkdv_lists* e = new pt_dkdv_lists();
  const size_t bi = sizeof(DkdvItem) * std::max<size_t>(packed.size(), 1);
  const size_t bs = sizeof(int4) * std::max<size_t>(splits.size(), 1);
  const size_t bc = sizeof(int) * (grid + 1);
  int rc = pool_alloc(&e->mem, bi + bs + bc, bm->device, s);
  if (rc) {
    delete e;
    return rc;
  }
  e->items = e->mem;
  e->splits = static_cast<char*>(e->mem) + bi;
  e->cta = static_cast<char*>(e->mem) + bi + bs;
  {  // one upload in the device layout: items | splits | CTA index
    std::vector<char> host(bi + bs + bc, 0);
    if (!packed.empty()) std::memcpy(host.data(), packed.data(), sizeof(DkdvItem) * packed.size());
    if (!splits.empty()) std::memcpy(host.data() + bi, splits.data(), sizeof(int4) * splits.size());
    std::memcpy(host.data() + bi + bs, cta.data(), bc);
    if ((rc = upload(e->mem, host.data(), host.size(), bm->device, s))) {
      pool_free(e->mem, s);
      delete e;
      return rc;
    }
  }
  e->g = g;
  e->hkv = Hkv;
  e->max_slots = max_slots;
  e->sms = sms;
  e->exact_fill = exact_fill;
  e->n_items = (int)packed.size();
  e->grid = grid;
  e->n_splits = (int)splits.size();
  e->n_slots = slot;
  e->next = bm->dkdv_lists;
  bm->dkdv_lists = e;
  *out = e;
  return 0;
}

// dQ rows of the q tiles that attend to nothing are zero: one memset per run
// of consecutive such tiles (the list is ascending).
int zero_empty_dq(const pt_dq_lists* L, void* dQ, int T, int Hq, int D, cudaStream_t s) {
  for (int i = 0; i < L->n_empty;) {
    int e = i + 1;
    while (e < L->n_empty && L->h_empty[e] == L->h_empty[e - 1] + 1) ++e;
    const int t0 = L->h_empty[i] * 128, t1 = std::min(T, L->h_empty[e - 1] * 128 + 128);
    if (cudaMemsetAsync(static_cast<__nv_bfloat16*>(dQ) + (size_t)t0 * Hq * D, 0,
                        sizeof(__nv_bfloat16) * (size_t)(t1 - t0) * Hq * D, s) != cudaSuccess) {
      set_error("backward: cudaMemsetAsync failed");
      return 3;
    }
    i = e;
  }
  return 0;
}

// Work items of the pipelined q-major kernel, kept on the map per head count:
// every (q tile, head) with at least one kv block, packed longest first onto
// the grid's CTAs by LPT list scheduling and stored grouped by CTA, plus the
// q tiles with no kv block at all (their dQ rows are zero).
// Packs the q-major items (q tile, q head, first list entry, kv blocks) of a
// map whose q tiles have row_cnt[t] kv blocks listed (nq tiles) onto `sms`
// CTAs, longest first onto the least loaded CTA (about two blocks of fixed
// work per item); *cta_out: per CTA (first item, end item, kv blocks, 0);
// *empty_out: the q tiles with no kv block.  Returns the grid, or -1 with
// the error set if one CTA would get more than 2^31 - 1 kv blocks.
int pack_dq_items(const int* row_cnt, int nq, int Hq, int sms, std::vector<int4>* packed_out,
                  std::vector<int4>* cta_out, std::vector<int>* empty_out) {
  std::vector<int4> items;
  std::vector<int> empty;
  int e0 = 0;
  for (int t = 0; t < nq; ++t) {
    const int n = row_cnt[t];
    if (n == 0) empty.push_back(t);
    for (int h = 0; h < Hq && n > 0; ++h) items.push_back(make_int4(t, h, e0, n));
    e0 += n;
  }
  std::stable_sort(items.begin(), items.end(), [](const int4& a, const int4& b) { return a.w > b.w; });
  const int grid = std::max(1, std::min<int>(sms, (int)items.size()));
  std::vector<std::vector<int>> bins(grid);
  std::vector<long long> blocks(grid, 0);
  {
    using Load = std::pair<long long, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int b = 0; b < grid; ++b) heap.push(Load(0, b));
    for (int i = 0; i < (int)items.size(); ++i) {
      Load l = heap.top();
      heap.pop();
      bins[l.second].push_back(i);
      blocks[l.second] += items[i].w;
      l.first += items[i].w + 2;  // about two blocks of fixed work per item
      heap.push(l);
    }
  }
  std::vector<int4> packed, cta(grid);
  packed.reserve(items.size());
  for (int b = 0; b < grid; ++b) {
    cta[b].x = (int)packed.size();
    for (int i : bins[b]) packed.push_back(items[i]);
    cta[b].y = (int)packed.size();
    if (blocks[b] > INT32_MAX) {
      set_error("backward kernel: too many kv blocks for one CTA");
      return -1;
    }
    cta[b].z = (int)blocks[b];
    cta[b].w = 0;
  }
  *packed_out = std::move(packed);
  *cta_out = std::move(cta);
  *empty_out = std::move(empty);
  return grid;
}

int prepare_dq_items(const pt_blockmap* cbm, int Hq, int sms, bool allow_build, cudaStream_t s,
                     const pt_dq_lists** out) {
  pt_blockmap* bm = const_cast<pt_blockmap*>(cbm);  // the list cache is the map's only mutable part
  std::lock_guard<std::mutex> lk(g_items_mu);
  for (const pt_dq_lists* e = bm->dq_lists; e; e = e->next)
    if (e->hq == Hq && e->sms == sms) {
      *out = e;
      return 0;
    }
  if (!allow_build) {
    set_error("block map's dQ work lists are not prepared for this head count (call pt_blockmap_prepare_bwd first)");
    return 1;
  }
  const int *row_cnt = nullptr, *col_cnt = nullptr;
  if (int rc = rowcol_counts(bm, &row_cnt, &col_cnt)) return rc;
  const int nq = bm->nq;
  std::vector<int4> packed, cta;
  std::vector<int> empty;
  const int grid = pack_dq_items(row_cnt, nq, Hq, sms, &packed, &cta, &empty);
  if (grid < 0) return 1;
  pt_dq_lists* e = new pt_dq_lists();
  if (!empty.empty()) {
    e->h_empty = static_cast<int*>(std::malloc(sizeof(int) * empty.size()));
    if (!e->h_empty) {
      delete e;
      set_error("out of host memory");
      return 4;
    }
    std::copy(empty.begin(), empty.end(), e->h_empty);
  }
  const size_t bi = sizeof(int4) * std::max<size_t>(packed.size(), 1), bc = sizeof(int4) * grid;
  int rc = pool_alloc(&e->mem, bi + bc, bm->device, s);
  if (rc) {
    std::free(e->h_empty);
    delete e;
    return rc;
  }
  e->items = e->mem;
  e->cta = static_cast<char*>(e->mem) + bi;
  {  // one upload in the device layout: items | CTA records
    std::vector<char> host(bi + bc, 0);
    if (!packed.empty()) std::memcpy(host.data(), packed.data(), sizeof(int4) * packed.size());
    std::memcpy(host.data() + bi, cta.data(), bc);
    if ((rc = upload(e->mem, host.data(), host.size(), bm->device, s))) {
      pool_free(e->mem, s);
      std::free(e->h_empty);
      delete e;
      return rc;
    }
  }
  e->n_empty = (int)empty.size();
  e->hq = Hq;
  e->sms = sms;
  e->grid = grid;
  e->n_items = (int)packed.size();
  e->next = bm->dq_lists;
  bm->dq_lists = e;
  *out = e;
  return 0;
}

// The one-pass kernel's register split adds up to 128 per thread at launch:
// a build with another count would leave its setmaxnreg.inc waiting, so it
// is then not used (the two-pass kernels run instead).
bool fused_regs_ok(int dev) {
  static int state[64] = {0};  // 0 unknown, 1 usable, -1 not
  if (dev < 0 || dev >= 64) return false;
  if (!state[dev]) {
    cudaFuncAttributes fa{};
    state[dev] = (cudaFuncGetAttributes(&fa, k_bwd_fused) == cudaSuccess && fa.numRegs == FusedL::REG_LAUNCH &&
                  fa.maxThreadsPerBlock >= FusedL::THREADS)
                     ? 1
                     : -1;
  }
  return state[dev] == 1;
}

template <int D>
int launch_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
               int Hq, int Hkv, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
               float* lse2, float* partial, size_t partial_bytes, bool allow_build, cudaStream_t s) {
  static int set_dkdv[64] = {0}, set_dq[64] = {0}, set_fused[64] = {0};
  const int dev = bm->device;
  const int Tpad = bm->nq * 128;
  // head_dim 64 with room in the workspace for an fp32 dQ accumulator: the
  // one-pass kernel (dQ summed in an order that varies between runs); else
  // the kv-major and q-major kernels, each output element written once
  float* dq_acc = nullptr;
  if constexpr (D == 64) {
    const size_t dq_bytes = sizeof(float) * (size_t)Tpad * Hq * D;
    if (partial && partial_bytes >= dq_bytes && fused_regs_ok(dev)) {
      dq_acc = partial;
      partial = reinterpret_cast<float*>(reinterpret_cast<char*>(partial) + dq_bytes);
      partial_bytes -= dq_bytes;
    }
  }
  int rc = dq_acc ? reserve_smem(k_bwd_fused, FusedL::BYTES, dev, set_fused)
                  : reserve_smem(k_bwd_dkdv<D>, DkdvL<D>::BYTES, dev, set_dkdv);
  if (!rc && !dq_acc) {
    if constexpr (D == 128)
      rc = reserve_smem(k_bwd_dq_pipe<D>, DqpL<D>::BYTES, dev, set_dq);
    else
      rc = reserve_smem(k_bwd_dq<D>, DqL<D>::BYTES, dev, set_dq);
  }
  if (rc) return rc;
  if (masks_missing(bm)) {
    set_error("backward kernel: block map has no tile masks");
    return 1;
  }
  const int sms = num_sms(dev);
  const int max_slots = partial ? (int)std::min<size_t>(partial_bytes / (sizeof(float) * 128 * 2 * D), 1 << 20) : 0;
  const pt_dkdv_lists* KL = nullptr;
  // the one-pass kernel's fixed work per item is small enough that cutting
  // columns exactly at each CTA's share pays; the kv-major kernels of the
  // two-pass backward keep the longest-first packing
  if ((rc = prepare_dkdv_items(bm, Hq / Hkv, Hkv, max_slots, sms, dq_acc != nullptr, allow_build, s, &KL))) return rc;
  const pt_dq_lists* QL = nullptr;
  if (D == 128 && (rc = prepare_dq_items(bm, Hq, sms, allow_build, s, &QL))) return rc;
  {
    const size_t sm = sizeof(float) * kPrepTokens * ((size_t)Hq + 1);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(k_bwd_prep<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess) {
      set_error("backward preprocess: %d heads need %zu bytes of shared memory", Hq, sm);
      return 3;
    }
    ProfScope ps(s, "bwd_prep");
    launch_pdl(k_bwd_prep<D>, dim3((unsigned)(Tpad / kPrepTokens)), dim3(256), sm, s, static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), LSE, T, Tpad, Hq, delta, lse2, reinterpret_cast<float4*>(dq_acc));
  }
  CUtensorMap mQ, mdO, mK, mV, mdQ;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mdO, dO, T, Hq, D, 128) ||
      !make_tmap_thd(&mK, K, T, Hkv, D, 128) || !make_tmap_thd(&mV, V, T, Hkv, D, 128) ||
      !make_tmap_thd(&mdQ, dQ, T, Hq, D, 128))
    return 3;
  BwdParams p{};
  p.ndelta = delta;
  p.nlse2 = lse2;
  p.T = T;
  p.Tpad = Tpad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  // dK, dV
  p.ptr = bm->k_ptr;
  p.idx = bm->q_idx;
  p.pidx = bm->pidxT;
  p.order = bm->k_order;
  p.masks = bm->mask_cols;
  p.out0 = static_cast<__nv_bfloat16*>(dK);
  p.out1 = static_cast<__nv_bfloat16*>(dV);
  p.n_major = bm->nk;
  p.items = static_cast<const DkdvItem*>(KL->items);
  p.n_items = KL->n_items;
  p.cta_ptr = static_cast<const int*>(KL->cta);
  p.partial = partial;
  p.dq_acc = dq_acc;
  int launches = 1;
  if (p.n_items > 0) {
    if (dq_acc) {
      CUtensorMap mAcc;
      if (!make_tmap_acc32(&mAcc, dq_acc, Tpad, Hq)) return 3;
      ProfScope ps(s, "bwd_fused");
      launch_pdl(k_bwd_fused, dim3(KL->grid), dim3(FusedL::THREADS), FusedL::BYTES, s, mQ, mdO, mK, mV, mAcc, p);
    } else {
      ProfScope ps(s, "bwd_dkdv");
      launch_pdl(k_bwd_dkdv<D>, dim3(KL->grid), dim3(BwdCfg<D>::THREADS), DkdvL<D>::BYTES, s, mQ, mdO, mK, mV, p);
    }
    ++launches;
  }
  if (dq_acc) {  // split columns and dQ in one launch
    const size_t n8 = (size_t)T * Hq * D / 8;
    const unsigned blocks = (unsigned)std::min<size_t>((n8 + 255) / 256, (size_t)sms * 8) + 16u * KL->n_splits;
    ProfScope ps(s, "bwd_fused_finalize");
    launch_pdl(k_fused_finalize, dim3(blocks), dim3(256), 0, s, static_cast<const int4*>(KL->splits), KL->n_splits,
               (const float*)partial, T, Hkv, static_cast<__nv_bfloat16*>(dK), static_cast<__nv_bfloat16*>(dV),
               reinterpret_cast<const float4*>(dq_acc), n8, scale, static_cast<uint4*>(dQ));
    count_launch(launches + 1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("backward launch failed: %s", cudaGetErrorString(e));
      return 3;
    }
    return 0;
  }
  if (KL->n_splits > 0) {
    ProfScope ps(s, "bwd_dkdv_finalize");
    launch_pdl(k_dkdv_finalize<D>, dim3(dim3(KL->n_splits, 16)), dim3(256), 0, s, static_cast<const int4*>(KL->splits), partial, T, Hkv, static_cast<__nv_bfloat16*>(dK), static_cast<__nv_bfloat16*>(dV));
    ++launches;
  }
  // dQ
  p.ptr = bm->q_ptr;
  p.idx = bm->kv_idx;
  p.pidx = bm->pidx;
  p.order = bm->q_order;
  p.masks = bm->mask_rows;
  p.out0 = static_cast<__nv_bfloat16*>(dQ);
  p.out1 = nullptr;
  p.n_major = bm->nq;
  p.items = nullptr;
  p.cta_ptr = nullptr;
  p.partial = nullptr;
  const int items = bm->nq * Hq;
  if (items > 0) {
    ProfScope ps(s, "bwd_dq");
    if constexpr (D == 128) {
      if ((rc = zero_empty_dq(QL, dQ, T, Hq, D, s))) return rc;
      p.dq_items = static_cast<const int4*>(QL->items);
      p.dq_cta = static_cast<const int4*>(QL->cta);
      if (QL->n_items > 0)
        launch_pdl(k_bwd_dq_pipe<D>, dim3(QL->grid), dim3(DqpCfg<D>::THREADS), DqpL<D>::BYTES, s, mQ, mdO, mK, mV, p);
    } else {
      launch_pdl(k_bwd_dq<D>, dim3(items < sms ? items : sms), dim3(BwdCfg<D>::THREADS), DqL<D>::BYTES, s, mQ, mdO, mK, mV, mdQ, p);
    }
    ++launches;
  }
  count_launch(launches);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("backward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

// head_dim 256: preprocess, then the dV, dK and dQ passes of k_bwd_wide.
int launch_bwd_wide(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
                    int Hq, int Hkv, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
                    float* lse2, float* partial, size_t partial_bytes, bool allow_build, cudaStream_t s) {
  constexpr int D = 256;
  static int set_v[64] = {0}, set_k[64] = {0}, set_q[64] = {0};
  const int dev = bm->device;
  int rc = reserve_smem(k_bwd_wide<WIDE_DV>, WideCfg<WIDE_DV>::BYTES, dev, set_v);
  if (!rc) rc = reserve_smem(k_bwd_wide<WIDE_DK>, WideCfg<WIDE_DK>::BYTES, dev, set_k);
  if (!rc) rc = reserve_smem(k_bwd_wide<WIDE_DQ>, WideCfg<WIDE_DQ>::BYTES, dev, set_q);
  if (rc) return rc;
  if (masks_missing(bm)) {
    set_error("backward kernel: block map has no tile masks");
    return 1;
  }
  const int sms = num_sms(dev);
  // kv-major items: long columns cut into chunks that write fp32 partial sums
  // (slots of 128 x 2D floats, of which each pass fills its D columns), when
  // the caller's workspace has room for them; the finalize kernel sums them
  const int max_slots = partial ? (int)std::min<size_t>(partial_bytes / (sizeof(float) * 128 * 2 * D), 1 << 20) : 0;
  const pt_dkdv_lists* KL = nullptr;
  const pt_dq_lists* QL = nullptr;
  if ((rc = prepare_dkdv_items(bm, Hq / Hkv, Hkv, max_slots, sms, false, allow_build, s, &KL))) return rc;
  if ((rc = prepare_dq_items(bm, Hq, sms, allow_build, s, &QL))) return rc;
  const int Tpad = bm->nq * 128;
  {
    const size_t sm = sizeof(float) * kPrepTokens * ((size_t)Hq + 1);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(k_bwd_prep<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess) {
      set_error("backward preprocess: %d heads need %zu bytes of shared memory", Hq, sm);
      return 3;
    }
    ProfScope ps(s, "bwd_prep");
    launch_pdl(k_bwd_prep<D>, dim3((unsigned)(Tpad / kPrepTokens)), dim3(256), sm, s, static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), LSE, T, Tpad, Hq, delta, lse2, static_cast<float4*>(nullptr));
  }
  CUtensorMap mQ, mdO, mK, mV, mQh, mdOh, mKh, mVh;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mdO, dO, T, Hq, D, 128) ||
      !make_tmap_thd(&mK, K, T, Hkv, D, 128) || !make_tmap_thd(&mV, V, T, Hkv, D, 128) ||
      !make_tmap_thd(&mQh, Q, T, Hq, D, 64) || !make_tmap_thd(&mdOh, dO, T, Hq, D, 64) ||
      !make_tmap_thd(&mKh, K, T, Hkv, D, 64) || !make_tmap_thd(&mVh, V, T, Hkv, D, 64))
    return 3;
  BwdParams p{};
  p.ndelta = delta;
  p.nlse2 = lse2;
  p.T = T;
  p.Tpad = Tpad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  int launches = 1;
  // dV and dK: kv-major lists and column masks
  p.ptr = bm->k_ptr;
  p.idx = bm->q_idx;
  p.pidx = bm->pidxT;
  p.masks = bm->mask_cols;
  p.items = static_cast<const DkdvItem*>(KL->items);
  p.cta_ptr = static_cast<const int*>(KL->cta);
  p.n_items = KL->n_items;
  p.out0 = static_cast<__nv_bfloat16*>(dK);
  p.out1 = static_cast<__nv_bfloat16*>(dV);
  p.partial = partial;
  if (p.n_items > 0) {
    const int4* splits = static_cast<const int4*>(KL->splits);
    {
      ProfScope ps(s, "bwd_dv");
      launch_pdl(k_bwd_wide<WIDE_DV>, dim3(KL->grid), dim3(320), WideCfg<WIDE_DV>::BYTES, s, mK, mK, mdOh, mQh, p);
    }
    if (KL->n_splits > 0) {
      ProfScope ps(s, "bwd_dkdv_finalize");
      launch_pdl(k_split_finalize<D>, dim3(KL->n_splits, 16), dim3(256), 0, s, splits, (const float*)partial, 2 * D, T,
                 Hkv, D, 0, static_cast<__nv_bfloat16*>(dV));
      ++launches;
    }
    {
      ProfScope ps(s, "bwd_dk");
      launch_pdl(k_bwd_wide<WIDE_DK>, dim3(KL->grid), dim3(320), WideCfg<WIDE_DK>::BYTES, s, mK, mV, mQh, mdOh, p);
    }
    if (KL->n_splits > 0) {
      ProfScope ps(s, "bwd_dkdv_finalize");
      launch_pdl(k_split_finalize<D>, dim3(KL->n_splits, 16), dim3(256), 0, s, splits, (const float*)partial, 2 * D, T,
                 Hkv, D, 0, static_cast<__nv_bfloat16*>(dK));
      ++launches;
    }
    launches += 2;
  }
  // dQ: q-major lists and row masks
  p.idx = bm->kv_idx;
  p.pidx = bm->pidx;
  p.masks = bm->mask_rows;
  p.items = nullptr;
  p.cta_ptr = nullptr;
  p.dq_items = static_cast<const int4*>(QL->items);
  p.dq_cta = static_cast<const int4*>(QL->cta);
  p.out0 = static_cast<__nv_bfloat16*>(dQ);
  p.out1 = nullptr;
  if ((rc = zero_empty_dq(QL, dQ, T, Hq, D, s))) return rc;
  if (QL->n_items > 0) {
    ProfScope ps(s, "bwd_dq");
    launch_pdl(k_bwd_wide<WIDE_DQ>, dim3(QL->grid), dim3(320), WideCfg<WIDE_DQ>::BYTES, s, mQ, mdO, mKh, mVh, p);
    ++launches;
  }
  count_launch(launches);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("backward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}


// head_dim 512: preprocess, then the dV, dK and dQ passes of k_bwd_d512, one
// per half of each output.
int launch_bwd_d512(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
                    int Hq, int Hkv, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
                    float* lse2, float* partial, size_t partial_bytes, bool allow_build, cudaStream_t s) {
  constexpr int D = 512;
  using C = Bwd512Cfg;
  static int set_v[64] = {0}, set_k[64] = {0}, set_q[64] = {0};
  const int dev = bm->device;
  int rc = reserve_smem(k_bwd_d512<D512_DV>, C::BYTES, dev, set_v);
  if (!rc) rc = reserve_smem(k_bwd_d512<D512_DK>, C::BYTES, dev, set_k);
  if (!rc) rc = reserve_smem(k_bwd_d512<D512_DQ>, C::BYTES, dev, set_q);
  if (rc) return rc;
  if (masks_missing(bm)) {
    set_error("backward kernel: block map has no tile masks");
    return 1;
  }
  const int sms = num_sms(dev);
  // kv-major items: long columns cut into chunks that write fp32 partial sums
  // of the pass's 256 columns (slots of 128 x 2D floats) when the workspace
  // has room; the finalize kernel sums them after each pass
  const int max_slots = partial ? (int)std::min<size_t>(partial_bytes / (sizeof(float) * 128 * 2 * D), 1 << 20) : 0;
  const pt_dkdv_lists* KL = nullptr;
  const pt_dq_lists* QL = nullptr;
  if ((rc = prepare_dkdv_items(bm, Hq / Hkv, Hkv, max_slots, sms, false, allow_build, s, &KL))) return rc;
  if ((rc = prepare_dq_items(bm, Hq, sms, allow_build, s, &QL))) return rc;
  const int Tpad = bm->nq * 128;
  {
    const size_t sm = sizeof(float) * kPrepTokens * ((size_t)Hq + 1);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(k_bwd_prep<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess) {
      set_error("backward preprocess: %d heads need %zu bytes of shared memory", Hq, sm);
      return 3;
    }
    ProfScope ps(s, "bwd_prep");
    launch_pdl(k_bwd_prep<D>, dim3((unsigned)(Tpad / kPrepTokens)), dim3(256), sm, s,
               static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), LSE, T, Tpad, Hq, delta,
               lse2, static_cast<float4*>(nullptr));
  }
  CUtensorMap mQ, mK, mV, mdO;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mK, K, T, Hkv, D, 128) ||
      !make_tmap_thd(&mV, V, T, Hkv, D, 128) || !make_tmap_thd(&mdO, dO, T, Hq, D, 128))
    return 3;
  BwdParams p{};
  p.ndelta = delta;
  p.nlse2 = lse2;
  p.T = T;
  p.Tpad = Tpad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  int launches = 1;
  // dV and dK: kv-major lists and column masks
  p.ptr = bm->k_ptr;
  p.idx = bm->q_idx;
  p.pidx = bm->pidxT;
  p.masks = bm->mask_cols;
  p.items = static_cast<const DkdvItem*>(KL->items);
  p.cta_ptr = static_cast<const int*>(KL->cta);
  p.n_items = KL->n_items;
  p.out0 = static_cast<__nv_bfloat16*>(dK);
  p.out1 = static_cast<__nv_bfloat16*>(dV);
  p.partial = partial;
  if (p.n_items > 0) {
    const int4* splits = static_cast<const int4*>(KL->splits);
    for (int m = 0; m < 2; ++m)
      for (int h = 0; h < 2; ++h) {
        p.half = h;
        {
          ProfScope ps(s, m == 0 ? "bwd_dv" : "bwd_dk");
          if (m == 0)
            launch_pdl(k_bwd_d512<D512_DV>, dim3(KL->grid), dim3(C::THREADS), C::BYTES, s, mQ, mK, mV, mdO, p);
          else
            launch_pdl(k_bwd_d512<D512_DK>, dim3(KL->grid), dim3(C::THREADS), C::BYTES, s, mQ, mK, mV, mdO, p);
        }
        ++launches;
        if (KL->n_splits > 0) {
          ProfScope ps(s, "bwd_dkdv_finalize");
          launch_pdl(k_split_finalize<256>, dim3(KL->n_splits, 16), dim3(256), 0, s, splits, (const float*)partial,
                     2 * D, T, Hkv, D, 256 * h, static_cast<__nv_bfloat16*>(m == 0 ? dV : dK));
          ++launches;
        }
      }
  }
  // dQ: q-major lists and row masks
  p.ptr = bm->q_ptr;
  p.idx = bm->kv_idx;
  p.pidx = bm->pidx;
  p.masks = bm->mask_rows;
  p.items = nullptr;
  p.cta_ptr = nullptr;
  p.dq_items = static_cast<const int4*>(QL->items);
  p.dq_cta = static_cast<const int4*>(QL->cta);
  p.out0 = static_cast<__nv_bfloat16*>(dQ);
  p.out1 = nullptr;
  if ((rc = zero_empty_dq(QL, dQ, T, Hq, D, s))) return rc;
  if (QL->n_items > 0) {
    for (int h = 0; h < 2; ++h) {
      p.half = h;
      ProfScope ps(s, "bwd_dq");
      launch_pdl(k_bwd_d512<D512_DQ>, dim3(QL->grid), dim3(C::THREADS), C::BYTES, s, mQ, mK, mV, mdO, p);
    }
    launches += 2;
  }
  count_launch(launches);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("backward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}
}  // namespace

int debug_pack_dq(const int* row_cnt, int nq, int Hq, int ctas, int32_t* items, long long cap_items, int32_t* cta_rec,
                  int32_t* n_items, int32_t* grid, int32_t* n_empty) {
  std::vector<int4> packed, cta;
  std::vector<int> empty;
  const int gr = pack_dq_items(row_cnt, nq, Hq, ctas, &packed, &cta, &empty);
  if (gr < 0) return 1;
  *n_items = (int32_t)packed.size();
  *grid = gr;
  *n_empty = (int32_t)empty.size();
  if ((long long)packed.size() > cap_items) {
    set_error("pt_debug_pack_dq: %zu items, room for %lld", packed.size(), cap_items);
    return 1;
  }
  for (size_t k = 0; k < packed.size(); ++k) {
    const int32_t v[4] = {packed[k].x, packed[k].y, packed[k].z, packed[k].w};
    std::memcpy(items + 4 * k, v, sizeof(v));
  }
  for (int b = 0; b < gr; ++b) {
    const int32_t v[4] = {cta[b].x, cta[b].y, cta[b].z, cta[b].w};
    std::memcpy(cta_rec + 4 * b, v, sizeof(v));
  }
  return 0;
}

int debug_pack_dkdv(const int* col_cnt, int nk, int g, int Hkv, int max_slots, int ctas, bool exact_fill, int32_t* items,
                    long long cap_items, int32_t* cta_ptr, int32_t* n_items, int32_t* n_slots, int32_t* grid) {
  std::vector<DkdvItem> packed;
  std::vector<int4> splits;
  std::vector<int> cta;
  int slots = 0;
  const int gr = pack_dkdv_items(col_cnt, nk, g, Hkv, max_slots, ctas, exact_fill, &packed, &splits, &cta, &slots);
  *n_items = (int32_t)packed.size();
  *n_slots = slots;
  *grid = gr;
  if ((long long)packed.size() > cap_items) {
    set_error("pt_debug_pack_dkdv: %zu items, room for %lld", packed.size(), cap_items);
    return 1;
  }
  for (size_t k = 0; k < packed.size(); ++k) {
    const DkdvItem& it = packed[k];
    const int32_t v[5] = {it.jb, it.hk, it.x0, it.x1, it.slot};
    std::memcpy(items + 5 * k, v, sizeof(v));
  }
  for (int b = 0; b <= gr; ++b) cta_ptr[b] = cta[b];
  return 0;
}

bool bwd_tc_supported(int D) { return D == 64 || D == 128 || D == 256 || D == 512; }

int prepare_bwd_noalloc(const pt_blockmap* bm, int Hq, int Hkv, int D, cudaStream_t s) {
  if (!bwd_tc_supported(D) || bm->BM != 128 || bm->BN != 128) return 0;  // those paths keep no lists
  const int sms = num_sms(bm->device);
  const pt_dkdv_lists* KL = nullptr;
  const pt_dq_lists* QL = nullptr;
  int rc = prepare_dkdv_items(bm, Hq / Hkv, Hkv, 0, sms, false, true, s, &KL);
  if (!rc && D >= 128) rc = prepare_dq_items(bm, Hq, sms, true, s, &QL);
  return rc;
}

int bwd_tc(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T, int Hq,
           int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta, float* lse2,
           float* partial, size_t partial_bytes, bool allow_build, cudaStream_t s) {
  switch (D) {
    case 64:
      return launch_bwd<64>(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, partial,
                            partial_bytes, allow_build, s);
    case 128:
      return launch_bwd<128>(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, partial,
                             partial_bytes, allow_build, s);
    case 256:
      return launch_bwd_wide(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, partial, partial_bytes,
                             allow_build, s);
    case 512:
      return launch_bwd_d512(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, partial, partial_bytes,
                             allow_build, s);
    default: set_error("tensor-core backward: head_dim %d not built", D); return 2;
  }
}

}  // namespace pt
