// pt_bwd_tc.cu -- tensor-core backward for bf16: dQ, dK, dV over the kept pairs.
//
// The backward of the block-sparse attention of "prefix_grouper_kernel.py"
// (the compiled FlexAttention backward it pads for) and of the drafter
// speed-up PR's GQA backward: with P = exp(s - LSE), Delta = rowsum(dO * O),
// dS = P * (dO V^T - Delta):  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,
// dK and dV summed over the q heads that share a kv head (native GQA: K and
// V are never repeated).  Empty tiles are skipped, partial tiles masked.
//
// Three launches, all on the caller's stream:
//  1. k_bwd_prep   (HBM-bound) Delta = rowsum(dO * O) and LSE * log2(e) into
//                  the workspace, [Hq, Tpad] each, Tpad = ceil(T/128)*128,
//                  padding rows set so they contribute nothing.
//  2. k_bwd_dkdv   persistent, kv-major: a work item is (kv block, kv head);
//                  K and V stay in shared memory while the q tiles of the
//                  block's column list stream through for each q head of the
//                  group.  Per step: S^T = K Q^T and dP^T = V dO^T into TMEM
//                  (kv rows in lanes); the compute warpgroup writes P^T and
//                  dS^T back over them as bf16; then dV += P^T dO and
//                  dK += dS^T Q read those operands straight from TMEM.
//  3. k_bwd_dq     persistent, q-major: a work item is (q tile, q head); Q and
//                  dO stay resident while the kv blocks of the tile's list
//                  stream through.  S = Q K^T, dP = dO V^T, dS into TMEM, then
//                  dQ += dS K.
// No atomics: every output element is written once, so results are
// deterministic.  TMEM per CTA: 512 columns (S 128, dP 128, accumulators).
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_bwd(cudaStream_t s) { return take_status_here(s); }

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
// One group of D/8 threads per (row, head): 16-byte loads of dO and O.
template <int D>
__global__ void k_bwd_prep(const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ O,
                           const float* __restrict__ LSE, int T, int Tpad, int Hq, float* __restrict__ delta,
                           float* __restrict__ lse2) {
  constexpr int TPR = D / 8;  // threads per row
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid / TPR;  // over Hq * Tpad, head-major
  const int sub = (int)(gid % TPR);
  if (row >= (long long)Hq * Tpad) return;
  const int h = (int)(row / Tpad), q = (int)(row % Tpad);
  float s = 0.f;
  if (q < T) {
    const uint4 a = *reinterpret_cast<const uint4*>(dO + ((size_t)q * Hq + h) * D + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(O + ((size_t)q * Hq + h) * D + sub * 8);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 x = __bfloat1622float2(pa[k]), y = __bfloat1622float2(pb[k]);
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
    }
  }
#pragma unroll
  for (int o = TPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, TPR);
  if (sub == 0) {
    delta[row] = s;
    float l = q < T ? LSE[(size_t)h * T + q] : -INFINITY;
    // rows that keep nothing (padding) get +inf so exp2(s - lse2) = 0
    lse2[row] = (l == -INFINITY) ? INFINITY : l * kLog2e;
  }
}

// ---------------------------------------------------------------------------
// shared configuration
// ---------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  static constexpr int NP = D / 64;
  static constexpr int PANEL = 128 * 128;
  static constexpr int TILE = NP * PANEL;
  static constexpr int STAGES = D == 64 ? 3 : 2;
  static constexpr int TM_S = 0, TM_DP = 128, TM_A0 = 256, TM_A1 = 256 + D;  // A0/A1: accumulators
  static_assert(TM_A1 + D <= 512 || D > 128, "TMEM budget");
};

struct BwdParams {
  const int* ptr;    // k_ptr (dkdv) or q_ptr (dq)
  const int* idx;    // q_idx or kv_idx
  const uint8_t* kind;
  const int* order;  // k_order or q_order
  const pt_tok* tok;
  const float* delta;  // [Hq, Tpad]
  const float* lse2;   // [Hq, Tpad]
  __nv_bfloat16* out0;  // dK (dkdv) or dQ (dq)
  __nv_bfloat16* out1;  // dV (dkdv)
  int T, Tpad, Hq, Hkv, n_major;
  float scale, scale_log2;
};

// P^T / dS^T (or dS) for 64 columns: pack pairs to bf16x2.
__device__ __forceinline__ void pack64(const uint32_t* v, uint32_t* out) {
#pragma unroll
  for (int c = 0; c < 32; ++c) out[c] = pack_bf16(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
}

// ---------------------------------------------------------------------------
// 2. dK / dV, kv-major
// ---------------------------------------------------------------------------
template <int D>
struct DkdvSmem {
  using C = BwdCfg<D>;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + C::TILE;
  static constexpr int OFF_ST = OFF_V + C::TILE;  // stages: Q | dO | lse2 | delta | tok
  static constexpr int ST_Q = 0, ST_DO = C::TILE, ST_L = 2 * C::TILE, ST_D = ST_L + 512, ST_T = ST_D + 512;
  static constexpr int ST_BYTES = ST_T + 1024;
  static constexpr int OFF_BAR = OFF_ST + C::STAGES * ST_BYTES;
  // kv_full kv_empty st_full[S] st_empty[S] s_full p_full acc_full acc_free mma_done
  static constexpr int NBAR = 2 + 2 * C::STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    k_bwd_dkdv(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
               const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, const BwdParams p) {
  using C = BwdCfg<D>;
  using L = DkdvSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 1;
  uint64_t* st_full = bars + 2;
  uint64_t* st_empty = st_full + C::STAGES;
  uint64_t* s_full = st_empty + C::STAGES;
  uint64_t* p_full = s_full + 1;
  uint64_t* acc_full = p_full + 1;
  uint64_t* acc_free = acc_full + 1;
  uint64_t* mma_done = acc_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int n_items = p.n_major * p.Hkv;

  if (threadIdx.x == 128) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(st_full + s, 1);
      mbar_init(st_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int jb = p.order[w / p.Hkv], hk = w % p.Hkv;
        const int e0 = p.ptr[jb], ncol = p.ptr[jb + 1] - e0;
        if (ncol == 0) continue;
        if (it > 0 && !(ok = mbar_wait(kv_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn) {
          tma_load_3d(smem + L::OFF_K + pn * C::PANEL, &mK, kv_full, pn * 64, hk, jb * 128);
          tma_load_3d(smem + L::OFF_V + pn * C::PANEL, &mV, kv_full, pn * 64, hk, jb * 128);
        }
        const int n = g * ncol;
        for (int x = 0; x < n; ++x) {
          const int h = hk * g + x / ncol, i = p.idx[e0 + x % ncol];
          const uint32_t s = sc % C::STAGES, u = sc / C::STAGES;
          if (u > 0 && !(ok = mbar_wait(st_empty + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
          mbar_expect_tx(st_full + s, 2 * C::TILE + 2048);
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn) {
            tma_load_3d(st + L::ST_Q + pn * C::PANEL, &mQ, st_full + s, pn * 64, h, i * 128);
            tma_load_3d(st + L::ST_DO + pn * C::PANEL, &mdO, st_full + s, pn * 64, h, i * 128);
          }
          bulk_load(st + L::ST_L, p.lse2 + (size_t)h * p.Tpad + i * 128, 512, st_full + s);
          bulk_load(st + L::ST_D, p.delta + (size_t)h * p.Tpad + i * 128, 512, st_full + s);
          bulk_load(st + L::ST_T, p.tok + (size_t)i * 128, 1024, st_full + s);
          ++sc;
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        mbar_wait_drain(kv_full, (it)&1, lim);
        for (uint32_t s = 0; s < C::STAGES && s < sc; ++s) {
          uint32_t last = sc - 1 - ((sc - 1 - s) % C::STAGES);
          mbar_wait_drain(st_full + s, (last / C::STAGES) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);
      const uint32_t sK = smem_u32(smem + L::OFF_K), sV = smem_u32(smem + L::OFF_V);
      const uint32_t sST = smem_u32(smem + L::OFF_ST);
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int jb = p.order[w / p.Hkv];
        const int ncol = p.ptr[jb + 1] - p.ptr[jb];
        if (ncol == 0) continue;
        const int n = g * ncol;
        if (!(ok = mbar_wait(kv_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int x = 0; x < n; ++x) {
          const uint32_t y = sc + x, s = y % C::STAGES;
          if (!(ok = mbar_wait(st_full + s, (y / C::STAGES) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t sQ = sST + s * L::ST_BYTES + L::ST_Q, sdO = sST + s * L::ST_BYTES + L::ST_DO;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_S, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), IDESC_S, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_DP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdO + off, 16, 1024), IDESC_S,
                   kk > 0);
          }
          mma_commit(s_full);
          if (!(ok = mbar_wait(p_full, y & 1, abort_flag))) break;
          if (x == 0 && it > 0 && !(ok = mbar_wait(acc_free, (it - 1) & 1, abort_flag))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acc = (x > 0 || kk > 0);
            mma_ts(tbase + C::TM_A0, tbase + C::TM_S + kk * 8, sdesc_sw128(sdO + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, acc);  // dV += P^T dO
            mma_ts(tbase + C::TM_A1, tbase + C::TM_DP + kk * 8, sdesc_sw128(sQ + kk * 2048, C::PANEL, 1024),
                   IDESC_ACC, acc);  // dK += dS^T Q
          }
          mma_commit(st_empty + s);
          if (x == n - 1) {
            mma_commit(kv_empty);
            mma_commit(acc_full);
          }
        }
        sc += n;
        ++it;
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute (kv row per thread)
    const int r = threadIdx.x;
    const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const int jb = p.order[w / p.Hkv], hk = w % p.Hkv;
      const int e0 = p.ptr[jb], ncol = p.ptr[jb + 1] - e0;
      const int kv = jb * 128 + r;
      if (ncol == 0) {
        if (kv < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          uint4* a = reinterpret_cast<uint4*>(p.out0 + ((size_t)kv * p.Hkv + hk) * D);
          uint4* b = reinterpret_cast<uint4*>(p.out1 + ((size_t)kv * p.Hkv + hk) * D);
          for (int c = 0; c < D / 8; ++c) a[c] = b[c] = z;
        }
        continue;
      }
      const pt_tok ktok = p.tok[kv];
      const int n = g * ncol;
      for (int x = 0; x < n; ++x) {
        const int e = e0 + x % ncol;
        const int q0 = p.idx[e] * 128;
        const bool partial = p.kind[e] == PT_KIND_PARTIAL;
        const uint32_t y = sc + x, s = y % C::STAGES;
        ok = mbar_wait(s_full, y & 1, abort_flag) && mbar_wait(st_full + s, (y / C::STAGES) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
        const float* l2 = reinterpret_cast<const float*>(st + L::ST_L);
        const float* dl = reinterpret_cast<const float*>(st + L::ST_D);
        const pt_tok* qt = reinterpret_cast<const pt_tok*>(st + L::ST_T);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[64], dr[64];
          tmem_ld32(tl + C::TM_S + half * 64, sr);
          tmem_ld32(tl + C::TM_S + half * 64 + 32, sr + 32);
          tmem_ld32(tl + C::TM_DP + half * 64, dr);
          tmem_ld32(tl + C::TM_DP + half * 64 + 32, dr + 32);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int cc = half * 64 + c;
            float pr = ex2(fmaf(__uint_as_float(sr[c]), p.scale_log2, -l2[cc]));
            if (partial) {
              const int qtin = qt[cc].tin;
              const bool keep = (kv <= q0 + cc) && (ktok.tin <= qtin) && (qtin < ktok.tout);
              pr = keep ? pr : 0.f;
            }
            sr[c] = __float_as_uint(pr);
            dr[c] = __float_as_uint(pr * (__uint_as_float(dr[c]) - dl[cc]));
          }
          uint32_t pk[32];
          pack64(sr, pk);
          tmem_st32(tl + C::TM_S + half * 32, pk);
          pack64(dr, pk);
          tmem_st32(tl + C::TM_DP + half * 32, pk);
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
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        // which 0: dV (A0, no scale) -> out1; which 1: dK (A1, scale) -> out0
        const float mul = which ? p.scale : 1.f;
        __nv_bfloat16* orow = (which ? p.out0 : p.out1) + ((size_t)kv * p.Hkv + hk) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tl + (which ? C::TM_A1 : C::TM_A0) + c * 32, v);
          tmem_ld_wait();
          if (kv < p.T) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              pk[k] = pack_bf16(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);
      sc += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// 3. dQ, q-major
// ---------------------------------------------------------------------------
template <int D>
struct DqSmem {
  using C = BwdCfg<D>;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + C::TILE;
  static constexpr int OFF_ST = OFF_DO + C::TILE;  // stages: K | V | tok
  static constexpr int ST_K = 0, ST_V = C::TILE, ST_T = 2 * C::TILE;
  static constexpr int ST_BYTES = ST_T + 1024;
  static constexpr int OFF_BAR = OFF_ST + C::STAGES * ST_BYTES;
  // res_full res_empty st_full[S] st_empty[S] s_full p_full acc_full acc_free mma_done
  static constexpr int NBAR = 2 + 2 * C::STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    k_bwd_dq(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
             const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, const BwdParams p) {
  using C = BwdCfg<D>;
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* res_full = bars;
  uint64_t* res_empty = bars + 1;
  uint64_t* st_full = bars + 2;
  uint64_t* st_empty = st_full + C::STAGES;
  uint64_t* s_full = st_empty + C::STAGES;
  uint64_t* p_full = s_full + 1;
  uint64_t* acc_full = p_full + 1;
  uint64_t* acc_free = acc_full + 1;
  uint64_t* mma_done = acc_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int n_items = p.n_major * p.Hq;

  if (threadIdx.x == 128) {
    mbar_init(res_full, 1);
    mbar_init(res_empty, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(st_full + s, 1);
      mbar_init(st_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mdO);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      uint32_t sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.order[w / p.Hq], h = w % p.Hq, hk = h / g;
        const int e0 = p.ptr[tile], n = p.ptr[tile + 1] - e0;
        if (n == 0) continue;
        if (it > 0 && !(ok = mbar_wait(res_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(res_full, 2 * C::TILE);
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn) {
          tma_load_3d(smem + L::OFF_Q + pn * C::PANEL, &mQ, res_full, pn * 64, h, tile * 128);
          tma_load_3d(smem + L::OFF_DO + pn * C::PANEL, &mdO, res_full, pn * 64, h, tile * 128);
        }
        for (int x = 0; x < n; ++x) {
          const int j = p.idx[e0 + x];
          const uint32_t s = sc % C::STAGES, u = sc / C::STAGES;
          if (u > 0 && !(ok = mbar_wait(st_empty + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* st = smem + L::OFF_ST + s * L::ST_BYTES;
          mbar_expect_tx(st_full + s, 2 * C::TILE + 1024);
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn) {
            tma_load_3d(st + L::ST_K + pn * C::PANEL, &mK, st_full + s, pn * 64, hk, j * 128);
            tma_load_3d(st + L::ST_V + pn * C::PANEL, &mV, st_full + s, pn * 64, hk, j * 128);
          }
          bulk_load(st + L::ST_T, p.tok + (size_t)j * 128, 1024, st_full + s);
          ++sc;
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        mbar_wait_drain(res_full, (it)&1, lim);
        for (uint32_t s = 0; s < C::STAGES && s < sc; ++s) {
          uint32_t last = sc - 1 - ((sc - 1 - s) % C::STAGES);
          mbar_wait_drain(st_full + s, (last / C::STAGES) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
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
        if (!(ok = mbar_wait(res_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int x = 0; x < n; ++x) {
          const uint32_t y = sc + x, s = y % C::STAGES;
          if (!(ok = mbar_wait(st_full + s, (y / C::STAGES) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t sK = sST + s * L::ST_BYTES + L::ST_K, sV = sST + s * L::ST_BYTES + L::ST_V;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_S, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), IDESC_S, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
            mma_ss(tbase + C::TM_DP, sdesc_sw128(sdO + off, 16, 1024), sdesc_sw128(sV + off, 16, 1024), IDESC_S,
                   kk > 0);
          }
          mma_commit(s_full);
          if (!(ok = mbar_wait(p_full, y & 1, abort_flag))) break;
          if (x == 0 && it > 0 && !(ok = mbar_wait(acc_free, (it - 1) & 1, abort_flag))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tbase + C::TM_A0, tbase + C::TM_DP + kk * 8, sdesc_sw128(sK + kk * 2048, C::PANEL, 1024), IDESC_ACC,
                   (x > 0 || kk > 0));  // dQ += dS K
          mma_commit(st_empty + s);
          if (x == n - 1) {
            mma_commit(res_empty);
            mma_commit(acc_full);
          }
        }
        sc += n;
        ++it;
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    const int r = threadIdx.x;
    const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const int tile = p.order[w / p.Hq], h = w % p.Hq;
      const int e0 = p.ptr[tile], n = p.ptr[tile + 1] - e0;
      const int q = tile * 128 + r;
      if (n == 0) {
        if (q < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          uint4* a = reinterpret_cast<uint4*>(p.out0 + ((size_t)q * p.Hq + h) * D);
          for (int c = 0; c < D / 8; ++c) a[c] = z;
        }
        continue;
      }
      const float l2 = p.lse2[(size_t)h * p.Tpad + q];
      const float dl = p.delta[(size_t)h * p.Tpad + q];
      const int q_tin = p.tok[q].tin;
      for (int x = 0; x < n; ++x) {
        const int e = e0 + x;
        const int k0 = p.idx[e] * 128;
        const bool partial = p.kind[e] == PT_KIND_PARTIAL;
        const uint32_t y = sc + x, s = y % C::STAGES;
        ok = mbar_wait(s_full, y & 1, abort_flag) && mbar_wait(st_full + s, (y / C::STAGES) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const pt_tok* kt = reinterpret_cast<const pt_tok*>(smem + L::OFF_ST + s * L::ST_BYTES + L::ST_T);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[64], dr[64];
          tmem_ld32(tl + C::TM_S + half * 64, sr);
          tmem_ld32(tl + C::TM_S + half * 64 + 32, sr + 32);
          tmem_ld32(tl + C::TM_DP + half * 64, dr);
          tmem_ld32(tl + C::TM_DP + half * 64 + 32, dr + 32);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int cc = half * 64 + c;
            float pr = ex2(fmaf(__uint_as_float(sr[c]), p.scale_log2, -l2));
            if (partial) {
              const pt_tok t = kt[cc];
              const bool keep = (k0 + cc <= q) && (t.tin <= q_tin) && (q_tin < t.tout);
              pr = keep ? pr : 0.f;
            }
            dr[c] = __float_as_uint(pr * (__uint_as_float(dr[c]) - dl));
          }
          uint32_t pk[32];
          pack64(dr, pk);
          tmem_st32(tl + C::TM_DP + half * 32, pk);
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
      __nv_bfloat16* orow = p.out0 + ((size_t)q * p.Hq + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::TM_A0 + c * 32, v);
        tmem_ld_wait();
        if (q < p.T) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16(__uint_as_float(v[2 * k]) * p.scale, __uint_as_float(v[2 * k + 1]) * p.scale);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);
      sc += n;
      ++it;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tbase, 512);
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

template <int D>
int launch_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
               int Hq, int Hkv, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
               float* lse2, cudaStream_t s) {
  static int set_dkdv[64] = {0}, set_dq[64] = {0};
  const int dev = bm->device;
  int rc = reserve_smem(k_bwd_dkdv<D>, DkdvSmem<D>::BYTES, dev, set_dkdv);
  if (!rc) rc = reserve_smem(k_bwd_dq<D>, DqSmem<D>::BYTES, dev, set_dq);
  if (rc) return rc;
  const int Tpad = bm->nq * 128;
  {
    const long long threads = (long long)Hq * Tpad * (D / 8);
    ProfScope ps(s, "bwd_prep");
    k_bwd_prep<D><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), LSE, T, Tpad, Hq, delta, lse2);
  }
  CUtensorMap mQ, mdO, mK, mV;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mdO, dO, T, Hq, D, 128) ||
      !make_tmap_thd(&mK, K, T, Hkv, D, 128) || !make_tmap_thd(&mV, V, T, Hkv, D, 128))
    return 3;
  BwdParams p{};
  p.tok = bm->tok;
  p.delta = delta;
  p.lse2 = lse2;
  p.T = T;
  p.Tpad = Tpad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  const int sms = num_sms(dev);
  // dK, dV
  p.ptr = bm->k_ptr;
  p.idx = bm->q_idx;
  p.kind = bm->kindT;
  p.order = bm->k_order;
  p.out0 = static_cast<__nv_bfloat16*>(dK);
  p.out1 = static_cast<__nv_bfloat16*>(dV);
  p.n_major = bm->nk;
  int items = bm->nk * Hkv;
  if (items > 0) {
    ProfScope ps(s, "bwd_dkdv");
    k_bwd_dkdv<D><<<items < sms ? items : sms, 192, DkdvSmem<D>::BYTES, s>>>(mQ, mdO, mK, mV, p);
  }
  // dQ
  p.ptr = bm->q_ptr;
  p.idx = bm->kv_idx;
  p.kind = bm->kind;
  p.order = bm->q_order;
  p.out0 = static_cast<__nv_bfloat16*>(dQ);
  p.out1 = nullptr;
  p.n_major = bm->nq;
  items = bm->nq * Hq;
  if (items > 0) {
    ProfScope ps(s, "bwd_dq");
    k_bwd_dq<D><<<items < sms ? items : sms, 192, DqSmem<D>::BYTES, s>>>(mQ, mdO, mK, mV, p);
  }
  count_launch(3);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("backward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

}  // namespace

bool bwd_tc_supported(int D) { return D == 64 || D == 128; }

int bwd_tc(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T, int Hq,
           int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta, float* lse2,
           cudaStream_t s) {
  switch (D) {
    case 64: return launch_bwd<64>(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, s);
    case 128: return launch_bwd<128>(dO, Q, K, V, O, LSE, T, Hq, Hkv, scale, bm, dQ, dK, dV, delta, lse2, s);
    default: set_error("tensor-core backward: head_dim %d not built", D); return 2;
  }
}

}  // namespace pt
