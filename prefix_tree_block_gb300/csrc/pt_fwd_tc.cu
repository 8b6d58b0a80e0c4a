// pt_fwd_tc.cu -- tensor-core forward for bf16: O and LSE over the kept pairs.
//
// "prefix_grouper_kernel.py", flex_shared_prefix_attention and its block
// mask: exact softmax attention in which every (q tile, kv block) pair the
// block map lists as empty is skipped, full pairs run unmasked, and partial
// pairs apply the tree mask element by element.
//
// Design (sm_103a, one persistent CTA per SM, 192 threads):
//   warp 4      TMA producer: Q tile once per work item, then K and V tiles
//               of each listed kv block through separate multi-stage rings
//               (128-byte swizzled 64-column panels), plus the kv block's
//               per-token tree coordinates by 1-D bulk copy with V.
//   warp 5      MMA issuer (one lane): S = Q K^T into one of two TMEM
//               buffers (M = 128 q rows, N = 128 kv, K = D), then
//               O += P V with P read from TMEM (M = 128, N = D, K = 128).
//               S of block j+1 is issued before PV of block j so the tensor
//               pipe has work while the softmax runs.
//   warps 0-3   softmax: thread t owns q row t of the tile; it loads its S
//               row from TMEM, masks partial blocks in registers, keeps the
//               running max and sum (base-2, scale folded in), writes P as
//               bf16 back over its S columns, and rescales O in TMEM only
//               when the running max grows by more than 2^8 (the final
//               division by l makes any fixed reference exact).
// TMEM: S0 cols [0,128), S1 [128,256), O [256, 256+D).  D = 256 fills all 512.
// Every wait is bounded; a timeout raises a CTA abort flag, records
// PT_ERR_TIMEOUT, drains copies and MMAs in flight and frees TMEM.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_fwd(cudaStream_t s) { return take_status_here(s); }

namespace {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NP = D / 64;        // 64-column panels per row
  static constexpr int PANEL = 128 * 128;  // bytes: 128 rows x 128 B
  static constexpr int TILE = NP * PANEL;
  static constexpr int KS = D == 64 ? 4 : (D == 128 ? 3 : 1);
  static constexpr int VS = D == 64 ? 4 : (D == 128 ? 2 : 1);
  static constexpr int TOKB = BN * (int)sizeof(pt_tok);
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + KS * TILE;
  static constexpr int OFF_TOK = OFF_V + VS * TILE;
  static constexpr int OFF_BAR = OFF_TOK + VS * TOKB;
  // q_full q_empty k_full[KS] k_empty[KS] v_full[VS] v_empty[VS] s_full[2] p_full[2] o_full o_free mma_done
  static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 2 + 2 + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TM_S0 = 0, TM_S1 = 128, TM_O = 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TM_O + D <= 512, "TMEM budget");
};

struct FwdParams {
  const int* q_ptr;
  const int* kv_idx;
  const uint8_t* kind;
  const int* q_order;
  const pt_tok* tok;
  __nv_bfloat16* O;
  float* LSE;
  int T, Hq, Hkv, nq;
  float scale_log2;  // softmax scale * log2(e)
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

template <int D>
__global__ void __launch_bounds__(192, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
             const __grid_constant__ CUtensorMap mV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + C::KS;
  uint64_t* v_full = k_empty + C::KS;
  uint64_t* v_empty = v_full + C::VS;
  uint64_t* s_full = v_empty + C::VS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* o_free = o_full + 1;
  uint64_t* mma_done = o_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.Hq / p.Hkv;
  const int n_items = p.nq * p.Hq;

  if (threadIdx.x == 128) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
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
      uint32_t kc = 0, vc = 0, it = 0;
      bool ok = true, q_issued = false;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.q_order[w / p.Hq], h = w % p.Hq, hk = h / g;
        const int e0 = p.q_ptr[tile], e1 = p.q_ptr[tile + 1];
        if (e1 == e0) continue;
        if (it > 0 && !(ok = mbar_wait(q_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(q_full, C::TILE);
#pragma unroll
        for (int pn = 0; pn < C::NP; ++pn)
          tma_load_3d(smem + C::OFF_Q + pn * C::PANEL, &mQ, q_full, pn * 64, h, tile * C::BM);
        q_issued = true;
        for (int e = e0; e < e1; ++e) {
          const int j = p.kv_idx[e];
          {
            const uint32_t s = kc % C::KS, u = kc / C::KS;
            if (u > 0 && !(ok = mbar_wait(k_empty + s, (u - 1) & 1, abort_flag))) break;
            mbar_expect_tx(k_full + s, C::TILE);
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn)
              tma_load_3d(smem + C::OFF_K + s * C::TILE + pn * C::PANEL, &mK, k_full + s, pn * 64, hk, j * C::BN);
            ++kc;
          }
          {
            const uint32_t s = vc % C::VS, u = vc / C::VS;
            if (u > 0 && !(ok = mbar_wait(v_empty + s, (u - 1) & 1, abort_flag))) break;
            mbar_expect_tx(v_full + s, C::TILE + C::TOKB);
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn)
              tma_load_3d(smem + C::OFF_V + s * C::TILE + pn * C::PANEL, &mV, v_full + s, pn * 64, hk, j * C::BN);
            bulk_load(smem + C::OFF_TOK + s * C::TOKB, p.tok + (size_t)j * C::BN, C::TOKB, v_full + s);
            ++vc;
          }
        }
        ++it;
      }
      if (!ok) {
        // drain: wait (bounded) for the last copy issued into each slot
        const long long lim = 20000000;
        if (q_issued) mbar_wait_drain(q_full, (it) & 1, lim);
        for (uint32_t s = 0; s < C::KS && s < kc; ++s) {
          uint32_t last = kc - 1 - ((kc - 1 - s) % C::KS);
          mbar_wait_drain(k_full + s, (last / C::KS) & 1, lim);
        }
        for (uint32_t s = 0; s < C::VS && s < vc; ++s) {
          uint32_t last = vc - 1 - ((vc - 1 - s) % C::VS);
          mbar_wait_drain(v_full + s, (last / C::VS) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      uint32_t kc = 0, vc = 0, sc = 0, it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int tile = p.q_order[w / p.Hq];
        const int e0 = p.q_ptr[tile], e1 = p.q_ptr[tile + 1];
        const int n = e1 - e0;
        if (n == 0) continue;
        if (!(ok = mbar_wait(q_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int jj = 0; jj <= n && ok; ++jj) {
          if (jj < n) {
            const uint32_t x = kc + jj, s = x % C::KS;
            if (!(ok = mbar_wait(k_full + s, (x / C::KS) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t b = (sc + jj) & 1;
            const uint32_t d_tmem = tbase + (b ? C::TM_S1 : C::TM_S0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
              mma_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + s * C::TILE + off, 16, 1024), IDESC_S,
                     kk > 0);
            }
            mma_commit(k_empty + s);
            mma_commit(s_full + b);
            if (jj == n - 1) mma_commit(q_empty);
          }
          if (jj >= 1) {
            const int i = jj - 1;
            const uint32_t b = (sc + i) & 1;
            if (!(ok = mbar_wait(p_full + b, ((sc + i) >> 1) & 1, abort_flag))) break;
            const uint32_t x = vc + i, s = x % C::VS;
            if (!(ok = mbar_wait(v_full + s, (x / C::VS) & 1, abort_flag))) break;
            if (i == 0 && it > 0 && !(ok = mbar_wait(o_free, (it - 1) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t a_tmem = tbase + (b ? C::TM_S1 : C::TM_S0);
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk) {
              mma_ts(tbase + C::TM_O, a_tmem + kk * 8, sdesc_sw128(sV + s * C::TILE + kk * 2048, C::PANEL, 1024),
                     IDESC_PV, (i > 0 || kk > 0));
            }
            mma_commit(v_empty + s);
            mma_commit(o_full);
          }
        }
        kc += n;
        vc += n;
        sc += n;
        ++it;
      }
      // every MMA issued so far must finish before TMEM is freed
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;  // q row within the tile, TMEM lane
    const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
    uint32_t sc = 0, vc = 0, pvc = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const int tile = p.q_order[w / p.Hq], h = w % p.Hq;
      const int e0 = p.q_ptr[tile], e1 = p.q_ptr[tile + 1];
      const int n = e1 - e0;
      const int q = tile * C::BM + t;
      if (n == 0) {
        if (q < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          uint4* dst = reinterpret_cast<uint4*>(p.O + ((size_t)q * p.Hq + h) * D);
          for (int c = 0; c < D / 8; ++c) dst[c] = z;
          p.LSE[(size_t)h * p.T + q] = -INFINITY;
        }
        continue;
      }
      const int q_tin = p.tok[q].tin;
      float m_use = -INFINITY, l = 0.f;
      for (int jj = 0; jj < n; ++jj) {
        const int e = e0 + jj;
        const int kd = p.kind[e];
        const int k0 = p.kv_idx[e] * C::BN;
        const uint32_t b = (sc + jj) & 1;
        ok = mbar_wait(s_full + b, ((sc + jj) >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = tl + (b ? C::TM_S1 : C::TM_S0);
        uint32_t sr[128];
        tmem_ld32(sb + 0, sr + 0);
        tmem_ld32(sb + 32, sr + 32);
        tmem_ld32(sb + 64, sr + 64);
        tmem_ld32(sb + 96, sr + 96);
        tmem_ld_wait();
        float mx = -INFINITY;
        if (kd == PT_KIND_PARTIAL) {
          const uint32_t x = vc + jj, s = x % C::VS;
          ok = mbar_wait(v_full + s, (x / C::VS) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const pt_tok* tk = reinterpret_cast<const pt_tok*>(smem + C::OFF_TOK + s * C::TOKB);
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const pt_tok kt = tk[c];
            const bool keep = (k0 + c <= q) && (kt.tin <= q_tin) && (q_tin < kt.tout);
            float v = keep ? __uint_as_float(sr[c]) : -INFINITY;
            sr[c] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
        }
        const float m_blk = mx * p.scale_log2;
        const bool grow = m_blk > m_use + kRescaleThreshold;
        float m_new = grow ? m_blk : m_use;
        if (__any_sync(0xffffffffu, grow && l > 0.f)) {
          // O holds contributions scaled to the old reference: wait for the PV
          // in flight, then rescale this warp's rows in place.
          ok = mbar_wait(o_full, (pvc + jj - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = (grow && l > 0.f) ? ex2(m_use - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tl + C::TM_O + c * 32, orr);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) orr[k] = __float_as_uint(__uint_as_float(orr[k]) * alpha);
            tmem_st32(tl + C::TM_O + c * 32, orr);
          }
          tmem_st_wait();
          l *= alpha;
        }
        m_use = m_new;
        const float ref = (m_use == -INFINITY) ? 0.f : m_use;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c]), p.scale_log2, -ref));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c + 1]), p.scale_log2, -ref));
          rs += p0 + p1;
          sr[c >> 1] = pack_bf16(p0, p1);
        }
        l += rs;
        tmem_st32(sb + 0, sr + 0);
        tmem_st32(sb + 32, sr + 32);
        tmem_st_wait();
        if (jj > 0) {
          ok = mbar_wait(o_full, (pvc + jj - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        tc_fence_before();
        mbar_arrive(p_full + b);
      }
      if (!ok) break;
      // epilogue: O / l and LSE
      ok = mbar_wait(o_full, (pvc + n - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.O + ((size_t)q * p.Hq + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(tl + C::TM_O + c * 32, orr);
        tmem_ld_wait();
        if (q < p.T) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16(__uint_as_float(orr[2 * k]) * inv, __uint_as_float(orr[2 * k + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      if (q < p.T) p.LSE[(size_t)h * p.T + q] = l > 0.f ? (m_use + log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      mbar_arrive(o_free);
      sc += n;
      vc += n;
      pvc += n;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

template <int D>
int launch_fwd(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, float scale,
               const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  using C = FwdCfg<D>;
  static int attr_set[64] = {0};
  int dev = bm->device;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_fwd_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) {
      set_error("forward kernel: cannot reserve %d bytes of shared memory: %s", C::SMEM_BYTES, cudaGetErrorString(e));
      return 3;
    }
    attr_set[dev] = 1;
  }
  CUtensorMap mQ, mK, mV;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mK, K, T, Hkv, D, 128) ||
      !make_tmap_thd(&mV, V, T, Hkv, D, 128))
    return 3;
  FwdParams p;
  p.q_ptr = bm->q_ptr;
  p.kv_idx = bm->kv_idx;
  p.kind = bm->kind;
  p.q_order = bm->q_order;
  p.tok = bm->tok;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.nq = bm->nq;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int n_items = bm->nq * Hq;
  const int grid = n_items < num_sms(dev) ? n_items : num_sms(dev);
  if (grid <= 0) return 0;
  {
    ProfScope ps(s, "fwd_tc");
    k_fwd_tc<D><<<grid, 192, C::SMEM_BYTES, s>>>(mQ, mK, mV, p);
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("forward kernel launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

}  // namespace

int fwd_tc(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
           const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  switch (D) {
    case 64: return launch_fwd<64>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    case 128: return launch_fwd<128>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    case 256: return launch_fwd<256>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    default: set_error("tensor-core forward: head_dim %d not built", D); return 2;
  }
}

}  // namespace pt
