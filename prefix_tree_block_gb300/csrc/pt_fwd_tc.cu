// pt_fwd_tc.cu -- tensor-core forward for bf16: O and LSE over the kept pairs.
//
// "prefix_grouper_kernel.py", flex_shared_prefix_attention and its block
// mask: exact softmax attention in which every (q tile, kv block) pair the
// block map lists as empty is skipped, full pairs run unmasked, and partial
// pairs apply the tree mask element by element (here: one bit per pair from
// the block map's precomputed 128 x 128 keep masks).
//
// Design (sm_103a, persistent CTAs: one per SM, two at head_dim 64):
//   NH softmax warpgroups (NH = 2 at head_dim 128, else 1).  A work item is
//   one q tile and NH q heads that share a kv head (grouped-query
//   attention), so every K/V tile loaded serves NH heads.  Warpgroup h owns
//   head h of the item; thread t of it owns q row t of the tile.  At head_dim
//   64 a CTA takes one head and half of TMEM, and two CTAs share each SM:
//   their softmax warpgroups, on independent items, fill each other's waits
//   (where two heads of one CTA would run in lockstep on the same K/V block).
//   producer warp   TMA: the NH Q tiles once per item, then K and V of each
//                   listed kv block through separate multi-stage rings
//                   (128-byte swizzled 64-column panels); with V, the tile's
//                   keep mask (partial tiles) and its slot id.
//   MMA warp(s)     one lane issues tcgen05.mma: S_h = Q_h K^T into TMEM
//                   (M = 128 q rows, N = 128 kv, K = D) and O_h += P_h V with
//                   P_h read from TMEM (M = 128, N = D, K = 128).  With two
//                   heads, head A's MMAs run while head B's softmax works and
//                   vice versa; with one head, S is double-buffered and S of
//                   block j+1 is issued before PV of block j.  At head_dim 64
//                   (P in its own columns) one warp issues the S products and
//                   a second warp the PV products: the tensor pipe runs one
//                   thread's MMAs into one accumulator after another with its
//                   latency (about 300 cycles) between chains, and short
//                   chains (4 and 8 MMAs) are all this head dim has, so two
//                   issuing threads keep it busy where one cannot.
//   softmax         load the S row from TMEM, clear masked entries, keep the
//                   running max and sum in base 2 with the scale folded in,
//                   write P as bf16 over the S columns, and rescale O in TMEM
//                   only when the running max grows by more than 2^8 (the
//                   final division by l makes any fixed reference exact).
// Every wait is bounded: a timeout raises a CTA abort flag, records
// PT_ERR_TIMEOUT, drains copies and MMAs in flight and frees TMEM.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_fwd(cudaStream_t s) { return take_status_here(s); }

namespace {

template <int D, int NH>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NP = D / 64;        // 64-column panels per row
  static constexpr int PANEL = 128 * 128;  // bytes: 128 rows x 128 B
  static constexpr int TILE = NP * PANEL;
  // Head_dim 64, one head per item: two CTAs share an SM (half of TMEM,
  // two-deep K and V rings, 256 threads each), so the softmax warpgroups of
  // two independent items fill each other's waits.
  static constexpr bool TWO = D == 64 && NH == 1;
  static constexpr int SB = (NH == 1 && !TWO) ? 2 : 1;  // S buffers per head
  // With TMEM to spare (head_dim 64) P goes to its own columns, so S of the
  // next block can be computed as soon as the softmax has loaded S, and the
  // next item's Q tiles load while this item runs.
  static constexpr bool OVL = D == 64;
  static constexpr int QB = OVL ? 2 : 1;  // Q buffers
  static constexpr int KS = TWO ? 2 : D == 64 ? 4 : (D == 128 ? (NH == 2 ? 2 : 3) : 1);
  static constexpr int VS = TWO ? 2 : D == 64 ? 4 : (D == 128 ? 2 : 1);
  static constexpr int MASKB = 128 * 16;  // one partial tile's row masks
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB * NH * TILE;
  static constexpr int OFF_V = OFF_K + KS * TILE;
  static constexpr int OFF_MASK = OFF_V + VS * TILE;
  // (head_dim 256) 2 KB per softmax warp to turn its 32 rows of a 32-column
  // O chunk into 64-byte row segments for the stores (see the epilogue); at
  // head_dim 128 the staging's registers cost the main loop more than it saves
  static constexpr bool OST = NH == 1 && !OVL;
  static constexpr int OFF_OST = OFF_MASK + VS * MASKB;
  static constexpr int OST_BYTES = OST ? NH * 4 * 2048 : 0;
  static constexpr int OFF_META = OFF_OST + OST_BYTES;
  static constexpr int OFF_BAR = OFF_META + 16 * ((VS * 4 + 15) / 16);
  // q_full[QB] q_empty[QB] k_full[KS] k_empty[KS] v_full[VS] v_empty[VS]
  // s_full[NH*SB] p_full[NH*SB] o_full[NH] o_free[NH] mma_done
  // (OVL) s_free[NH] p_free[NH] o_written[NH] mma_done2
  static constexpr int NBAR = 2 * QB + 2 * KS + 2 * VS + 2 * NH * SB + 2 * NH + 1 + (OVL ? 3 * NH + 1 : 0);
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0;                            // S(h, b) at (h * SB + b) * 128
  static constexpr int TM_P = NH * SB * 128;                // (OVL) packed P(h) at TM_P + h * 64
  static constexpr int TM_O = TM_P + (OVL ? NH * 64 : 0);  // O(h) at TM_O + h * D
  // softmax warpgroups, the producer warp and the MMA warp; with OVL a
  // second MMA warp: one issues the S products, the other the PV products,
  // so the tensor pipe overlaps their chains (one thread's MMAs into one
  // accumulator after another run with the pipe's latency between chains)
  // (TWO) the producer and MMA warps fill a second warpgroup (one warp
  // idle); registers move to the softmax warpgroup (setmaxnreg), the split
  // adding up to the launch's 128 per thread (the kernel must be built with 128)
  // (NH = 2) the producer and MMA warps fill a third warpgroup (two warps
  // idle), so that the softmax warpgroups can take registers with setmaxnreg:
  // with ten warps one SM sub-partition holds three of them and its 16 K
  // registers cap every thread at 168, the launch's count; 216 for the
  // softmax and 72 for the rest add up to it
  static constexpr bool SPLIT = TWO || NH == 2;
  static constexpr int THREADS = TWO ? 256 : NH == 2 ? 384 : NH * 128 + (OVL ? 96 : 64);
  static constexpr int CTAS_PER_SM = TWO ? 2 : 1;
  static constexpr int TMEM_COLS = TWO ? 256 : 512;
  static constexpr int REG_SOFTMAX = TWO ? 184 : 216, REG_CTRL = 72, REG_LAUNCH = TWO ? 128 : 168;
  static_assert(!SPLIT || NH * 128 * REG_SOFTMAX + (THREADS - NH * 128) * REG_CTRL == THREADS * REG_LAUNCH,
                "register split");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TM_O + NH * D <= TMEM_COLS, "TMEM budget");
};

struct FwdParams {
  const int* q_ptr;
  const int* kv_idx;
  const int* pidx;
  const int* q_order;
  const uint32_t* mask_rows;
  __nv_bfloat16* O;
  float* LSE;
  int T, Hq, Hkv, nq;
  float scale_log2;  // softmax scale * log2(e)
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Work item w -> q tile, first head, number of heads (1..NH).
template <int NH>
__device__ __forceinline__ void decode_item(const FwdParams& p, int w, int& tile, int& h0, int& nh) {
  const int g = p.Hq / p.Hkv;
  if (NH == 1) {
    tile = p.q_order[w / p.Hq];
    h0 = w % p.Hq;
    nh = 1;
  } else {
    const int np = (g + 1) >> 1;
    const int per_tile = p.Hkv * np;
    tile = p.q_order[w / per_tile];
    const int rem = w % per_tile, hk = rem / np, pr = rem % np;
    h0 = hk * g + 2 * pr;
    nh = min(2, g - 2 * pr);
  }
}

// Item of CTA b in round r of a grid of G: rounds alternate direction over
// the longest-first item order (boustrophedon), so no CTA takes the largest
// item of every round.
__device__ __forceinline__ int snake_item(int r, int b, int G) { return r * G + ((r & 1) ? G - 1 - b : b); }

template <int NH>
__host__ __device__ __forceinline__ int fwd_items(int nq, int Hq, int Hkv) {
  if (NH == 1) return nq * Hq;
  const int g = Hq / Hkv;
  return nq * Hkv * ((g + 1) / 2);
}

template <int D, int NH>
__global__ void __launch_bounds__(FwdCfg<D, NH>::THREADS, FwdCfg<D, NH>::CTAS_PER_SM)
    k_fwd_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
             const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO, const FwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = FwdCfg<D, NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;              // [QB]
  uint64_t* q_empty = q_full + C::QB;       // [QB]
  uint64_t* k_full = q_empty + C::QB;
  uint64_t* k_empty = k_full + C::KS;
  uint64_t* v_full = k_empty + C::KS;
  uint64_t* v_empty = v_full + C::VS;
  uint64_t* s_full = v_empty + C::VS;       // [NH][SB]
  uint64_t* p_full = s_full + NH * C::SB;   // [NH][SB]
  uint64_t* o_full = p_full + NH * C::SB;   // [NH]
  uint64_t* o_free = o_full + NH;           // [NH]
  uint64_t* mma_done = o_free + NH;
  uint64_t* s_free = mma_done + 1;          // [NH] (OVL) S(h) loaded by the softmax
  uint64_t* p_free = s_free + NH;           // [NH] (OVL) PV(h) done reading P(h)
  uint64_t* o_written = p_free + NH;        // [NH] (OVL) the warpgroup's O rows are in shared memory
  uint64_t* mma_done2 = o_written + NH;     // (OVL) the PV warp's MMAs are complete
  int* meta = reinterpret_cast<int*>(smem + C::OFF_META);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = fwd_items<NH>(p.nq, p.Hq, p.Hkv);
  constexpr int PRODUCER = NH * 4, ISSUER = NH * 4 + 1, ISSUER_PV = NH * 4 + 2;

  if (threadIdx.x == PRODUCER * 32) {
    for (int b = 0; b < C::QB; ++b) {
      mbar_init(q_full + b, 1);
      // OVL: each softmax warpgroup's O store, made from the item's Q buffer,
      // frees it; else the item's last S MMA does
      mbar_init(q_empty + b, C::OVL ? NH : 1);
    }
    if (C::OVL) {
      for (int h = 0; h < NH; ++h) {
        mbar_init(s_free + h, 128);
        mbar_init(p_free + h, 1);
        mbar_init(o_written + h, 128);
      }
      mbar_init(mma_done2, 1);
    }
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < NH * C::SB; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
    }
    for (int h = 0; h < NH; ++h) {
      mbar_init(o_full + h, 1);
      mbar_init(o_free + h, 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mQ);
    prefetch_tmap(&mK);
    prefetch_tmap(&mV);
    if (C::OVL) prefetch_tmap(&mO);
  }
  if (warp == ISSUER) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // the roles, one lambda each, run by the warps the dispatch below picks: producer
  const auto producer_role = [&]() {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kc = 0, vc = 0, it = 0;
      bool ok = true, q_issued = false;
      for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
        const int w = snake_item(rr, blockIdx.x, gridDim.x);
        if (w >= n_items) continue;
        int tile, h0, nh;
        decode_item<NH>(p, w, tile, h0, nh);
        const int e0 = p.q_ptr[tile], e1 = p.q_ptr[tile + 1];
        if (e1 == e0) continue;
        const uint32_t qb = it % C::QB;
        q_issued = false;  // this item's Q not issued yet
        if (it >= C::QB && !(ok = mbar_wait(q_empty + qb, (it / C::QB - 1) & 1, abort_flag))) break;
        mbar_expect_tx(q_full + qb, nh * C::TILE);
        for (int h = 0; h < nh; ++h)
#pragma unroll
          for (int pn = 0; pn < C::NP; ++pn)
            tma_load_3d(smem + C::OFF_Q + (qb * NH + h) * C::TILE + pn * C::PANEL, &mQ, q_full + qb, pn * 64, h0 + h,
                        tile * C::BM);
        q_issued = true;
        const int hk = h0 / (p.Hq / p.Hkv);
        for (int e = e0; e < e1; ++e) {
          const int j = p.kv_idx[e];
          const int slot = p.pidx[e];
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
            meta[s] = slot;  // made visible by the arrive below (release)
            mbar_expect_tx(v_full + s, C::TILE + (slot >= 0 ? C::MASKB : 0));
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn)
              tma_load_3d(smem + C::OFF_V + s * C::TILE + pn * C::PANEL, &mV, v_full + s, pn * 64, hk, j * C::BN);
            if (slot >= 0)
              bulk_load(smem + C::OFF_MASK + s * C::MASKB, p.mask_rows + (size_t)slot * 512, C::MASKB, v_full + s);
            ++vc;
          }
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        // Q loads issued: `it` items completed, plus this one if its Q went out
        const uint32_t nql = it + (q_issued ? 1 : 0);
        for (uint32_t b = 0; b < C::QB && b < nql; ++b) {
          const uint32_t last = nql - 1 - ((nql - 1 - b) % C::QB);
          mbar_wait_drain(q_full + b, (last / C::QB) & 1, lim);
        }
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
  };
  // MMA issuer
  const auto issuer_role = [&]() {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      uint32_t kc = 0, vc = 0, it = 0;
      uint32_t sc[NH], itv[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) sc[h] = itv[h] = 0;
      bool ok = true;

      uint32_t qb = 0;  // Q buffer of the current item
      auto issue_s = [&](int h, uint32_t u, uint32_t ks) {
        const uint32_t b = u % C::SB;
        const uint32_t d_tmem = tbase + C::TM_S + (h * C::SB + b) * 128;
        const uint32_t qa = sQ + (qb * NH + h) * C::TILE, ka = sK + ks * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
          mma_ss(d_tmem, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), IDESC_S, kk > 0);
        }
        mma_commit(s_full + h * C::SB + b);
      };
      auto issue_pv = [&](int h, uint32_t u, uint32_t vs, bool first) {
        const uint32_t b = u % C::SB;
        // P packed in place over S, or in its own columns
        const uint32_t a_tmem = tbase + (C::OVL ? C::TM_P + h * 64 : C::TM_S + (h * C::SB + b) * 128);
        const uint32_t va = sV + vs * C::TILE;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ts(tbase + C::TM_O + h * D, a_tmem + kk * 8, sdesc_sw128(va + kk * 2048, C::PANEL, 1024), IDESC_PV,
                 (!first || kk > 0));
      };

      for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
        const int w = snake_item(rr, blockIdx.x, gridDim.x);
        if (w >= n_items) continue;
        int tile, h0, nh;
        decode_item<NH>(p, w, tile, h0, nh);
        const int n = p.q_ptr[tile + 1] - p.q_ptr[tile];
        if (n == 0) continue;
        qb = it % C::QB;
        if (!(ok = mbar_wait(q_full + qb, (it / C::QB) & 1, abort_flag))) break;
        tc_fence_after();
        for (int jj = 0; jj <= n && ok; ++jj) {
          const uint32_t ks = (kc + jj) % C::KS;
          if (jj < n && !C::OVL) {  // (OVL: tested with the group's other barriers)
            if (!(ok = mbar_wait(k_full + ks, ((kc + jj) / C::KS) & 1, abort_flag))) break;
            tc_fence_after();
          }
          if constexpr (C::OVL) {
            // S of block jj for every head once K(jj) is in and the softmax
            // has loaded each head's previous S, the barriers tested together
            // and the heads' MMAs issued back to back.
            if (jj < n) {
              uint64_t* bars[1 + NH];
              uint32_t par[1 + NH];
              bars[0] = k_full + ks;
              par[0] = ((kc + jj) / C::KS) & 1;
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                const uint32_t u = sc[h] + jj;
                bars[1 + h] = (h < nh && u >= 1) ? s_free + h : nullptr;
                par[1 + h] = (u - 1) & 1;
              }
              if (!(ok = mbar_wait_all<1 + NH>(bars, par, abort_flag))) break;
              tc_fence_after();
              for (int h = 0; h < nh; ++h) issue_s(h, sc[h] + jj, ks);
              mma_commit(k_empty + ks);  // (OVL: the Q buffer is freed by the epilogue's O store)
            }
            // (the PV products of this item: the PV warp)
          } else if (NH == 1) {
            if (jj < n) {
              issue_s(0, sc[0] + jj, ks);
              mma_commit(k_empty + ks);
              if (jj == n - 1) mma_commit(q_empty + qb);
            }
            if (jj >= 1) {
              const int i = jj - 1;
              const uint32_t u = sc[0] + i, vs = (vc + i) % C::VS;
              if (!(ok = mbar_wait(p_full + (u % C::SB), (u / C::SB) & 1, abort_flag))) break;
              if (!(ok = mbar_wait(v_full + vs, ((vc + i) / C::VS) & 1, abort_flag))) break;
              if (i == 0 && itv[0] > 0 && !(ok = mbar_wait(o_free, (itv[0] - 1) & 1, abort_flag))) break;
              tc_fence_after();
              issue_pv(0, u, vs, i == 0);
              mma_commit(o_full);
              mma_commit(v_empty + vs);
            }
          } else {
            for (int h = 0; h < nh && ok; ++h) {
              if (jj >= 1) {
                const int i = jj - 1;
                const uint32_t u = sc[h] + i, vs = (vc + i) % C::VS;
                if (!(ok = mbar_wait(p_full + h * C::SB, u & 1, abort_flag))) break;
                if (h == 0 && !(ok = mbar_wait(v_full + vs, ((vc + i) / C::VS) & 1, abort_flag))) break;
                if (i == 0 && itv[h] > 0 && !(ok = mbar_wait(o_free + h, (itv[h] - 1) & 1, abort_flag))) break;
                tc_fence_after();
                issue_pv(h, u, vs, i == 0);
                // two heads: O is committed once per item; S_h(jj), issued
                // next, is committed after this PV, which the softmax relies on
                if (i == n - 1) mma_commit(o_full + h);
                if (h == nh - 1) mma_commit(v_empty + vs);
              }
              if (jj < n) {
                issue_s(h, sc[h] + jj, ks);
                if (h == nh - 1) {
                  mma_commit(k_empty + ks);
                  if (jj == n - 1) mma_commit(q_empty + qb);
                }
              }
            }
          }
        }
        kc += n;
        vc += n;
        for (int h = 0; h < nh; ++h) {
          sc[h] += n;
          itv[h] += 1;
        }
        ++it;
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  };
  // PV issuer (OVL)
  const auto pv_role = [&]() {
    // ------------------------------------------------------------ PV issuer (OVL)
    // PV of block i for every head of the item once V(i) and that head's P
    // tile are in (and, on the item's first block, the epilogue has read
    // the previous item's O); each head's MMAs go out as soon as its own
    // barriers are complete.
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      uint32_t vc = 0;
      uint32_t sc[NH], itv[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) sc[h] = itv[h] = 0;
      bool ok = true;
      for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
        const int w = snake_item(rr, blockIdx.x, gridDim.x);
        if (w >= n_items) continue;
        int tile, h0, nh;
        decode_item<NH>(p, w, tile, h0, nh);
        const int n = p.q_ptr[tile + 1] - p.q_ptr[tile];
        if (n == 0) continue;
        for (int i = 0; i < n && ok; ++i) {
          const uint32_t vs = (vc + i) % C::VS;
          if (!(ok = mbar_wait(v_full + vs, ((vc + i) / C::VS) & 1, abort_flag))) break;
          for (int h = 0; h < nh && ok; ++h) {
            const uint32_t u = sc[h] + i;
            uint64_t* bars[2] = {p_full + h, (i == 0 && itv[h] > 0) ? o_free + h : nullptr};
            const uint32_t par[2] = {u & 1, (itv[h] - 1) & 1};
            if (!(ok = mbar_wait_all<2>(bars, par, abort_flag))) break;
            tc_fence_after();
            // P(h) in its own TMEM columns
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk)
              mma_ts(tbase + C::TM_O + h * D, tbase + C::TM_P + h * 64 + kk * 8,
                     sdesc_sw128(sV + vs * C::TILE + kk * 2048, C::PANEL, 1024), IDESC_PV, (i > 0 || kk > 0));
            mma_commit(p_free + h);
            if (i == n - 1) mma_commit(o_full + h);
          }
          if (!ok) break;
          mma_commit(v_empty + vs);
        }
        vc += n;
        for (int h = 0; h < nh; ++h) {
          sc[h] += n;
          itv[h] += 1;
        }
      }
      mma_commit(mma_done2);
      mbar_wait_drain(mma_done2, 0, 200000000);
    }
    __syncwarp();
  };
  // softmax warpgroups
  const auto softmax_role = [&]() {
    // ------------------------------------------------------------ softmax
    const int h = warp >> 2;                   // head slot of this warpgroup
    const int r = threadIdx.x & 127;           // q row within the tile, TMEM lane
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t o_col = C::TM_O + h * D;
    uint32_t sc = 0, vc = 0, pvc = 0, itv = 0;
    uint32_t qi = 0;  // items with kv blocks so far: the Q buffer of an item is qi % QB
    bool ok = true;
    for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
      const int w = snake_item(rr, blockIdx.x, gridDim.x);
      if (w >= n_items) continue;
      int tile, h0, nh;
      decode_item<NH>(p, w, tile, h0, nh);
      const int e0 = p.q_ptr[tile], n = p.q_ptr[tile + 1] - e0;
      if (h >= nh) {  // this warpgroup has no head in the item; the V ring still advances
        vc += n;
        qi += n > 0 ? 1 : 0;
        continue;
      }
      const int head = h0 + h;
      const int q = tile * C::BM + r;
      if (n == 0) {
        if (q < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          uint4* dst = reinterpret_cast<uint4*>(p.O + ((size_t)q * p.Hq + head) * D);
          for (int c = 0; c < D / 8; ++c) dst[c] = z;
          p.LSE[(size_t)head * p.T + q] = -INFINITY;
        }
        continue;
      }
      float m_use = -INFINITY, l = 0.f;
      for (int jj = 0; jj < n; ++jj) {
        const uint32_t u = sc + jj, b = u % C::SB;
        const uint32_t x = vc + jj, vs = x % C::VS;
        ok = mbar_wait(s_full + h * C::SB + b, (u / C::SB) & 1, abort_flag) &&
             mbar_wait(v_full + vs, (x / C::VS) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = tl + C::TM_S + (h * C::SB + b) * 128;
        uint32_t sr[128];
        tmem_ld32(sb + 0, sr + 0);
        tmem_ld32(sb + 32, sr + 32);
        tmem_ld32(sb + 64, sr + 64);
        tmem_ld32(sb + 96, sr + 96);
        const int slot = meta[vs];
        uint4 mk = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
        if (slot >= 0) mk = reinterpret_cast<const uint4*>(smem + C::OFF_MASK + vs * C::MASKB)[r];
        tmem_ld_wait();
        if (C::OVL) {  // S is in registers: the MMA may compute the next S over it
          tc_fence_before();
          mbar_arrive(s_free + h);
        }
        // eight independent max chains (instruction-level parallelism)
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
        if (slot >= 0) {
          const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            const float v0 = ((mw[c >> 5] >> (c & 31)) & 1u) ? __uint_as_float(sr[c]) : -INFINITY;
            const float v1 = ((mw[c >> 5] >> ((c + 1) & 31)) & 1u) ? __uint_as_float(sr[c + 1]) : -INFINITY;
            sr[c] = __float_as_uint(v0);
            sr[c + 1] = __float_as_uint(v1);
            m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], v0, v1);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; c += 2)
            m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        }
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float m_blk = mx * p.scale_log2;
        const bool grow = m_blk > m_use + kRescaleThreshold;
        const float m_new = grow ? m_blk : m_use;
        // P of this block against the new reference first: the O rescale
        // below then holds only the packed P, not the 128 scores, and the
        // exponentials overlap the PV still in flight
        const float ref = (m_new == -INFINITY) ? 0.f : m_new;
        // scale and shift two columns per packed fma, the row sum in four
        // packed accumulators (eight chains)
        const unsigned long long sc2 = f2_pack(p.scale_log2, p.scale_log2), nref2 = f2_pack(-ref, -ref);
        unsigned long long r4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nref2), x0, x1);
          const float p0 = ex2_mix(x0, c), p1 = ex2_mix(x1, c + 1);
          r4[(c >> 1) & 3] = f2_add(r4[(c >> 1) & 3], f2_pack(p0, p1));
          sr[c >> 1] = pack_bf16(p0, p1);
        }
        float r8[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) f2_unpack(r4[k], r8[2 * k], r8[2 * k + 1]);
        const float l_blk = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
        if (C::OVL && u >= 1) {
          // PV of the previous block must be done: it reads the P columns
          // written below and accumulates into the O a rescale touches
          ok = mbar_wait(p_free + h, (u - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, grow && l > 0.f)) {
          // O holds contributions scaled to the old reference: rescale this
          // warp's rows in place once the PV in flight is done.  With two
          // heads that is already known (S(j) was committed after PV(j-1));
          // with one head, wait for it.
          if (NH == 1 && !C::OVL) {
            ok = mbar_wait(o_full + h, (pvc + jj - 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const float alpha = (grow && l > 0.f) ? ex2(m_use - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tl + o_col + c * 32, orr);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) orr[k] = __float_as_uint(__uint_as_float(orr[k]) * alpha);
            tmem_st32(tl + o_col + c * 32, orr);
          }
          tmem_st_wait();
          l *= alpha;
        }
        m_use = m_new;
        l += l_blk;
        const uint32_t pb = C::OVL ? tl + C::TM_P + h * 64 : sb;  // P: own columns, or over S
        tmem_st32(pb + 0, sr + 0);
        tmem_st32(pb + 32, sr + 32);
        tmem_st_wait();
        if (NH == 1 && !C::OVL && jj > 0) {
          ok = mbar_wait(o_full + h, (pvc + jj - 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        tc_fence_before();
        mbar_arrive(p_full + h * C::SB + b);
      }
      if (!ok) break;
      // epilogue: O / l and LSE (one head: O committed per PV; two heads: once per item)
      ok = mbar_wait(o_full + h, ((NH == 1 && !C::OVL) ? (pvc + n - 1) : itv) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if constexpr (C::OVL) {
        // O / l into this item's Q tile of the head (the MMAs that read it are
        // done: o_full follows the last S), in the tile's 128-byte-swizzled
        // layout, then one TMA store of the tile; the store's reads free the
        // buffer (the warpgroup of a one-head item also arrives for the idle one)
        const uint32_t qbuf = qi % C::QB;
        uint8_t* obuf = smem + C::OFF_Q + (qbuf * NH + h) * C::TILE;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tl + o_col + c * 32, orr);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16(__uint_as_float(orr[2 * k]) * inv, __uint_as_float(orr[2 * k + 1]) * inv);
          uint8_t* prow = obuf + (c >> 1) * C::PANEL + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int chunk = ((c & 1) * 4 + k) ^ (r & 7);
            *reinterpret_cast<uint4*>(prow + chunk * 16) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                                                                      pk[4 * k + 3]);
          }
        }
        fence_proxy_async_smem();  // the rows, written by this thread, for the TMA store
        mbar_arrive(o_written + h);
        if (r == 0) {  // one thread stores the tile once every row is in (a bounded wait)
          ok = mbar_wait(o_written + h, itv & 1, abort_flag);
          if (ok) {
#pragma unroll
            for (int pn = 0; pn < C::NP; ++pn) tma_store_3d(&mO, obuf + pn * C::PANEL, pn * 64, head, tile * C::BM);
            bulk_commit();
            bulk_wait_read0();
            mbar_arrive_cnt(q_empty + qbuf, h == 0 ? (uint32_t)(NH - nh + 1) : 1u);
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      } else if constexpr (C::OST) {
        // Each thread holds one row's 64 bytes of a 32-column chunk; stored
        // as they are, a warp instruction writes 32 rows.  The warp stages the
        // chunk in shared memory (16-byte pieces XOR-swizzled by row) and
        // reads it back so that four lanes cover one row's 64 bytes: each
        // store instruction then writes 8 rows of 64 contiguous bytes.
        uint8_t* wst = smem + C::OFF_OST + (warp & (NH * 4 - 1)) * 2048;
        const int lw = lane, rr = lw >> 2, kk = lw & 3;  // read-back: row rr (+ 8i), piece kk
        const int row0 = tile * C::BM + (warp & 3) * 32;  // first q row of this warp
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tl + o_col + c * 32, orr);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16(__uint_as_float(orr[2 * k]) * inv, __uint_as_float(orr[2 * k + 1]) * inv);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(wst + lw * 64 + ((k ^ (lw & 3)) * 16)) =
                make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = rr + 8 * i;  // 0..31 within the warp
            const uint4 v = *reinterpret_cast<const uint4*>(wst + row * 64 + ((kk ^ (row & 3)) * 16));
            const int qr = row0 + row;
            if (qr < p.T)
              *reinterpret_cast<uint4*>(p.O + ((size_t)qr * p.Hq + head) * D + c * 32 + kk * 8) = v;
          }
          __syncwarp();
        }
      } else {
        __nv_bfloat16* orow = p.O + ((size_t)q * p.Hq + head) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tl + o_col + c * 32, orr);
          tmem_ld_wait();
          store_rows32(orow + c * 32, (size_t)p.Hq * D, q, p.T, orr, inv);  // 8 row segments per store
        }
      }
      if (q < p.T) p.LSE[(size_t)head * p.T + q] = l > 0.f ? (m_use + log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      mbar_arrive(o_free + h);
      sc += n;
      vc += n;
      pvc += n;
      ++itv;
      ++qi;
    }
    if (!ok) *abort_flag = 1;
    if (C::OVL && r == 0) bulk_wait0();  // this warpgroup's O stores have landed
  };
  if constexpr (C::SPLIT) {
    // whole warpgroups take their registers first, so that each setmaxnreg
    // dominates the code of its warpgroup (ptxas then allocates each region
    // to its own count)
    if (warp >= PRODUCER) {
      regs_dec<C::REG_CTRL>();
      if (warp == PRODUCER)
        producer_role();
      else if (warp == ISSUER)
        issuer_role();
      else if (C::OVL && warp == ISSUER_PV)
        pv_role();  // (the other warps of this warpgroup have no role)
    } else {
      regs_inc<C::REG_SOFTMAX>();
      softmax_role();
    }
  } else {
    if (warp == PRODUCER)
      producer_role();
    else if (warp == ISSUER)
      issuer_role();
    else if (C::OVL && warp == ISSUER_PV)
      pv_role();
    else
      softmax_role();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == ISSUER) tmem_dealloc(tbase, C::TMEM_COLS);
}

template <int D, int NH>
int launch_fwd(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, float scale,
               const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  using C = FwdCfg<D, NH>;
  static int attr_set[64] = {0};
  int dev = bm->device;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_fwd_tc<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) {
      set_error("forward kernel: cannot reserve %d bytes of shared memory: %s", C::SMEM_BYTES, cudaGetErrorString(e));
      return 3;
    }
    attr_set[dev] = 1;
  }
  if constexpr (C::SPLIT) {
    // the register split adds up to the launch's count per thread: a build
    // with another count would leave setmaxnreg.inc waiting, so it is refused
    static int regs_ok[64] = {0};
    if (dev >= 0 && dev < 64 && !regs_ok[dev]) {
      cudaFuncAttributes fa{};
      if (cudaFuncGetAttributes(&fa, k_fwd_tc<D, NH>) != cudaSuccess || fa.numRegs != C::REG_LAUNCH) {
        set_error("forward kernel built with %d registers per thread, %d expected", fa.numRegs, C::REG_LAUNCH);
        return 3;
      }
      regs_ok[dev] = 1;
    }
  }
  if (masks_missing(bm)) {
    set_error("forward kernel: block map has no tile masks");
    return 1;
  }
  CUtensorMap mQ, mK, mV, mO;
  if (!make_tmap_thd(&mQ, Q, T, Hq, D, 128) || !make_tmap_thd(&mK, K, T, Hkv, D, 128) ||
      !make_tmap_thd(&mV, V, T, Hkv, D, 128) || !make_tmap_thd(&mO, O, T, Hq, D, 128))
    return 3;
  FwdParams p;
  p.q_ptr = bm->q_ptr;
  p.kv_idx = bm->kv_idx;
  p.pidx = bm->pidx;
  p.q_order = bm->q_order;
  p.mask_rows = bm->mask_rows;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.nq = bm->nq;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int n_items = fwd_items<NH>(bm->nq, Hq, Hkv);
  const int slots = num_sms(dev) * C::CTAS_PER_SM;
  const int grid = n_items < slots ? n_items : slots;
  if (grid <= 0) return 0;
  {
    ProfScope ps(s, "fwd_tc");
    launch_pdl(k_fwd_tc<D, NH>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, mQ, mK, mV, mO, p);
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("forward kernel launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}


// ---------------------------------------------------------------------------
// head_dim 512 (tensor cores)
//
// A 128-row Q tile is 128 KB at this head dim and a 128 x 512 fp32 O
// accumulator would take all of TMEM, so the kernel keeps the item's Q tile
// resident in shared memory, streams K and V through a ring of four 16 KB
// 64-column panels, and runs each item (q tile, q head) as two passes over
// its kv blocks, one per 256-column half of O:
//   pass 0  online softmax: S = Q K^T (8 K panels, K = 512), P over S in
//           TMEM, O[:, 0:256] += P V[:, 0:256] (one N = 256 product from the
//           four V panels of the half), the running max and sum as in the
//           other forward kernels;
//   pass 1  S again, P = exp2(s * scale * log2(e) - m) against the final
//           reference m of pass 0 (no rescaling), O[:, 256:512] += P V.
// Each block's 8 K panels and the previous block's 4 V panels are loaded in
// the order the MMAs consume them (K(j), V(j-1), K(j+1), V(j), ...), so
// every group is a multiple of four panels and a block's V panels always sit
// in ring slots 0..3, the contiguous operand an N = 256 MMA reads.  S is
// double-buffered (2 x 128 TMEM columns) beside the 256-column O half: S of
// block j+1 is computed while the softmax works on block j.
// ---------------------------------------------------------------------------
struct Fwd512Cfg {
  static constexpr int D = 512, NP = 8, PANEL = 128 * 128;
  static constexpr int RING = 4;
  static constexpr int MASKB = 128 * 16;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + NP * PANEL;
  static constexpr int OFF_MASK = OFF_RING + RING * PANEL;
  static constexpr int OFF_META = OFF_MASK + 2 * MASKB;
  static constexpr int OFF_BAR = OFF_META + 16;
  // q_full q_empty ring_full[4] ring_empty[4] s_full[2] p_full[2] o_full
  // o_free m_full[2] m_empty[2] mma_done
  static constexpr int NBAR = 2 + 2 * RING + 2 + 2 + 2 + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_O = 256;  // S(b) at b * 128; O half at 256
  static constexpr int THREADS = 128 + 64;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(Fwd512Cfg::THREADS, 1)
    k_fwd_d512(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const FwdParams p) {
  pdl_wait();  // launched with programmatic dependent launch
  using C = Fwd512Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 1;
  uint64_t* ring_full = q_empty + 1;         // [RING]
  uint64_t* ring_empty = ring_full + C::RING;  // [RING]
  uint64_t* s_full = ring_empty + C::RING;   // [2]
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* o_full = p_full + 2;
  uint64_t* o_free = o_full + 1;
  uint64_t* m_full = o_free + 1;             // [2]
  uint64_t* m_empty = m_full + 2;            // [2]
  uint64_t* mma_done = m_empty + 2;
  int* meta = reinterpret_cast<int*>(smem + C::OFF_META);  // mask slot of each mask buffer (-1: full tile)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.nq * p.Hq;
  constexpr int PRODUCER = 4, ISSUER = 5;
  const int g = p.Hq / p.Hkv;

  if (threadIdx.x == PRODUCER * 32) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(ring_full + s, 1);
      mbar_init(ring_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
      mbar_init(m_full + b, 1);
      mbar_init(m_empty + b, 128);
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
      uint32_t c = 0, mc = 0, it = 0;  // ring panels, mask buffers, items with blocks
      bool ok = true, q_issued = false;
      auto ring_load = [&](const CUtensorMap* map, int col, int hk, int row) -> bool {
        const uint32_t s = c % C::RING, u = c / C::RING;
        if (u > 0 && !mbar_wait(ring_empty + s, (u - 1) & 1, abort_flag)) return false;
        mbar_expect_tx(ring_full + s, C::PANEL);
        tma_load_3d(smem + C::OFF_RING + s * C::PANEL, map, ring_full + s, col, hk, row);
        ++c;
        return true;
      };
      for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
        const int w = snake_item(rr, blockIdx.x, gridDim.x);
        if (w >= n_items) continue;
        const int tile = p.q_order[w / p.Hq], head = w % p.Hq, hk = head / g;
        const int e0 = p.q_ptr[tile], n = p.q_ptr[tile + 1] - e0;
        if (n == 0) continue;
        q_issued = false;
        if (it > 0 && !(ok = mbar_wait(q_empty, (it - 1) & 1, abort_flag))) break;
        mbar_expect_tx(q_full, C::NP * C::PANEL);
        for (int pn = 0; pn < C::NP; ++pn)
          tma_load_3d(smem + C::OFF_Q + pn * C::PANEL, &mQ, q_full, pn * 64, head, tile * 128);
        q_issued = true;
        for (int hf = 0; hf < 2 && ok; ++hf) {
          for (int jj = 0; jj <= n && ok; ++jj) {
            if (jj < n) {
              const int j = p.kv_idx[e0 + jj], slot = p.pidx[e0 + jj];
              // the block's keep mask (partial tiles) into its mask buffer
              const uint32_t mb = mc % 2, mu = mc / 2;
              if (mu > 0 && !(ok = mbar_wait(m_empty + mb, (mu - 1) & 1, abort_flag))) break;
              meta[mb] = slot;  // made visible by the arrive below (release)
              mbar_expect_tx(m_full + mb, slot >= 0 ? C::MASKB : 0);
              if (slot >= 0)
                bulk_load(smem + C::OFF_MASK + mb * C::MASKB, p.mask_rows + (size_t)slot * 512, C::MASKB, m_full + mb);
              ++mc;
              for (int pn = 0; pn < C::NP && ok; ++pn) ok = ring_load(&mK, pn * 64, hk, j * 128);
            }
            if (jj >= 1 && ok) {
              const int j = p.kv_idx[e0 + jj - 1];
              for (int q4 = 0; q4 < 4 && ok; ++q4) ok = ring_load(&mV, (hf * 4 + q4) * 64, hk, j * 128);
            }
          }
        }
        ++it;
      }
      if (!ok) {
        const long long lim = 20000000;
        if (q_issued) mbar_wait_drain(q_full, (it) & 1, lim);
        for (uint32_t s = 0; s < C::RING && s < c; ++s) {
          const uint32_t last = c - 1 - ((c - 1 - s) % C::RING);
          mbar_wait_drain(ring_full + s, (last / C::RING) & 1, lim);
        }
        for (uint32_t b = 0; b < 2 && b < mc; ++b) {
          const uint32_t last = mc - 1 - ((mc - 1 - b) % 2);
          mbar_wait_drain(m_full + b, (last / 2) & 1, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == ISSUER) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sR = smem_u32(smem + C::OFF_RING);
      uint32_t c = 0, sc = 0, pvc = 0, it = 0, passes = 0;
      bool ok = true;
      for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
        const int w = snake_item(rr, blockIdx.x, gridDim.x);
        if (w >= n_items) continue;
        const int tile = p.q_order[w / p.Hq];
        const int n = p.q_ptr[tile + 1] - p.q_ptr[tile];
        if (n == 0) continue;
        if (!(ok = mbar_wait(q_full, it & 1, abort_flag))) break;
        tc_fence_after();
        for (int hf = 0; hf < 2 && ok; ++hf) {
          for (int jj = 0; jj <= n && ok; ++jj) {
            if (jj < n) {
              // S(u) = Q K_j^T into buffer u % 2, accumulated over the 8 panels
              const uint32_t u = sc + jj, b = u % 2;
              for (int pn = 0; pn < C::NP && ok; ++pn) {
                const uint32_t s = c % C::RING;
                if (!(ok = mbar_wait(ring_full + s, (c / C::RING) & 1, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tbase + C::TM_S + b * 128, sdesc_sw128(sQ + pn * C::PANEL + kk * 32, 16, 1024),
                         sdesc_sw128(sR + s * C::PANEL + kk * 32, 16, 1024), IDESC_S, (pn > 0 || kk > 0));
                mma_commit(ring_empty + s);
                ++c;
              }
              if (!ok) break;
              mma_commit(s_full + b);
              if (hf == 1 && jj == n - 1) mma_commit(q_empty);  // the item's last read of Q
            }
            if (jj >= 1) {
              // O half += P(u) V_half for block jj-1: P over S in TMEM, the four V
              // panels of the half in ring slots 0..3 (one N = 256 operand)
              const int i = jj - 1;
              const uint32_t u = sc + i, b = u % 2;
              if (!(ok = mbar_wait(p_full + b, (u / 2) & 1, abort_flag))) break;
              if (i == 0 && passes > 0 && !(ok = mbar_wait(o_free, (passes - 1) & 1, abort_flag))) break;
              for (int q4 = 0; q4 < 4 && ok; ++q4)
                ok = mbar_wait(ring_full + (c + q4) % C::RING, ((c + q4) / C::RING) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(tbase + C::TM_O, tbase + C::TM_S + b * 128 + kk * 8,
                       sdesc_sw128(sR + (c % C::RING) * C::PANEL + kk * 2048, C::PANEL, 1024), IDESC_PV,
                       (i > 0 || kk > 0));
              for (int q4 = 0; q4 < 4; ++q4) mma_commit(ring_empty + (c + q4) % C::RING);
              c += 4;
              mma_commit(o_full);
              ++pvc;
            }
          }
          sc += n;
          ++passes;
        }
        ++it;
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, 200000000);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (q row per thread)
    const int r = threadIdx.x;  // q row within the tile, TMEM lane
    const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t sc = 0, pvc = 0, mc = 0, passes = 0;
    bool ok = true;
    for (int rr = 0; rr * (int)gridDim.x < n_items && ok; ++rr) {
      const int w = snake_item(rr, blockIdx.x, gridDim.x);
      if (w >= n_items) continue;
      const int tile = p.q_order[w / p.Hq], head = w % p.Hq;
      const int n = p.q_ptr[tile + 1] - p.q_ptr[tile];
      const int q = tile * 128 + r;
      __nv_bfloat16* orow = p.O + ((size_t)q * p.Hq + head) * C::D;
      if (n == 0) {
        if (q < p.T) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c8 = 0; c8 < C::D / 8; ++c8) reinterpret_cast<uint4*>(orow)[c8] = z;
          p.LSE[(size_t)head * p.T + q] = -INFINITY;
        }
        continue;
      }
      float m_use = -INFINITY, l = 0.f;
      for (int hf = 0; hf < 2 && ok; ++hf) {
        for (int jj = 0; jj < n; ++jj) {
          const uint32_t u = sc + jj, b = u % 2;
          const uint32_t mb = mc % 2;
          ok = mbar_wait(s_full + b, (u / 2) & 1, abort_flag) && mbar_wait(m_full + mb, (mc / 2) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = tl + C::TM_S + b * 128;
          uint32_t sr[128];
          tmem_ld32(sb + 0, sr + 0);
          tmem_ld32(sb + 32, sr + 32);
          tmem_ld32(sb + 64, sr + 64);
          tmem_ld32(sb + 96, sr + 96);
          const int slot = meta[mb];
          uint4 mk = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
          if (slot >= 0) mk = reinterpret_cast<const uint4*>(smem + C::OFF_MASK + mb * C::MASKB)[r];
          mbar_arrive(m_empty + mb);  // the mask is in registers
          ++mc;
          tmem_ld_wait();
          if (slot >= 0) {
            const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (!((mw[c >> 5] >> (c & 31)) & 1u)) sr[c] = __float_as_uint(-INFINITY);
          }
          float ref = m_use;
          if (hf == 0) {
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; c += 2)
              m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float m_blk = mx * p.scale_log2;
            const bool grow = m_blk > m_use + kRescaleThreshold;
            const float m_new = grow ? m_blk : m_use;
            if (__any_sync(0xffffffffu, grow && l > 0.f)) {
              // O holds contributions against the old reference: once the PV in
              // flight is done, rescale this warp's rows in place
              ok = mbar_wait(o_full, (pvc + jj - 1) & 1, abort_flag);
              if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const float alpha = (grow && l > 0.f) ? ex2(m_use - m_new) : 1.f;
#pragma unroll 1
              for (int c = 0; c < 256 / 32; ++c) {
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
            ref = m_new;
          }
          const float rf = (ref == -INFINITY) ? 0.f : ref;
          // scale and shift two columns per packed fma, the row sum in four
          // packed accumulators (eight chains)
          const unsigned long long sc2 = f2_pack(p.scale_log2, p.scale_log2), nrf2 = f2_pack(-rf, -rf);
          unsigned long long r4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nrf2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            r4[(c >> 1) & 3] = f2_add(r4[(c >> 1) & 3], f2_pack(p0, p1));
            sr[c >> 1] = pack_bf16(p0, p1);
          }
          float r8[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f2_unpack(r4[k], r8[2 * k], r8[2 * k + 1]);
          if (hf == 0) l += ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
          tmem_st32(sb + 0, sr + 0);  // P over S (bf16 pairs in the first 64 columns)
          tmem_st32(sb + 32, sr + 32);
          tmem_st_wait();
          if (jj > 0) {
            // never more than one PV behind: the rescale above and the
            // epilogue's waits rely on the parity of o_full
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
        // epilogue of the pass: this half of O / l
        ok = mbar_wait(o_full, (pvc + n - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tl + C::TM_O + c * 32, orr);
          tmem_ld_wait();
          store_rows32(orow + hf * 256 + c * 32, (size_t)p.Hq * C::D, q, p.T, orr, inv);
        }
        tc_fence_before();
        mbar_arrive(o_free);
        sc += n;
        pvc += n;
        ++passes;
      }
      if (!ok) break;
      if (q < p.T) p.LSE[(size_t)head * p.T + q] = l > 0.f ? (m_use + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == ISSUER) tmem_dealloc(tbase, 512);
}

int launch_fwd512(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, float scale,
                  const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  using C = Fwd512Cfg;
  static int attr_set[64] = {0};
  int dev = bm->device;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_fwd_d512, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) {
      set_error("forward kernel: cannot reserve %d bytes of shared memory: %s", C::SMEM_BYTES, cudaGetErrorString(e));
      return 3;
    }
    attr_set[dev] = 1;
  }
  if (masks_missing(bm)) {
    set_error("forward kernel: block map has no tile masks");
    return 1;
  }
  CUtensorMap mQ, mK, mV;
  if (!make_tmap_thd(&mQ, Q, T, Hq, C::D, 128) || !make_tmap_thd(&mK, K, T, Hkv, C::D, 128) ||
      !make_tmap_thd(&mV, V, T, Hkv, C::D, 128))
    return 3;
  FwdParams p;
  p.q_ptr = bm->q_ptr;
  p.kv_idx = bm->kv_idx;
  p.pidx = bm->pidx;
  p.q_order = bm->q_order;
  p.mask_rows = bm->mask_rows;
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
    launch_pdl(k_fwd_d512, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, mQ, mK, mV, p);
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

namespace {
// One thread waits on an mbarrier that nothing will ever complete: the same
// bounded wait the attention kernels use runs out after about a second,
// records PT_ERR_TIMEOUT in this unit's status word and the kernel returns.
__global__ void k_wait_timeout_probe() {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, &abort_flag);
  }
}

// y = 2^x with the MUFU instruction (method 0) or the FMA-pipe polynomial
// (method 1) the softmax loops can mix, for tests of the polynomial's accuracy.
__global__ void k_exp2_probe(const float* __restrict__ x, float* __restrict__ y, long long n, int method) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    y[i] = method == 0 ? ex2(x[i]) : ex2_poly(x[i]);
}
}  // namespace

int exp2_probe(const float* x, float* y, long long n, int method, cudaStream_t s) {
  if (n <= 0) return 0;
  const long long blocks = (n + 255) / 256;
  k_exp2_probe<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(x, y, n, method);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("exp2 probe launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

int wait_timeout_probe(cudaStream_t s) {
  k_wait_timeout_probe<<<1, 32, 0, s>>>();
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("timeout probe launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

int fwd_tc(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
           const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  switch (D) {
    case 64: return launch_fwd<64, 1>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    case 128: return launch_fwd<128, 2>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    case 256: return launch_fwd<256, 1>(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    case 512: return launch_fwd512(Q, K, V, T, Hq, Hkv, scale, bm, O, LSE, s);
    default: set_error("tensor-core forward: head_dim %d not built", D); return 2;
  }
}

}  // namespace pt
