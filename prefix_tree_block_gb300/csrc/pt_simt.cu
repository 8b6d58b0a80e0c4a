// pt_simt.cu -- CUDA-core forward and backward (fp32 math) for fp32 inputs
// and for bf16 head dims the tensor-core kernels do not cover.
//
// "prefix_grouper_kernel.py", _kernel_options_for_dtype: fp32 inputs need a
// tighter numerical floor than bf16; here fp32 stays on fp32 FMAs (tf32
// tensor cores would miss a 1e-5 max-abs bound).  One warp owns one
// (row, head): lanes split head_dim, a shuffle reduction forms each score,
// and the row walks only the kv blocks its q tile lists, evaluating the
// tree mask on partial blocks.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {

int take_status_simt(cudaStream_t s) { return take_status_here(s); }

namespace {

// NPL values of a head_dim row per lane: 8 up to head_dim 256, 16 up to 512
// (head dims the tensor-core kernels do not take; "flex" fails beyond 256 on
// sm_103, per the drafter PR's testing notes).
constexpr int kMaxHeadDim = 512;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int NPL, class E>
__device__ __forceinline__ void load_row(const E* p, int D, float* r) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    int d = lane + 32 * i;
    r[i] = d < D ? to_f(p[d]) : 0.f;
  }
}

template <int NPL, class E>
__device__ __forceinline__ float dot_row(const float* a, const E* p, int D) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    int d = lane + 32 * i;
    if (d < D) s += a[i] * to_f(p[d]);
  }
  return warp_sum(s);
}

__device__ __forceinline__ bool tree_keep(const pt_tok* tok, int q_tin, int kv) {
  pt_tok t = tok[kv];
  return t.tin <= q_tin && q_tin < t.tout;
}

template <class E, int NPL>
__global__ void k_fwd(const E* __restrict__ Q, const E* __restrict__ K, const E* __restrict__ V, int T, int Hq,
                      int Hkv, int D, float scale, const int* __restrict__ q_ptr, const int* __restrict__ kv_idx,
                      const uint8_t* __restrict__ kind, const pt_tok* __restrict__ tok, int BM, int BN,
                      int generic, const uint32_t* __restrict__ masks, const int* __restrict__ pidx,
                      E* __restrict__ O, float* __restrict__ LSE) {
  long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)T * Hq) return;
  const int q = (int)(w / Hq), h = (int)(w % Hq), hk = h / (Hq / Hkv);
  float qv[NPL], acc[NPL];
  load_row<NPL>(Q + ((long long)q * Hq + h) * D, D, qv);
#pragma unroll
  for (int i = 0; i < NPL; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  // tree maps: ancestor test plus kv <= q; other maps (generic): the partial
  // tile's keep bits, over the whole tile
  const int qt = q / BM, q_tin = generic ? 0 : tok[q].tin;
  for (int e = q_ptr[qt]; e < q_ptr[qt + 1]; ++e) {
    const int k0 = kv_idx[e] * BN;
    const bool partial = kind[e] == PT_KIND_PARTIAL;
    const int k1 = generic ? min(k0 + BN, T) : min(min(k0 + BN, T), q + 1);
    const uint32_t* mrow = (generic && partial) ? masks + ((size_t)pidx[e] * 128 + (q - qt * BM)) * 4 : nullptr;
    for (int kv = k0; kv < k1; ++kv) {
      if (partial && (mrow ? !((mrow[(kv - k0) >> 5] >> ((kv - k0) & 31)) & 1u) : !tree_keep(tok, q_tin, kv)))
        continue;
      const E* kr = K + ((long long)kv * Hkv + hk) * D;
      const E* vr = V + ((long long)kv * Hkv + hk) * D;
      float s = dot_row<NPL>(qv, kr, D) * scale;
      float mn = fmaxf(m, s);
      float c = expf(m - mn), p = expf(s - mn);
      l = l * c + p;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        int d = lane + 32 * i;
        acc[i] = acc[i] * c + (d < D ? p * to_f(vr[d]) : 0.f);
      }
      m = mn;
    }
  }
  E* orow = O + ((long long)q * Hq + h) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    int d = lane + 32 * i;
    if (d < D) from_f(orow + d, acc[i] * inv);
  }
  if (lane == 0) LSE[(long long)h * T + q] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <class E, int NPL>
__global__ void k_delta(const E* __restrict__ dO, const E* __restrict__ O, int T, int Hq, int D,
                        float* __restrict__ delta) {
  long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= (long long)T * Hq) return;
  const int q = (int)(w / Hq), h = (int)(w % Hq);
  float a[NPL];
  load_row<NPL>(dO + ((long long)q * Hq + h) * D, D, a);
  float s = dot_row<NPL>(a, O + ((long long)q * Hq + h) * D, D);
  if ((threadIdx.x & 31) == 0) delta[(long long)h * T + q] = s;
}

template <class E, int NPL>
__global__ void k_dq(const E* __restrict__ dO, const E* __restrict__ Q, const E* __restrict__ K,
                     const E* __restrict__ V, const float* __restrict__ LSE, const float* __restrict__ delta, int T,
                     int Hq, int Hkv, int D, float scale, const int* __restrict__ q_ptr,
                     const int* __restrict__ kv_idx, const uint8_t* __restrict__ kind, const pt_tok* __restrict__ tok,
                     int BM, int BN, int generic, const uint32_t* __restrict__ masks,
                     const int* __restrict__ pidx, E* __restrict__ dQ) {
  long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)T * Hq) return;
  const int q = (int)(w / Hq), h = (int)(w % Hq), hk = h / (Hq / Hkv);
  float qv[NPL], dov[NPL], acc[NPL];
  load_row<NPL>(Q + ((long long)q * Hq + h) * D, D, qv);
  load_row<NPL>(dO + ((long long)q * Hq + h) * D, D, dov);
#pragma unroll
  for (int i = 0; i < NPL; ++i) acc[i] = 0.f;
  const float lse = LSE[(long long)h * T + q], dl = delta[(long long)h * T + q];
  const int qt = q / BM, q_tin = generic ? 0 : tok[q].tin;
  for (int e = q_ptr[qt]; e < q_ptr[qt + 1]; ++e) {
    const int k0 = kv_idx[e] * BN;
    const bool partial = kind[e] == PT_KIND_PARTIAL;
    const int k1 = generic ? min(k0 + BN, T) : min(min(k0 + BN, T), q + 1);
    const uint32_t* mrow = (generic && partial) ? masks + ((size_t)pidx[e] * 128 + (q - qt * BM)) * 4 : nullptr;
    for (int kv = k0; kv < k1; ++kv) {
      if (partial && (mrow ? !((mrow[(kv - k0) >> 5] >> ((kv - k0) & 31)) & 1u) : !tree_keep(tok, q_tin, kv)))
        continue;
      const E* kr = K + ((long long)kv * Hkv + hk) * D;
      const E* vr = V + ((long long)kv * Hkv + hk) * D;
      float p = expf(dot_row<NPL>(qv, kr, D) * scale - lse);
      float ds = p * (dot_row<NPL>(dov, vr, D) - dl);
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        int d = lane + 32 * i;
        if (d < D) acc[i] += ds * to_f(kr[d]);
      }
    }
  }
  E* out = dQ + ((long long)q * Hq + h) * D;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    int d = lane + 32 * i;
    if (d < D) from_f(out + d, acc[i] * scale);
  }
}

template <class E, int NPL>
__global__ void k_dkv(const E* __restrict__ dO, const E* __restrict__ Q, const E* __restrict__ K,
                      const E* __restrict__ V, const float* __restrict__ LSE, const float* __restrict__ delta, int T,
                      int Hq, int Hkv, int D, float scale, const int* __restrict__ k_ptr,
                      const int* __restrict__ q_idx, const uint8_t* __restrict__ kindT,
                      const pt_tok* __restrict__ tok, int BM, int BN, int generic,
                      const uint32_t* __restrict__ masks, const int* __restrict__ pidxT, E* __restrict__ dK,
                      E* __restrict__ dV) {
  long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)T * Hkv) return;
  const int kv = (int)(w / Hkv), hk = (int)(w % Hkv), g = Hq / Hkv;
  float kr[NPL], vr[NPL], dk[NPL], dv[NPL];
  load_row<NPL>(K + ((long long)kv * Hkv + hk) * D, D, kr);
  load_row<NPL>(V + ((long long)kv * Hkv + hk) * D, D, vr);
#pragma unroll
  for (int i = 0; i < NPL; ++i) dk[i] = dv[i] = 0.f;
  const pt_tok ktok = generic ? pt_tok{0, 0} : tok[kv];
  const int kb = kv / BN;
  for (int e = k_ptr[kb]; e < k_ptr[kb + 1]; ++e) {
    const int q0 = q_idx[e] * BM;
    const bool partial = kindT[e] == PT_KIND_PARTIAL;
    const int qa = generic ? q0 : max(q0, kv), qb = min(q0 + BM, T);
    const uint32_t* mcol = (generic && partial) ? masks + ((size_t)pidxT[e] * 128 + (kv - kb * BN)) * 4 : nullptr;
    for (int q = qa; q < qb; ++q) {
      if (partial) {
        if (mcol) {
          if (!((mcol[(q - q0) >> 5] >> ((q - q0) & 31)) & 1u)) continue;
        } else {
          int qt = tok[q].tin;
          if (!(ktok.tin <= qt && qt < ktok.tout)) continue;
        }
      }
      for (int h = hk * g; h < (hk + 1) * g; ++h) {
        const E* qrow = Q + ((long long)q * Hq + h) * D;
        const E* dorow = dO + ((long long)q * Hq + h) * D;
        float p = expf(dot_row<NPL>(kr, qrow, D) * scale - LSE[(long long)h * T + q]);
        float ds = p * (dot_row<NPL>(vr, dorow, D) - delta[(long long)h * T + q]);
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          int d = lane + 32 * i;
          if (d < D) {
            dv[i] += p * to_f(dorow[d]);
            dk[i] += ds * to_f(qrow[d]);
          }
        }
      }
    }
  }
  E* ko = dK + ((long long)kv * Hkv + hk) * D;
  E* vo = dV + ((long long)kv * Hkv + hk) * D;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    int d = lane + 32 * i;
    if (d < D) {
      from_f(ko + d, dk[i] * scale);
      from_f(vo + d, dv[i]);
    }
  }
}

unsigned grid_for_warps(long long warps, int block) { return (unsigned)((warps * 32 + block - 1) / block); }

template <class E, int NPL>
int fwd_impl(const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
             const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  const int block = 256;
  const bool generic = bm->producer != PT_PRODUCER_TREE;  // masks from the tile bitmasks
  ProfScope ps(s, "fwd_simt");
  k_fwd<E, NPL><<<grid_for_warps((long long)T * Hq, block), block, 0, s>>>(
      (const E*)Q, (const E*)K, (const E*)V, T, Hq, Hkv, D, scale, bm->q_ptr, bm->kv_idx, bm->kind, bm->tok, bm->BM,
      bm->BN, generic ? 1 : 0, bm->mask_rows, bm->pidx, (E*)O, LSE);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("fp32 forward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

template <class E, int NPL>
int bwd_impl(const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int T,
             int Hq, int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV, float* delta,
             cudaStream_t s) {
  const int block = 256;
  const bool generic = bm->producer != PT_PRODUCER_TREE;  // masks from the tile bitmasks
  ProfScope ps(s, "bwd_simt");
  k_delta<E, NPL><<<grid_for_warps((long long)T * Hq, block), block, 0, s>>>((const E*)dO, (const E*)O, T, Hq, D, delta);
  k_dq<E, NPL><<<grid_for_warps((long long)T * Hq, block), block, 0, s>>>(
      (const E*)dO, (const E*)Q, (const E*)K, (const E*)V, LSE, delta, T, Hq, Hkv, D, scale, bm->q_ptr, bm->kv_idx,
      bm->kind, bm->tok, bm->BM, bm->BN, generic ? 1 : 0, bm->mask_rows, bm->pidx, (E*)dQ);
  k_dkv<E, NPL><<<grid_for_warps((long long)T * Hkv, block), block, 0, s>>>(
      (const E*)dO, (const E*)Q, (const E*)K, (const E*)V, LSE, delta, T, Hq, Hkv, D, scale, bm->k_ptr, bm->q_idx,
      bm->kindT, bm->tok, bm->BM, bm->BN, generic ? 1 : 0, bm->mask_cols, bm->pidxT, (E*)dK, (E*)dV);
  count_launch(3);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("fp32 backward launch failed: %s", cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

}  // namespace

int fwd_simt(bool bf16, const void* Q, const void* K, const void* V, int T, int Hq, int Hkv, int D, float scale,
             const pt_blockmap* bm, void* O, float* LSE, cudaStream_t s) {
  if (D > kMaxHeadDim) return 2;
  if (D <= 256)
    return bf16 ? fwd_impl<__nv_bfloat16, 8>(Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, s)
                : fwd_impl<float, 8>(Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, s);
  return bf16 ? fwd_impl<__nv_bfloat16, 16>(Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, s)
              : fwd_impl<float, 16>(Q, K, V, T, Hq, Hkv, D, scale, bm, O, LSE, s);
}

int bwd_simt(bool bf16, const void* dO, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             int T, int Hq, int Hkv, int D, float scale, const pt_blockmap* bm, void* dQ, void* dK, void* dV,
             float* delta, cudaStream_t s) {
  if (D > kMaxHeadDim) return 2;
  if (D <= 256)
    return bf16 ? bwd_impl<__nv_bfloat16, 8>(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, s)
                : bwd_impl<float, 8>(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, s);
  return bf16 ? bwd_impl<__nv_bfloat16, 16>(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, s)
              : bwd_impl<float, 16>(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, s);
}

}  // namespace pt
