// pt_noalloc.cu -- pt_attn_bwd_noalloc: the backward pass without any device
// allocation, for callers that cannot call cudaMalloc.
//
// Some programs that embed this library own all device memory themselves: a
// serving process or a training framework that hands every byte out through
// its own allocator, and gives a plugin no hook to allocate more.  Others run
// the backward on a latency-critical path where cudaMalloc, which can
// synchronise the device, is not acceptable.  pt_attn_bwd asks its caller for
// scratch (Delta and LSE*log2(e) rows); this variant takes that scratch from a
// fixed array compiled into the library instead, so the caller passes only
// inputs and outputs.
//
// The array below is a file-scope __device__ object: every GPU that loads the
// library holds it (kNoallocScratchBytes) until the process exits.  In host
// code its name is only a host-side stand-in, not a device address, so the
// address handed to kernels is looked up with cudaGetSymbolAddress, once per
// device, with that device current.
#include <cmath>
#include <mutex>

#include "pt.h"
#include "pt_internal.h"

namespace {

// Room for two fp32 row statistics of Hq * ceil(T/128)*128 entries each:
// 2^21 floats (8 MiB) covers, for example, Hq = 32 heads at T = 32768.
constexpr size_t kNoallocScratchFloats = size_t(1) << 21;
constexpr size_t kNoallocScratchBytes = kNoallocScratchFloats * sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on `dev` (the current device); looked
// up on the first call for that device.
float* scratch_for_device(int dev) {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      pt::set_error("pt_attn_bwd_noalloc: cudaGetSymbolAddress failed on device %d: %s", dev, cudaGetErrorString(e));
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" size_t pt_bwd_noalloc_max_scratch_bytes(void) { return kNoallocScratchBytes; }

extern "C" pt_status pt_attn_bwd_noalloc(const void* dO, const void* Q, const void* K, const void* V,
                                         const void* O, const float* LSE, pt_dtype dtype, int32_t T, int32_t Hq,
                                         int32_t Hkv, int32_t D, float scale, const pt_blockmap* bm, void* dQ,
                                         void* dK, void* dV, cudaStream_t stream) {
  // Same checks as pt_attn_bwd, done here so nothing below allocates.
  if (!bm) {
    pt::set_error("pt_attn_bwd_noalloc: block map is NULL");
    return PT_ERR_INVALID_ARG;
  }
  if (T != bm->T || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || (dtype != PT_BF16 && dtype != PT_F32)) {
    pt::set_error("pt_attn_bwd_noalloc: bad shape or dtype (T=%d vs map T=%d, Hq=%d, Hkv=%d, D=%d)", T, bm->T, Hq,
                  Hkv, D);
    return PT_ERR_INVALID_ARG;
  }
  if (D > 512) {  // as pt_attn_bwd: head dims above 256 run on the CUDA-core kernels, up to 512
    pt::set_error("pt_attn_bwd_noalloc: head_dim %d outside 1..512", D);
    return PT_ERR_UNSUPPORTED;
  }
  if (T == 0) return PT_OK;
  const void* ptrs[] = {dO, Q, K, V, O, LSE, dQ, dK, dV};
  for (const void* p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) {
      pt::set_error("pt_attn_bwd_noalloc: tensor pointers must be non-NULL and 16-byte aligned");
      return PT_ERR_INVALID_ARG;
    }
  const size_t tpad = ((size_t)T + 127) / 128 * 128;
  const size_t half = round256(sizeof(float) * tpad * Hq);
  if (2 * half > kNoallocScratchBytes) {
    pt::set_error(
        "pt_attn_bwd_noalloc: needs %zu bytes of scratch for T=%d, Hq=%d but the built-in array holds %zu; "
        "use pt_attn_bwd with a caller workspace",
        2 * half, T, Hq, kNoallocScratchBytes);
    return PT_ERR_INVALID_ARG;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || dev != bm->device) {
    pt::set_error("pt_attn_bwd_noalloc: current device %d is not the block map's device %d", dev, bm->device);
    return PT_ERR_INVALID_ARG;
  }
  float* base = scratch_for_device(dev);
  if (!base) return PT_ERR_CUDA;
  float* delta = base;
  float* lse2 = reinterpret_cast<float*>(reinterpret_cast<char*>(base) + half);
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)D);
  // Both kernel families overwrite every scratch entry they later read, so
  // the previous call's contents never need clearing.
  int rc;
  if (dtype == PT_BF16 && bm->BM == 128 && bm->BN == 128 && pt::bwd_tc_supported(D))
    rc = pt::bwd_tc(dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, lse2, nullptr, 0, false, stream);
  else if (dtype == PT_BF16 && D % 8 != 0) {
    pt::set_error("pt_attn_bwd_noalloc: bf16 needs head_dim %% 8 == 0 (got %d)", D);
    return PT_ERR_UNSUPPORTED;
  } else
    rc = pt::bwd_simt(dtype == PT_BF16, dO, Q, K, V, O, LSE, T, Hq, Hkv, D, scale, bm, dQ, dK, dV, delta, stream);
  switch (rc) {
    case 0: return PT_OK;
    case 1: return PT_ERR_INVALID_ARG;
    case 2: return PT_ERR_UNSUPPORTED;
    default: return PT_ERR_CUDA;
  }
}
