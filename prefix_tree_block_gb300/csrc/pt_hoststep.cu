// Forward and backward of the prefix-tree attention from pinned host memory.
//
// The pages run the attention on tensors already on the GPU ("prefix_grouper_kernel.py",
// flex_shared_prefix_attention); a training step still has to bring each
// batch's Q, K, V and the upstream gradient in and take the gradients out.
// This object owns two device copies of every buffer and alternates between
// them, so a step's uploads (on one stream) and the previous step's
// downloads (on another) overlap the kernels of the step in between (on the
// caller's stream).  Events order each buffer set's reuse:
//   uploads into set b    after the kernels of the step that last used b,
//   kernels on set b      after this step's uploads and after the downloads
//                         of the step that last used b,
//   downloads from set b  after this step's kernels.
#include <cstring>
#include <new>

#include "pt.h"
#include "pt_internal.h"

struct pt_hoststep {
  int device;
  pt_dtype dtype;
  int32_t T, Hq, Hkv, D;
  size_t bq, bk, blse;  // bytes of a [T, Hq, D] tensor, a [T, Hkv, D] tensor, LSE [Hq, T]
  struct Set {
    void* mem;
    char *Q, *K, *V, *dO, *O, *dQ, *dK, *dV;
    float* LSE;
  } set[2];
  void* ws;
  size_t ws_bytes;
  cudaStream_t up, down;
  cudaEvent_t in_ready[2], do_ready[2], computed[2], out_done[2];
  bool used[2];
  int64_t n;
};

namespace {

void destroy(pt_hoststep* h) {
  if (!h) return;
  if (h->up) cudaStreamSynchronize(h->up);
  if (h->down) cudaStreamSynchronize(h->down);
  for (int b = 0; b < 2; ++b) {
    if (h->set[b].mem) cudaFree(h->set[b].mem);
    cudaEvent_t* evs[4] = {h->in_ready, h->do_ready, h->computed, h->out_done};
    for (cudaEvent_t* e : evs)
      if (e[b]) cudaEventDestroy(e[b]);
  }
  if (h->ws) cudaFree(h->ws);
  if (h->up) cudaStreamDestroy(h->up);
  if (h->down) cudaStreamDestroy(h->down);
  delete h;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

pt_status pt_hoststep_create(pt_dtype dtype, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, pt_hoststep** out) {
  if (!out) {
    pt::set_error("pt_hoststep_create: NULL out");
    return PT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if ((dtype != PT_BF16 && dtype != PT_F32) || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) {
    pt::set_error("pt_hoststep_create: bad dtype or sizes (T=%d Hq=%d Hkv=%d D=%d)", T, Hq, Hkv, D);
    return PT_ERR_INVALID_ARG;
  }
  // the head dims pt_attn_fwd and pt_attn_bwd take, refused here before any buffer is made
  if (D > 512 || (dtype == PT_BF16 && D % 8 != 0)) {
    pt::set_error("pt_hoststep_create: head_dim %d unsupported (1..512, a multiple of 8 for bf16)", D);
    return PT_ERR_UNSUPPORTED;
  }
  pt_hoststep* h = new (std::nothrow) pt_hoststep;
  if (!h) return PT_ERR_NOMEM;
  std::memset(h, 0, sizeof(*h));
  cudaGetDevice(&h->device);
  h->dtype = dtype;
  h->T = T;
  h->Hq = Hq;
  h->Hkv = Hkv;
  h->D = D;
  const size_t es = dtype == PT_BF16 ? 2 : 4;
  h->bq = (size_t)T * Hq * D * es;
  h->bk = (size_t)T * Hkv * D * es;
  h->blse = (size_t)Hq * T * sizeof(float);
  const size_t q = round256(h->bq), k = round256(h->bk), l = round256(h->blse);
  for (int b = 0; b < 2; ++b) {
    pt_hoststep::Set& s = h->set[b];
    if (cudaMalloc(&s.mem, 4 * q + 4 * k + l + 256) != cudaSuccess) {
      cudaGetLastError();
      pt::set_error("pt_hoststep_create: device allocation of %zu bytes failed", 4 * q + 4 * k + l);
      destroy(h);
      return PT_ERR_NOMEM;
    }
    char* p = static_cast<char*>(s.mem);
    s.Q = p;
    s.dO = p + q;
    s.O = p + 2 * q;
    s.dQ = p + 3 * q;
    s.K = p + 4 * q;
    s.V = s.K + k;
    s.dK = s.K + 2 * k;
    s.dV = s.K + 3 * k;
    s.LSE = reinterpret_cast<float*>(s.K + 4 * k);
  }
  h->ws_bytes = pt_bwd_workspace_bytes(T, Hq, D);
  if (h->ws_bytes && cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    pt::set_error("pt_hoststep_create: workspace allocation of %zu bytes failed", h->ws_bytes);
    destroy(h);
    return PT_ERR_NOMEM;
  }
  if (cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&h->down, cudaStreamNonBlocking) != cudaSuccess) {
    pt::set_error("pt_hoststep_create: stream creation failed");
    destroy(h);
    return PT_ERR_CUDA;
  }
  for (int b = 0; b < 2; ++b) {
    cudaEvent_t* evs[4] = {h->in_ready, h->do_ready, h->computed, h->out_done};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(&e[b], cudaEventDisableTiming) != cudaSuccess) {
        pt::set_error("pt_hoststep_create: event creation failed");
        destroy(h);
        return PT_ERR_CUDA;
      }
  }
  *out = h;
  return PT_OK;
}

pt_status pt_hoststep_run(pt_hoststep* h, const void* hQ, const void* hK, const void* hV, const void* hdO, float scale,
                          const pt_blockmap* bm, void* hdQ, void* hdK, void* hdV, cudaStream_t stream) {
  if (!h || !bm || (h->T > 0 && (!hQ || !hK || !hV || !hdO || !hdQ || !hdK || !hdV))) {
    pt::set_error("pt_hoststep_run: NULL argument");
    return PT_ERR_INVALID_ARG;
  }
  if (bm->T != h->T) {
    pt::set_error("pt_hoststep_run: map has T = %d, buffers were made for T = %d", bm->T, h->T);
    return PT_ERR_INVALID_ARG;
  }
  const int b = (int)(h->n & 1);
  pt_hoststep::Set& s = h->set[b];
  auto cuda_fail = [](const char* what) {
    pt::set_error("pt_hoststep_run: %s failed: %s", what, cudaGetErrorString(cudaGetLastError()));
    return PT_ERR_CUDA;
  };
  // uploads: K, V, Q (the forward's inputs) first, then dO
  if (h->used[b] && cudaStreamWaitEvent(h->up, h->computed[b], 0) != cudaSuccess) return cuda_fail("wait");
  if (cudaMemcpyAsync(s.K, hK, h->bk, cudaMemcpyHostToDevice, h->up) != cudaSuccess ||
      cudaMemcpyAsync(s.V, hV, h->bk, cudaMemcpyHostToDevice, h->up) != cudaSuccess ||
      cudaMemcpyAsync(s.Q, hQ, h->bq, cudaMemcpyHostToDevice, h->up) != cudaSuccess ||
      cudaEventRecord(h->in_ready[b], h->up) != cudaSuccess ||
      cudaMemcpyAsync(s.dO, hdO, h->bq, cudaMemcpyHostToDevice, h->up) != cudaSuccess ||
      cudaEventRecord(h->do_ready[b], h->up) != cudaSuccess)
    return cuda_fail("upload");
  // kernels on the caller's stream
  if (cudaStreamWaitEvent(stream, h->in_ready[b], 0) != cudaSuccess ||
      (h->used[b] && cudaStreamWaitEvent(stream, h->out_done[b], 0) != cudaSuccess))
    return cuda_fail("wait");
  pt_status st = pt_attn_fwd(s.Q, s.K, s.V, h->dtype, h->T, h->Hq, h->Hkv, h->D, scale, bm, s.O, s.LSE, stream);
  if (st != PT_OK) return st;
  if (cudaStreamWaitEvent(stream, h->do_ready[b], 0) != cudaSuccess) return cuda_fail("wait");
  st = pt_attn_bwd(s.dO, s.Q, s.K, s.V, s.O, s.LSE, h->dtype, h->T, h->Hq, h->Hkv, h->D, scale, bm, s.dQ, s.dK, s.dV,
                   h->ws, h->ws_bytes, stream);
  if (st != PT_OK) return st;
  if (cudaEventRecord(h->computed[b], stream) != cudaSuccess) return cuda_fail("record");
  // downloads once the kernels are done
  if (cudaStreamWaitEvent(h->down, h->computed[b], 0) != cudaSuccess ||
      cudaMemcpyAsync(hdK, s.dK, h->bk, cudaMemcpyDeviceToHost, h->down) != cudaSuccess ||
      cudaMemcpyAsync(hdV, s.dV, h->bk, cudaMemcpyDeviceToHost, h->down) != cudaSuccess ||
      cudaMemcpyAsync(hdQ, s.dQ, h->bq, cudaMemcpyDeviceToHost, h->down) != cudaSuccess ||
      cudaEventRecord(h->out_done[b], h->down) != cudaSuccess)
    return cuda_fail("download");
  h->used[b] = true;
  ++h->n;
  return PT_OK;
}

pt_status pt_hoststep_sync(pt_hoststep* h, cudaStream_t stream) {
  if (!h) {
    pt::set_error("pt_hoststep_sync: NULL object");
    return PT_ERR_INVALID_ARG;
  }
  for (int b = 0; b < 2; ++b)
    if (h->used[b] && cudaStreamWaitEvent(stream, h->out_done[b], 0) != cudaSuccess) {
      pt::set_error("pt_hoststep_sync: %s", cudaGetErrorString(cudaGetLastError()));
      return PT_ERR_CUDA;
    }
  return PT_OK;
}

pt_status pt_hoststep_last_forward(pt_hoststep* h, void* hO, float* hLSE) {
  if (!h || h->n == 0 || (h->T > 0 && (!hO || !hLSE))) {
    pt::set_error("pt_hoststep_last_forward: NULL argument or no step run yet");
    return PT_ERR_INVALID_ARG;
  }
  const int b = (int)((h->n - 1) & 1);
  if (cudaEventSynchronize(h->computed[b]) != cudaSuccess ||
      cudaMemcpy(hO, h->set[b].O, h->bq, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(hLSE, h->set[b].LSE, h->blse, cudaMemcpyDeviceToHost) != cudaSuccess) {
    pt::set_error("pt_hoststep_last_forward: %s", cudaGetErrorString(cudaGetLastError()));
    return PT_ERR_CUDA;
  }
  return PT_OK;
}

void pt_hoststep_free(pt_hoststep* h) { destroy(h); }

}  // extern "C"
