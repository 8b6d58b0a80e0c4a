// pt_bwd_tc.cu -- tensor-core backward for bf16 (placeholder until written).
#include "pt_device.cuh"
#include "pt_internal.h"

namespace pt {
int take_status_bwd(cudaStream_t s) { return take_status_here(s); }
int bwd_tc(const void*, const void*, const void*, const void*, const void*, const float*, int, int, int, int, float,
           const pt_blockmap*, void*, void*, void*, float*, float*, cudaStream_t) {
  set_error("tensor-core backward not built yet");
  return 2;
}
}  // namespace pt
