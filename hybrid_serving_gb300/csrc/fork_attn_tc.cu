// fork_attn_tc.cu -- tensor-core ForkAttention (bf16, d = 128) for sm_103a.
// Placeholder until the tcgen05 kernel lands: declines every call so that
// the CUDA-core path runs.
#include "device.cuh"

hs_status hs_fork_attn_tc_launch(const hs_round_caps*, const void*, int, int, int, float, const void*, const void*,
                                 const void*, int, void*, int32_t*, cudaStream_t) {
  return HS_EUNSUPPORTED;
}
