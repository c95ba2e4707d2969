// bf16 grouped GEMMs on tcgen05 tensor cores (placeholder until the kernels land).
#include "common.cuh"

namespace moe {

int launch_gmm_bf16_gate_up(const void*, const void*, const void*, const int32_t*, int, int, int,
                            int, void*, void*, int32_t*, cudaStream_t) {
  return MOE_ERR_UNSUPPORTED;
}
int launch_gmm_bf16_down(const void*, const void*, const int32_t*, int, int, int, int, void*,
                         int32_t*, cudaStream_t) {
  return MOE_ERR_UNSUPPORTED;
}
int launch_mlp_grad_bf16(const void*, const void*, const void*, const void*, const int32_t*, int,
                         int, int, int, const void*, const void*, const void*, void*, void*,
                         void*, void*, void*, int32_t*, cudaStream_t) {
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
