// Mixture-of-experts block (placeholder until the MoE kernels land).
#include "common.cuh"
#include "internal.h"
#include "layer.h"

namespace qwen {

qwen_status moe_forward(qwen_layer_s*, const bf16*, const float*, bf16*, int, int32_t*, float*,
                        float*, uint8_t*, const WorkspaceLayout&, cudaStream_t) {
  return QWEN_ERR_UNSUPPORTED;
}

}  // namespace qwen
