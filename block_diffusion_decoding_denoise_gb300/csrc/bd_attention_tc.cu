// Tensor-core block attention (placeholder until the bf16 kernel lands).
#include "bd_attention.cuh"

namespace bd {
bd_status attention_tc(const AttnParams &, cudaStream_t) { return BD_ERR_UNSUPPORTED; }
}  // namespace bd
