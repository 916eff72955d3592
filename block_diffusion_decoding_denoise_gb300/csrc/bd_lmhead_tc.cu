// Tensor-core LM head (placeholder until the tcgen05 kernel lands).
#include "bd_confidence.cuh"

namespace bd {
bool lmhead_tc_supported(const ConfParams &) { return false; }
int lmhead_tc_num_partials(int) { return 0; }
bd_status lmhead_tc(const ConfParams &, cudaStream_t) { return BD_ERR_UNSUPPORTED; }
}  // namespace bd
