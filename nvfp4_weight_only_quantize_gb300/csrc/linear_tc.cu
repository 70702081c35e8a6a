// Tensor-core (tcgen05) path of the NVFP4 LoRA linear.
#include "linear.cuh"

namespace qerl {

size_t tc_fwd_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }
size_t tc_bwd_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }
qerl_status tc_linear_fwd(const FwdArgs &, char *, size_t, cudaStream_t) { return QERL_ERR_SHAPE; }
qerl_status tc_linear_bwd(const BwdArgs &, char *, size_t, cudaStream_t) { return QERL_ERR_SHAPE; }

}  // namespace qerl
