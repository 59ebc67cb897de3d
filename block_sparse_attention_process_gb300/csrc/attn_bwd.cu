// placeholder: replaced by the dK/dV and dQ kernels
#include "internal.h"
namespace bsa {
bsa_status dkv_launch(const bsa_bwd_args*, const bsa_mask_info*, float, cudaStream_t) {
  return fail(BSA_ERR_UNSUPPORTED, "dkv not built yet");
}
bsa_status dq_launch(const bsa_bwd_args*, const bsa_mask_info*, float, cudaStream_t) {
  return fail(BSA_ERR_UNSUPPORTED, "dq not built yet");
}
}  // namespace bsa
