// fwd_fp8.cu -- placeholder until the FP8 prefill kernel lands.
#include "launch.h"
namespace attn {
cudaError_t launch_fwd_fp8(const FwdArgs &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                           cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace attn
