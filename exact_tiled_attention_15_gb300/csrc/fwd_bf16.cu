// fwd_bf16.cu -- bf16 prefill entry (attn_fwd): instantiates the shared
// tcgen05 kernel of fwd_kernel.cuh for head dimensions 64 and 128.
#include "fwd_kernel.cuh"

namespace attn {

cudaError_t launch_fwd_bf16(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream) {
  if (a.D == 128) return fwd::launch<fwd::Bf16, 128>(a, tq, tk, tv, stream);
  if (a.D == 64) return fwd::launch<fwd::Bf16, 64>(a, tq, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
