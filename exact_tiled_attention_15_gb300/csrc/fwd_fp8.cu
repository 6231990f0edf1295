// fwd_fp8.cu -- FP8 e4m3 prefill entry (attn_fwd_fp8): instantiates the shared
// tcgen05 kernel of fwd_kernel.cuh with kind::f8f6f4 MMAs, head dimension 128
// (one 128 x 128 scale tile spans the head dimension).
#include "fwd_kernel.cuh"

namespace attn {

cudaError_t launch_fwd_fp8(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           cudaStream_t stream) {
  if (a.D == 128) return fwd::launch<fwd::Fp8, 128>(a, tq, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
