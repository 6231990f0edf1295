// fwd_fp8.cu -- FP8 e4m3 prefill entry (attn_fwd_fp8): instantiates the shared
// tcgen05 kernel of fwd_kernel.cuh with kind::f8f6f4 MMAs, head dimension 128
// (one 128 x 128 scale tile spans the head dimension).  Head dimension 64 runs
// on the same kernel: its tensor maps are 64 columns wide with 128-column
// boxes, so TMA reads the upper 64 columns of every tile as zeros, which add
// nothing to Q K^T and make the upper half of O zero; only D columns of O are
// written.
#include "fwd_kernel.cuh"

namespace attn {

cudaError_t launch_fwd_fp8(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           cudaStream_t stream) {
  if (a.D == 128 || a.D == 64) return fwd::launch<fwd::Fp8, 128>(a, tq, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
