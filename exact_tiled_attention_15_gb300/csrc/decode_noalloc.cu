// decode_noalloc.cu -- attn_decode_noalloc: the split-K decode with its scratch
// in a fixed static device array instead of a caller-provided workspace.
//
// Who needs it: callers that are handed only input and output buffers and have
// no way to obtain device scratch -- a custom-op or plugin interface without a
// workspace slot, or a serving loop that must not call cudaMalloc (which can
// synchronise the device) and has no memory pool of its own.  This entry point
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
//
// The scratch is the file-scope array below.  Its size is fixed at
// ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB); every GPU on which this module is
// loaded keeps those 16 MiB until the process exits.  In host code the array's
// name is only a host-side stand-in, never a device address: its device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on that device.  That first call
// therefore makes runtime calls beyond the launches (the lookup) and should
// come before any stream capture.
//
// Every call shares the one array and leaves its contents behind.  The decode
// kernels write every scratch entry they later read, so nothing has to start
// at zero.  Calls whose GPU work overlaps (different streams, or different
// host threads on the same device) race on the array and give wrong results:
// serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device, looked up on first use.
void *scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" attn_status attn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                                           const int32_t *seqlens, void *o, float *lse, int B, int Hq, int Hkv,
                                           int Lmax, int D, float scale, attn_stream_t stream) {
  const size_t need = attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D);
  if (need == 0) return ATTN_ERR_INVALID_ARG;  // sizes that attn_decode would reject
  if (need > (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH_LIMIT;
  if (!q || !kcache || !vcache || !seqlens || !o) return ATTN_ERR_INVALID_ARG;
  void *ws = scratch_address();
  if (!ws) return ATTN_ERR_CUDA;
  return attn_decode(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, Lmax, D, scale, ws,
                     (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
