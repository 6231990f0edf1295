// attn_api.cu -- the C ABI (include/attn.h): argument checks, TMA descriptor
// set-up and kernel dispatch.  Every argument check runs on the host before
// any CUDA call, so a bad call returns a status and leaves the GPU untouched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <mutex>

#include "../../include/attn.h"
#include "launch.h"

namespace {

// Device error word: a bounded wait that ran out records ATTN_ERR_TIMEOUT here.
__device__ unsigned g_attn_error;

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per pipeline wait

// attn_debug_stall_role_waits: when set, kernels that support it first wait
// for a signal nothing gives, with the waits between warp roles bounded by
// kStallWaitNs, so that those waits run out.
std::atomic<int> g_debug_stall{0};
constexpr uint64_t kStallWaitNs = 1000000ull;  // 1 ms

uint64_t role_wait_ns() {
  return g_debug_stall.load(std::memory_order_relaxed) ? kStallWaitNs : kDefaultTimeoutNs;
}
int debug_stall() { return g_debug_stall.load(std::memory_order_relaxed); }

// attn_debug_skew_roles: when set, forward kernels that support it run with
// fixed delays in some warp roles, so that others run ahead of them.
std::atomic<int> g_debug_skew{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

// Device address of the error word on the current device (nullptr on failure).
unsigned *error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned *>(p);
  }
  return g_err_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sm103_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  return major == 10 && minor == 3;
}

// 3-D tiled tensor map over a dense [planes, rows, cols] array.
bool make_tmap(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem_bytes, uint64_t cols,
               uint64_t rows, uint64_t planes, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * elem_bytes, cols * rows * elem_bytes};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

attn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return ATTN_ERR_CUDA;
}

bool bad_scale(float s) { return !(s > 0.f) || !std::isfinite(s); }

attn_status check_prefill(const void *q, const void *k, const void *v, const void *o, int B, int Hq, int Hkv,
                          int Sq, int Sk, int D, float scale) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (bad_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  // TMA coordinates are 32-bit: keep every plane count and row count in range.
  if ((int64_t)B * Hq > (1LL << 30) || (int64_t)B * Hkv > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

}  // namespace

extern "C" {

const char *attn_status_str(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_NO_DEVICE: return "ATTN_ERR_NO_DEVICE";
    case ATTN_ERR_SCRATCH_LIMIT: return "ATTN_ERR_SCRATCH_LIMIT";
    case ATTN_ERR_BAD_INDEX: return "ATTN_ERR_BAD_INDEX";
  }
  return "ATTN_ERR_UNKNOWN";
}

const char *attn_version(void) { return "0.1.0"; }

attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int causal, float scale, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_fwd");
  attn_status st = check_prefill(q, k, v, o, B, Hq, Hkv, Sq, Sk, D, scale);
  if (st != ATTN_OK) return st;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  CUtensorMap tq, tk, tv;
  if (!make_tmap(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sq, (uint64_t)B * Hq, 64, 128) ||
      !make_tmap(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, (uint64_t)B * Hkv, 64, 128) ||
      !make_tmap(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, (uint64_t)B * Hkv, 64, 128))
    return ATTN_ERR_CUDA;
  attn::FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.skew = g_debug_skew.load(std::memory_order_relaxed);
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_fwd_bf16(a, tq, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D) {
  return attn_decode_multi_workspace_bytes(B, Hq, Hkv, 1, Lmax, D);
}

size_t attn_decode_multi_workspace_bytes(int B, int Hq, int Hkv, int T, int Lmax, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || T > 16 || Lmax < 1 || D < 1 || Hq % Hkv != 0) return 0;
  const int chunk = attn::decode_chunk(B, Hq, Hkv, T, Lmax);
  const size_t ns = (size_t)attn::decode_nsplit(Lmax, chunk);
  const size_t rows = (size_t)B * Hq * T * ns;
  size_t o_bytes = rows * (size_t)D * sizeof(float);
  o_bytes = (o_bytes + 255) / 256 * 256;
  return o_bytes + rows * sizeof(float);
}

attn_status attn_decode(const void *q, const void *kcache, const void *vcache, const int32_t *seqlens, void *o,
                        float *lse, int B, int Hq, int Hkv, int Lmax, int D, float scale, void *workspace,
                        size_t workspace_bytes, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_decode");
  if (!q || !kcache || !vcache || !seqlens || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || D < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (bad_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv > (1LL << 30) || (int64_t)B * Hq > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  CUtensorMap tk, tv;
  if (!make_tmap(&tk, kcache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Lmax, (uint64_t)B * Hkv, 64, 64) ||
      !make_tmap(&tv, vcache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Lmax, (uint64_t)B * Hkv, 64, 64))
    return ATTN_ERR_CUDA;
  attn::DecodeArgs a{};
  a.q = q;
  a.seqlens = seqlens;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.D = D;
  a.T = 1;
  a.causal = 0;
  a.chunk = attn::decode_chunk(B, Hq, Hkv, 1, Lmax);
  a.nsplit = attn::decode_nsplit(Lmax, a.chunk);
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  const size_t rows = (size_t)B * Hq * a.nsplit;
  size_t o_bytes = (rows * (size_t)D * sizeof(float) + 255) / 256 * 256;
  a.part_o = static_cast<float *>(workspace);
  a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
  return from_cuda(attn::launch_decode(a, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

attn_status attn_decode_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                              const int32_t *seqlens, void *o, float *lse, int B, int Hq, int Hkv, int page_size,
                              int max_blocks, int num_pages, int D, float scale, void *workspace,
                              size_t workspace_bytes, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_decode_paged");
  if (!q || !k_pages || !v_pages || !block_table || !seqlens || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_pages < 1 || D < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (page_size < 1 || (int64_t)max_blocks * page_size > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  if (bad_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens) | reinterpret_cast<uintptr_t>(block_table)) & 3u) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID_ARG;
  const int Lmax = max_blocks * page_size;
  if (workspace_bytes < attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128 && page_size != 256)
    return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * Hkv > (1LL << 30) || (int64_t)B * Hq > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  const uint32_t box_rows = page_size < 64 ? (uint32_t)page_size : 64u;
  CUtensorMap tk, tv;
  if (!make_tmap(&tk, k_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, page_size, (uint64_t)num_pages * Hkv, 64,
                 box_rows) ||
      !make_tmap(&tv, v_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, page_size, (uint64_t)num_pages * Hkv, 64,
                 box_rows))
    return ATTN_ERR_CUDA;
  attn::DecodeArgs a{};
  a.q = q;
  a.seqlens = seqlens;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.D = D;
  a.T = 1;
  a.causal = 0;
  a.chunk = attn::decode_chunk(B, Hq, Hkv, 1, Lmax);
  a.nsplit = attn::decode_nsplit(Lmax, a.chunk);
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  const size_t rows = (size_t)B * Hq * a.nsplit;
  size_t o_bytes = (rows * (size_t)D * sizeof(float) + 255) / 256 * 256;
  a.part_o = static_cast<float *>(workspace);
  a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
  return from_cuda(attn::launch_decode(a, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

attn_status attn_decode_multi(const void *q, const void *kcache, const void *vcache, const int32_t *seqlens, void *o,
                              float *lse, int B, int Hq, int Hkv, int T, int Lmax, int D, int causal, float scale,
                              void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_decode_multi");
  if (!q || !kcache || !vcache || !seqlens || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || D < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (T < 1 || T > 16) return ATTN_ERR_UNSUPPORTED;
  if (bad_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_decode_multi_workspace_bytes(B, Hq, Hkv, T, Lmax, D)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv > (1LL << 30) || (int64_t)B * Hq * T > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  CUtensorMap tk, tv;
  if (!make_tmap(&tk, kcache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Lmax, (uint64_t)B * Hkv, 64, 64) ||
      !make_tmap(&tv, vcache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Lmax, (uint64_t)B * Hkv, 64, 64))
    return ATTN_ERR_CUDA;
  attn::DecodeArgs a{};
  a.q = q;
  a.seqlens = seqlens;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.D = D;
  a.T = T;
  a.causal = causal ? 1 : 0;
  a.chunk = attn::decode_chunk(B, Hq, Hkv, T, Lmax);
  a.nsplit = attn::decode_nsplit(Lmax, a.chunk);
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  const size_t rows = (size_t)B * Hq * T * a.nsplit;
  size_t o_bytes = (rows * (size_t)D * sizeof(float) + 255) / 256 * 256;
  a.part_o = static_cast<float *>(workspace);
  a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
  return from_cuda(attn::launch_decode(a, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

attn_status attn_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8, const float *q_scale,
                         const float *k_scale, const float *v_scale, void *o, float *lse, int B, int Hq, int Hkv,
                         int Sq, int Sk, int D, int causal, float scale, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_fwd_fp8");
  attn_status st = check_prefill(q8, k8, v8, o, B, Hq, Hkv, Sq, Sk, D, scale);
  if (st != ATTN_OK) return st;
  if (!q_scale || !k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  // 128-column boxes: for D = 64 the upper 64 columns of a box lie outside the
  // tensor and arrive as zeros
  CUtensorMap tq, tk, tv;
  if (!make_tmap(&tq, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, Sq, (uint64_t)B * Hq, 128, 128) ||
      !make_tmap(&tk, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, Sk, (uint64_t)B * Hkv, 128, 128) ||
      !make_tmap(&tv, v8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, Sk, (uint64_t)B * Hkv, 128, 128))
    return ATTN_ERR_CUDA;
  attn::FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.skew = g_debug_skew.load(std::memory_order_relaxed);
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_fwd_fp8(a, tq, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq, int D) {
  if (B < 1 || Hq < 1 || Sq < 1 || D < 1) return 0;
  const size_t rows = (size_t)B * Hq * Sq;
  return (rows * D * sizeof(float) + 255) / 256 * 256 + rows * sizeof(float);
}

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                     void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                     float scale, void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_bwd");
  attn_status st = check_prefill(q, k, v, o, B, Hq, Hkv, Sq, Sk, D, scale);
  if (st != ATTN_OK) return st;
  if (!lse || !dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Sq, D)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sq, (uint64_t)B * Hq, 64, 128) ||
      !make_tmap(&tdo, dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sq, (uint64_t)B * Hq, 64, 128) ||
      !make_tmap(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, (uint64_t)B * Hkv, 64, 128) ||
      !make_tmap(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, Sk, (uint64_t)B * Hkv, 64, 128))
    return ATTN_ERR_CUDA;
  const size_t rows = (size_t)B * Hq * Sq;
  float *dq_acc = static_cast<float *>(workspace);
  // fp32 dQ accumulator, reduced into by TMA in 128-row x 32-column boxes
  CUtensorMap tdq;
  if (!make_tmap(&tdq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, Sq, (uint64_t)B * Hq, 32, 128))
    return ATTN_ERR_CUDA;
  attn::BwdArgs a{};
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = dq_acc;
  a.dvec = reinterpret_cast<float *>(static_cast<char *>(workspace) + (rows * D * sizeof(float) + 255) / 256 * 256);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd(a, tq, tk, tv, tdo, tdq, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

// Host-side checks of one tensor of a rotate + quantise call (no CUDA call).
attn_status check_quant_tensor(const void *x, const uint8_t *codes, const float *scales, int B, int H, int S) {
  if (!x || !codes || !scales) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return ATTN_ERR_INVALID_ARG;
  if ((int64_t)B * H > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;  // TMA plane coordinate
  return ATTN_OK;
}

// Adds one checked tensor to the launch.
// For D = 64 the kernel still reads two 64-column slabs (the second lies
// outside the tensor and arrives as zeros) and stores 128-column boxes of
// codes, whose upper 64 columns lie outside the tensor and are dropped.
attn_status add_quant_tensor(attn::QuantArgs &a, const void *x, uint8_t *codes, float *scales, int B, int H, int S,
                             int D, int rotate) {
  const int i = a.n;
  if (!make_tmap(&a.tmx[i], x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, S, (uint64_t)B * H, 64, 128) ||
      !make_tmap(&a.tmc[i], codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D, S, (uint64_t)B * H, 128, 128))
    return ATTN_ERR_CUDA;
  a.scales[i] = scales;
  a.nts[i] = (S + 127) / 128;
  a.rotate[i] = rotate ? 1 : 0;
  a.first[i + 1] = a.first[i] + (long)a.nts[i] * B * H;
  a.n = i + 1;
  return ATTN_OK;
}

attn_status launch_quant(attn::QuantArgs &a, attn_stream_t stream) {
  a.timeout_ns = kDefaultTimeoutNs;
  a.wait_ns = role_wait_ns();
  a.stall = debug_stall();
  a.err = error_word();
  if (!a.err) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_rotate_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

attn_status attn_rotate_quantize_fp8(const void *x, uint8_t *codes, float *scales, const float *signs, int B, int H,
                                     int S, int D, attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_rotate_quantize_fp8");
  if (D < 1) return ATTN_ERR_INVALID_ARG;
  if (signs && (reinterpret_cast<uintptr_t>(signs) & 3u)) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_quant_tensor(x, codes, scales, B, H, S);
  if (st != ATTN_OK) return st;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  attn::QuantArgs a{};
  a.signs = signs;
  a.d = D;
  st = add_quant_tensor(a, x, codes, scales, B, H, S, D, signs != nullptr);
  if (st != ATTN_OK) return st;
  return launch_quant(a, stream);
}

attn_status attn_rotate_quantize_fp8_many(const attn_quant_tensor *tensors, int n, const float *signs, int D,
                                          attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_rotate_quantize_fp8_many");
  if (!tensors || n < 1) return ATTN_ERR_INVALID_ARG;
  if (n > ATTN_QUANT_MAX_TENSORS) return ATTN_ERR_UNSUPPORTED;
  if (D < 1) return ATTN_ERR_INVALID_ARG;
  bool any_rot = false;
  for (int i = 0; i < n; ++i) any_rot |= tensors[i].rotate != 0;
  if (any_rot && (!signs || (reinterpret_cast<uintptr_t>(signs) & 3u))) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const attn_quant_tensor &t = tensors[i];
    const attn_status st = check_quant_tensor(t.x, t.codes, t.scales, t.B, t.H, t.S);
    if (st != ATTN_OK) return st;
  }
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!sm103_device()) return ATTN_ERR_NO_DEVICE;
  attn::QuantArgs a{};
  a.signs = any_rot ? signs : nullptr;
  a.d = D;
  for (int i = 0; i < n; ++i) {
    const attn_quant_tensor &t = tensors[i];
    attn_status st = add_quant_tensor(a, t.x, t.codes, t.scales, t.B, t.H, t.S, D, t.rotate);
    if (st != ATTN_OK) return st;
  }
  return launch_quant(a, stream);
}

void attn_debug_stall_role_waits(int enable) { g_debug_stall.store(enable ? 1 : 0, std::memory_order_relaxed); }

void attn_debug_skew_roles(int enable) { g_debug_skew.store(enable ? 1 : 0, std::memory_order_relaxed); }

attn_status attn_get_error(attn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned *p = error_word();
  if (!p) return ATTN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return v == 0 ? ATTN_OK : static_cast<attn_status>(v);
}

}  // extern "C"
