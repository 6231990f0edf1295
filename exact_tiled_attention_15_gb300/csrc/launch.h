// launch.h -- host-side launchers shared between the kernel translation units
// and the C ABI layer (attn_api.cu).  Internal: not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdint>

namespace attn {

// An NVTX range named after the entry point, open for the duration of the
// call (its host-side work and launches), so that profilers and tracing tools
// show each call of the library on the timeline.  Costs a pointer check when
// no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

// Query heads one decode CTA covers: nhpc * T query rows fit the 16 MMA rows.
inline int decode_heads_per_cta(int Hq, int Hkv, int T) {
  const int g = Hq / Hkv, n = 16 / T;
  return n < g ? n : g;
}
// Keys per split of the decode kernel for these sizes (a multiple of 64);
// T = query tokens per sequence.
int decode_chunk(int B, int Hq, int Hkv, int T, int Lmax);
// Number of key splits for a cache of Lmax rows.
inline int decode_nsplit(int Lmax, int chunk) { return (Lmax + chunk - 1) / chunk; }

struct DecodeArgs {
  const void *q;
  const int32_t *seqlens;
  const int32_t *block_table;  // nullptr: contiguous cache; else [B, max_blocks] page ids
  int max_blocks, page_size, num_pages;
  void *o;
  float *lse;
  float *part_o;    // [B, Hq, nsplit, D]
  float *part_lse;  // [B, Hq, nsplit], log2 domain
  int B, Hq, Hkv, Lmax, D, chunk, nsplit;
  int T, causal;  // query tokens per sequence; bottom-right causal mask among them
  float scale;
  uint64_t timeout_ns;  // waits on copies
  uint64_t wait_ns;     // waits of one warp role on another (producer <-> consumers)
  int stall;            // test hook: the consumer warps first wait for a signal nothing gives
  unsigned *err;
};

// Launch split kernel + combine kernel.  tmap_k / tmap_v describe the caches as
// 3-D tensors (D, Lmax, B*Hkv) with 64 x 64 boxes and 128-byte swizzle, or for a
// paged cache the pools as (D, page_size, num_pages*Hkv) with 64 x
// min(page_size, 64) boxes.
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                          cudaStream_t stream);

struct FwdArgs {
  void *o;
  float *lse;
  const float *q_scale, *k_scale, *v_scale;  // FP8 only
  int B, Hq, Hkv, Sq, Sk, D, causal;
  float scale;
  uint64_t timeout_ns;  // waits on copies and on a CTA's own tensor-core work
  uint64_t wait_ns;     // waits of one warp role on another inside a CTA
  int stall;            // test hook: the softmax first waits for a signal nothing gives
  int skew;             // test hook: fixed delays that let one warp role run ahead of another
  unsigned *err;
};

// bf16 prefill.  tmap_q/k/v: 3-D tensors (D, S, B*H) with 64 x 128 boxes, 128B swizzle.
cudaError_t launch_fwd_bf16(const FwdArgs &a, const CUtensorMap &tmap_q, const CUtensorMap &tmap_k,
                            const CUtensorMap &tmap_v, cudaStream_t stream);

// FP8 prefill.  tmap_q/k/v: 3-D tensors (D, S, B*H) of bytes with 128 x 128 boxes.
cudaError_t launch_fwd_fp8(const FwdArgs &a, const CUtensorMap &tmap_q, const CUtensorMap &tmap_k,
                           const CUtensorMap &tmap_v, cudaStream_t stream);

struct BwdArgs {
  const void *o, *dout;  // bf16 [B, Hq, Sq, D]
  const float *lse;      // [B, Hq, Sq]
  void *dq, *dk, *dv;    // bf16 outputs
  float *dq_acc;         // workspace [B, Hq, Sq, D] fp32
  float *dvec;           // workspace [B, Hq, Sq]
  int B, Hq, Hkv, Sq, Sk, D, causal;
  float scale;
  uint64_t timeout_ns;  // waits on copies and on a CTA's own tensor-core work
  uint64_t wait_ns;     // waits of one warp role on another inside a CTA
  int stall;            // test hook: the compute warps first wait for a signal nothing gives
  unsigned *err;
};

// Backward: Dvec + zero accumulator, main kernel, dQ conversion.  tq/tk/tv/tdo:
// 3-D tensor maps (D, S, B*H) with 64 x 128 boxes, 128-byte swizzle.
cudaError_t launch_bwd(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdq, cudaStream_t stream);

// Hadamard rotation + per-128x128-tile e4m3 quantisation of up to
// kQuantMaxTensors bf16 [B, H, S, 128] tensors in one launch.  Per tensor i:
// tmx[i] maps x as [B*H, S, 128] bf16 (64 x 128 boxes), tmc[i] the codes as
// [B*H, S, 128] uint8 (128 x 128 boxes), both 128-byte swizzled; its tiles are
// the launch's tiles first[i] .. first[i+1] - 1, nts[i] per (b, h) matrix;
// rotate[i] selects y = x H diag(signs) / sqrt(128) (else y = x).
constexpr int kQuantMaxTensors = 4;
struct QuantArgs {
  CUtensorMap tmx[kQuantMaxTensors], tmc[kQuantMaxTensors];
  float *scales[kQuantMaxTensors];
  long first[kQuantMaxTensors + 1];
  int nts[kQuantMaxTensors];
  int rotate[kQuantMaxTensors];
  int n;
  int d;                // head dimension, 64 or 128 (a 64-wide tensor is read as 128 columns, the upper 64 zero)
  const float *signs;  // [d] of +-1; read only when some rotate[i] is set
  uint64_t timeout_ns;  // waits on copies and on a CTA's own tensor-core work
  uint64_t wait_ns;     // waits of one warp role on another inside a CTA
  int stall;            // test hook: the epilogue warps first wait for a signal nothing gives
  unsigned *err;
};
cudaError_t launch_rotate_quantize(const QuantArgs &a, cudaStream_t stream);

}  // namespace attn
