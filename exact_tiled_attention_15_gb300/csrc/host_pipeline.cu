// host_pipeline.cu -- attn_fwd for inputs and outputs in host memory.
//
// The (batch, KV head) units of prefill attention are independent problems
// (each query head reads only its own group's K and V: "Fast Inference and
// Training at Scale" §6.2), so a call over host buffers is cut into chunks of
// consecutive units, and for each chunk the host-to-device copy, the kernel
// and the device-to-host copy run on three streams, three chunk buffers deep:
// while chunk c computes, chunk c+1 is copied in and chunk c-1 is copied out.
// Every chunk is an ordinary attn_fwd call on device pointers, so the result
// is the same as one attn_fwd over the whole tensors on device copies.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/attn.h"
#include "launch.h"

namespace {

constexpr int kBuffers = 3;
constexpr int kTargetChunks = 8;
constexpr long kMinCtas = 2 * 152;  // keep each chunk's launch at two waves of SMs or more
constexpr int kMaxDevices = 16;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct Plan {
  long units, per_chunk;       // (batch, KV head) units, units per chunk
  size_t q_unit, kv_unit, lse_unit;  // bytes per unit
  size_t q_off, k_off, v_off, o_off, lse_off, buffer;  // layout of one chunk buffer
};

bool make_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, Plan &p) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1 || Hq % Hkv != 0) return false;
  const long g = Hq / Hkv;
  p.units = (long)B * Hkv;
  const long qblocks = (Sq + 255) / 256;  // the prefill kernel's CTAs per query head
  long per = (p.units + kTargetChunks - 1) / kTargetChunks;
  const long min_units = (kMinCtas + g * qblocks - 1) / (g * qblocks);
  if (per < min_units) per = min_units;
  if (per > p.units) per = p.units;
  p.per_chunk = per;
  p.q_unit = (size_t)g * Sq * D * 2;
  p.kv_unit = (size_t)Sk * D * 2;
  p.lse_unit = (size_t)g * Sq * 4;
  p.q_off = 0;
  p.k_off = align256(p.q_off + per * p.q_unit);
  p.v_off = align256(p.k_off + per * p.kv_unit);
  p.o_off = align256(p.v_off + per * p.kv_unit);
  p.lse_off = align256(p.o_off + per * p.q_unit);
  p.buffer = align256(p.lse_off + per * p.lse_unit);
  return true;
}

// Two copy streams and the per-buffer events, made once per thread and device.
struct Streams {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in_done[kBuffers] = {}, comp_done[kBuffers] = {}, out_done[kBuffers] = {};
};
thread_local Streams g_streams[kMaxDevices];

cudaError_t streams_for_device(Streams *&s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  s = &g_streams[dev];
  if (s->ready) return cudaSuccess;
  e = cudaStreamCreateWithFlags(&s->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s->d2h, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->start, cudaEventDisableTiming);
  for (int b = 0; e == cudaSuccess && b < kBuffers; ++b) {
    e = cudaEventCreateWithFlags(&s->in_done[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->comp_done[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->out_done[b], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) s->ready = true;
  return e;
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D) {
  Plan p;
  if (!make_plan(B, Hq, Hkv, Sq, Sk, D, p)) return 0;
  return kBuffers * p.buffer;
}

attn_status attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                          int Sq, int Sk, int D, int causal, float scale, void *workspace, size_t workspace_bytes,
                          attn_stream_t stream) {
  attn::NvtxRange nvtx_range("attn_fwd_host");
  Plan p;
  if (!q || !k || !v || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!make_plan(B, Hq, Hkv, Sq, Sk, D, p)) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < kBuffers * p.buffer) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  Streams *s = nullptr;
  if (streams_for_device(s) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaStream_t comp = reinterpret_cast<cudaStream_t>(stream);
  const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
             *hv = static_cast<const char *>(v);
  char *ho = static_cast<char *>(o), *hl = reinterpret_cast<char *>(lse);
  char *ws = static_cast<char *>(workspace);
  // nothing touches the workspace before earlier work on the caller's stream is done
  if (cudaEventRecord(s->start, comp) != cudaSuccess || cudaStreamWaitEvent(s->h2d, s->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(s->d2h, s->start, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const long nchunks = (p.units + p.per_chunk - 1) / p.per_chunk;
  for (long c = 0; c < nchunks; ++c) {
    const int b = (int)(c % kBuffers);
    const long n0 = c * p.per_chunk, nu = (p.units - n0 < p.per_chunk) ? p.units - n0 : p.per_chunk;
    char *buf = ws + b * p.buffer;
    cudaError_t e = cudaSuccess;
    // in: after the buffer's previous chunk has been copied out
    if (c >= kBuffers) e = cudaStreamWaitEvent(s->h2d, s->out_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(buf + p.q_off, hq + n0 * p.q_unit, nu * p.q_unit, cudaMemcpyHostToDevice, s->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(buf + p.k_off, hk + n0 * p.kv_unit, nu * p.kv_unit, cudaMemcpyHostToDevice, s->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(buf + p.v_off, hv + n0 * p.kv_unit, nu * p.kv_unit, cudaMemcpyHostToDevice, s->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(s->in_done[b], s->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, s->in_done[b], 0);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    // compute: the chunk's units are consecutive (batch, KV head) pairs, i.e.
    // one batch entry of nu KV heads and nu * (Hq / Hkv) query heads
    const attn_status st = attn_fwd(buf + p.q_off, buf + p.k_off, buf + p.v_off, buf + p.o_off,
                                    lse ? reinterpret_cast<float *>(buf + p.lse_off) : nullptr, 1,
                                    (int)(nu * (Hq / Hkv)), (int)nu, Sq, Sk, D, causal, scale, stream);
    if (st != ATTN_OK) return st;
    e = cudaEventRecord(s->comp_done[b], comp);
    // out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s->d2h, s->comp_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ho + n0 * p.q_unit, buf + p.o_off, nu * p.q_unit, cudaMemcpyDeviceToHost, s->d2h);
    if (e == cudaSuccess && lse)
      e = cudaMemcpyAsync(hl + n0 * p.lse_unit, buf + p.lse_off, nu * p.lse_unit, cudaMemcpyDeviceToHost, s->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(s->out_done[b], s->d2h);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  // the caller's stream continues once the last chunk is back in host memory
  const int last = (int)((nchunks - 1) % kBuffers);
  if (cudaStreamWaitEvent(comp, s->out_done[last], 0) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
