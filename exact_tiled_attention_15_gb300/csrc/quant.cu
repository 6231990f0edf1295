// quant.cu -- fused Hadamard rotation + per-tile FP8 e4m3 quantisation.
//
// "FlashAttention scaling, multi-GPU training and weight quantization" §1
// (FlashAttention-3): before the FP8 attention, Q and K are multiplied by a
// random orthogonal matrix to spread outliers (incoherent processing) and
// each small tile is quantised with its own scale (block quantisation).
// Here R = H_D diag(s) / sqrt(D) (Sylvester Hadamard H_D, signs s), one tile =
// 128 rows x 128 columns of a (b, h) matrix, scale = max |y| / 448 (1 for an
// all-zero tile), code = e4m3(y / scale) rounded to nearest even and held at
// +-448.  HBM-bound: each bf16 input byte is read once and each code written
// once.
//
// Persistent CTAs (two per SM) walk the tiles; per tile 256 threads = 64 rows x
// 4 lanes per pass, 2 passes, and the next tile's loads are in flight while the
// current one is transformed.
// A lane holds 32 consecutive columns; the 128-point fast Walsh-Hadamard
// transform runs 5 butterfly stages inside the lane and 2 across the row's
// four lanes (xor shuffles).  The tile's amax is reduced across the CTA before
// any code is written; codes are y * (1 / scale) rounded by the e4m3
// conversion.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "launch.h"

namespace attn {
namespace qnt {

constexpr int TR = 128;  // rows per tile
constexpr int DQ = 128;  // head dimension (one tile wide)
constexpr int THREADS = 256;
constexpr int LPR = 4;                             // lanes per row
constexpr int CPL = DQ / LPR;                      // 32 consecutive columns per lane
constexpr int PASSES = TR / (THREADS / LPR);       // 2

// Loads one tile's rows for this thread (2 rows x 64 bytes).
__device__ __forceinline__ void load_tile(uint4 (&raw)[PASSES][4], const __nv_bfloat16 *__restrict__ x, long t,
                                          int nts, int S, int rloc, int sub) {
  const long bh = t / nts;
  const int tile = (int)(t % nts);
  const size_t base = ((size_t)bh * S + (size_t)tile * TR) * DQ;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int row = ps * (THREADS / LPR) + rloc;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + base + (size_t)row * DQ) + sub * 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[ps][k] = (tile * TR + row < S) ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
  }
}

// Persistent: CTA c handles tiles c, c + gridDim.x, ... (tile index = bh * nts
// + tile row), loading the next tile while it transforms the current one.
__global__ void __launch_bounds__(THREADS, 2) rotate_quantize_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                     uint8_t *__restrict__ codes,
                                                                     float *__restrict__ scales,
                                                                     const float *__restrict__ signs, int S, int nts,
                                                                     long ntiles) {
  __shared__ float s_red[2][THREADS / 32];
  const int rloc = threadIdx.x / LPR;  // row within a pass
  const int sub = threadIdx.x % LPR;   // 32-column segment of the row
  uint4 nxt[PASSES][4];
  if ((long)blockIdx.x < ntiles) load_tile(nxt, x, blockIdx.x, nts, S, rloc, sub);
  int parity = 0;
  for (long t = blockIdx.x; t < ntiles; t += gridDim.x, parity ^= 1) {
  const long bh = t / nts;
  const int tile = (int)(t % nts);
  const size_t base = ((size_t)bh * S + (size_t)tile * TR) * DQ;
  uint4 raw[PASSES][4];
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps)
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[ps][k] = nxt[ps][k];
  if (t + gridDim.x < ntiles) load_tile(nxt, x, t + gridDim.x, nts, S, rloc, sub);
  float y[PASSES][CPL];
  float amax = 0.f;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    float *v = y[ps];
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(raw[ps]);
#pragma unroll
    for (int k = 0; k < CPL / 2; ++k) {
      const float2 f = __bfloat1622float2(h2[k]);
      v[2 * k] = f.x;
      v[2 * k + 1] = f.y;
    }
    if (signs) {
      // butterflies over column bits 0..4 (inside the lane)
#pragma unroll
      for (int h = 1; h < CPL; h <<= 1)
#pragma unroll
        for (int i = 0; i < CPL; ++i)
          if (!(i & h)) {
            const float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
          }
      // butterflies over column bits 5..6 (lane bits 0..1 of the row's quad)
#pragma unroll
      for (int st = 1; st < LPR; st <<= 1)
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const float o = __shfl_xor_sync(0xffffffffu, v[k], st);
          v[k] = (sub & st) ? (o - v[k]) : (v[k] + o);
        }
      // y_j = s_j (x H)_j / sqrt(D); "+ 0" turns an exact -0 into +0
#pragma unroll
      for (int k = 0; k < CPL; ++k) v[k] = v[k] * (__ldg(&signs[sub * CPL + k]) * 0.08838834764831845f) + 0.f;
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k) amax = fmaxf(amax, fabsf(v[k]));
  }
  // tile amax across the CTA
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // (double-buffered by tile parity, so one barrier per tile suffices)
  if ((threadIdx.x & 31) == 0) s_red[parity][threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) m = fmaxf(m, s_red[parity][w]);
  const float sc = m > 0.f ? m / 448.f : 1.f;
  if (threadIdx.x == 0) scales[(size_t)bh * nts + tile] = sc;
  const float inv = 1.f / sc;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int row = ps * (THREADS / LPR) + rloc;
    if (tile * TR + row >= S) continue;
    uint32_t w[CPL / 4];
#pragma unroll
    for (int k = 0; k < CPL / 4; ++k) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[ps][4 * k] * inv, y[ps][4 * k + 1] * inv),
                                                   __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y[ps][4 * k + 2] * inv, y[ps][4 * k + 3] * inv),
                                                   __NV_SATFINITE, __NV_E4M3);
      w[k] = lo | (hi << 16);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(codes + base + (size_t)row * DQ) + sub * 2;
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  }
}

}  // namespace qnt

cudaError_t launch_rotate_quantize(const void *x, uint8_t *codes, float *scales, const float *signs, int B, int H,
                                   int S, cudaStream_t stream) {
  const int nts = (S + qnt::TR - 1) / qnt::TR;
  const long ntiles = (long)nts * B * H;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long grid = ntiles < 2L * sms ? ntiles : 2L * sms;  // two resident CTAs per SM
  qnt::rotate_quantize_kernel<<<(unsigned)grid, qnt::THREADS, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(x), codes, scales, signs, S, nts, ntiles);
  return cudaGetLastError();
}

}  // namespace attn
