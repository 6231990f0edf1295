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
// Persistent CTAs of 128 threads, two per SM.  Tiles arrive by TMA in a
// two-stage shared-memory ring (128-byte swizzle, so the row reads below are
// free of bank conflicts); one thread owns one row and keeps it as 64 fp32
// pairs (column m, column m + 64), so the 128-point fast Walsh-Hadamard
// transform runs six butterfly stages on packed f32x2 adds and subtracts and
// the seventh inside each pair, with no shuffles.  The tile's amax is reduced
// across the CTA, the codes y * (1 / scale) are rounded by the e4m3
// conversion into a swizzled shared-memory tile, and a TMA store writes it.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace qnt {

constexpr int TR = 128;                 // rows per tile = threads per CTA
constexpr int DQ = 128;                 // head dimension (one tile wide)
constexpr int THREADS = TR;
constexpr int NW = THREADS / 32;
constexpr int NP = DQ / 2;              // fp32 pairs per row
constexpr int NSTAGE = 2;               // input ring depth
constexpr int BOX = 128 * 128;          // 128 rows x 128 bytes
constexpr int IN_TILE = 2 * BOX;        // a bf16 tile: two 64-column boxes
constexpr int OFF_IN = 0;
constexpr int OFF_OUT = OFF_IN + NSTAGE * IN_TILE;  // e4m3 codes of one tile
constexpr int OFF_SC = OFF_OUT + BOX;               // (s_m, s_{m+64}) / sqrt(D)
constexpr int OFF_RED = OFF_SC + NP * 8;            // amax partials, two parities
constexpr int OFF_BAR = OFF_RED + 2 * NW * 4;
constexpr int SMEM = OFF_BAR + NSTAGE * 8 + 1024;   // + alignment slack
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
// element i (0..7) of eight packed bf16, as fp32 (exact)
__device__ __forceinline__ float bf16_at(const uint4 &v, int i) {
  const uint32_t w = word_of(v, i / 2);
  return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
}

__global__ void __launch_bounds__(THREADS, 2)
    rotate_quantize_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmc,
                           float *__restrict__ scales, const float *__restrict__ signs, int nts, long ntiles,
                           uint64_t timeout_ns, unsigned *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  const float4 *s_sc4 = reinterpret_cast<const float4 *>(smem + OFF_SC);
  float *s_red = reinterpret_cast<float *>(smem + OFF_RED);
  uint8_t *out = smem + OFF_OUT;
  const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
  const bool rotate = signs != nullptr;
  const long t0 = blockIdx.x, step = gridDim.x;
  const int my_n = t0 < ntiles ? (int)((ntiles - 1 - t0) / step + 1) : 0;

  if (r == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
  }
  if (rotate && r < NP)
    reinterpret_cast<float2 *>(smem + OFF_SC)[r] =
        make_float2(__ldg(&signs[r]) * kInvSqrtD, __ldg(&signs[r + NP]) * kInvSqrtD);
  __syncthreads();
  // tile t = (b*H + h) * nts + row tile; its two 64-column boxes go to stage s
  auto load = [&](int s, long t) {
    const int z = (int)(t / nts), y = (int)(t % nts) * TR;
    mbar_arrive_expect_tx(&full[s], IN_TILE);
    tma_load_3d(smem + OFF_IN + s * IN_TILE, &tmx, &full[s], 0, y, z);
    tma_load_3d(smem + OFF_IN + s * IN_TILE + BOX, &tmx, &full[s], 64, y, z);
  };
  if (r == 0) {
    tma_prefetch_desc(&tmx);
    tma_prefetch_desc(&tmc);
    for (int s = 0; s < NSTAGE && s < my_n; ++s) load(s, t0 + s * step);
  }
  int consumed = 0;
  for (int it = 0; it < my_n; ++it) {
    const long t = t0 + it * step;
    const int s = it % NSTAGE;
    // (every thread takes the same branch: the barrier ANDs the outcomes)
    if (!__syncthreads_and(mbar_wait(&full[s], (it / NSTAGE) & 1, timeout_ns, err))) break;
    consumed = it + 1;
    const uint8_t *in = smem + OFF_IN + s * IN_TILE;
    uint64_t P[NP];  // pair m = (column m, column m + 64)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 a = *reinterpret_cast<const uint4 *>(in + sw(r, c));
      const uint4 b = *reinterpret_cast<const uint4 *>(in + BOX + sw(r, c));
#pragma unroll
      for (int i = 0; i < 8; ++i) P[c * 8 + i] = f2_pack(bf16_at(a, i), bf16_at(b, i));
    }
    if (rotate) {
      // butterflies over column bits 0..5 (between pairs)
#pragma unroll
      for (int h = 1; h < NP; h <<= 1)
#pragma unroll
        for (int m = 0; m < NP; ++m)
          if (!(m & h)) {
            const uint64_t a = P[m], b = P[m + h];
            P[m] = f2_add(a, b);
            P[m + h] = f2_sub(a, b);
          }
      // column bit 6 (inside each pair), then y_j = s_j (x H)_j / sqrt(D)
#pragma unroll
      for (int m = 0; m < NP; m += 2) {
        const float4 c = s_sc4[m / 2];
        float a0, b0, a1, b1;
        f2_unpack(P[m], a0, b0);
        f2_unpack(P[m + 1], a1, b1);
        P[m] = f2_mul(f2_pack(a0 + b0, a0 - b0), f2_pack(c.x, c.y));
        P[m + 1] = f2_mul(f2_pack(a1 + b1, a1 - b1), f2_pack(c.z, c.w));
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int m = 0; m < NP; ++m) {
      float a, b;
      f2_unpack(P[m], a, b);
      amax = fmax3(amax, fabsf(a), fabsf(b));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_red[(it & 1) * NW + warp] = amax;
    if (r == 0) bulk_wait_read_all();  // the previous tile's codes have left the output buffer
    __syncthreads();
    // every thread has read stage s: refill it
    if (r == 0 && it + NSTAGE < my_n) load(s, t + NSTAGE * step);
    float mt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) mt = fmaxf(mt, s_red[(it & 1) * NW + w]);
    const float sc = mt > 0.f ? mt / 448.f : 1.f;
    const float inv = 1.f / sc;
    // y * inv + 0: an exact -0 becomes +0 (code 0x00)
    const uint64_t inv2 = f2_pack(inv, inv), zero2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // 16 codes: columns 16c .. 16c+15
      float q[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int m = (c % 4) * 16 + e;
        float lo, hi;
        f2_unpack(f2_fma(P[m], inv2, zero2), lo, hi);
        q[e] = c < 4 ? lo : hi;
      }
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t a = __nv_cvt_float2_to_fp8x2(make_float2(q[4 * k], q[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t b =
            __nv_cvt_float2_to_fp8x2(make_float2(q[4 * k + 2], q[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
        w[k] = a | (b << 16);
      }
      *reinterpret_cast<uint4 *>(out + sw(r, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (r == 0) {
      // rows past the end of the sequence fall outside the tensor map and are dropped
      tma_store_3d(&tmc, out, 0, (int)(t % nts) * TR, (int)(t / nts));
      bulk_commit_group();
      scales[t] = sc;
    }
  }
  if (r == 0) {
    bulk_wait_all();
    // after a failed wait, let the loads still in flight land before leaving
    for (int it = consumed; it < my_n && it < consumed + NSTAGE; ++it)
      mbar_wait(&full[it % NSTAGE], (it / NSTAGE) & 1, timeout_ns, err);
  }
}

}  // namespace qnt

cudaError_t launch_rotate_quantize(const CUtensorMap &tmx, const CUtensorMap &tmc, float *scales, const float *signs,
                                   int B, int H, int S, uint64_t timeout_ns, unsigned *err, cudaStream_t stream) {
  const int nts = (S + qnt::TR - 1) / qnt::TR;
  const long ntiles = (long)nts * B * H;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(qnt::rotate_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, qnt::SMEM);
  if (e != cudaSuccess) return e;
  const long grid = ntiles < 2L * sms ? ntiles : 2L * sms;  // two resident CTAs per SM
  qnt::rotate_quantize_kernel<<<(unsigned)grid, qnt::THREADS, qnt::SMEM, stream>>>(tmx, tmc, scales, signs, nts,
                                                                                  ntiles, timeout_ns, err);
  return cudaGetLastError();
}

}  // namespace attn
