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
// The rotation is a 128 x 128 x 128 product per tile, so it runs on the tensor
// core: z = x B with B = H_D diag(s) (entries +-1, exact in bf16; the identity
// when there is no rotation), products exact, fp32 accumulation in TMEM.
// One launch takes up to four tensors (e.g. Q and K rotated with the same
// signs, V not); their tiles form one sequence that the CTAs split.  A head
// dimension of 64 uses the same 128-column tiles: its upper 64 input columns
// arrive from TMA as zeros, B keeps only its leading 64 x 64 block (H_64 is
// the leading block of H_128), and the upper 64 columns of the codes fall
// outside the output tensor map and are not stored.
// Persistent, one CTA per SM, warp roles:
//   warp 0      TMA producer: bf16 tiles into a four-stage shared-memory ring
//               (two 64-column boxes, 128-byte swizzle = the K-major operand
//               layout of the tensor core);
//   warp 1      allocates TMEM and issues the products of each tile (with the
//               tile's B: rotation or identity) into one of four 128-column
//               accumulators;
//   warps 2-9   two epilogue warpgroups taking alternate tiles: each thread
//               reads its row of z from TMEM, y = z / sqrt(D) (y = z without
//               rotation), the tile amax is reduced across the group, codes
//               y * (1 / scale) are rounded by the e4m3 conversion into a
//               swizzled shared-memory tile that a TMA store writes out.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace qnt {

constexpr int TR = 128;    // rows per tile
constexpr int DQ = 128;    // columns of a tile: the head dimension (a 64-wide one is read with zeros above)
constexpr int NST = 4;     // input ring depth (tiles)
constexpr int NG = 2;      // epilogue warpgroups; group g takes the CTA's tiles g, g + NG, ...
constexpr int NACC = 4;    // TMEM accumulators of 128 columns (two per group)
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_EPI = 2;
constexpr int THREADS = 32 * (WARP_EPI + 4 * NG);
constexpr int BOX = 128 * 128;     // 128 rows x 128 bytes
constexpr int IN_TILE = 2 * BOX;   // a bf16 tile: two 64-column boxes
constexpr int OFF_B = 0;                          // B^T of the rotation, K-major like the input tiles
constexpr int OFF_BI = OFF_B + IN_TILE;           // the identity, same layout
constexpr int OFF_IN = OFF_BI + IN_TILE;
constexpr int OFF_OUT = OFF_IN + NST * IN_TILE;   // e4m3 codes, one tile per group
constexpr int OFF_RED = OFF_OUT + NG * BOX;       // amax partials [NG][4]
constexpr int OFF_BAR = OFF_RED + NG * 4 * 4;
constexpr int NBAR = 2 * NST + 2 * NACC + 2;      // full, empty, acc_full, acc_empty, mma_done, never
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;      // TMEM base, tiles landed (seen by the MMA warp), loads issued
constexpr int SMEM = OFF_MISC + 16 + 1024;        // + alignment slack
constexpr uint32_t TMEM_COLS = NACC * DQ;
// instruction descriptor: f32 accumulate, A and B bf16, both K-major, N = 128, M = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(DQ >> 3) << 17) | ((uint32_t)(TR >> 4) << 24);
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1 / sqrt(128)
static_assert(SMEM <= 227 * 1024, "shared memory budget");
static_assert(TMEM_COLS <= 512, "TMEM budget");

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Tensor i of the launch's tile t and the tile's index lt within that tensor.
__device__ __forceinline__ int tensor_of(const QuantArgs &a, long t, long &lt) {
  int i = 0;
  while (i + 1 < a.n && t >= a.first[i + 1]) ++i;
  lt = t - a.first[i];
  return i;
}

__global__ void __launch_bounds__(THREADS, 1) rotate_quantize_kernel(const __grid_constant__ QuantArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *full = bars, *empty = bars + NST, *acc_full = bars + 2 * NST, *acc_empty = acc_full + NACC;
  uint64_t *mma_done = acc_empty + NACC;
  uint64_t *never = mma_done + 1;  // test hook: no thread ever arrives on it
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  float *s_red = reinterpret_cast<float *>(smem + OFF_RED);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long t0 = blockIdx.x, step = gridDim.x, ntiles = a.first[a.n];
  const int my_n = t0 < ntiles ? (int)((ntiles - 1 - t0) / step + 1) : 0;
  const uint64_t timeout_ns = a.timeout_ns, wait_ns = a.wait_ns;  // copies / own products; other roles
  unsigned *const err = a.err;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < NACC; ++k) {
      mbar_init(&acc_full[k], 1);
      mbar_init(&acc_empty[k], 4);  // one arrival per warp of the group
    }
    mbar_init(mma_done, 1);
    mbar_init(never, 1);
    mbar_init_fence();
    misc[1] = 0;  // tiles whose loads the MMA warp saw land
    misc[2] = 0;  // tiles whose loads the producer issued
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&misc[0], TMEM_COLS);
    tmem_relinquish();
  }
  // B^T[n][k] = s_n H[n][k] = s_n (-1)^popcount(n & k) (H is symmetric) for
  // the rotation, delta(n, k) for the identity; +-1 is 0x3f80 / 0xbf80 in bf16.
  // For a.d = 64 only the 64 x 64 block n, k < 64 is nonzero (H_64 is the
  // leading block of H_128): the zero upper columns of x add nothing and the
  // upper columns of y come out zero.
  bool any_rot = false;
  for (int i = 0; i < a.n; ++i) any_rot |= a.rotate[i] != 0;
  if (tid < 2 * DQ) {
    const int n = tid % DQ;
    const bool rot = tid < DQ;
    const int d = a.d;
    const uint32_t neg = rot && any_rot && __ldg(&a.signs[n & (d - 1)]) < 0.f;
    uint8_t *bt = smem + (rot ? OFF_B : OFF_BI);
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {  // eight columns k = 8c .. 8c + 7
      // outside the d x d block (d is 64 or 128, a multiple of 8): zero
      const uint32_t keep = (n < d && 8 * c < d) ? 0xffffffffu : 0u;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t h[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int k = 8 * c + 2 * e + i;
          h[i] = rot ? (0x3f80u | (((__popc(n & k) & 1u) ^ neg) << 15)) : (k == n ? 0x3f80u : 0u);
        }
        w[e] = (h[0] | (h[1] << 16)) & keep;
      }
      *reinterpret_cast<uint4 *>(bt + (c >> 3) * BOX + sw(n, c & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();  // the tensor core reads B through the async proxy
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < a.n; ++i) tma_prefetch_desc(&a.tmx[i]);
      for (int it = 0; it < my_n; ++it) {
        const int s = it % NST;
        if (it >= NST && !mbar_wait(&empty[s], ((it / NST) + 1) & 1, wait_ns, err)) break;
        long lt;
        const int i = tensor_of(a, t0 + it * step, lt);
        const int z = (int)(lt / a.nts[i]), y = (int)(lt % a.nts[i]) * TR;
        uint8_t *dst = smem + OFF_IN + s * IN_TILE;
        mbar_arrive_expect_tx(&full[s], IN_TILE);
        tma_load_3d(dst, &a.tmx[i], &full[s], 0, y, z);
        tma_load_3d(dst + BOX, &a.tmx[i], &full[s], 64, y, z);
        misc[2] = it + 1;
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint64_t da0 = sdesc_sw128(smem_u32(smem + OFF_IN), 16, 1024);
      const uint64_t db_rot = sdesc_sw128(smem_u32(smem + OFF_B), 16, 1024);
      const uint64_t db_id = sdesc_sw128(smem_u32(smem + OFF_BI), 16, 1024);
      for (int it = 0; it < my_n; ++it) {
        const int s = it % NST, acc = it % NACC;
        if (!mbar_wait(&full[s], (it / NST) & 1, timeout_ns, err)) break;
        misc[1] = it + 1;
        if (it >= NACC && !mbar_wait(&acc_empty[acc], ((it / NACC) + 1) & 1, wait_ns, err)) break;
        tc_fence_after();
        long lt;
        const uint64_t db = a.rotate[tensor_of(a, t0 + it * step, lt)] ? db_rot : db_id;
        const uint64_t da = sdesc_add(da0, s * IN_TILE);
#pragma unroll
        for (int kk = 0; kk < DQ / 16; ++kk) {  // 16 columns (32 bytes) per product
          const uint32_t o = (kk >> 2) * BOX + (kk & 3) * 32;
          mma_ss(tmem + acc * DQ, sdesc_add(da, o), sdesc_add(db, o), IDESC, kk > 0);
        }
        tc_commit(&empty[s]);
        tc_commit(&acc_full[acc]);
      }
      // every product issued has completed before TMEM is released
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, timeout_ns, err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - WARP_EPI) / 4, q = warp & 3;  // TMEM lanes 32q .. 32q + 31
    const int r = 32 * q + lane;                        // row of the tile
    const bool leader = warp == WARP_EPI + 4 * g && lane == 0;
    uint8_t *out = smem + OFF_OUT + g * BOX;
    float *red = s_red + g * 4;
    // test hook: wait for a signal nothing gives, so that this wait runs out
    const bool go = !a.stall || __all_sync(0xffffffffu, mbar_wait(never, 0, wait_ns, err));
    for (int it = g; it < my_n; it += NG) {
      const int acc = it % NACC;
      long lt;
      const int ti = tensor_of(a, t0 + it * step, lt);
      // y = z / sqrt(d) for a rotation, y = x otherwise
      const float ys = a.rotate[ti] ? (a.d == 64 ? 0.125f : kInvSqrtD) : 1.f;
      bool ok = go && __all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (it / NACC) & 1, wait_ns, err));
      uint32_t v[128];
      float amax = 0.f;
      if (ok) {
        tc_fence_after();
        tmem_ld128(tmem + ((uint32_t)(32 * q) << 16) + acc * DQ, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);  // the accumulator is in registers: free it
#pragma unroll
        for (int e = 0; e < 128; e += 2)
          amax = fmax3(amax, fabsf(__uint_as_float(v[e])), fabsf(__uint_as_float(v[e + 1])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[q] = amax;
      }
      if (leader) bulk_wait_read_all();  // the previous tile's codes have left the output buffer
      if (!named_barrier_and(1 + g, 128, ok)) break;
      // max |y| = (max |z|) * ys: rounding z * ys is monotone in |z|
      const float mt = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) * ys;
      const float sc = mt > 0.f ? mt / 448.f : 1.f;
      const float inv = 1.f / sc;
      // y = z * ys, then y * inv + 0: an exact -0 becomes +0 (code 0x00)
      const uint64_t c2 = f2_pack(ys, ys), inv2 = f2_pack(inv, inv), zero2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 16 codes: columns 16c .. 16c + 15
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float qv[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = 16 * c + 4 * k + 2 * h;
            const uint64_t y2 = f2_mul(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2);
            f2_unpack(f2_fma(y2, inv2, zero2), qv[2 * h], qv[2 * h + 1]);
          }
          const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(qv[0], qv[1]), __NV_SATFINITE, __NV_E4M3);
          const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(qv[2], qv[3]), __NV_SATFINITE, __NV_E4M3);
          w[k] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4 *>(out + sw(r, c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      named_barrier_sync(1 + g, 128);
      if (leader) {
        // rows past the end of the sequence fall outside the tensor map and are dropped
        tma_store_3d(&a.tmc[ti], out, 0, (int)(lt % a.nts[ti]) * TR, (int)(lt / a.nts[ti]));
        bulk_commit_group();
        a.scales[ti][lt] = sc;
      }
    }
    if (leader) bulk_wait_all();
  }

  // after a failed wait, let the loads still in flight land before leaving
  __syncthreads();
  if (warp == WARP_TMA && lane == 0) {
    const int issued = (int)misc[2], consumed = (int)misc[1];
    for (int it = consumed; it < issued; ++it) mbar_wait(&full[it % NST], (it / NST) & 1, timeout_ns, err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace qnt

cudaError_t launch_rotate_quantize(const QuantArgs &a, cudaStream_t stream) {
  const long ntiles = a.first[a.n];
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(qnt::rotate_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, qnt::SMEM);
  if (e != cudaSuccess) return e;
  const long grid = ntiles < sms ? ntiles : sms;  // one resident CTA per SM
  qnt::rotate_quantize_kernel<<<(unsigned)grid, qnt::THREADS, qnt::SMEM, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
