// fwd_bf16.cu -- bf16 prefill attention forward on the sm_103a tensor cores.
//
// The method: "Fast Inference and Training at Scale" §6.21 (Idea 1, tiling):
// Q is cut into row tiles and K, V into column tiles that live on chip; the
// scores of one (Q tile, K tile) pair never reach HBM; a running max and a
// running sum (the online softmax; update printed in "Hardware Co-Design",
// FlashAttention section) stitch the tiles together, and only O (plus the
// per-row log-sum-exp, "Week 13. GPUs and FlashAttention" step 2) is written.
// The loop order is Q-outer / KV-inner and the grid spans (batch, head, Q
// block), as FlashAttention-2 does ("FlashAttention scaling, multi-GPU
// training and weight quantization" §1); division by the row sum is deferred
// to the end; with a causal mask, key tiles wholly above the diagonal are
// never visited (Week 13, step 2).
//
// GB300 mapping, one CTA = two 128-row Q tiles of one (batch, query head):
//   warp 8      TMA producer: Q once, then K_j / V_j into 2-stage rings
//               (cp.async.bulk.tensor, 128-byte swizzle, mbarrier tx counts);
//   warp 9      MMA issuer (one thread): S_i = Q_i K_j^T with tcgen05.mma
//               (both operands in shared memory, fp32 accumulator in TMEM),
//               then O_i += P_i V_j with P_i read from TMEM;
//   warps 0-3   softmax of Q tile 0, one thread per query row (TMEM lane);
//   warps 4-7   softmax of Q tile 1.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 after it.
// P_i (bf16 pairs) overwrites the first 64 columns of S_i.  The running
// max is only moved when the new maximum exceeds it by more than 8 (log2
// units), so O is rescaled rarely; probabilities then stay below 2^8.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <climits>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace fwd {

constexpr int BM = 128;          // query rows per Q tile
constexpr int BN = 128;          // keys per K/V tile
constexpr int NQT = 2;           // Q tiles per CTA
constexpr int NSTAGE = 2;        // K and V ring depth
constexpr int HALF = 128 * 128;  // 128 rows x 128 bytes: one swizzled 64-column half of a bf16 tile
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int THREADS = 10 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int NH = D / 64;       // 128-byte halves per row
  static constexpr int TILE = NH * HALF;  // one 128 x D bf16 tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * TILE;
  static constexpr int OFF_V = OFF_K + NSTAGE * TILE;
  static constexpr int OFF_BAR = OFF_V + NSTAGE * TILE;
  static constexpr int NBAR = 1 + 4 * NSTAGE + 3 * NQT + 1;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEMPTR + 16 + 1024;
  __device__ static constexpr uint32_t col_s(int i) { return (uint32_t)(i * BN); }
  __device__ static constexpr uint32_t col_o(int i) { return (uint32_t)(NQT * BN + i * D); }
  // instruction descriptors (kind::f16): f32 accumulate, bf16 A and B, M = 128
  static constexpr uint32_t IDESC_QK =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static constexpr uint32_t IDESC_PV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) /* B (V) MN-major */ |
                                       ((uint32_t)(D >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct Params {
  __nv_bfloat16 *o;
  float *lse;
  int B, Hq, Hkv, Sq, Sk, causal, g, nqb;
  float scale_log2;
  uint64_t timeout_ns;
  unsigned *err;
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1, *k_empty = k_full + NSTAGE;
  uint64_t *v_full = k_empty + NSTAGE, *v_empty = v_full + NSTAGE;
  uint64_t *s_full = v_empty + NSTAGE, *p_full = s_full + NQT, *o_full = p_full + NQT;
  uint64_t *done_bar = o_full + NQT;
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEMPTR);

  const int bh = blockIdx.x;  // b * Hq + hq
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / p.g;
  const int q0 = (p.nqb - 1 - (int)blockIdx.y) * (NQT * BM);  // latest (heaviest) query blocks first
  const int off = p.Sk - p.Sq;                                 // causal alignment: key j <= row + off
  int kv_end = p.Sk;
  if (p.causal) kv_end = min(p.Sk, min(q0 + NQT * BM - 1, p.Sq - 1) + off + 1);
  const int nkv = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (nkv == 0) {  // no query row of this block may attend to any key
    if (threadIdx.x < NQT * BM) {
      const int row = q0 + threadIdx.x;
      if (row < p.Sq) {
        uint4 *orow = reinterpret_cast<uint4 *>(p.o + ((size_t)bh * p.Sq + row) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
        if (p.lse) p.lse[(size_t)bh * p.Sq + row] = -CUDART_INF_F;
      }
    }
    return;
  }

  if (warp == WARP_MMA) {
    tmem_alloc(tmem_ptr, TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < NQT; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], BM);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(done_bar, 1);
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_arrive_expect_tx(q_full, NQT * C::TILE);
#pragma unroll
      for (int i = 0; i < NQT; ++i)
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_Q + i * C::TILE + h * HALF, &tmq, q_full, h * 64, q0 + i * BM, bh);
      const int zk = b * p.Hkv + hkv;
      int nk = 0, nv = 0;
      for (int j = 0; j < nkv; ++j) {
        const int slot = j % NSTAGE;
        const uint32_t par = ((j / NSTAGE) - 1) & 1;
        if (j >= NSTAGE && !mbar_wait(&k_empty[slot], par, p.timeout_ns, p.err)) break;
        mbar_arrive_expect_tx(&k_full[slot], C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_K + slot * C::TILE + h * HALF, &tmk, &k_full[slot], h * 64, j * BN, zk);
        nk = j + 1;
        if (j >= NSTAGE && !mbar_wait(&v_empty[slot], par, p.timeout_ns, p.err)) break;
        mbar_arrive_expect_tx(&v_full[slot], C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_V + slot * C::TILE + h * HALF, &tmv, &v_full[slot], h * 64, j * BN, zk);
        nv = j + 1;
      }
      // Leave only once every copy issued here has landed.
      mbar_wait(q_full, 0, p.timeout_ns, p.err);
      for (int t = max(0, nk - NSTAGE); t < nk; ++t) mbar_wait(&k_full[t % NSTAGE], (t / NSTAGE) & 1, p.timeout_ns, p.err);
      for (int t = max(0, nv - NSTAGE); t < nv; ++t) mbar_wait(&v_full[t % NSTAGE], (t / NSTAGE) & 1, p.timeout_ns, p.err);
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t qs = smem_u32(smem + C::OFF_Q), ks = smem_u32(smem + C::OFF_K), vs = smem_u32(smem + C::OFF_V);
      bool ok = mbar_wait(q_full, 0, p.timeout_ns, p.err);
      tc_fence_after();
      for (int j = 0; ok && j < nkv; ++j) {
        const int slot = j % NSTAGE;
        const uint32_t par = (j / NSTAGE) & 1;
        if (!mbar_wait(&k_full[slot], par, p.timeout_ns, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < NQT; ++i) {
          // S_i = Q_i K_j^T: K-major operands, 16 columns of D per instruction.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(tmem + C::col_s(i), sdesc_sw128(qs + i * C::TILE + o, 16, 1024),
                   sdesc_sw128(ks + slot * C::TILE + o, 16, 1024), C::IDESC_QK, kk > 0);
          }
          tc_commit(&s_full[i]);
        }
        tc_commit(&k_empty[slot]);
        if (!mbar_wait(&v_full[slot], par, p.timeout_ns, p.err)) break;
#pragma unroll
        for (int i = 0; i < NQT; ++i) {
          if (!mbar_wait(&p_full[i], j & 1, p.timeout_ns, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O_i += P_i V_j: P from TMEM (8 columns = 16 keys per instruction),
          // V MN-major (rows = keys, 128-byte swizzled halves of D apart by HALF).
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + C::col_o(i), tmem + C::col_s(i) + kk * 8,
                   sdesc_sw128(vs + slot * C::TILE + kk * 16 * 128, HALF, 1024), C::IDESC_PV, (j > 0 || kk > 0));
          tc_commit(&o_full[i]);
        }
        tc_commit(&v_empty[slot]);
      }
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, p.timeout_ns, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int i = warp >> 2;                     // Q tile
    const int r = (warp & 3) * 32 + lane;        // row within the tile = TMEM lane
    const int row = q0 + i * BM + r;             // query row
    const uint32_t taddr = tmem + (((warp & 3) * 32) << 16);
    const uint32_t s_col = C::col_s(i), o_col = C::col_o(i);
    const int lim = p.causal ? min(p.Sk - 1, row + off) : p.Sk - 1;  // last key this row may see
    const float sl2 = p.scale_log2;
    float m_use = -CUDART_INF_F;  // running max in log2 units (moved lazily)
    float l = 0.f;                // running sum relative to m_use
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[i], j & 1, p.timeout_ns, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(taddr + s_col + c * 32, s[c]);
      const int kb = j * BN;
      if (kb + BN - 1 > lim) {  // diagonal or ragged tile: mask keys past lim
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kb + c * 32 + e > lim) s[c][e] = __float_as_uint(-CUDART_INF_F);
      }
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(s[c][e]));
      const float m_new = fmaxf(m_use, mx * sl2);
      float alpha = 1.f;
      const bool moved = m_new > m_use + RESCALE_THRESHOLD;  // also true on the first finite max
      if (moved) {
        alpha = fast_exp2(m_use - m_new);  // 0 if nothing accumulated yet
        m_use = m_new;
      }
      const float mb = (m_use == -CUDART_INF_F) ? 0.f : m_use;
      float rs = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(s[c][e]), sl2, -mb));
          const float p1 = fast_exp2(fmaf(__uint_as_float(s[c][e + 1]), sl2, -mb));
          rs += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + e / 2] = pack_bf16x2(p0, p1);
        }
      l = l * alpha + rs;
      tmem_st32(taddr + s_col, pk[0]);
      tmem_st32(taddr + s_col + 32, pk[1]);
      // Rescale O_i by alpha once P_{j-1} V_{j-1} has landed (warp-uniform).
      if (__any_sync(0xffffffffu, moved && j > 0 && alpha != 0.f)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&o_full[i], (j - 1) & 1, p.timeout_ns, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(taddr + o_col + c * 32, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(taddr + o_col + c * 32, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[i]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[i], (nkv - 1) & 1, p.timeout_ns, p.err));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4 *orow = reinterpret_cast<uint4 *>(p.o + ((size_t)bh * p.Sq + min(row, p.Sq - 1)) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(taddr + o_col + c * 32, ov);
        uint32_t pkd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkd[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
        if (row < p.Sq) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            orow[c * 4 + e] = make_uint4(pkd[4 * e], pkd[4 * e + 1], pkd[4 * e + 2], pkd[4 * e + 3]);
        }
      }
      if (p.lse && row < p.Sq)
        p.lse[(size_t)bh * p.Sq + row] = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   cudaStream_t st) {
  using C = Cfg<D>;
  Params p;
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.causal = a.causal;
  p.g = a.Hq / a.Hkv;
  p.nqb = (a.Sq + NQT * BM - 1) / (NQT * BM);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.timeout_ns = a.timeout_ns;
  p.err = a.err;
  if (p.nqb > 65535) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.Hq), (unsigned)p.nqb);
  fwd_bf16_kernel<D><<<grid, THREADS, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd_bf16(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream) {
  if (a.D == 128) return fwd::launch<128>(a, tq, tk, tv, stream);
  if (a.D == 64) return fwd::launch<64>(a, tq, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
