// bwd.cu -- attention backward with recomputation on the sm_103a tensor cores.
//
// "Fast Inference and Training at Scale" §6.21 (Idea 2) and "Week 13. GPUs and
// FlashAttention" step 2: the forward keeps only O and the per-row
// log-sum-exp; the backward recomputes the scores tile by tile and never
// stores an S x S matrix.  With S = scale Q K^T, P = exp(S - LSE):
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - rowsum(dO o O)),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Kernel 1 (bwd_pre_kernel): Dvec = rowsum(dO o O) in fp32, and zeroes the fp32
// dQ accumulator.
// Kernel 2 (bwd_kernel): one CTA per (128-key tile, KV head, batch) walks
// every visible 128-row query tile of the KV head's query-head group:
//   warp 8      TMA: K_j, V_j once; Q_i and dO_i into a 2-stage ring; adds
//               each staged scale * dQ_i into the fp32 accumulator with TMA
//               reduce-add (full 128-byte lines, no per-thread atomics);
//   warp 9      one thread issues tcgen05.mma, per item i in the order
//                 dP^T_i = V_j dO_i^T; [P^T_i ready] dV += P^T_i dO_i;
//                 S^T_{i+1} = K_j Q_{i+1}^T (S^T_0 before the loop);
//                 [dS^T_i ready] dK += dS^T_i Q_i, dQ_i = dS_i K_j
//               (S^T, dP^T from shared-memory operands, fp32 in TMEM, one lane
//               per key; P^T, dS^T read from TMEM; dS staged in shared memory,
//               MN-major, for dQ; dV, dK stay in TMEM for the whole CTA).  The
//               next item's S^T runs while dS^T_i is computed, so the compute
//               warps go from dS^T_i straight to P^T_{i+1};
//   warps 0-7   one thread per (key, half of the query tile): stage the
//               item's LSE and Dvec in shared memory; once S^T is in TMEM,
//               P^T = exp2(S^T scale log2e - LSE log2e) to TMEM (bf16), kept
//               in registers (fp32); once dP^T is, dS^T = P^T o (dP^T - Dvec)
//               to TMEM (bf16) and shared memory; at the end dK (times scale)
//               and dV are written once as bf16;
//   warps 12-15 one thread per query row: once dQ_i is in TMEM, stage
//               scale * dQ_i in the item's Q / dO ring slot, which its MMAs
//               no longer need (warps 10-11 idle).
// Registers: launched at 128 per thread; the compute warpgroups take 176,
// the producer / MMA warpgroup keeps 56 and the dQ warpgroup 96
// (2 x 256 x 176 + 128 x 56 + 128 x 96 = 64,512 of the 65,536 launched; per
// sub-partition one warp of each: 32 x 504 of its 16,384).
// Kernel 3 (bwd_post_kernel): dQ = bf16(accumulator).
// TMEM columns: S^T [0,128) (then P^T bf16 in [0,32) and [64,96)), dP^T
// [128,256) (then dS^T bf16 likewise, then dQ_i [128,256)), dV [256,384),
// dK [384,512).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace bwd {

// Register reallocation between warpgroups (every warp of the warpgroup
// executes it): give back registers down to N, or take more up to N.
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

constexpr int BM = 128;          // query rows per Q tile
constexpr int BN = 128;          // keys per CTA
constexpr int NS = 2;            // Q / dO ring depth
constexpr int HALF = 128 * 128;  // 128 rows x 128 bytes
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_DQ = 12;
constexpr int THREADS = 16 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 384;
constexpr uint32_t COL_DQ = COL_DPT;  // dQ_i goes over dP^T / dS^T once dK_i has read dS^T

template <int D>
struct Cfg {
  static constexpr int NH = D / 64;
  static constexpr int TILE = NH * HALF;  // 128 x D bf16
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;        // NS stages of Q
  static constexpr int OFF_DO = OFF_Q + NS * TILE;  // NS stages of dO
  static constexpr int OFF_DS = OFF_DO + NS * TILE; // dS^T staging: 128 keys x 128 queries bf16
  static constexpr int OFF_LSE = OFF_DS + 2 * HALF;  // 128 x (LSE log2, Dvec) of the current item
  static constexpr int OFF_BAR = OFF_LSE + 128 * 2 * 4;
  static constexpr int NBAR = 1 + 4 * NS + 8;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEMPTR + 16 + 1024;
  // M = 128; K-major A and B (S^T, dP^T)
  static constexpr uint32_t IDESC_SS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BM >> 3) << 17) |
                                       ((uint32_t)(128 >> 4) << 24);
  // A from TMEM (K-major), B MN-major, N = D (dV, dK)
  static constexpr uint32_t IDESC_TS = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                       ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  // A and B MN-major, N = D (dQ = dS K)
  static constexpr uint32_t IDESC_DQ = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                                       ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // Box bx (fp32 columns 32bx .. 32bx+31) of a 128-row dQ tile staged in ring
  // slot `slot`: the first D/64 boxes over the slot's Q tile, the rest over its
  // dO tile (128 rows x 128 bytes each, 1024-byte aligned).
  static __device__ __forceinline__ uint8_t *dq_box(uint8_t *smem, int slot, int bx) {
    return smem + slot * TILE + (bx < NH ? OFF_Q + bx * HALF : OFF_DO + (bx - NH) * HALF);
  }
};

struct Params {
  const float *lse;   // [B, Hq, Sq] natural log (forward output)
  const float *dvec;  // [B, Hq, Sq] rowsum(dO o O)
  float *dq_acc;      // [B, Hq, Sq, D] fp32
  __nv_bfloat16 *dk, *dv;
  int B, Hq, Hkv, Sq, Sk, causal, g, nqt;
  float scale, scale_log2;
  uint64_t timeout_ns;  // waits on copies and on the CTA's own tensor-core work
  uint64_t wait_ns;     // waits of one warp role on another
  int stall;            // test hook: the compute warps first wait for a signal nothing gives
  unsigned *err;
};

// Byte offset of the 16-byte chunk c (queries 8c .. 8c+7) of key row k in the
// dS^T staging buffer (two 64-query slabs, 128-byte rows, 128-byte swizzle).
__device__ __forceinline__ uint32_t ds_off(int k, int c) {
  return (c >> 3) * HALF + k * 128 + (((c & 7) ^ (k & 7)) << 4);
}

// P^T of one key row over 32 queries: from S^T (raw scores, fp32) and the
// per-query LSE (log2 units) in shared memory, to fp32 (kept for dS^T) and
// packed bf16 pairs.  Element e is visible iff elo <= e < ehi (MASK only); a
// row without any visible key (LSE = -inf) is always masked, so the exp2 of
// +inf it may produce is never selected.
template <bool MASK>
__device__ __forceinline__ void p_chunk(const uint32_t (&sv)[32], const float4 *l2v, float scale_log2, int elo,
                                        int ehi, float *pf, uint32_t (&pp)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 l4 = l2v[e / 4];
    const float l2[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float pr = fast_exp2(fmaf(__uint_as_float(sv[e + u]), scale_log2, -l2[u]));
      if (MASK) pr = (e + u >= elo && e + u < ehi) ? pr : 0.f;
      pf[e + u] = pr;
    }
    pp[e / 2] = pack_bf16x2(pf[e], pf[e + 1]);
    pp[e / 2 + 1] = pack_bf16x2(pf[e + 2], pf[e + 3]);
  }
}

// dS^T = P^T o (dP^T - Dvec) of one key row over 32 queries, packed bf16 pairs
// (masked elements have P = 0, hence dS = 0).
__device__ __forceinline__ void ds_chunk(const float *pf, const uint32_t (&dpv)[32], const float4 *dvv,
                                         uint32_t (&dd)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 d4 = dvv[e / 4];
    const float dq[4] = {d4.x, d4.y, d4.z, d4.w};
    float dsv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) dsv[u] = pf[e + u] * (__uint_as_float(dpv[e + u]) - dq[u]);
    dd[e / 2] = pack_bf16x2(dsv[0], dsv[1]);
    dd[e / 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
  }
}

// TMEM column (relative to S^T or dP^T) of the bf16 P^T / dS^T values of
// 32-query chunk c: chunks 0, 1 over fp32 chunk 0, chunks 2, 3 over fp32
// chunk 2, so each half of the warps overwrites only columns it has read.
__device__ __forceinline__ constexpr uint32_t pcol(int c) { return (c >> 1) * 64 + (c & 1) * 16; }

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
               const __grid_constant__ CUtensorMap tmdq, Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *kv_full = bars;
  // per ring slot: Q landed, dO landed, dQ columns 0-63 / 64-127 staged
  uint64_t *q_full = bars + 1, *o_full = q_full + NS, *dq_half = o_full + NS;  // dq_half[2 * slot + h]
  uint64_t *s_full = dq_half + 2 * NS, *dp_full = s_full + 1, *p_ready = dp_full + 1, *ds_ready = p_ready + 1;
  uint64_t *dq_full = ds_ready + 1, *dq_free = dq_full + 1;
  uint64_t *done_bar = dq_free + 1;
  uint64_t *never = done_bar + 1;  // test hook: no thread ever arrives on it
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEMPTR);

  const int nkt = (p.Sk + BN - 1) / BN;
  const int j = (int)(blockIdx.x % nkt);    // key tile
  const int bkv = (int)(blockIdx.x / nkt);  // batch x KV head
  const int b = bkv / p.Hkv, kvh = bkv % p.Hkv;
  const int kj0 = j * BN;
  const int off = p.Sk - p.Sq;  // causal: key k visible to query q iff k <= q + off
  // query tiles that see at least one key of this tile (a suffix of 0..nqt-1)
  int qt0 = 0;
  if (p.causal) {
    qt0 = max(0, (kj0 - off) / BM - 1);
    while (qt0 < p.nqt && min(qt0 * BM + BM - 1, p.Sq - 1) + off < kj0) ++qt0;
  }
  const int nvis = p.nqt - qt0;
  const int nitems = nvis * p.g;  // item it: query head kvh*g + it / nvis, query tile qt0 + it % nvis
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (nitems == 0) {  // no query sees these keys: zero gradients
    for (int idx = threadIdx.x; idx < BN * D / 8; idx += THREADS) {
      const int k = idx / (D / 8), c = idx % (D / 8);
      if (kj0 + k < p.Sk) {
        const size_t o = ((size_t)bkv * p.Sk + kj0 + k) * D + c * 8;
        *reinterpret_cast<uint4 *>(p.dk + o) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(p.dv + o) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  if (warp == WARP_MMA) {
    tmem_alloc(tmem_ptr, TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&o_full[s], 1);
      mbar_init(&dq_half[2 * s], 4);  // one arrival per dQ warp
      mbar_init(&dq_half[2 * s + 1], 4);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);  // one arrival per dQ warp
    mbar_init(done_bar, 1);
    mbar_init(never, 1);
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  if (warp >> 2 == 2) {  // producer / MMA warpgroup (warps 10, 11 idle)
    reg_dealloc<56>();
    if (warp == WARP_TMA) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmdo);
        mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h) {
          tma_load_3d(smem + C::OFF_K + h * HALF, &tmk, kv_full, h * 64, kj0, bkv);
          tma_load_3d(smem + C::OFF_V + h * HALF, &tmv, kv_full, h * 64, kj0, bkv);
        }
        // Item i's Q and dO go into ring slot i % NS.  Once item r's MMAs are
        // done, the dQ warps stage scale * dQ_r (fp32, boxes of 128 rows x 32
        // columns) in that slot: columns 0-63 over its Q tile, then 64-127 over
        // its dO tile.  This thread adds each half into the accumulator with
        // TMA reduce-add and reloads the part it occupied with item r + NS as
        // soon as the reduce has read it (Q first: the next products need it
        // first).
        auto load_q = [&](int it) {
          const int slot = it % NS, hq = kvh * p.g + it / nvis, q0 = (qt0 + it % nvis) * BM;
          mbar_arrive_expect_tx(&q_full[slot], C::TILE);
#pragma unroll
          for (int h = 0; h < C::NH; ++h)
            tma_load_3d(smem + C::OFF_Q + slot * C::TILE + h * HALF, &tmq, &q_full[slot], h * 64, q0, b * p.Hq + hq);
        };
        auto load_do = [&](int it) {
          const int slot = it % NS, hq = kvh * p.g + it / nvis, q0 = (qt0 + it % nvis) * BM;
          mbar_arrive_expect_tx(&o_full[slot], C::TILE);
#pragma unroll
          for (int h = 0; h < C::NH; ++h)
            tma_load_3d(smem + C::OFF_DO + slot * C::TILE + h * HALF, &tmdo, &o_full[slot], h * 64, q0,
                        b * p.Hq + hq);
        };
        int nq = 0, ndo = 0;  // items whose Q / dO loads are issued
        for (; nq < nitems && nq < NS; ++nq, ++ndo) {
          load_q(nq);
          load_do(ndo);
        }
        for (int r = 0; r < nitems; ++r) {
          const int slot = r % NS;
          const int hq = kvh * p.g + r / nvis, q0 = (qt0 + r % nvis) * BM;
          // rows past Sq fall outside the tensor map and are dropped
          if (!mbar_wait(&dq_half[2 * slot], (r / NS) & 1, p.wait_ns, p.err)) break;
#pragma unroll
          for (int bx = 0; bx < C::NH; ++bx)
            tma_reduce_add_3d(&tmdq, C::dq_box(smem, slot, bx), bx * 32, q0, b * p.Hq + hq);
          bulk_commit_group();
          bulk_wait_read_all();
          if (nq < nitems) load_q(nq++);
          if (!mbar_wait(&dq_half[2 * slot + 1], (r / NS) & 1, p.wait_ns, p.err)) break;
#pragma unroll
          for (int bx = C::NH; bx < D / 32; ++bx)
            tma_reduce_add_3d(&tmdq, C::dq_box(smem, slot, bx), bx * 32, q0, b * p.Hq + hq);
          bulk_commit_group();
          bulk_wait_read_all();
          if (ndo < nitems) load_do(ndo++);
        }
        bulk_wait_all();  // the accumulator is complete before the CTA ends
        // Leave only once every copy issued here has landed.
        mbar_wait(kv_full, 0, p.timeout_ns, p.err);
        for (int t = max(0, nq - NS); t < nq; ++t) mbar_wait(&q_full[t % NS], (t / NS) & 1, p.timeout_ns, p.err);
        for (int t = max(0, ndo - NS); t < ndo; ++t) mbar_wait(&o_full[t % NS], (t / NS) & 1, p.timeout_ns, p.err);
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issue
      if (lane == 0) {
        const uint32_t ks = smem_u32(smem + C::OFF_K), vs = smem_u32(smem + C::OFF_V),
                       qs = smem_u32(smem + C::OFF_Q), dos = smem_u32(smem + C::OFF_DO),
                       dss = smem_u32(smem + C::OFF_DS);
        // descriptors built once: K-major reads (LBO 16) and MN-major reads (LBO = half tile),
        // advanced per product by byte offsets
        const uint64_t k_km = sdesc_sw128(ks, 16, 1024), v_km = sdesc_sw128(vs, 16, 1024),
                       q_km = sdesc_sw128(qs, 16, 1024), do_km = sdesc_sw128(dos, 16, 1024),
                       q_mn = sdesc_sw128(qs, HALF, 1024), do_mn = sdesc_sw128(dos, HALF, 1024),
                       ds_mn = sdesc_sw128(dss, HALF, 1024), k_mn = sdesc_sw128(ks, HALF, 1024);
        // S^T = K Q^T into [0, 128): K-major operands, 32 bytes of D per instruction
        auto issue_st = [&](int it) {
          const uint64_t q_k = sdesc_add(q_km, (it % NS) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(tmem + COL_ST, sdesc_add(k_km, o), sdesc_add(q_k, o), C::IDESC_SS, kk > 0);
          }
          tc_commit(s_full);
        };
        bool ok = mbar_wait(kv_full, 0, p.timeout_ns, p.err) && mbar_wait(&q_full[0], 0, p.timeout_ns, p.err);
        if (ok) {
          tc_fence_after();
          issue_st(0);
        }
        for (int it = 0; ok && it < nitems; ++it) {
          const uint32_t so = (it % NS) * C::TILE;
          // dP^T = V dO^T into [128, 256), which holds the previous dQ until the dQ warps have read it
          if (it > 0 && !mbar_wait(dq_free, (it - 1) & 1, p.wait_ns, p.err)) break;
          if (!mbar_wait(&o_full[it % NS], (it / NS) & 1, p.timeout_ns, p.err)) break;
          tc_fence_after();
          const uint64_t do_k = sdesc_add(do_km, so);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(tmem + COL_DPT, sdesc_add(v_km, o), sdesc_add(do_k, o), C::IDESC_SS, kk > 0);
          }
          tc_commit(dp_full);
          // dV += P^T dO: A from TMEM (16 queries = 8 columns per instruction),
          // B = dO MN-major (rows = queries)
          if (!mbar_wait(p_ready, it & 1, p.wait_ns, p.err)) break;
          tc_fence_after();
          const uint64_t do_m = sdesc_add(do_mn, so), q_m = sdesc_add(q_mn, so);
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ts(tmem + COL_DV, tmem + COL_ST + pcol(kk >> 1) + (kk & 1) * 8, sdesc_add(do_m, kk * 16 * 128),
                   C::IDESC_TS, (it > 0 || kk > 0));
          // Then, in whichever order their inputs arrive: the next item's S^T
          // (into [0, 128), behind dV, the last reader of P^T there; the
          // compute warps have read S^T_i), once its Q has landed; and
          // dK += dS^T Q (A from TMEM, B = Q MN-major) followed by dQ = dS K
          // into [128, 256) (A = dS staged as dS^T rows = keys: MN-major,
          // B = K MN-major; 16 keys per instruction), once dS^T is ready.
          bool st_done = it + 1 >= nitems, kq_done = false;
          const uint64_t t_start = globaltimer_ns();
          while (!(st_done && kq_done)) {
            if (!kq_done && mbar_try_wait(ds_ready, it & 1)) {
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < BM / 16; ++kk)
                mma_ts(tmem + COL_DK, tmem + COL_DPT + pcol(kk >> 1) + (kk & 1) * 8, sdesc_add(q_m, kk * 16 * 128),
                       C::IDESC_TS, (it > 0 || kk > 0));
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_ss(tmem + COL_DQ, sdesc_add(ds_mn, kk * 16 * 128), sdesc_add(k_mn, kk * 16 * 128), C::IDESC_DQ,
                       kk > 0);
              tc_commit(dq_full);
              kq_done = true;
            } else if (!st_done && mbar_try_wait(&q_full[(it + 1) % NS], ((it + 1) / NS) & 1)) {
              tc_fence_after();
              issue_st(it + 1);
              st_done = true;
            } else {
              const uint64_t el = globaltimer_ns() - t_start;
              if ((!kq_done && el > p.wait_ns) || (!st_done && el > p.timeout_ns)) {
                record_error(p.err, kErrTimeout);
                ok = false;
                break;
              }
            }
          }
        }
        tc_commit(done_bar);
        mbar_wait(done_bar, 0, p.timeout_ns, p.err);
      }
    }
  } else if (warp >= WARP_DQ) {
    reg_dealloc<96>();
    // ------------------------------------------------------- dQ read-out
    // Warp w reads TMEM lanes 32*(w%4) .. +31 (query rows of the item's tile)
    // and stages scale * dQ_i as 128-row x 32-column fp32 boxes with the
    // 128-byte swizzle in the item's Q / dO slot (the first half of the boxes
    // over its Q tile, the second over its dO tile); the TMA thread adds them
    // into the accumulator.
    static_assert(D == 64 || D == 128, "dQ is read out in 64-column pieces");
    const int quad = warp & 3;
    const int rq = quad * 32 + lane;
    const uint32_t taddr = tmem + ((quad * 32) << 16);
    // boxes bx0 .. bx0 + nbox - 1 from v[32 * vb ..]
    auto stage = [&](const uint32_t (&v)[64], int slot, int bx0, int nbox, int vb) {
#pragma unroll
      for (int bx = 0; bx < 2; ++bx)
        if (bx < nbox) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t *w = v + (vb + bx) * 32 + 4 * j;
            *reinterpret_cast<float4 *>(C::dq_box(smem, slot, bx0 + bx) + rq * 128 + ((j ^ (rq & 7)) << 4)) =
                make_float4(__uint_as_float(w[0]) * p.scale, __uint_as_float(w[1]) * p.scale,
                            __uint_as_float(w[2]) * p.scale, __uint_as_float(w[3]) * p.scale);
          }
        }
    };
    for (int it = 0; it < nitems; ++it) {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, p.wait_ns, p.err))) break;
      tc_fence_after();
      const int slot = it % NS;
      uint32_t v[64];
      tmem_ld64(taddr + COL_DQ, v);  // columns 0 .. 63
      if constexpr (D == 128) {
        stage(v, slot, 0, 2, 0);  // over the item's Q tile
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dq_half[2 * slot]);
        tmem_ld64(taddr + COL_DQ + 64, v);  // columns 64 .. 127, over its dO tile
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);  // the next item's dP^T may overwrite these columns
      if constexpr (D == 64) {
        stage(v, slot, 0, 1, 0);  // columns 0 .. 31 over the item's Q tile
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dq_half[2 * slot]);
        stage(v, slot, 1, 1, 1);  // columns 32 .. 63 over its dO tile
      } else {
        stage(v, slot, 2, 2, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dq_half[2 * slot + 1]);
    }
  } else {
    reg_alloc<176>();
    // ------------------------------------------------------- compute warps
    // Warp w reads TMEM lanes 32*(w%4) .. +31 and takes one half of the
    // columns: the queries half*64 .. +63 of S^T / dP^T, then the dQ (or dK,
    // dV) columns half*D/2 .. +D/2-1.
    const int quad = warp & 3, half = warp >> 2;
    const int k = quad * 32 + lane;  // key within the tile (S^T, dP^T, dK, dV rows); query row of dQ
    const int key = kj0 + k;
    const uint32_t taddr = tmem + ((quad * 32) << 16);
    uint8_t *ds_stage = smem + C::OFF_DS;
    float *s_l2 = reinterpret_cast<float *>(smem + C::OFF_LSE), *s_dv = s_l2 + BM;
    // queries this key is visible to: qlo <= q < qhi (causal: q >= key - off;
    // a key past the end is visible to none)
    const long long qlo = p.causal ? (long long)key - off : -1;
    const long long qhi = key < p.Sk ? p.Sq : -1;
    // this thread's share of an item's per-query values: half 0 the LSE (as
    // log2), half 1 Dvec, for query q0 + k.  Loaded one item ahead, before the
    // dQ reductions that would otherwise queue in front of it.
    auto item_value = [&](int i) -> float {
      const int hq = kvh * p.g + i / nvis, qt = (qt0 + i % nvis) * BM + k;
      if (qt >= p.Sq) return 0.f;
      const size_t r = ((size_t)b * p.Hq + hq) * p.Sq + qt;
      return half ? __ldg(&p.dvec[r]) : __ldg(&p.lse[r]) * 1.4426950408889634f;
    };
    float nval = item_value(0);
    // test hook: wait for a signal nothing gives, so that this wait runs out
    bool ok = !p.stall || named_barrier_and(1, 256, mbar_wait(never, 0, p.wait_ns, p.err));
    for (int it = 0; ok && it < nitems; ++it) {
      const int q0 = (qt0 + it % nvis) * BM;
      named_barrier_sync(1, 256);  // every compute thread is done with the previous item's values
      (half ? s_dv : s_l2)[k] = nval;
      // the barrier publishes the staged values
      if (!named_barrier_and(1, 256, mbar_wait(s_full, it & 1, p.wait_ns, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T of this thread's 64 queries (two chunks of 32), kept in fp32 for dS^T
      float pf[64];
      int elo[2], ehi[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = half * 2 + cc;
        const int qc = q0 + c * 32;
        // element e of this chunk (query qc + e) is visible iff elo <= e < ehi
        elo[cc] = (int)max(-1LL, min(33LL, qlo - qc));
        ehi[cc] = (int)max(-1LL, min(33LL, qhi - qc));
        const float4 *l2v = reinterpret_cast<const float4 *>(s_l2 + c * 32);
        uint32_t sv[32], pp[16];
        tmem_ld32(taddr + COL_ST + c * 32, sv);
        if (__all_sync(0xffffffffu, elo[cc] <= 0 && ehi[cc] >= 32))  // whole chunk visible to every key of the warp
          p_chunk<false>(sv, l2v, p.scale_log2, 0, 32, pf + cc * 32, pp);
        else
          p_chunk<true>(sv, l2v, p.scale_log2, elo[cc], ehi[cc], pf + cc * 32, pp);
        // bf16 P^T of chunk c goes over fp32 columns this warp has already read
        tmem_st16(taddr + COL_ST + pcol(c), pp);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);
      // dS^T once dP^T is in TMEM (its product ran while P^T was computed)
      if (!named_barrier_and(1, 256, mbar_wait(dp_full, it & 1, p.wait_ns, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = half * 2 + cc;
        uint32_t dpv[32], dd[16];
        tmem_ld32(taddr + COL_DPT + c * 32, dpv);
        ds_chunk(pf + cc * 32, dpv, reinterpret_cast<const float4 *>(s_dv + c * 32), dd);
        tmem_st16(taddr + COL_DPT + pcol(c), dd);
#pragma unroll
        for (int u = 0; u < 4; ++u)  // queries c*32 + 8u .. +7
          *reinterpret_cast<uint4 *>(ds_stage + ds_off(k, c * 4 + u)) =
              make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // dS^T stores before the tensor core reads them
      tc_fence_before();
      mbar_arrive(ds_ready);
      if (it + 1 < nitems) nval = item_value(it + 1);
    }
    // ---------------------------------------------------- dK, dV epilogue
    // once every product of the CTA has completed
    if (ok) ok = named_barrier_and(1, 256, mbar_wait(done_bar, 0, p.timeout_ns, p.err));
    if (ok) {
      tc_fence_after();
      const size_t o = ((size_t)bkv * p.Sk + min(key, p.Sk - 1)) * D + half * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t col = half * (D / 2) + c * 32;
        uint32_t a[32], bv[32];
        tmem_ld32(taddr + COL_DK + col, a);
        tmem_ld32(taddr + COL_DV + col, bv);
        uint32_t pk[16], pv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
          pv[e] = pack_bf16x2(__uint_as_float(bv[2 * e]), __uint_as_float(bv[2 * e + 1]));
        }
        if (key < p.Sk) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            reinterpret_cast<uint4 *>(p.dk + o)[c * 4 + e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            reinterpret_cast<uint4 *>(p.dv + o)[c * 4 + e] = make_uint4(pv[4 * e], pv[4 * e + 1], pv[4 * e + 2], pv[4 * e + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Dvec = rowsum(dO o O) per query row; zero the dQ accumulator.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dout,
                                                      float *__restrict__ dvec, float *__restrict__ dq_acc,
                                                      long rows) {
  const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f;
  for (int d = lane * 2; d < D; d += 64) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(o + row * D + d));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(dout + row * D + d));
    acc += a.x * c.x + a.y * c.y;
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) dvec[row] = acc;
  for (int d = lane * 4; d < D; d += 128) *reinterpret_cast<float4 *>(dq_acc + row * D + d) = make_float4(0, 0, 0, 0);
}

template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq,
                                                       long n4) {
  const long i = (long)blockIdx.x * 256 + threadIdx.x;
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4 *>(dq_acc)[i];
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  reinterpret_cast<uint2 *>(dq)[i] = w;
}

template <int D>
cudaError_t launch(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   const CUtensorMap &tdo, const CUtensorMap &tdq, cudaStream_t st) {
  using C = Cfg<D>;
  const long rows = (long)a.B * a.Hq * a.Sq;
  bwd_pre_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.o),
                                                                  static_cast<const __nv_bfloat16 *>(a.dout),
                                                                  a.dvec, a.dq_acc, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Params p;
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq_acc = a.dq_acc;
  p.dk = static_cast<__nv_bfloat16 *>(a.dk);
  p.dv = static_cast<__nv_bfloat16 *>(a.dv);
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.causal = a.causal;
  p.g = a.Hq / a.Hkv;
  p.nqt = (a.Sq + BM - 1) / BM;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.timeout_ns = a.timeout_ns;
  p.wait_ns = a.wait_ns;
  p.stall = a.stall;
  p.err = a.err;
  if ((long)((a.Sk + BN - 1) / BN) * a.B * a.Hkv > 0x7fffffffL) return cudaErrorNotSupported;
  e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(((a.Sk + BN - 1) / BN) * a.B * a.Hkv));
  bwd_kernel<D><<<grid, THREADS, C::SMEM, st>>>(tq, tk, tv, tdo, tdq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long n4 = rows * D / 4;
  bwd_post_kernel<D><<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(a.dq_acc, static_cast<__nv_bfloat16 *>(a.dq), n4);
  return cudaGetLastError();
}

}  // namespace bwd

cudaError_t launch_bwd(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdq, cudaStream_t stream) {
  if (a.D == 128) return bwd::launch<128>(a, tq, tk, tv, tdo, tdq, stream);
  if (a.D == 64) return bwd::launch<64>(a, tq, tk, tv, tdo, tdq, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
