// fwd_kernel.cuh -- prefill attention forward on the sm_103a tensor cores,
// shared by the bf16 (fwd_bf16.cu) and FP8 e4m3 (fwd_fp8.cu) entry points.
//
// The method: "Fast Inference and Training at Scale" §6.21 (Idea 1, tiling):
// Q is cut into row tiles and K, V into column tiles that live on chip; the
// scores of one (Q tile, K tile) pair never reach HBM; a running max and a
// running sum (the online softmax; update printed in "Hardware Co-Design",
// FlashAttention section) stitch the tiles together, and only O (plus the
// per-row log-sum-exp, "Week 13. GPUs and FlashAttention" step 2) is written.
// The loop order is Q-outer / KV-inner and the grid spans (Q block, batch x
// head), as FlashAttention-2 does ("FlashAttention scaling, multi-GPU
// training and weight quantization" §1); division by the row sum is deferred
// to the end; with a causal mask, key tiles wholly above the diagonal are
// never visited (Week 13, step 2).  The FP8 variant follows FlashAttention-3
// (same page, §1): e4m3 operands on the FP8 tensor cores with one scale per
// 128 x 128 tile.
//
// GB300 mapping, one CTA = two 128-row Q tiles of one (batch, query head):
//   warp 8      TMA producers (cp.async.bulk.tensor, 128-byte swizzle,
//               mbarrier tx counts): lane 0 loads Q once and streams K_j
//               into a 2-stage ring, lane 1 streams V_j into a 3-stage ring
//               (FP8: 3 and 3, K slots handed back with the V slots);
//   warp 9      MMA issuer (one thread): S_i = Q_i K_j^T with tcgen05.mma
//               (both operands in shared memory, fp32 accumulator in TMEM),
//               then O_i += P_i V_j with P_i read from TMEM.  Issue order
//               P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1): while one Q tile's
//               softmax runs, the tensor core works on the other tile
//               (FP8: P_i from shared memory, order S_0(j+1), S_1(j+1),
//               P_0 V_j, P_1 V_j, each S once its tile's softmax has read
//               the previous one);
//   warps 0-3   softmax of Q tile 0, one thread per query row (TMEM lane);
//   warps 4-7   softmax of Q tile 1.
// The softmax uses the packed fp32x2 FMA/ADD and three-input max of sm_100+.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 after it.
// P_i overwrites the first columns of S_i (FP8: P_i in shared memory, two
// buffers per Q tile after the V ring).  The running max only moves when
// the new maximum exceeds it by more than a threshold (log2 units), so O is
// rescaled rarely.
//
// FP8 specifics: S_ij is dequantised by one scalar sq_i * sk_j * scale;
// probabilities are multiplied by 2^4 * sv_j / max_j sv_j before the e4m3
// rounding (so they stay in e4m3's normal range and carry the value tile's
// scale), and the output is multiplied back by max_j sv_j / 2^4.
#pragma once
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace fwd {

constexpr int BM = 128;          // query rows per Q tile
constexpr int BN = 128;          // keys per K/V tile
constexpr int NQT = 2;           // Q tiles per CTA
constexpr int HALF = 128 * 128;  // 128 rows x 128 bytes: one 128-byte-swizzled slab of a tile
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int THREADS = 10 * 32;

constexpr uint32_t TMEM_COLS = 512;

struct Bf16 {
  static constexpr bool kFp8 = false;
  static constexpr int kElem = 2;        // bytes per element
  static constexpr int kMmaK = 16;       // K elements per MMA instruction (32 bytes)
  // Lazy-rescale threshold, log2 units: the running max moves (and O is
  // rescaled) only when a tile's max exceeds it by more than this, so P stays
  // <= 2^32 -- well inside bf16's range -- and l <= Sk * 2^32, l * |V| (the
  // fp32 O accumulator) far below fp32's 2^128 for any plausible V.  Fewer
  // rescales: under outlier keys the max jumps often by a few units.
  static constexpr float kThresh = 32.f;
  static constexpr float kPre = 0.f;     // log2 of the probability pre-scale
  static constexpr uint32_t kTypeBits = (1u << 7) | (1u << 10);  // A and B bf16
  // Commit o_full after every P.V (else only after each tile's last one).
  static constexpr bool kOFullEachTile = true;
  static constexpr int kNSK = 2, kNSV = 3;  // K and V ring depths
  // K slot j is handed back by the commit that releases V slot j (one key
  // tile later than its own commit would), saving a commit per key tile;
  // needs equal ring depths.
  static constexpr bool kKRelByV = false;
  // P_i goes back into S_i's TMEM columns, so S_i(j+1) waits for P_i V_j.
  static constexpr bool kPSmem = false;
};

struct Fp8 {
  static constexpr bool kFp8 = true;
  static constexpr int kElem = 1;
  static constexpr int kMmaK = 32;
  static constexpr float kThresh = 4.f;
  static constexpr float kPre = 4.f;
  static constexpr uint32_t kTypeBits = 0u;  // A and B e4m3
  // A commit costs ~71 cycles of the tensor pipe, and an FP8 key tile has
  // only ~1024 cycles of products: the per-tile o_full commits are dropped.
  // The O rescale of tile j needs P_i V_{j-1} landed; the V release of key
  // tile j-1, committed after both tiles' P V_{j-1}, says so.
  static constexpr bool kOFullEachTile = false;
  // For the same reason K slots go back with the V release: K_j is free once
  // P_1 V_j is done (S_1(j) came before it).  Three stages of each keep the
  // loads ahead (four measured no faster: 224 KB of shared memory with the P
  // buffers, against 198 KB).
  static constexpr int kNSK = 3, kNSV = 3;
  static constexpr bool kKRelByV = true;
  // P_i goes to shared memory (two 16 KB buffers per Q tile) and P.V reads
  // both operands from there.  S_i's columns are free as soon as the softmax
  // has read them, so S_i(j+1) runs during softmax_i(j) instead of after
  // P_i V_j: the softmax phases follow each other without waiting for the
  // products, which is what the FP8 tile (products half as long as bf16's,
  // as many exponentials) is bound by.  bf16 keeps P in TMEM: its products
  // already fill the tensor core and shared memory.
  static constexpr bool kPSmem = true;
};

template <class T, int D>
struct Cfg {
  static constexpr int NSK = T::kNSK, NSV = T::kNSV;
  static_assert(!T::kKRelByV || NSK == NSV, "K released with V needs equal ring depths");
  static constexpr int NH = D * T::kElem / 128;  // 128-byte slabs per row
  static constexpr int TILE = NH * HALF;         // one 128 x D tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * TILE;
  static constexpr int OFF_V = OFF_K + NSK * TILE;
  static constexpr int NP = T::kPSmem ? 2 * NQT : 0;  // P buffers in shared memory, two per Q tile
  static constexpr int OFF_P = OFF_V + NSV * TILE;
  static constexpr int OFF_BAR = OFF_P + NP * HALF;
  static constexpr int NBAR = 1 + 2 * NSK + 2 * NSV + 5 * NQT + 2;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEMPTR + 16 + 1024;
  static constexpr int P_REGS = BN * T::kElem / 4;  // 32-bit TMEM columns holding one P row
  __device__ static constexpr uint32_t col_s(int i) { return (uint32_t)(i * BN); }
  __device__ static constexpr uint32_t col_o(int i) { return (uint32_t)(NQT * BN + i * D); }
  // instruction descriptors: f32 accumulate, M = 128; V (B of P.V) is MN-major
  static constexpr uint32_t IDESC_QK =
      (1u << 4) | T::kTypeBits | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static constexpr uint32_t IDESC_PV =
      (1u << 4) | T::kTypeBits | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static_assert(NH >= 1, "tile rows must span at least one 128-byte slab");
  static_assert(!T::kPSmem || BN * T::kElem == 128, "a P row in shared memory is one 128-byte swizzle row");
  static_assert(!T::kPSmem || T::kKRelByV, "with P in shared memory K slots go back with the V release");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(NQT * BN + NQT * D <= (int)TMEM_COLS, "TMEM budget");
};

struct Params {
  __nv_bfloat16 *o;
  float *lse;
  const float *q_scale, *k_scale, *v_scale;  // FP8 only
  int B, Hq, Hkv, Sq, Sk, causal, g, nqb, nqt, nkt;
  int dout;  // columns of O (and its row stride): D, or 64 for FP8 inputs read as 128 columns
  int hc;  // (batch, head) pairs per launch-order chunk
  float scale_log2;
  uint64_t timeout_ns;  // waits on copies and on the CTA's own tensor-core work
  uint64_t wait_ns;     // waits of one role on another (softmax <-> MMA issuer)
  int stall;            // test hook: the softmax first waits for a signal nothing gives
  unsigned *err;
};

// both operands in shared memory
template <class T>
__device__ __forceinline__ void mma_smem(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (T::kFp8) mma_ss_f8(d, a, b, idesc, acc);
  else mma_ss(d, a, b, idesc, acc);
}

template <class T>
__device__ __forceinline__ void mma_pv(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (T::kFp8) mma_ts_f8(d, a_tmem, b, idesc, acc);
  else mma_ts(d, a_tmem, b, idesc, acc);
}

// Test hook, compiled only into the kSkew instantiation: a fixed 20 us delay
// of one warp role, so that the others run ahead of it.
__device__ __forceinline__ void skew_delay() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 20000ull) {
  }
}

// kSkew: the issuing thread pauses after each S commit and tile 0's softmax
// before each wait for S, so the other tile's softmax and the issuing thread
// get ahead of it (the barrier-phase cases of the P-in-shared-memory order).
template <class T, int D, bool kSkew = false>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, Params p) {
  using C = Cfg<T, D>;
  constexpr int NSK = C::NSK, NSV = C::NSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1, *k_empty = k_full + NSK;
  uint64_t *v_full = k_empty + NSK, *v_empty = v_full + NSV;
  // p_full: one per Q tile; with P in shared memory two per Q tile (key tile
  // parity), since a tile's softmax may then finish key tile j + 1 before the
  // issuing thread has waited for its P of key tile j
  uint64_t *s_full = v_empty + NSV, *p_full = s_full + NQT, *o_full = p_full + 2 * NQT;
  uint64_t *s_free = o_full + NQT;  // P in shared memory: the softmax has read S_i
  uint64_t *done_bar = s_free + NQT;
  uint64_t *never = done_bar + 1;  // test hook: no thread ever arrives on it
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEMPTR);

  // Launch order: (batch, head) pairs in chunks of p.hc, whose K and V fit in
  // L2 together; inside a chunk the latest (heaviest, under a causal mask)
  // query blocks of all its heads first, so the light ones end the launch.
  int bh, qx;
  {
    const long lin = blockIdx.x, per_chunk = (long)p.hc * p.nqb;
    const long chunk = lin / per_chunk, r = lin % per_chunk;
    const long heads = min((long)p.hc, (long)p.B * p.Hq - chunk * p.hc);  // pairs in this chunk
    qx = (int)(r / heads);
    bh = (int)(chunk * p.hc + r % heads);  // b * Hq + hq
  }
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / p.g;
  const int q0 = (p.nqb - 1 - qx) * (NQT * BM);
  const int off = p.Sk - p.Sq;                                 // causal alignment: key j <= row + off
  // key tiles each Q tile visits (a prefix 0 .. nkv_t[i]-1)
  int nkv_t[NQT];
#pragma unroll
  for (int i = 0; i < NQT; ++i) {
    const int first = q0 + i * BM, last = min(first + BM - 1, p.Sq - 1);
    int end = p.Sk;
    if (last < first) end = 0;  // the tile lies past the last query row
    else if (p.causal) end = min(p.Sk, last + off + 1);
    nkv_t[i] = end > 0 ? (end + BN - 1) / BN : 0;
  }
  const int nkv = max(nkv_t[0], nkv_t[1]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (nkv == 0) {  // no query row of this block may attend to any key
    if (threadIdx.x < NQT * BM) {
      const int row = q0 + threadIdx.x;
      if (row < p.Sq) {
        uint4 *orow = reinterpret_cast<uint4 *>(p.o + ((size_t)bh * p.Sq + row) * p.dout);
        for (int c = 0; c < p.dout / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
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
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < NQT; ++i) {  // p_full, s_free: one arrival per softmax warp
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[2 * i], BM / 32);
      mbar_init(&p_full[2 * i + 1], BM / 32);
      mbar_init(&o_full[i], 1);
      mbar_init(&s_free[i], BM / 32);
    }
    mbar_init(done_bar, 1);
    mbar_init(never, 1);
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producers
    const int zk = b * p.Hkv + hkv;
    if (lane == 0) {  // Q, then the K ring
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      mbar_arrive_expect_tx(q_full, NQT * C::TILE);
#pragma unroll
      for (int i = 0; i < NQT; ++i)
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_Q + i * C::TILE + h * HALF, &tmq, q_full, h * (128 / T::kElem), q0 + i * BM,
                      bh);
      int nk = 0;
      for (int j = 0; j < nkv; ++j) {
        const int slot = j % NSK;
        uint64_t *freed = T::kKRelByV ? &v_empty[slot] : &k_empty[slot];
        if (j >= NSK && !mbar_wait(freed, ((j / NSK) - 1) & 1, p.timeout_ns, p.err)) break;
        mbar_arrive_expect_tx(&k_full[slot], C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_K + slot * C::TILE + h * HALF, &tmk, &k_full[slot], h * (128 / T::kElem),
                      j * BN, zk);
        nk = j + 1;
      }
      // Leave only once every copy issued here has landed.
      mbar_wait(q_full, 0, p.timeout_ns, p.err);
      for (int t = max(0, nk - NSK); t < nk; ++t) mbar_wait(&k_full[t % NSK], (t / NSK) & 1, p.timeout_ns, p.err);
    } else if (lane == 1) {  // the V ring
      tma_prefetch_desc(&tmv);
      int nv = 0;
      for (int j = 0; j < nkv; ++j) {
        const int slot = j % NSV;
        if (j >= NSV && !mbar_wait(&v_empty[slot], ((j / NSV) - 1) & 1, p.timeout_ns, p.err)) break;
        mbar_arrive_expect_tx(&v_full[slot], C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(smem + C::OFF_V + slot * C::TILE + h * HALF, &tmv, &v_full[slot], h * (128 / T::kElem),
                      j * BN, zk);
        nv = j + 1;
      }
      for (int t = max(0, nv - NSV); t < nv; ++t) mbar_wait(&v_full[t % NSV], (t / NSV) & 1, p.timeout_ns, p.err);
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issue
    // One thread issues both Q tiles' chains in the order
    // P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1): while one tile's softmax runs the
    // tensor core works on the other tile, and each group of MMAs runs
    // contiguously so its result is ready as early as possible.
    if (lane == 0) {
      const uint32_t qs = smem_u32(smem + C::OFF_Q), ks = smem_u32(smem + C::OFF_K), vs = smem_u32(smem + C::OFF_V);
      // base descriptors (start address + constant offsets below)
      const uint64_t dq0 = sdesc_sw128(qs, 16, 1024), dk0 = sdesc_sw128(ks, 16, 1024),
                     dv0 = sdesc_sw128(vs, HALF, 1024);
      // S_i = Q_i K_j^T: K-major operands, 32 bytes of the head dimension per instruction
      auto issue_s = [&](int i, int j) {
        const int slot = j % NSK;
        const uint64_t dq = sdesc_add(dq0, i * C::TILE), dk = sdesc_add(dk0, slot * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / T::kMmaK; ++kk) {
          const uint32_t o = (kk >> 2) * HALF + (kk & 3) * 32;
          mma_smem<T>(tmem + C::col_s(i), sdesc_add(dq, o), sdesc_add(dk, o), C::IDESC_QK, kk > 0);
        }
        if (!T::kPSmem) tc_commit(&s_full[i]);
      };
      // O_i += P_i V_j: P from TMEM (8 columns per instruction), V MN-major
      // (rows = keys; 128-byte slabs of the head dimension HALF bytes apart)
      auto issue_pv = [&](int i, int j) -> bool {
        if (!mbar_wait(&p_full[i], j & 1, p.wait_ns, p.err)) return false;
        tc_fence_after();
        const int slot = j % NSV;
        const uint64_t dv = sdesc_add(dv0, slot * C::TILE);
#pragma unroll
        for (int kk = 0; kk < BN / T::kMmaK; ++kk)
          mma_pv<T>(tmem + C::col_o(i), tmem + C::col_s(i) + kk * 8, sdesc_add(dv, kk * T::kMmaK * 128), C::IDESC_PV,
                    (j > 0 || kk > 0));
        if (T::kOFullEachTile || j + 1 == nkv_t[i]) tc_commit(&o_full[i]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, p.timeout_ns, p.err) && mbar_wait(&k_full[0], 0, p.timeout_ns, p.err);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < NQT; ++i)
          if (nkv_t[i] > 0) issue_s(i, 0);
        if (T::kPSmem) tc_commit(&s_full[0]);  // one signal for both tiles' scores
        if (!T::kKRelByV) tc_commit(&k_empty[0]);
      }
      if constexpr (T::kPSmem) {
        // O_i += P_i V_j with P_i in shared memory (buffer j & 1, K-major,
        // 128-byte swizzle: 32 keys = 32 bytes of each row per instruction).
        // Issue order S_0(j+1), S_1(j+1), P_0 V_j, P_1 V_j: each S as soon as
        // its tile's softmax has read the previous one, and one commit on
        // s_full[0] for both (a commit costs ~74 cycles of the tensor pipe;
        // tile 0's softmax waits the ~120 ns of S_1 more).  P_i V_j precedes
        // S_i(j+2), so the softmax's wait for S(j+2) also tells it that
        // buffer j & 1 is free again.
        const uint64_t dp0 = sdesc_sw128(smem_u32(smem + C::OFF_P), 16, 1024);
        // The issuing thread sets the pace here, so its loop carries as few
        // instructions as possible: ring slots and phases as counters, and
        // the key tiles both Q tiles visit (now and next) in a loop of their
        // own without per-tile checks.  K_{j+1} and V_j share the ring depth.
        static_assert(NSK == NSV, "one slot counter for both rings");
        int ks = 1 % NSK, kph = NSK == 1 ? 1 : 0;  // slot and phase of K_{j+1}
        int vsl = 0, vph = 0;                      // slot and phase of V_j
        auto step = [](int &slot, int &ph) {
          if (++slot == NSK) {
            slot = 0;
            ph ^= 1;
          }
        };
        auto wait_p = [&](int i, int j) -> bool {
          return mbar_wait(&p_full[2 * i + (j & 1)], (j >> 1) & 1, p.wait_ns, p.err);
        };
        auto issue_s_slot = [&](int i) {
          const uint64_t dq = sdesc_add(dq0, i * C::TILE), dk = sdesc_add(dk0, ks * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / T::kMmaK; ++kk) {
            const uint32_t o = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_smem<T>(tmem + C::col_s(i), sdesc_add(dq, o), sdesc_add(dk, o), C::IDESC_QK, kk > 0);
          }
        };
        auto issue_pv_smem = [&](int i, int j) {
          const uint64_t dp = sdesc_add(dp0, (2 * i + (j & 1)) * HALF);
          const uint64_t dv = sdesc_add(dv0, vsl * C::TILE);
#pragma unroll
          for (int kk = 0; kk < BN / T::kMmaK; ++kk)
            mma_smem<T>(tmem + C::col_o(i), sdesc_add(dp, kk * T::kMmaK * T::kElem),
                        sdesc_add(dv, kk * T::kMmaK * 128), C::IDESC_PV, (j > 0 || kk > 0));
        };
        const int jb = max(0, min(nkv_t[0], nkv_t[1]) - 1);  // j < jb: both tiles visit j and j + 1
        int j = 0;
        for (; ok && j < jb; ++j) {
          ok = mbar_wait(&k_full[ks], kph, p.timeout_ns, p.err) && mbar_wait(&s_free[0], j & 1, p.wait_ns, p.err);
          if (!ok) break;
          tc_fence_after();
          issue_s_slot(0);
          if (!(ok = mbar_wait(&s_free[1], j & 1, p.wait_ns, p.err))) break;
          tc_fence_after();
          issue_s_slot(1);
          tc_commit(&s_full[0]);
          step(ks, kph);
          if constexpr (kSkew) skew_delay();
          if (!(ok = mbar_wait(&v_full[vsl], vph, p.timeout_ns, p.err) && wait_p(0, j))) break;
          tc_fence_after();
          issue_pv_smem(0, j);
          if (!(ok = wait_p(1, j))) break;
          tc_fence_after();
          issue_pv_smem(1, j);
          tc_commit(&v_empty[vsl]);  // also frees K slot j (K_j's last product, S_1(j), came before)
          step(vsl, vph);
        }
        // the last key tiles: a tile may stop earlier (causal) or see no key at all
        for (; ok && j < nkv; ++j) {
          if (j + 1 < nkv) {
            if (!(ok = mbar_wait(&k_full[ks], kph, p.timeout_ns, p.err))) break;
            tc_fence_after();
#pragma unroll
            for (int i = 0; i < NQT; ++i) {
              // a tile whose last key tile is j must also have read S(j)
              // before s_full completes the phase of S(j+1): a waiter two
              // phases behind would read the parity wrongly
              if (ok && j < nkv_t[i]) {
                ok = mbar_wait(&s_free[i], j & 1, p.wait_ns, p.err);
                if (ok && j + 1 < nkv_t[i]) {
                  tc_fence_after();
                  issue_s_slot(i);
                }
              }
            }
            if (!ok) break;
            tc_commit(&s_full[0]);
            step(ks, kph);
            if constexpr (kSkew) skew_delay();
          }
          if (!(ok = mbar_wait(&v_full[vsl], vph, p.timeout_ns, p.err))) break;
#pragma unroll
          for (int i = 0; i < NQT; ++i) {
            if (ok && j < nkv_t[i]) {
              ok = wait_p(i, j);
              if (ok) {
                tc_fence_after();
                issue_pv_smem(i, j);
                if (j + 1 == nkv_t[i]) tc_commit(&o_full[i]);
              }
            }
          }
          if (!ok) break;
          tc_commit(&v_empty[vsl]);
          step(vsl, vph);
        }
      } else {
        for (int j = 0; ok && j < nkv; ++j) {
          const bool next = j + 1 < nkv;
          if (!mbar_wait(&v_full[j % NSV], (j / NSV) & 1, p.timeout_ns, p.err)) break;
          tc_fence_after();
          if (j < nkv_t[0] && !issue_pv(0, j)) break;
          if (next) {
            if (!mbar_wait(&k_full[(j + 1) % NSK], ((j + 1) / NSK) & 1, p.timeout_ns, p.err)) break;
            tc_fence_after();
            if (j + 1 < nkv_t[0]) issue_s(0, j + 1);
          }
          if (j < nkv_t[1] && !issue_pv(1, j)) break;
          tc_commit(&v_empty[j % NSV]);
          if (next) {
            if (j + 1 < nkv_t[1]) issue_s(1, j + 1);
            if (!T::kKRelByV) tc_commit(&k_empty[(j + 1) % NSK]);
          }
        }
      }
      // every product issued above has completed before the CTA moves on
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, p.timeout_ns, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int i = warp >> 2;               // Q tile
    const int r = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
    const int row = q0 + i * BM + r;       // query row
    const int my_nkv = nkv_t[i];
    const uint32_t taddr = tmem + (((warp & 3) * 32) << 16);
    const uint32_t s_col = C::col_s(i), o_col = C::col_o(i);
    const int lim = p.causal ? min(p.Sk - 1, row + off) : p.Sk - 1;  // last key this row may see
    const int zk = b * p.Hkv + hkv;
    // FP8: per-tile dequantisation scalars; the largest V scale of the row block
    float cq = 1.f, sv_ref = 1.f, lsv_ref = 0.f, ks_next = 0.f, vs_next = 0.f;
    if constexpr (T::kFp8) {
      cq = __ldg(&p.q_scale[(size_t)bh * p.nqt + (q0 + i * BM) / BM]);
      float mv = 0.f;
      for (int j = lane; j < nkv; j += 32) mv = fmaxf(mv, __ldg(&p.v_scale[(size_t)zk * p.nkt + j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
      sv_ref = fmaxf(mv, 1e-30f);
      lsv_ref = __log2f(sv_ref);
      // key tile j's K and V scales are loaded during tile j - 1, off the critical path
      if (my_nkv > 0) {
        ks_next = __ldg(&p.k_scale[(size_t)zk * p.nkt]);
        vs_next = __ldg(&p.v_scale[(size_t)zk * p.nkt]);
      }
    }
    float m_use = -CUDART_INF_F;  // running max in log2 units (moved lazily)
    float l = 0.f;                // running sum relative to m_use (gives the LSE)
    float l_o = 0.f;              // the sum O is divided by (below)
    // test hook: wait for a signal nothing gives, so that this wait runs out
    bool ok = !p.stall || __all_sync(0xffffffffu, mbar_wait(never, 0, p.wait_ns, p.err));
    for (int j = 0; ok && j < my_nkv; ++j) {
      float cj = p.scale_log2, e_off = T::kPre;
      if constexpr (T::kFp8) {
        cj *= cq * ks_next;
        e_off += __log2f(fmaxf(vs_next, 1e-30f)) - lsv_ref;
        if (j + 1 < my_nkv) {
          ks_next = __ldg(&p.k_scale[(size_t)zk * p.nkt + j + 1]);
          vs_next = __ldg(&p.v_scale[(size_t)zk * p.nkt + j + 1]);
        }
      }
      if constexpr (kSkew) {
        if (i == 0) skew_delay();
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[T::kPSmem ? 0 : i], j & 1, p.wait_ns, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[128];
      tmem_ld128(taddr + s_col, s);
      if constexpr (T::kPSmem) {  // S_i's columns may take the next key tile's scores now
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[i]);
      }
      const int kb = j * BN;
      const bool masked = kb + BN - 1 > lim;  // diagonal or ragged tile
      if (masked) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (kb + e > lim) s[e] = __float_as_uint(-CUDART_INF_F);
      }
      float mx4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx4[u] = __uint_as_float(s[u]);
#pragma unroll
      for (int e = 4; e + 8 <= 128; e += 8)  // s[4 .. 123], two groups of four per step
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mx4[u] = fmax3(mx4[u], __uint_as_float(s[e + u]), __uint_as_float(s[e + 4 + u]));
#pragma unroll
      for (int u = 0; u < 4; ++u) mx4[u] = fmaxf(mx4[u], __uint_as_float(s[124 + u]));
      const float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
      const float m_new = fmaxf(m_use, mx * cj);
      float alpha = 1.f;
      const bool moved = m_new > m_use + T::kThresh;  // also true on the first finite max
      // O holds earlier tiles' sums only once the max was finite; alpha may
      // then underflow to exactly 0 (a jump of > 126 in log2 units), and O
      // must still be multiplied by it.
      const bool rescale_o = moved && j > 0 && m_use != -CUDART_INF_F;
      if (moved) {
        alpha = fast_exp2(m_use - m_new);  // 0 if nothing accumulated yet
        m_use = m_new;
      }
      const float bias = e_off - ((m_use == -CUDART_INF_F) ? 0.f : m_use);
      const uint64_t c2 = f2_pack(cj, cj), b2 = f2_pack(bias, bias);
      uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      uint32_t pk[C::P_REGS];
#pragma unroll
      for (int e = 0; e < 128; e += 8) {
        float pr[8];
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
          const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[e + u]), __uint_as_float(s[e + u + 1])), c2, b2);
          f2_unpack(x2, pr[u], pr[u + 1]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) pr[u] = fast_exp2(pr[u]);
        acc2[0] = f2_add(acc2[0], f2_add(f2_pack(pr[0], pr[1]), f2_pack(pr[2], pr[3])));
        acc2[1] = f2_add(acc2[1], f2_add(f2_pack(pr[4], pr[5]), f2_pack(pr[6], pr[7])));
        if constexpr (T::kFp8) {
#pragma unroll
          for (int u = 0; u < 8; u += 4) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(pr[u], pr[u + 1]), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi =
                __nv_cvt_float2_to_fp8x2(make_float2(pr[u + 2], pr[u + 3]), __NV_SATFINITE, __NV_E4M3);
            pk[(e + u) / 4] = lo | (hi << 16);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; u += 2) pk[(e + u) / 2] = pack_bf16x2(pr[u], pr[u + 1]);
        }
      }
      float r0, r1, r2, r3;
      f2_unpack(acc2[0], r0, r1);
      f2_unpack(acc2[1], r2, r3);
      const float rs = (r0 + r1) + (r2 + r3);
      // The tile's largest probability enters P rounded to bf16 (e4m3).  With
      // the running max moved lazily it is 2^x with 0 < x <= the threshold,
      // not 1, so its rounding is up to half an ulp of it; the sum that O is
      // divided by takes that rounding too, so a row dominated by one key
      // still comes out as that key's value row.  (The LSE keeps the exact sum.)
      const float pm = fast_exp2(fmaf(mx, cj, bias));  // as computed for that score above
      float pm_r;
      if constexpr (T::kFp8) {
        const __half_raw hr = __nv_cvt_fp8_to_halfraw(__nv_cvt_float_to_fp8(pm, __NV_SATFINITE, __NV_E4M3), __NV_E4M3);
        pm_r = __half2float(__half(hr));
      } else {
        pm_r = __bfloat162float(__float2bfloat16_rn(pm));
      }
      const float back = T::kFp8 ? fast_exp2(-e_off) : 1.f;
      l = l * alpha + rs * back;
      l_o = l_o * alpha + (rs + (pm_r - pm)) * back;
      if constexpr (T::kPSmem) {
        // row r of buffer j & 1: 16-byte chunk c at position c ^ (r & 7) (the
        // 128-byte swizzle); eight consecutive rows cover all 32 banks
        uint8_t *prow = smem + C::OFF_P + (2 * i + (j & 1)) * HALF + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(prow + ((c ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < C::P_REGS / 32; ++c) {
          uint32_t chunk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) chunk[e] = pk[c * 32 + e];
          tmem_st32(taddr + s_col + c * 32, chunk);
        }
      }
      // Rescale O_i by alpha once P_{j-1} V_{j-1} has landed (warp-uniform).
      // With P in TMEM and no per-tile o_full, S_i(j) (issued after it)
      // implies it; with P in shared memory S_i(j) may come first, and the V
      // release of key tile j-1 (committed after both tiles' P V_{j-1}) does.
      if (__any_sync(0xffffffffu, rescale_o)) {
        bool landed = true;
        if constexpr (T::kOFullEachTile)
          landed = __all_sync(0xffffffffu, mbar_wait(&o_full[i], (j - 1) & 1, p.wait_ns, p.err));
        else if constexpr (T::kPSmem)
          landed = __all_sync(0xffffffffu,
                              mbar_wait(&v_empty[(j - 1) % NSV], ((j - 1) / NSV) & 1, p.wait_ns, p.err));
        if (!landed) {
          tmem_st_wait();  // no store of P may still be in flight when the CTA ends
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
      if constexpr (T::kPSmem) fence_proxy_async_smem();  // P's stores before the tensor core reads them
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[T::kPSmem ? 2 * i + (j & 1) : i]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok && my_nkv > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&o_full[i], T::kOFullEachTile ? (my_nkv - 1) & 1 : 0, p.wait_ns, p.err));
    if (ok) {
      tc_fence_after();
      const float out_scale = T::kFp8 ? sv_ref * fast_exp2(-T::kPre) : 1.f;
      const float inv = l_o > 0.f ? out_scale / l_o : 0.f;
      uint4 *orow = reinterpret_cast<uint4 *>(p.o + ((size_t)bh * p.Sq + min(row, p.Sq - 1)) * p.dout);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        if (T::kFp8 && c * 32 >= p.dout) break;  // the zero columns of a 64-wide FP8 head
        uint32_t ov[32];
        if (my_nkv > 0) {
          tmem_ld32(taddr + o_col + c * 32, ov);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
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

template <class T, int D>
cudaError_t launch(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   cudaStream_t st) {
  using C = Cfg<T, D>;
  Params p;
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.causal = a.causal;
  p.g = a.Hq / a.Hkv;
  p.nqb = (a.Sq + NQT * BM - 1) / (NQT * BM);
  p.nqt = (a.Sq + BM - 1) / BM;
  p.nkt = (a.Sk + BN - 1) / BN;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.dout = a.D;
  // chunks of (batch, head) pairs whose K and V take ~48 MB of L2, used when
  // the causal mask makes the lightest query block cost under half the
  // heaviest; otherwise all blocks cost about the same and the order stays
  // head by head (a head's blocks then share its K and V in L2 at once)
  {
    const bool skewed = a.causal && 2L * std::max(0L, (long)a.Sk - a.Sq + NQT * BM) < (long)a.Sk;
    const double kv_per_head = 2.0 * a.Sk * D * T::kElem / p.g;
    const long hc = skewed ? (long)(48.0e6 / kv_per_head) : 1;
    p.hc = (int)std::max(1L, std::min(hc, (long)a.B * a.Hq));
  }
  p.timeout_ns = a.timeout_ns;
  p.wait_ns = a.wait_ns;
  p.stall = a.stall;
  p.err = a.err;
  if ((long)p.nqb * a.B * a.Hq > 0x7fffffffL) return cudaErrorNotSupported;
  auto kern = fwd_kernel<T, D, false>;
  if constexpr (T::kPSmem) {  // the skew hook exists for the P-in-shared-memory order only
    if (a.skew) kern = fwd_kernel<T, D, true>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((long)p.nqb * a.B * a.Hq));
  kern<<<grid, THREADS, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace fwd
}  // namespace attn
