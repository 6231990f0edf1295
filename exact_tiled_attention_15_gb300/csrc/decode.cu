// decode.cu -- split-K grouped-query decode against a contiguous KV cache.
//
// One query token per sequence ("Fast Inference and Training at Scale" §6.1)
// attends over that sequence's cached keys and values.  The work is bound by
// HBM: every cached K and V byte is read once, and with grouped-query heads
// (§6.2) one read of a key/value head serves all Hq/Hkv query heads of its
// group ("Week 13. GPUs and FlashAttention", step 1: decode intensity is about
// Hq/Hkv FLOP per byte).
//
// Kernel 1 (decode_split_kernel), one CTA per (key split, KV head [, head
// chunk], sequence):
//   * a producer warp streams 64-key tiles of K and V into a 3-stage shared
//     memory ring with TMA (cp.async.bulk.tensor, 128-byte swizzle);
//   * four consumer warps each take 16 keys of a tile: S = Q K^T with the
//     group's query heads as the 16 rows of a warp MMA, the online-softmax
//     update (running max m, running sum l, rescale by 2^(m_old - m_new)),
//     then O += P V with P taken straight from the score registers;
//   * the four warps' (m, l, O) are merged and the split's normalised O and
//     log2-LSE go to the workspace.
// Kernel 2 (decode_combine_kernel) merges the splits of each (sequence, head)
// with log-sum-exp weights -- the same running max / running sum update
// ("Hardware Co-Design", FlashAttention section) applied to whole splits.  It
// is launched as a programmatic dependent of kernel 1, so it is resident and
// waiting when the last splits finish instead of paying a launch gap.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace dec {

// Device error word code of an out-of-range device-resident index (a
// sequence length or a block-table entry): ATTN_ERR_BAD_INDEX of attn.h.
constexpr unsigned kErrBadIndex = 7u;
constexpr int KS = 64;                      // keys per pipeline stage
constexpr int NST = 3;                      // pipeline stages
constexpr int NCW = 4;                      // consumer warps, 16 keys of a stage each
constexpr int THREADS = (NCW + 1) * 32;     // + one producer warp
constexpr int MROWS = 16;                   // query heads per CTA (rows of the warp MMA)
constexpr int HALF_BYTES = KS * 128;        // one 64-column (128-byte) half of a tile
constexpr int TARGET_CTAS = 4864;           // aim: ~16 CTAs per SM over the whole call

template <int D>
struct Cfg {
  static constexpr int NHALF = D / 64;
  static constexpr int TILE_BYTES = NHALF * HALF_BYTES;  // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = NST * STAGE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + (2 * NST + 1) * 8 + 16 + 1024;  // + barriers, flag, alignment
  static constexpr int NK = D / 16;  // k-steps of Q.K^T
  static constexpr int NT = D / 8;   // 8-column tiles of O
  static_assert(NCW * MROWS * D * 4 + 2 * NCW * MROWS * 4 <= BAR_OFF, "merge scratch must fit in the ring");
};

struct Params {
  const __nv_bfloat16 *q;
  const int32_t *seqlens;
  const int32_t *block_table;  // paged cache only: [B, max_blocks]
  int max_blocks, page_size, box_rows, num_pages;
  float *part_o;
  float *part_lse;
  int B, Hq, Hkv, Lmax, chunk, nsplit, g, nhc;
  int T;       // query tokens per sequence (1 = plain decode)
  int nhpc;    // query heads per CTA: nhpc * T <= 16 MMA rows
  int causal;  // T > 1: token t sits at position L - T + t and sees keys <= it
  float scale_log2;
  uint64_t timeout_ns;  // waits on copies
  uint64_t wait_ns;     // waits of one warp role on another
  int stall;            // test hook: the consumers first wait for a signal nothing gives
  unsigned *err;
};

// Byte offset of 16-byte chunk c (0 .. D/8-1) of row `row` inside one tile as
// TMA writes it: 64-column halves, 128-byte rows, chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t tile_off(int row, int c) {
  return (c >> 3) * HALF_BYTES + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// PAGED: K/V live in a page pool [num_pages, Hkv, page_size, D]; position t
// of sequence b is row t % page_size of page block_table[b, t / page_size]
// ("Fast Inference and Training at Scale" §6.3, PagedAttention).  Each 64-key
// stage is then gathered by boxes of min(page_size, 64) rows.
template <int D, bool PAGED>
__global__ void __launch_bounds__(THREADS, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *empty = full + NST;
  uint64_t *cbar = empty + NST;  // consumer-warp barrier (bounded, unlike bar.sync)
  int *s_fail = reinterpret_cast<int *>(cbar + 1);
  uint64_t *never = cbar + 2;  // test hook: no thread ever arrives on it

  // one-dimensional grid: split fastest, then (KV head, head chunk), then sequence
  const long cta = blockIdx.x;
  const int split = (int)(cta % p.nsplit);
  const long rest = cta / p.nsplit;
  const int kvh = (int)(rest % ((long)p.Hkv * p.nhc)) / p.nhc, hc = (int)(rest % ((long)p.Hkv * p.nhc)) % p.nhc;
  const int b = (int)(rest / ((long)p.Hkv * p.nhc));
  // The merge kernel may be scheduled as soon as every CTA of this grid has
  // started; it waits for this grid's results before reading them.
  griddep_launch_dependents();
  const int seq_len = p.seqlens[b];
  const int L = max(0, min(seq_len, p.Lmax));
  // a length outside [0, Lmax] is clamped; one CTA per sequence reports it
  if ((seq_len < 0 || seq_len > p.Lmax) && split == 0 && kvh == 0 && hc == 0 && threadIdx.x == 0)
    record_error(p.err, kErrBadIndex);
  const int s0 = split * p.chunk;
  if (s0 >= L) return;  // the whole CTA leaves together, before any barrier
  const int s1 = min(s0 + p.chunk, L);
  const int nst = (s1 - s0 + KS - 1) / KS;
  const int T = p.T;
  const int h0 = kvh * p.g + hc * p.nhpc;
  const int nh = min(p.nhpc, p.g - hc * p.nhpc);
  const int nrows = nh * T;  // MMA row r = (query head h0 + r / T, token r % T)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCW);
    }
    mbar_init(cbar, NCW * 32);
    mbar_init(never, 1);
    *s_fail = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NCW) {  // ---------------------------------------------- producer
    if constexpr (!PAGED) {
      if (lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        const int z = b * p.Hkv + kvh;
        int issued = 0;
        for (int t = 0; t < nst; ++t) {
          const int slot = t % NST;
          if (t >= NST && !mbar_wait(&empty[slot], ((t / NST) - 1) & 1, p.wait_ns, p.err)) break;
          uint8_t *kt = smem + slot * C::STAGE_BYTES;
          uint8_t *vt = kt + C::TILE_BYTES;
          mbar_arrive_expect_tx(&full[slot], C::STAGE_BYTES);
          const int y = s0 + t * KS;
#pragma unroll
          for (int hf = 0; hf < C::NHALF; ++hf) {
            tma_load_3d(kt + hf * HALF_BYTES, &tmk, &full[slot], hf * 64, y, z);
            tma_load_3d(vt + hf * HALF_BYTES, &tmv, &full[slot], hf * 64, y, z);
          }
          issued = t + 1;
        }
        // Do not leave while a copy this thread issued may still be landing.
        for (int t = max(0, issued - NST); t < issued; ++t)
          mbar_wait(&full[t % NST], (t / NST) & 1, p.timeout_ns, p.err);
      }
    } else {
      // The whole warp walks the block table, 32 entries per coalesced load;
      // lane 0 issues the copies.
      if (lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
      }
      const int32_t *table = p.block_table + (size_t)b * p.max_blocks;
      int win = -1, entry = 0;  // entries win .. win+31 of the table, one per lane
      bool bad = false;         // this lane met a live entry outside the pool
      int issued = 0;
      for (int t = 0; t < nst; ++t) {
        const int slot = t % NST;
        if (t >= NST && !__all_sync(0xffffffffu, mbar_wait(&empty[slot], ((t / NST) - 1) & 1, p.wait_ns, p.err)))
          break;
        uint8_t *kt = smem + slot * C::STAGE_BYTES;
        uint8_t *vt = kt + C::TILE_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], C::STAGE_BYTES);
        const int y = s0 + t * KS;
        for (int r = 0; r < KS; r += p.box_rows) {
          const int pos = y + r;
          int page = 0;  // rows past the sequence's end come from page 0 and are masked
          if (pos < L) {
            const int blk = pos / p.page_size;
            if (win < 0 || blk >= win + 32) {
              win = blk;
              entry = (blk + lane < p.max_blocks) ? __ldg(&table[blk + lane]) : 0;
              // an entry outside the pool is read as page 0; if this sequence
              // reads it, that is reported once the copies are issued
              const bool out = (unsigned)entry >= (unsigned)p.num_pages;
              bad |= out && (blk + lane) * p.page_size < L;
              entry = out ? 0 : entry;
            }
            page = __shfl_sync(0xffffffffu, entry, blk - win);
          }
          if (lane == 0) {
            const int z = page * p.Hkv + kvh, off = pos % p.page_size;
#pragma unroll
            for (int hf = 0; hf < C::NHALF; ++hf) {
              tma_load_3d(kt + hf * HALF_BYTES + r * 128, &tmk, &full[slot], hf * 64, off, z);
              tma_load_3d(vt + hf * HALF_BYTES + r * 128, &tmv, &full[slot], hf * 64, off, z);
            }
          }
        }
        issued = t + 1;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(p.err, kErrBadIndex);
      if (lane == 0)
        for (int t = max(0, issued - NST); t < issued; ++t)
          mbar_wait(&full[t % NST], (t / NST) & 1, p.timeout_ns, p.err);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int gid = lane >> 2, tq = lane & 3;
  const int mat = lane >> 3, r8 = lane & 7;

  // Q as the A operand: row r = (query head h0 + r / T, token r % T); rows
  // >= nrows are zero.  q is [B, Hq, T, D].
  uint32_t qa[C::NK][4];
  {
    const bool ok0 = gid < nrows, ok1 = gid + 8 < nrows;
    const int r0 = ok0 ? gid : 0, r1 = ok1 ? gid + 8 : 0;
    const uint32_t *q0 =
        reinterpret_cast<const uint32_t *>(p.q + (((size_t)b * p.Hq + h0 + r0 / T) * T + r0 % T) * D);
    const uint32_t *q1 =
        reinterpret_cast<const uint32_t *>(p.q + (((size_t)b * p.Hq + h0 + r1 / T) * T + r1 % T) * D);
#pragma unroll
    for (int ks = 0; ks < C::NK; ++ks) {
      qa[ks][0] = ok0 ? q0[ks * 8 + tq] : 0u;
      qa[ks][1] = ok1 ? q1[ks * 8 + tq] : 0u;
      qa[ks][2] = ok0 ? q0[ks * 8 + 4 + tq] : 0u;
      qa[ks][3] = ok1 ? q1[ks * 8 + 4 + tq] : 0u;
    }
  }

  float oacc[C::NT][4];
#pragma unroll
  for (int i = 0; i < C::NT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  // last key each of this lane's two rows may see (bottom-right causal for T > 1)
  const int lim[2] = {p.causal ? L - T + gid % T : L - 1, p.causal ? L - T + (gid + 8) % T : L - 1};
  float m[2] = {-CUDART_INF_F, -CUDART_INF_F};  // running max (log2 units), rows gid and gid+8
  float l[2] = {0.f, 0.f};                       // running sum, this lane's share

  uint32_t cphase = 0;  // completed phases of cbar
  auto consumers_sync = [&]() -> bool {
    mbar_arrive(cbar);
    return mbar_wait(cbar, (cphase++) & 1, p.timeout_ns, p.err);
  };

  // test hook: wait for a signal nothing gives, so that this wait runs out
  bool ok = !p.stall || mbar_wait(never, 0, p.wait_ns, p.err);
  for (int t = 0; ok && t < nst; ++t) {
    const int slot = t % NST;
    if (!mbar_wait(&full[slot], (t / NST) & 1, p.timeout_ns, p.err)) {
      ok = false;
      break;
    }
    uint8_t *kt = smem + slot * C::STAGE_BYTES;
    uint8_t *vt = kt + C::TILE_BYTES;
    const int base = s0 + t * KS;
    const int nvalid = min(KS, s1 - base);
    if (nvalid < KS) {
      // Last tile of the sequence: rows past its end hold whatever the cache
      // holds there.  Their probabilities are 0, but 0 * NaN is NaN, so zero
      // the V rows before the P.V product.
      constexpr int CH = C::NHALF * 8;  // 16-byte chunks per row
      for (int i = threadIdx.x; i < (KS - nvalid) * CH; i += NCW * 32) {
        const int row = nvalid + i / CH, c = i % CH;
        *reinterpret_cast<uint4 *>(vt + (c >> 3) * HALF_BYTES + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      if (!consumers_sync()) {
        ok = false;
        break;
      }
    }
    const int kb = warp * 16;  // this warp's keys within the tile
    if (kb < nvalid) {
      const uint32_t kt_u = smem_u32(kt), vt_u = smem_u32(vt);
      float s[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::NK; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt_u + tile_off(kb + (mat >> 1) * 8 + r8, ks * 2 + (mat & 1)), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qa[ks], b0, b1);
        mma_bf16_16816(s[1], qa[ks], b2, b3);
      }
      // scale into log2 units, mask keys past the split, row maxima
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = base + kb + nt * 8 + 2 * tq + (i & 1);
          const float v = (key < s1 && key <= lim[i >> 1]) ? s[nt][i] * p.scale_log2 : -CUDART_INF_F;
          s[nt][i] = v;
          mx[i >> 1] = fmaxf(mx[i >> 1], v);
        }
      float alpha[2], mb[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mn = fmaxf(m[r], mx[r]);
        mb[r] = (mn == -CUDART_INF_F) ? 0.f : mn;  // no key yet: exponentiate against 0, not -inf
        alpha[r] = fast_exp2(m[r] - mb[r]);        // 0 while nothing has been accumulated
        m[r] = mn;
      }
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float e = fast_exp2(s[nt][i] - mb[i >> 1]);
          s[nt][i] = e;
          ps[i >> 1] += e;
        }
      l[0] = l[0] * alpha[0] + ps[0];
      l[1] = l[1] * alpha[1] + ps[1];
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          oacc[nt][0] *= alpha[0];
          oacc[nt][1] *= alpha[0];
          oacc[nt][2] *= alpha[1];
          oacc[nt][3] *= alpha[1];
        }
      }
      // P as the A operand straight from the score registers (bf16)
      const uint32_t pa[4] = {pack_bf16x2(s[0][0], s[0][1]), pack_bf16x2(s[0][2], s[0][3]),
                              pack_bf16x2(s[1][0], s[1][1]), pack_bf16x2(s[1][2], s[1][3])};
#pragma unroll
      for (int dp = 0; dp < C::NT / 2; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vt_u + tile_off(kb + (mat & 1) * 8 + r8, dp * 2 + (mat >> 1)), b0, b1, b2, b3);
        mma_bf16_16816(oacc[2 * dp], pa, b0, b1);
        mma_bf16_16816(oacc[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ------------------------------------------------ merge the four warps' state
  if (!ok) atomicExch(s_fail, 1);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  // every consumer is done with the ring
  if (!consumers_sync() || *reinterpret_cast<volatile int *>(s_fail)) return;

  float *so = reinterpret_cast<float *>(smem);  // [NCW][MROWS][D]
  float *sm = so + NCW * MROWS * D;             // [NCW][MROWS]
  float *sl = sm + NCW * MROWS;                 // [NCW][MROWS]
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = gid + 8 * r;
    if (tq == 0) {
      sm[warp * MROWS + row] = m[r];
      sl[warp * MROWS + row] = l[r];
    }
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      float2 v = make_float2(oacc[nt][2 * r], oacc[nt][2 * r + 1]);
      *reinterpret_cast<float2 *>(&so[(warp * MROWS + row) * D + nt * 8 + 2 * tq]) = v;
    }
  }
  if (!consumers_sync()) return;
  for (int idx = threadIdx.x; idx < nrows * D; idx += NCW * 32) {
    const int row = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm[w * MROWS + row]);
    float tot = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float mw = sm[w * MROWS + row];
      const float f = (mw == -CUDART_INF_F) ? 0.f : fast_exp2(mw - M);
      tot += f * sl[w * MROWS + row];
      acc += f * so[(w * MROWS + row) * D + d];
    }
    // partial rows are (b, head, token), splits innermost
    const size_t ri = ((((size_t)b * p.Hq + h0 + row / T) * T + row % T) * p.nsplit) + split;
    const bool empty_row = !(tot > 0.f);  // no key of this split is visible to the row
    p.part_o[ri * D + d] = empty_row ? 0.f : acc / tot;
    if (d == 0) p.part_lse[ri] = empty_row ? -CUDART_INF_F : M + __log2f(tot);
  }
}

struct CombineParams {
  const int32_t *seqlens;
  const float *part_o;
  const float *part_lse;
  __nv_bfloat16 *o;
  float *lse;
  int Hq, T, Lmax, chunk, nsplit;
};

// One CTA per (sequence, query head), one thread per output column.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(CombineParams p) {
  const int bh = blockIdx.x;  // (b, head, token) row
  const int b = bh / (p.Hq * p.T);
  const int d = threadIdx.x;
  griddep_wait();  // launched early (programmatic dependent launch): wait for the splits
  const int L = max(0, min(p.seqlens[b], p.Lmax));
  const int ns = (L + p.chunk - 1) / p.chunk;
  if (ns == 0) {  // empty sequence
    p.o[(size_t)bh * D + d] = __float2bfloat16(0.f);
    if (d == 0 && p.lse) p.lse[bh] = -CUDART_INF_F;
    return;
  }
  const float *pl = p.part_lse + (size_t)bh * p.nsplit;
  const float *po = p.part_o + (size_t)bh * p.nsplit * D;
  float M = -CUDART_INF_F;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, pl[s]);
  if (M == -CUDART_INF_F) {  // the row sees no key (a causal token before the cache start)
    p.o[(size_t)bh * D + d] = __float2bfloat16(0.f);
    if (d == 0 && p.lse) p.lse[bh] = -CUDART_INF_F;
    return;
  }
  float tot = 0.f, acc = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = exp2f(pl[s] - M);
    tot += w;
    acc += w * po[(size_t)s * D + d];
  }
  p.o[(size_t)bh * D + d] = __float2bfloat16(acc / tot);
  if (d == 0 && p.lse) p.lse[bh] = (M + log2f(tot)) * 0.69314718055994530942f;
}

template <int D, bool PAGED>
cudaError_t launch(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv, cudaStream_t st) {
  using C = Cfg<D>;
  const int g = a.Hq / a.Hkv;
  const int nhpc = decode_heads_per_cta(a.Hq, a.Hkv, a.T);
  const int nhc = (g + nhpc - 1) / nhpc;
  Params p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.seqlens = a.seqlens;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.page_size = a.page_size;
  p.num_pages = a.num_pages;
  p.box_rows = a.page_size < KS ? a.page_size : KS;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Lmax = a.Lmax;
  p.chunk = a.chunk;
  p.nsplit = a.nsplit;
  p.g = g;
  p.nhc = nhc;
  p.T = a.T;
  p.nhpc = nhpc;
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.timeout_ns = a.timeout_ns;
  p.wait_ns = a.wait_ns;
  p.stall = a.stall;
  p.err = a.err;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long nctas = (long)a.nsplit * a.Hkv * nhc * a.B;
  if (nctas > 0x7fffffffL || (long)a.B * a.Hq * a.T > 0x7fffffffL) return cudaErrorNotSupported;
  dim3 grid((unsigned)nctas);
  decode_split_kernel<D, PAGED><<<grid, THREADS, C::SMEM_BYTES, st>>>(tmk, tmv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineParams c;
  c.seqlens = a.seqlens;
  c.part_o = a.part_o;
  c.part_lse = a.part_lse;
  c.o = static_cast<__nv_bfloat16 *>(a.o);
  c.lse = a.lse;
  c.Hq = a.Hq;
  c.T = a.T;
  c.Lmax = a.Lmax;
  c.chunk = a.chunk;
  c.nsplit = a.nsplit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq * a.T);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, c);
}

}  // namespace dec

int decode_chunk(int B, int Hq, int Hkv, int T, int Lmax) {
  const int g = Hq / Hkv;
  const int nhpc = decode_heads_per_cta(Hq, Hkv, T);
  const long units = (long)B * Hkv * ((g + nhpc - 1) / nhpc);
  // With T query tokens every split writes T times the partial output that the
  // combine reads back; fewer, longer splits keep that traffic small (4-token
  // decode of 64 sequences: 10 -> 4 splits, 0.83 -> 0.90 of the copy bandwidth).
  const long target = dec::TARGET_CTAS / (T < 3 ? T : 3);
  long ns = (target + units - 1) / units;
  if (ns < 1) ns = 1;
  long chunk = (Lmax + ns - 1) / ns;
  chunk = (chunk + dec::KS - 1) / dec::KS * dec::KS;
  if (chunk < dec::KS) chunk = dec::KS;
  return (int)chunk;
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                          cudaStream_t stream) {
  const bool paged = a.block_table != nullptr;
  if (a.D == 128) return paged ? dec::launch<128, true>(a, tmap_k, tmap_v, stream)
                               : dec::launch<128, false>(a, tmap_k, tmap_v, stream);
  if (a.D == 64) return paged ? dec::launch<64, true>(a, tmap_k, tmap_v, stream)
                              : dec::launch<64, false>(a, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
