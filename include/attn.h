/*
 * attn.h -- C ABI of the exact tiled attention library for GB300 (sm_103a).
 *
 * The operation (all entry points):  O = softmax(scale * Q K^T + mask) V, with
 * the per-row log-sum-exp LSE_i = log sum_j exp(scale * q_i . k_j) over the
 * allowed keys (natural log).  Problem statement: "Fast Inference and Training
 * at Scale" §6.21 (the attention formula, Q, K, V of N x d_k); the method
 * (tiles, running max / running sum, never writing the score matrix):
 * the same section's "Idea 1", "Week 13. GPUs and FlashAttention" step 2 and
 * "Hardware Co-Design" (FlashAttention section, the online-softmax update).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers owned by the caller (attn_fwd_host takes
 *     its tensors in host memory); the library keeps no pointer after a call
 *     returns and allocates no device memory (every workspace is passed in).
 *   - Layouts are dense row-major ("contiguous"): Q/O [B, Hq, Sq, D],
 *     K/V [B, Hkv, Sk, D], LSE [B, Hq, Sq].  Every tensor pointer must be
 *     16-byte aligned.
 *   - Grouped-query attention ("Fast Inference and Training at Scale" §6.2):
 *     Hq must be a multiple of Hkv; query head h reads key/value head
 *     h / (Hq / Hkv) (contiguous groups).  Hkv == Hq is MHA, Hkv == 1 is MQA.
 *   - causal != 0 masks key j for query i unless j <= i + (Sk - Sq) (aligned at
 *     the bottom right; plain j <= i when Sq == Sk).  A query row with no
 *     allowed key gets O = 0 and LSE = -inf.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are detected on the host before any
 *     CUDA call and return a status without touching the GPU.  A launch
 *     failure returns ATTN_ERR_CUDA.  Device-side faults of the pipeline (a
 *     bounded wait that ran out) are recorded in a device error word that
 *     attn_get_error() reads.
 *   - Size limits: B * Hq and B * Hkv (decode: B * Hq * T; paged: num_pages *
 *     Hkv) at most 2^30 (the TMA coordinate range) and at most 2^31 - 1 CTAs
 *     per launch; beyond them a call returns ATTN_ERR_UNSUPPORTED.  There is
 *     no other limit on the batch or head counts.
 *   - The library is stateless apart from that error word, a per-device
 *     cache of kernel attributes and, for attn_fwd_host, two CUDA streams and
 *     ten events per calling thread and device; calls may come from several
 *     host threads.
 */
#ifndef EXACT_TILED_ATTENTION_ATTN_H
#define EXACT_TILED_ATTENTION_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0 */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head dim other than 64/128) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (reported by attn_get_error) */
  ATTN_ERR_NO_DEVICE = 5,   /* no usable sm_103 device for this call */
  ATTN_ERR_SCRATCH_LIMIT = 6, /* attn_decode_noalloc: sizes need more than its fixed scratch */
  ATTN_ERR_BAD_INDEX = 7      /* a decode read a device-resident index out of range (reported by attn_get_error) */
} attn_status;

/*
 * attn_fwd -- bf16 prefill forward (causal or not, MHA/GQA/MQA).
 *   q   [B, Hq,  Sq, D] bf16          o   [B, Hq, Sq, D] bf16 (written)
 *   k,v [B, Hkv, Sk, D] bf16          lse [B, Hq, Sq] fp32 natural-log LSE
 *                                         (written; may be NULL to skip)
 *   B, Hq, Hkv, Sq, Sk >= 1; D in {64, 128} else ATTN_ERR_UNSUPPORTED;
 *   scale > 0 and finite (usually 1/sqrt(D)).
 * Arithmetic: bf16 products accumulated in fp32 by the tensor cores; softmax
 * in fp32; the probabilities enter the P.V product rounded to bf16; O is
 * divided by the fp32 row sum once at the end and rounded to bf16.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                     float scale, attn_stream_t stream);

/* attn_fwd_host_workspace_bytes -- device scratch for attn_fwd_host (three
 * chunk buffers); 0 on invalid sizes. */
size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D);

/*
 * attn_fwd_host -- attn_fwd for q, k, v, o (and lse, nullable) in HOST memory,
 * same layouts and arguments.  The (batch, KV head) units are independent
 * problems ("Fast Inference and Training at Scale" §6.2: each query head reads
 * only its group's K and V), so the call is cut into chunks of consecutive
 * units whose host-to-device copies, kernels and device-to-host copies overlap
 * on three streams; each chunk is an attn_fwd call, so the results equal
 * attn_fwd's on device copies of the same data.
 *   workspace: device memory >= attn_fwd_host_workspace_bytes(...), 256-byte
 *   aligned, owned by the caller.
 *   Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 *   the copies to overlap; pageable memory works but serialises them.
 * Asynchronous: work before the call on `stream` is ordered before it, and
 * `stream` waits until o and lse are back in host memory; the host must not
 * read o before synchronising the stream.  On first use per calling thread and
 * device it creates two CUDA streams and ten events, kept until process exit.
 * Errors: as attn_fwd; ATTN_ERR_INVALID_ARG for a short or misaligned
 * workspace.
 */
attn_status attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                          void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* attn_bwd_workspace_bytes -- scratch for attn_bwd (fp32 dQ accumulator and
 * rowsum(dO o O)); 0 on invalid sizes. */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq, int D);

/*
 * attn_bwd -- gradients of attn_fwd with recomputation ("Fast Inference and
 * Training at Scale" §6.21, Idea 2; "Week 13. GPUs and FlashAttention"
 * step 2: only O and the log-sum-exp are kept from the forward).
 *   q, k, v, o as for attn_fwd; lse [B, Hq, Sq] fp32 from attn_fwd;
 *   dout [B, Hq, Sq, D] bf16 (gradient of O).
 *   dq [B, Hq, Sq, D], dk/dv [B, Hkv, Sk, D] bf16 (written).  With GQA the
 *   gradient of a key/value head sums over its group's query heads.
 *   workspace >= attn_bwd_workspace_bytes(B, Hq, Sq, D), 256-byte aligned.
 *   D in {64, 128}.  causal, scale as for attn_fwd.
 * dS and P enter the tensor-core products as bf16; dQ is accumulated in fp32.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Sq, int Sk,
                     int D, int causal, float scale, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream);

/*
 * attn_decode_workspace_bytes -- size in bytes of the scratch attn_decode needs
 * for these sizes (partial outputs of the key splits).  0 on invalid sizes.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D);

/*
 * attn_decode -- one query token per sequence against a contiguous KV cache
 * ("Fast Inference and Training at Scale" §6.1: the new token's query attends
 * over every cached position, the cache already holding its own K and V).
 *   q       [B, Hq, D] bf16            o   [B, Hq, D] bf16 (written)
 *   kcache, vcache [B, Hkv, Lmax, D] bf16
 *   seqlens [B] int32 device array, 0 <= seqlens[b] <= Lmax; rows at or beyond
 *           seqlens[b] are never read into the result.  seqlens[b] == 0 gives
 *           O = 0, LSE = -inf.  A value outside [0, Lmax] is clamped into it
 *           and recorded as ATTN_ERR_BAD_INDEX for attn_get_error (that
 *           sequence's output is then meaningless; the others are unaffected).
 *   lse     [B, Hq] fp32 natural-log LSE (may be NULL)
 *   workspace: device scratch of at least attn_decode_workspace_bytes(...)
 *           bytes, 256-byte aligned; contents on entry do not matter; calls that
 *           share one workspace must not overlap on the GPU.
 *   Hq / Hkv <= 16 heads share a key/value head per block of work (larger
 *   groups are split); D in {64, 128}.
 * Keys are split into chunks processed in parallel, each with its own running
 * max and sum; the partial results are merged with log-sum-exp weights.
 */
attn_status attn_decode(const void *q, const void *kcache, const void *vcache,
                        const int32_t *seqlens, void *o, float *lse,
                        int B, int Hq, int Hkv, int Lmax, int D, float scale,
                        void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_multi_workspace_bytes -- scratch for attn_decode_multi (0 on
 * invalid sizes).
 */
size_t attn_decode_multi_workspace_bytes(int B, int Hq, int Hkv, int T, int Lmax, int D);

/*
 * attn_decode_multi -- T query tokens per sequence against its KV cache: the
 * verification step of speculative decoding, or a short chunk of prefill
 * ("Week 13. GPUs and FlashAttention", step 1: draft verification scores
 * gamma + 1 tokens per sequence in one pass).  The cache already holds the T
 * new tokens' K and V (seqlens[b] counts them).
 *   q [B, Hq, T, D] bf16, o [B, Hq, T, D] bf16, lse [B, Hq, T] fp32 (may be NULL)
 *   kcache, vcache [B, Hkv, Lmax, D] bf16, seqlens [B] int32 as for attn_decode.
 *   1 <= T <= 16 (else ATTN_ERR_UNSUPPORTED).
 *   causal != 0: token t sits at position seqlens[b] - T + t and sees keys at
 *           positions <= its own (bottom-right alignment); a token whose
 *           position is negative sees nothing (O = 0, LSE = -inf).
 *           causal == 0: every token sees all seqlens[b] keys.
 *   workspace: at least attn_decode_multi_workspace_bytes(B, Hq, Hkv, T, Lmax, D)
 *           bytes, 256-byte aligned.
 * With T = 1 this is attn_decode.
 */
attn_status attn_decode_multi(const void *q, const void *kcache, const void *vcache, const int32_t *seqlens,
                              void *o, float *lse, int B, int Hq, int Hkv, int T, int Lmax, int D, int causal,
                              float scale, void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_paged -- attn_decode against a paged KV cache ("Fast Inference
 * and Training at Scale" §6.3, PagedAttention: the cache lives in fixed-size
 * blocks reached through a per-sequence block table).
 *   k_pages, v_pages [num_pages, Hkv, page_size, D] bf16: the shared page pool.
 *   block_table [B, max_blocks] int32: position t of sequence b is row
 *           t % page_size of page block_table[b, t / page_size].  Only the
 *           entries covering positions < seqlens[b] are read; an entry
 *           outside [0, num_pages) is read as page 0 (no fault) and recorded
 *           as ATTN_ERR_BAD_INDEX for attn_get_error (that sequence's output is
 *           then meaningless; the others are unaffected).
 *   seqlens [B] int32, 0 <= seqlens[b] <= max_blocks * page_size.
 *   page_size in {16, 32, 64, 128, 256} else ATTN_ERR_UNSUPPORTED.
 *   workspace: at least attn_decode_workspace_bytes(B, Hq, Hkv,
 *           max_blocks * page_size, D) bytes, 256-byte aligned.
 *   q, o, lse, D, scale and errors as for attn_decode.
 */
attn_status attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *block_table, const int32_t *seqlens, void *o, float *lse,
                              int B, int Hq, int Hkv, int page_size, int max_blocks, int num_pages, int D,
                              float scale, void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* Size of the fixed device scratch array used by attn_decode_noalloc. */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

/*
 * attn_decode_noalloc -- attn_decode without a workspace argument; it
 * allocates nothing.  (The pages have no counterpart of this call: it exists
 * for callers, not for the method.)
 *   For callers that cannot obtain device scratch: code handed only input and
 *   output buffers (a custom-op or plugin interface with no workspace slot), or
 *   a serving loop that must not call cudaMalloc, which may synchronise the
 *   device.  No cudaMalloc, cudaFree or allocating library call is made.
 *   Arguments, layouts, results and errors are those of attn_decode.  The
 *   scratch is one static device array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES
 *   (16 MiB) that each GPU running this call keeps until the process exits.
 *   Sizes whose attn_decode_workspace_bytes() exceeds it return
 *   ATTN_ERR_SCRATCH_LIMIT before any GPU work.  The need is about
 *   B * Hq * nsplit * (D + 1) * 4 bytes with nsplit ~ 4864 / (B * Hkv) key
 *   splits (at most ceil(Lmax / 64)); e.g. 64 sequences, 32 query / 8 KV
 *   heads, D = 128 need 10.1 MiB whatever Lmax is.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make it before any
 *   stream capture.  All calls share the array: calls whose GPU work overlaps
 *   race and return wrong results, so serialise them.  Nothing in the array
 *   needs to start at zero.
 */
attn_status attn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                                const int32_t *seqlens, void *o, float *lse,
                                int B, int Hq, int Hkv, int Lmax, int D, float scale,
                                attn_stream_t stream);

/*
 * attn_fwd_fp8 -- FP8 e4m3 prefill forward with block quantisation
 * ("FlashAttention scaling, multi-GPU training and weight quantization" §1,
 * FlashAttention-3: FP8 tensor cores, tiles scaled independently).
 *   q8 [B, Hq, Sq, D], k8/v8 [B, Hkv, Sk, D]: e4m3 codes (OCP E4M3, 1 byte).
 *   q_scale [B, Hq,  ceil(Sq/128), ceil(D/128)] fp32, k_scale/v_scale
 *   [B, Hkv, ceil(Sk/128), ceil(D/128)] fp32: the real value of element
 *   (b,h,s,d) is e4m3(code) * scale[b,h,s/128,d/128].
 *   o [B, Hq, Sq, D] bf16, lse [B, Hq, Sq] fp32 (may be NULL).
 *   D = 64 or 128 (one scale tile spans the head dimension; D = 64 runs
 *   on the D = 128 kernel with the upper 64 columns read as zeros, at the
 *   D = 128 cost).  ATTN_ERR_UNSUPPORTED for any other D.
 * Scores are dequantised with one scalar per (query tile, key tile); the
 * probabilities enter the P.V product as e4m3 with the value tile's scale
 * folded in.
 */
attn_status attn_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                         const float *q_scale, const float *k_scale, const float *v_scale,
                         void *o, float *lse, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                         int causal, float scale, attn_stream_t stream);

/*
 * attn_rotate_quantize_fp8 -- prepares attn_fwd_fp8's inputs: optional Hadamard
 * rotation, then block quantisation to e4m3 with one fp32 scale per 128 x 128
 * tile ("FlashAttention scaling, multi-GPU training and weight quantization"
 * §1, FlashAttention-3: incoherent processing and block quantisation).
 *   x      [B, H, S, D] bf16, D = 64 or 128 (else ATTN_ERR_UNSUPPORTED)
 *   signs  [D] fp32 of +-1, or NULL for no rotation (use NULL for V and the
 *          same signs for Q and K, which leaves Q K^T unchanged)
 *   codes  [B, H, S, D] e4m3 bytes (written)
 *   scales [B, H, ceil(S/128), 1] fp32 (written)
 * With signs, y = x R, R = H_D diag(signs) / sqrt(D) (Sylvester Hadamard);
 * else y = x.  Per tile: scale = max |y| / 448 (1 if the tile is all zero),
 * code = e4m3(y / scale), nearest even, saturating at +-448.
 */
attn_status attn_rotate_quantize_fp8(const void *x, uint8_t *codes, float *scales, const float *signs, int B, int H,
                                     int S, int D, attn_stream_t stream);

/* One tensor of attn_rotate_quantize_fp8_many (layouts as for attn_rotate_quantize_fp8). */
typedef struct attn_quant_tensor {
  const void *x;   /* [B, H, S, D] bf16, 16-byte aligned, read */
  uint8_t *codes;  /* [B, H, S, D] e4m3 bytes, 16-byte aligned, written */
  float *scales;   /* [B, H, ceil(S/128), 1] fp32, written */
  int B, H, S;
  int rotate; /* nonzero: y = x R with the call's signs; zero: y = x */
} attn_quant_tensor;

#define ATTN_QUANT_MAX_TENSORS 4

/*
 * attn_rotate_quantize_fp8_many -- attn_rotate_quantize_fp8 for up to
 * ATTN_QUANT_MAX_TENSORS tensors in one launch, e.g. the three inputs of
 * attn_fwd_fp8: Q and K rotated with the same signs (so Q K^T is unchanged),
 * V not.  The tensors' tiles are shared out over one persistent grid, so the
 * launch's fixed costs (start, ramp, drain) are paid once.
 *   tensors  host array of n descriptors (read during the call only)
 *   signs    [D] fp32 of +-1, device; may be NULL when no tensor rotates
 *   D        head dimension of every tensor, 64 or 128
 * Results are identical to one attn_rotate_quantize_fp8 call per tensor.
 * ATTN_ERR_INVALID_ARG for a NULL or misaligned pointer, a size < 1, n < 1 or
 * a rotating tensor without signs; ATTN_ERR_UNSUPPORTED for n >
 * ATTN_QUANT_MAX_TENSORS, D not 64 or 128, or B * H > 2^30.  Tensors must not
 * overlap one another's outputs.
 */
attn_status attn_rotate_quantize_fp8_many(const attn_quant_tensor *tensors, int n, const float *signs, int D,
                                          attn_stream_t stream);

/*
 * attn_get_error -- synchronises `stream`, then returns and clears the device
 * error word of the current device: ATTN_OK, or the first device-side error
 * since the last call: ATTN_ERR_TIMEOUT if a bounded pipeline wait ran out
 * (its kernel then returned early and its outputs are invalid),
 * ATTN_ERR_BAD_INDEX if a decode met a sequence length outside [0, Lmax] or a
 * block-table entry outside [0, num_pages).  ATTN_ERR_CUDA if the
 * synchronisation failed.
 */
attn_status attn_get_error(attn_stream_t stream);

/*
 * attn_debug_stall_role_waits -- test hook for the failure path of the
 * pipelines (no page defines it).  Inside a CTA of the prefill forward
 * (attn_fwd, attn_fwd_fp8), the backward (attn_bwd), the rotate + quantise
 * kernel (attn_rotate_quantize_fp8, _many) and the decode split kernel
 * (attn_decode, _paged, _multi, _noalloc), warp roles wait on one another
 * (the softmax for the scores, the tensor-core issuer for the probabilities,
 * the producer for a freed stage, ...), each wait bounded in time.  With
 * enable != 0, every such call made afterwards first has its softmax
 * (backward: gradient; quantise: epilogue; decode: consumer) warps wait for a
 * signal that nothing gives, and the bound of the waits between
 * roles is cut to 1 ms: those waits run out, the kernel records
 * ATTN_ERR_TIMEOUT (returned by the next attn_get_error()) and the outputs of
 * that call are invalid.  Waits for data copies and for a CTA's own
 * tensor-core work keep the normal bound (4 s), so a CTA that gives up still
 * lets every copy and product it started complete and frees its tensor
 * memory before it ends; the GPU context stays usable.  enable = 0 restores
 * normal operation.  Process-wide; for tests only.
 */
void attn_debug_stall_role_waits(int enable);

/*
 * attn_debug_skew_roles -- test hook for the synchronisation of the FP8
 * prefill forward (attn_fwd_fp8; no page defines it).  There the issuing
 * thread asks for the next key tile's scores before it consumes the current
 * probabilities, so a warp role may run up to a key tile ahead of another.
 * With enable != 0, every attn_fwd_fp8 call made afterwards runs a build of
 * the kernel in which the issuing thread pauses 20 us after each request for
 * scores and the softmax warps of each CTA's first query tile pause 20 us
 * before each wait for scores, so that the other roles get as far ahead as
 * the protocol allows.  Results and error reporting are those of a normal
 * call (only slower); a protocol that miscounted a barrier phase would show
 * as ATTN_ERR_TIMEOUT from attn_get_error().  enable = 0 restores normal
 * operation.  Process-wide; for tests only.
 */
void attn_debug_skew_roles(int enable);

/* Human-readable name of a status code (static string). */
const char *attn_status_str(attn_status status);

/* Library version string, e.g. "0.1.0". */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* EXACT_TILED_ATTENTION_ATTN_H */
