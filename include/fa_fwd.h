/*
 * fa_fwd.h -- C ABI of the GB300 (sm_103a) tiled FlashAttention forward.
 *
 * One operation: O = softmax(scale * Q K^T + mask) V for every query row,
 * computed tile by tile with a per-row online softmax (running max m, running
 * sum l, rescale of the O accumulator), never materialising S or P, plus the
 * per-row log-sum-exp LSE = scale * m + ln(l) for a backward pass.
 *
 * Where the operation is defined:
 *   - attention itself and its blockwise / online-softmax form:
 *     "FlashAttention correctness verification" (ai6s.net), sections
 *     "Standard Attention vs FlashAttention: mathematical equivalence" and
 *     "Formal verification outline" (loop invariant, inductive step
 *     L_{i+1} = L_i exp(m_i - m_{i+1}) + l_{i+1});
 *   - scale, mask and the softmax max / sum outputs kept for the backward:
 *     "FlashAttentionScore" operator doc (gitcode ops-transformer), sections
 *     "Function description" (forward formula) and "Parameter description"
 *     (softmaxMaxOut / softmaxSumOut);
 *   - BNSD layout, GQA (Hq % Hkv == 0), per-batch actual sequence lengths,
 *     compact per-Q-block KV-block lists with invalid slots, LSE semantics
 *     P = exp(scale*S - LSE): "BSA (Block Sparse Attention) PyPTO
 *     implementation notes", sections 1 "Overview", 3.2 "Core design
 *     strategies" and 3.3 "Data layout and tiling";
 *   - top-k gathered keys shared by all heads (sparse MLA, MQA) and the
 *     exact-running-max versus lazy-rescale switch (threshold in log2 units):
 *     "Sparse-MLA training forward: exact running max vs lazy rescale"
 *     (cf-1.com), sections "Background: sparse MLA and top-k gathered KV" and
 *     "Verifying the threshold branch from source".
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are caller-owned DEVICE memory on the current
 *     device, contiguous, and must stay valid until the work on `stream` has
 *     finished.  The library keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Argument errors are returned
 *     synchronously and nothing is launched.  Device-side errors are
 *     reported later through fa_check_status().
 *   - The dense / GQA / block-sparse paths allocate nothing (a bf16 V is
 *     converted to fp16 tile by tile inside the kernel), except a dense
 *     problem with too few (batch, head, query-tile) units to fill half the
 *     GPU: its units' KV tiles are split into up to fa_set_max_kv_split()
 *     pieces whose partial O / l and LSE (fp32) go to stream-ordered scratch
 *     and are merged by a second kernel (the blockwise merge of
 *     "FlashAttention correctness verification", ai6s.net, section "Standard
 *     Attention vs FlashAttention: mathematical equivalence", in log-sum-exp
 *     form).  The top-k path with a bf16 key latent converts the latent to
 *     fp16 into stream-ordered scratch.  Scratch comes from cudaMallocAsync
 *     on the device's default memory pool and is released on `stream` after
 *     use; fa_fwd_noalloc uses a fixed array instead and allocates nothing at
 *     all (a split that does not fit it runs unsplit).  Why scratch at all:
 *     the split's partial results must outlive the kernel that writes them
 *     until the merge kernel reads them, and the top-k kernel reads each
 *     latent row many times (once per token that lists it), so converting
 *     it once per call is cheaper than converting it at every gather.
 */
#ifndef FA_FWD_H_
#define FA_FWD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define FA_OK                   0
#define FA_ERR_NULL            -1  /* a required pointer is NULL                      */
#define FA_ERR_SHAPE           -2  /* a size <= 0, Hq % Hkv != 0, both sparse modes,  */
                                   /* block != 128, max_sel / topk out of range, ...  */
#define FA_ERR_UNSUPPORTED     -3  /* (D, Dv, dtype, mode) combination not built      */
#define FA_ERR_ALIGN           -4  /* tensor base not 16-byte aligned (lse: 4 bytes)  */
#define FA_ERR_THRESHOLD       -5  /* rescale_threshold outside [0, 15] or not finite */
#define FA_ERR_CUDA            -6  /* a CUDA call failed; see fa_last_cuda_error()    */
#define FA_ERR_DEVICE_TIMEOUT  -7  /* a bounded on-chip wait expired (kernel bailed)  */
#define FA_ERR_RANGE           -8  /* a bf16 value outside the fp16 range (|x| >      */
                                   /* 65504) met an fp16 product (V; with top-k also  */
                                   /* Q and the key latent), or fa_bwd with fp16      */
                                   /* inputs met a dS beyond that range               */
#define FA_ERR_SCRATCH         -9  /* fa_fwd_noalloc, top-k: the bf16 key latent     */
                                   /* needs more than its fixed scratch               */
                                   /* (B*Skv*D*2 > 32 MiB)                            */

/* ---- mask_mode flag word ----------------------------------------------- */
/* bits 0-3: mask */
#define FA_MASK_NONE             0  /* every key j < kv_len is visible                */
#define FA_MASK_CAUSAL           1  /* key j masked for query i when j > i (top-left) */
#define FA_MASK_CAUSAL_DIAG_BLOCK 2 /* block-sparse only: j > i masked only inside    */
                                    /* the diagonal block (key block == query block)  */
/* element type of q, k, v and o (default bf16) */
#define FA_DTYPE_FP16        0x100
/* top-k only: V is the first Dv columns of every K row (shared MLA latent);   */
/* `v` may then be NULL */
#define FA_V_FROM_K          0x200
/* bf16 q / o with an fp16 copy of the value operand made beforehand by      */
/* fa_convert_v_fp16 (e.g. once for a KV cache read by many calls): `v`, or   */
/* with FA_V_FROM_K the key latent `k`, is fp16; skips the conversion */
#define FA_V_FP16            0x400

/* ---- sparse descriptors ------------------------------------------------ */

/* Compact per-Q-block KV-block lists ("Mask2Idx", BSA notes section 1).
 * The entry for batch b, query head h, query block qb, slot s is
 *   idx[b*stride_b + h*stride_h + qb*max_sel + s]   (device int32)
 * Query block qb covers rows [qb*block, qb*block + block); a valid entry e
 * names keys [e*block, e*block + block).  An entry < 0 or >= ceil(Skv/block)
 * is an invalid slot and contributes nothing.  stride_h = 0 shares one list
 * among all heads.  Each valid slot counts once (a block listed twice counts
 * twice).  Slots are visited in list order.  block must be 128, 1 <= max_sel
 * <= 512. */
typedef struct {
  const int32_t* idx;
  int32_t max_sel;
  int32_t block;
  int64_t stride_b;
  int64_t stride_h;
} fa_block_sparse_t;

/* Top-k gathered keys, shared by all query heads (sparse MLA / MQA).
 * The entry for batch b, query row i, slot w is idx[b*stride_b + i*topk + w]
 * (device int32); an entry < 0 or >= kv_len is an invalid slot. */
typedef struct {
  const int32_t* idx;
  int32_t topk;
  int64_t stride_b;
} fa_topk_t;

/* ---- the forward ------------------------------------------------------- */
/*
 * fa_fwd -- attention forward with online softmax and LSE output.
 *
 *   q    [B, Hq,  Sq,  D ]  bf16 or fp16 (FA_DTYPE_FP16), contiguous BNSD
 *   k    [B, Hkv, Skv, D ]  same type
 *   v    [B, Hkv, Skv, Dv]  same type (NULL with FA_V_FROM_K)
 *   o    [B, Hq,  Sq,  Dv]  same type, written in full (padding rows too)
 *   lse  [B, Hq,  Sq]       fp32, natural log over scaled scores,
 *                           +inf for a row with no valid key or a padding row
 *   query head h reads KV head h / (Hq / Hkv).
 *   scale          multiplies Q K^T before the softmax (typically 1/sqrt(D)).
 *   mask_mode      FA_MASK_* | FA_DTYPE_FP16 | FA_V_FROM_K.
 *   seqlens        NULL, or device int32[B]: actual length of batch b, applied
 *                  to queries and keys alike; rows i >= seqlens[b] are padding
 *                  (O = 0, LSE = +inf) and keys j >= seqlens[b] are masked.
 *                  Padding rows of k and v must hold finite values.
 *   kv_block_idx   NULL, or host pointer to a block-sparse descriptor (its
 *                  idx array is device memory).
 *   topk_idx       NULL, or host pointer to a top-k descriptor.  At most one
 *                  of kv_block_idx / topk_idx may be set.
 *   rescale_threshold  0 = exact running max (O and l are rescaled whenever a
 *                  row max grows); t > 0 = lazy rescale: the running max is
 *                  kept until a block's max exceeds it by more than t in
 *                  log2 units of scaled scores (t = 8 is the usual lazy
 *                  setting).  Range [0, 15] so that p <= 2^t fits the fp16 P
 *                  operand.  Every setting targets the same exact result.
 *   stream         cudaStream_t, as void*.
 *
 * Supported (D, Dv): dense / causal / ragged / GQA / block-sparse: D = Dv in
 * {64, 128}; top-k: D = 576, Dv = 512 with FA_V_FROM_K.
 * Returns FA_OK or a negative FA_ERR_* code (nothing launched on error).
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale,
           int mask_mode, const int32_t* seqlens,
           const fa_block_sparse_t* kv_block_idx, const fa_topk_t* topk_idx,
           float rescale_threshold, void* stream);

/* ---- optional terms of the operator ------------------------------------ */
/*
 * The "FlashAttentionScore" operator doc (gitcode ops-transformer), sections
 * "Function description" (forward formula: s = scale * Q K^T + pse, masked,
 * softmax, times V) and "Parameter description" (atten_mask, pse_type,
 * sparse_mode, pre_tokens / next_tokens):
 *
 *   window       0: no window.
 *                1: sparse_mode 0, key j visible from query i when
 *                   i - pre_tokens <= j <= i + next_tokens (a band);
 *                2: sparse_mode 3, bottom-right causal: j <= i + kv_len - q_len,
 *                   so the last query of a sequence sees up to its last key
 *                   (kv_len, q_len: the batch's actual lengths when seqlens
 *                   is given, else Skv, Sq).
 *                Top-left causal (sparse_mode 2) is FA_MASK_CAUSAL in
 *                mask_mode; it may be combined with a window (both apply).
 *   pre_tokens, next_tokens   window 1 only (any int; values beyond +-(Sq + Skv)
 *                act as unbounded).
 *   atten_mask   NULL, or DEVICE uint8 with element (b, h, i, j) at
 *                atten_mask[b*mask_stride_b + h*mask_stride_h + i*mask_stride_q + j];
 *                a nonzero byte masks key j for query i.  Strides in
 *                elements, >= 0 (0 broadcasts over batch or head); the base,
 *                mask_stride_q, mask_stride_h and mask_stride_b must be
 *                multiples of 16 bytes and Skv a multiple of 16 (16-byte loads).
 *   alibi        0: none; 1: pse_type 2, the position bias -slope_h * |i - j|
 *                added after the scale; 2: pse_type 3, -slope_h * sqrt(|i - j|);
 *                slope_h = 2^(-8 (h + 1) / Hq).
 *   pse          NULL, or DEVICE bias of q's type (bf16, or fp16 with
 *                FA_DTYPE_FP16), element (b, h, i, j) at
 *                pse[b*pse_stride_b + h*pse_stride_h + i*pse_stride_q + j];
 *                strides in elements, >= 0 (0 broadcasts), multiples of 8,
 *                the base 16-byte aligned and Skv a multiple of 8.
 *   pse_type     with pse: 0 adds it after the scale (s = scale Q K^T + pse),
 *                1 before (s = scale (Q K^T + pse)).  pse and alibi are
 *                exclusive (the doc's pse_type picks one).
 *   keep_prob    0 (a zero-initialised struct) or 1: no dropout.  In
 *                (0, 1): dropout after the softmax,
 *                O = (P * M / keep_prob) V with LSE still the softmax's
 *                ("FlashAttentionScoreGrad" pytest framework write-up,
 *                section 5.2).  M follows its section 5.3 generator:
 *                element (b, h, i, j), at index e of the row-major
 *                [B, Hq, Sq, Skv] grid, is kept when byte e % 16 of the
 *                Philox4x32-10 output for counter offset / 16 + e / 16
 *                (counter words: its low and high 32 bits, then 0, 0; key:
 *                the seed's low and high 32 bits; bytes of the four output
 *                words in order, low byte first) is below keep_prob * 255.
 *                offset and Skv must be multiples of 16.
 *   seed, offset the generator's seed and stream offset (in elements).
 *
 * A row whose keys are all masked gets O = 0 and LSE = +inf, as in fa_fwd.
 */
typedef struct {
  int32_t window;
  int32_t pre_tokens;
  int32_t next_tokens;
  int32_t alibi;
  const uint8_t* atten_mask;
  int64_t mask_stride_b;
  int64_t mask_stride_h;
  int64_t mask_stride_q;
  const void* pse;
  int64_t pse_stride_b;
  int64_t pse_stride_h;
  int64_t pse_stride_q;
  int32_t pse_type;
  float keep_prob;
  uint64_t seed;
  uint64_t offset;
} fa_extras_t;

/* fa_fwd with the optional terms above (`extras` is a host pointer, required).
 * Dense / causal / ragged / GQA problems only (no block-sparse or top-k
 * descriptors), D = Dv in {64, 128}, ceil(Skv / 128) <= 512; mask_mode
 * FA_MASK_NONE or FA_MASK_CAUSAL plus the dtype flags.  Every other argument
 * and output as fa_fwd.  Errors: FA_ERR_NULL (extras NULL), FA_ERR_SHAPE
 * (window, alibi or pse_type out of range, pse with alibi, negative stride,
 * Skv too long, keep_prob outside [0, 1], a dropout offset or Skv not a
 * multiple of 16), FA_ERR_ALIGN (mask or pse layout), FA_ERR_UNSUPPORTED (D, Dv), and those of
 * fa_fwd.  Allocates nothing. */
int fa_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale,
               int mask_mode, const int32_t* seqlens, const fa_extras_t* extras,
               float rescale_threshold, void* stream);

/* ---- FP8 inputs ---------------------------------------------------------- */
#define FA_FP8_E4M3  0   /* e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits, max 448 */
#define FA_FP8_E5M2  1   /* e5m2:  1 sign, 5 exponent (bias 15), 2 mantissa bits, max 57344 */

/* fa_fwd_fp8 -- the forward on FP8 query / key / value with full-quantisation
 * dequant scales ("FlashAttentionScore" operator doc, gitcode ops-transformer,
 * parameter table: d_scale_q / d_scale_k / d_scale_v), formed as the
 * "FlashAttentionScoreGrad" pytest framework write-up, section 5.1, gives
 * them: per (batch, head) along S in blocks of 128 rows, the attention then
 * runs on x_q * d_scale.
 *   q8 [B, Hq, Sq, D], k8 [B, Hkv, Skv, D], v8 [B, Hkv, Skv, Dv]: DEVICE
 *      bytes in fp8_format (FA_FP8_E4M3 or FA_FP8_E5M2), 16-byte aligned;
 *   d_scale_q [B, Hq, ceil(Sq / 128)], d_scale_k [B, Hkv, ceil(Skv / 128)],
 *      d_scale_v [B, Hkv, ceil(Skv / 128)]: DEVICE fp32;
 *   o [B, Hq, Sq, Dv]: fp16; lse, scale, seqlens, rescale_threshold as fa_fwd;
 *   mask_mode: FA_MASK_NONE or FA_MASK_CAUSAL (no dtype flags);
 *   extras: NULL, or the optional terms of fa_fwd_ext (a pse tensor is fp16).
 * D = Dv in {64, 128}, ceil(Skv / 128) <= 512.  Q and K are copied to fp16
 * exactly (both formats lie inside fp16) and the kernel scales S of each
 * (query block, key block) pair by d_q d_k, so the scores see the exact x_q
 * values; V is copied as x_q * d_v rounded once to fp16.  The copies live in
 * stream-ordered scratch.  Errors as fa_fwd_ext, plus
 * FA_ERR_NULL for a missing scale and FA_ERR_SHAPE for an unknown format. */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* d_scale_q,
               const float* d_scale_k, const float* d_scale_v, int fp8_format, void* o, float* lse,
               int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
               const int32_t* seqlens, const fa_extras_t* extras, float rescale_threshold,
               void* stream);

/* fa_fwd that also writes the output's rounding residual
 *   o_lo = fp32(O) - O rounded to o's type,
 * itself rounded to that type, same layout as o (rows past Sq / padded heads
 * untouched), so that o + o_lo carries O to about twice o's precision for a
 * backward that recomputes with it ("Sparse-MLA training forward: exact
 * running max vs lazy rescale" (cf-1.com), section "Tests: order-invariance
 * verification", the precise-dpsum test).  o_lo: DEVICE memory, 16-byte
 * aligned; FA_ERR_NULL / FA_ERR_ALIGN otherwise.  Every other argument and
 * return code as fa_fwd. */
int fa_fwd_o_lo(const void* q, const void* k, const void* v, void* o, void* o_lo, float* lse,
                int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale,
                int mask_mode, const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
                const fa_topk_t* topk_idx, float rescale_threshold, void* stream);

/* fa_bwd -- gradients of the dense forward for an upstream gradient dout:
 *   P = exp(scale * Q K^T - LSE) recomputed from the forward's LSE,
 *   d_row = rowsum(dout * (o + o_lo)),   dV = P^T dout,
 *   dS = P * (dout V^T - d_row),   dQ = scale dS K,   dK = scale dS^T Q
 * ("BSA PyPTO implementation notes" (gitcode pypto-gym), sections 3.2
 * "Core design strategies" (recomputation), 8.4 (d_row precomputed) and 1
 * (dV unscaled, dQ / dK scaled)).  GQA: dK / dV sum over the heads of a group.
 * q, o, dout, dq: [B, Hq, Sq, D]; k, v, dk, dv: [B, Hkv, Skv, D]; lse:
 * [B, Hq, Sq] fp32 as fa_fwd wrote it; all DEVICE memory, bf16 (or fp16 with
 * FA_DTYPE_FP16 in mask_mode), 16-byte aligned (lse 4).  o_lo: the residual
 * from fa_fwd_o_lo, or NULL; without it the dpsum uses the rounded output, and
 * on causal problems dQ / dK then lose about an order of magnitude in
 * accuracy.  mask_mode: FA_MASK_NONE or FA_MASK_CAUSAL (top-left), plus
 * FA_DTYPE_FP16; seqlens as fa_fwd.  D = Dv, 64 or 128 (FA_ERR_UNSUPPORTED
 * otherwise).  Rows past a batch's length get zero gradients.  S, P, dP and
 * dS are materialised for a batch of (KV head, head of its group) planes at a
 * time and every product is a cuBLAS tensor-core GEMM of the inputs' type
 * accumulating in fp32 (S and dP exact, P and dS as hi + lo pairs of that
 * type).  With fp16 inputs a |dS| beyond 65504 cannot be held by the pair:
 * the gradients are then not finite and fa_check_status() reports
 * FA_ERR_RANGE.  Stream-ordered scratch (cudaMallocAsync, freed on `stream`):
 * d_row; fp32 dq; fp32 dk and dv with two rows per key (the products of the
 * hi and lo parts, summed at the end); k with every row twice (16-bit);
 * 8 * Sq * Skv bytes per plane of a batch (S and dP in fp32, then the P and
 * dS pairs in place), batches of up to 1 GiB (at least one plane).  Calls from several host threads
 * serialise their enqueueing on one lock per process.  Returns FA_OK or a
 * negative FA_ERR_* code (nothing launched on an argument error). */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* o_lo,
           const float* lse, const void* dout, void* dq, void* dk, void* dv, int B, int Hq,
           int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
           const int32_t* seqlens, void* stream);

/*
 * fa_fwd_noalloc -- fa_fwd without any memory allocation.  (The pages define
 * no counterpart: this is an interface for callers, not part of the method.)
 *
 * For callers that cannot let a library allocate device memory: programs that
 * hand out all device memory from their own fixed arena and account for every
 * byte, and latency-critical call sites where a driver allocation (and the
 * synchronisation it may imply) is not acceptable.  fa_fwd takes
 * stream-ordered scratch from the device's memory pool in two cases: the fp16
 * copy of a bf16 key latent (top-k path) and the fp32 partial results of a
 * dense problem split along its KV tiles (too few units to fill half the
 * GPU).  This entry point puts either into one fixed array inside the
 * library's device image instead (32 MiB, held by every device that loads
 * the library until the process exits) and calls no cudaMalloc, cudaFree or
 * other allocating routine.  Every other call allocates nothing in either
 * entry point.
 *
 * Same arguments, layouts and results as fa_fwd (bit for bit, whenever the
 * split pieces fit the array).  Differences:
 *   - top-k calls with a bf16 key latent of B*Skv*D*2 bytes > 32 MiB are
 *     rejected with FA_ERR_SCRATCH before any CUDA call (fp16 latents need
 *     no scratch);
 *   - a split dense problem whose pieces, kv_split * B*Hq*Sq * (4*Dv + 4)
 *     bytes, exceed 32 MiB runs unsplit (same result, slower);
 *   - the first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture;
 *   - every call shares the one array, which keeps the last call's contents:
 *     calls whose work overlaps on the GPU (different streams without
 *     ordering between them) race on it.  Serialise them, e.g. on one stream.
 */
int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale,
                   int mask_mode, const int32_t* seqlens,
                   const fa_block_sparse_t* kv_block_idx, const fa_topk_t* topk_idx,
                   float rescale_threshold, void* stream);

/*
 * fa_convert_v_fp16 -- fp16 copy of a bf16 tensor (the V operand).
 *
 * The P.V product runs on fp16 operands (fp16 keeps three more mantissa bits
 * of the probabilities than bf16); fa_fwd converts a bf16 V itself (inside
 * the kernel; the top-k latent into scratch), or takes this copy with
 * FA_V_FP16.  v_bf16 and v_fp16 are device pointers, 16-byte
 * aligned, n_elems a positive multiple of 8.  bf16 -> fp16 is exact for
 * 2^-14 <= |v| <= 65504; larger magnitudes become inf and are reported as
 * FA_ERR_RANGE by fa_check_status.  Asynchronous on `stream`.
 */
int fa_convert_v_fp16(const void* v_bf16, void* v_fp16, int64_t n_elems, void* stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_RANGE (the first
 * error seen since the last call), or FA_ERR_CUDA if the synchronisation
 * itself failed. */
int fa_check_status(void* stream);

/* Sets the limit of every bounded on-chip wait (nanoseconds, default 2e9);
 * values <= 0 restore the default.  Affects launches made after the call. */
void fa_set_wait_timeout_ns(int64_t ns);

/* Most pieces a dense unit's KV tiles are split into when the problem has
 * too few units to fill half the GPU (default 8, the maximum; 1 never
 * splits).  Pieces have at least two KV tiles.  Returns FA_OK, or
 * FA_ERR_SHAPE for n outside [1, 8].  Affects calls made after it. */
int fa_set_max_kv_split(int n);

/* Failure-detection probe: one warp waits, with the same bounded wait as the
 * attention kernels, on an mbarrier that nothing ever arrives at, so that the
 * wait runs out after the limit set by fa_set_wait_timeout_ns, sets the
 * timeout bit of the status word and returns.  The next fa_check_status()
 * reports FA_ERR_DEVICE_TIMEOUT; the context stays usable.  Asynchronous on
 * `stream`; FA_OK once launched, FA_ERR_CUDA if the launch failed. */
int fa_wait_probe(void* stream);

/* Static string for a return code. */
const char* fa_strerror(int code);

/* The cudaError_t of the last FA_ERR_CUDA (0 if none), and its name. */
int fa_last_cuda_error(void);
const char* fa_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_FWD_H_ */
