/*
 * ffpa.h -- C ABI of libffpa: exact scaled-dot-product attention forward for
 * large head dimensions (D = 64..1024) on NVIDIA GB300 (sm_103a).
 *
 * The operation (FFPA API reference, "ffpa_attn.ffpa_attn_func", parameters
 * `query`, `key`, `value`, `attn_mask`, `is_causal`, `scale`, `enable_gqa`
 * and "Returns"; README, "Split-D and TiledMMA"):
 *
 *     O[b,h,i,:] = sum_k softmax_k( scale * Q[b,h,i,:].K[b,h/g,k,:] + M[b,h,i,k] ) V[b,h/g,k,:]
 *
 * with g = Hq / Hkv query heads per key/value head, M an optional boolean
 * (true keeps, false removes) or additive mask broadcast to [B,Hq,Nq,Nkv],
 * and, when causal, key k visible to query row i only if k <= i + (Nkv - Nq)
 * (queries aligned to the tail of the keys).  The optional LSE output is the
 * natural logarithm of sum_k exp(scale * q.k + M), in fp32 ("CUDA
 * convention", FFPA API reference, "ffpa_attn_varlen_func", `return_lse`).
 * A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Conventions shared by every entry point:
 *  - Pointers named q, k, v, o, lse, mask, cu_seqlens_* are DEVICE pointers:
 *    device (or managed) memory of one sm_103 GPU, all of them on the same
 *    GPU (else FFPA_ERR_INVALID; another arch is FFPA_ERR_UNSUPPORTED).
 *    `scale` is a HOST pointer.  The library never allocates, frees or synchronises on the
 *    caller's behalf (ffpa_last_device_error excepted); work is enqueued on
 *    `stream` and runs asynchronously.  The caller owns every buffer and
 *    must keep it alive until the stream has passed this work.
 *  - Strides are in ELEMENTS.  The last (D) stride must be 1.  For q, k and
 *    v every other stride times the element size must be a multiple of 16
 *    bytes and the base pointer 16-byte aligned (tensor-memory-accelerator
 *    loads); o must satisfy the same rules (16-byte vector stores).
 *  - Inputs are bf16 or fp16 (all three the same type); O has the input type.
 *    lse is 4-byte aligned; a mask is aligned to its element size.
 *  - Return codes: FFPA_OK, or the first failed check; nothing is enqueued
 *    when the result is not FFPA_OK.
 *
 * Per-call options: every entry point has an `_ex` form taking a
 * `const ffpa_options*` last (NULL = defaults; the plain form passes NULL).
 * The options carry the call's device status word, its wait time limit,
 * the kernel choice and a test hook; nothing the caller sets outlives the
 * call.
 *
 * Thread safety and shared state.  The entry points may be called
 * concurrently from several host threads on any streams.  What the library
 * shares between calls is exactly:
 *  - facts looked up once per device and never changed afterwards (compute
 *    capability, the address of the device's fallback status word) and the
 *    shared-memory limit raised once per kernel and device;
 *  - one FALLBACK STATUS WORD per device, written by the kernels of every
 *    call made without an options status word (ffpa_options.status = NULL)
 *    when one of their waits runs out.  ffpa_last_device_error(stream) reads
 *    and clears that word, so a timeout of such a call on one stream is
 *    reported to whichever caller next checks any stream of that device.
 *    Callers that need the failure of one call attributed to that call pass
 *    their own status word in the options.
 * A call leaves the calling thread's current CUDA device as it found it.
 */
#ifndef FFPA_H_
#define FFPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ffpa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  FFPA_OK = 0,
  FFPA_ERR_DTYPE = 1,          /* input dtype other than bf16/fp16 (API reference: TypeError) */
  FFPA_ERR_INVALID = 2,        /* bad shape, stride, pointer or option (API reference: ValueError) */
  FFPA_ERR_UNSUPPORTED = 3,    /* head dim or device not covered (API reference: NotImplementedError) */
  FFPA_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, attribute, device query) */
  FFPA_ERR_DEVICE_TIMEOUT = 5  /* a kernel pipeline wait exceeded its time limit (see below) */
} ffpa_status;

typedef enum { FFPA_BF16 = 0, FFPA_FP16 = 1 } ffpa_dtype;

typedef enum {
  FFPA_MASK_NONE = 0,
  FFPA_MASK_BOOL = 1,      /* uint8, nonzero = the element participates */
  FFPA_MASK_ADD_F32 = 2,   /* float32 additive bias (may hold -inf) */
  FFPA_MASK_ADD_QTYPE = 3  /* additive bias in the input dtype (bf16/fp16) */
} ffpa_mask_kind;

/* Kernel choice (ffpa_options.kernel).  The library has four forward
 * kernels with identical results:
 *   - single-CTA: one CTA per 128-row query tile and output slice of at most
 *     256 columns (any D; S is recomputed once per slice);
 *   - CTA pair: two SMs share each 256-query tile and each load half of every
 *     K/V tile (D in {128, 256, 512});
 *   - column split: a cluster of C SMs shares each 128-query tile, each SM
 *     owns an equal share of the output columns, key tiles are dealt
 *     round-robin and the P tiles are exchanged, so S is computed once (D a
 *     multiple of 64 from 128 to 1024; C = 2 up to D = 512, 3 up to 768, 4
 *     up to 1024; D is padded with zero columns to 2, 4, 6, 8, 12 or 16
 *     chunks of 64, which are read as zeros and not stored);
 *   - dual tile: one SM owns two 128-query tiles of a head, loads each K/V
 *     tile once for both and overlaps one tile's softmax with the other's
 *     products (dense batches, D in {64, 128}).
 *   FFPA_VARIANT_AUTO   (0) the fastest one measured for the shape (default:
 *                           column split for D > 256 (multiples of 64), CTA
 *                           pair for dense D = 256, dual tile for dense
 *                           D in {64, 128}, single-CTA otherwise)
 *   FFPA_VARIANT_SINGLE (1) always the single-CTA kernel
 *   FFPA_VARIANT_PAIR   (2) the CTA-pair kernel wherever D allows it
 *   FFPA_VARIANT_SPLIT  (3) the column-split kernel wherever D allows it
 *   FFPA_VARIANT_DUAL   (4) the dual-tile kernel wherever D and the layout allow it
 * Where the chosen kernel does not support D, the single-CTA kernel runs.
 * The backward has one kernel set and ignores the choice. */
enum {
  FFPA_VARIANT_AUTO = 0,
  FFPA_VARIANT_SINGLE = 1,
  FFPA_VARIANT_PAIR = 2,
  FFPA_VARIANT_SPLIT = 3,
  FFPA_VARIANT_DUAL = 4
};

/* Options of one call (all fields zero = the defaults). */
typedef struct ffpa_options {
  /* Device int (4-byte aligned, on the call's GPU) or NULL.  When a wait
   * inside this call's kernels runs past its limit, the kernel stores
   * FFPA_ERR_DEVICE_TIMEOUT there (drains its own copies, frees its tensor
   * memory and returns).  The library never clears it: the caller zeroes
   * it before the call and reads it after the stream has passed the call.
   * NULL selects the device's shared fallback word (ffpa_last_device_error). */
  int* status;
  /* Time limit of every in-kernel wait, in nanoseconds; 0 = 2e9 (2 s). */
  uint64_t wait_timeout_ns;
  /* FFPA_VARIANT_* (forward only); any other value is FFPA_ERR_INVALID. */
  int kernel;
  /* TEST HOOK, not for production use: nonzero makes this call's kernels
   * skip the first tensor copy of each CTA, so that the pipeline wait that
   * depends on it runs out and reports FFPA_ERR_DEVICE_TIMEOUT (no fault,
   * no hang). */
  int test_drop_first_copy;
} ffpa_options;

/*
 * Dense attention forward (FFPA API reference, "ffpa_attn.ffpa_attn_func").
 *
 *   q   [B, Hq,  Nq,  D]   strides q_str  = (b, h, n, d)
 *   k   [B, Hkv, Nkv, D]   strides k_str
 *   v   [B, Hkv, Nkv, D]   strides v_str
 *   o   [B, Hq,  Nq,  D]   strides o_str  (written)
 *   lse [B, Hq, Nq] fp32 contiguous, or NULL when not wanted (written)
 *   mask: NULL with FFPA_MASK_NONE, else broadcastable to [B, Hq, Nq, Nkv]
 *         with element strides mask_str (0 on a broadcast dimension).
 *   scale: NULL selects 1/sqrt(D) (API reference, `scale`).
 *   is_causal: tail-aligned causal masking; requires Nkv >= Nq.
 *   enable_gqa: must be nonzero when Hq != Hkv (API reference, `enable_gqa`).
 *
 * Checks, in order: dt (FFPA_ERR_DTYPE); sizes >= 0, Hq, Hkv >= 1
 * (INVALID); 64 <= D <= 1024 and D % 8 == 0 (UNSUPPORTED; a D that is not a
 * multiple of 64 is zero-padded to whole 64-column chunks and runs on the
 * single-CTA kernel; README "End-to-End Inference": head dims divisible by
 * 8, e.g. 120); Hq % Hkv,
 * enable_gqa, causal with Nkv < Nq, null pointers, strides, alignment, mask
 * kind, non-finite scale (INVALID); device is sm_103 (UNSUPPORTED).  An
 * empty problem (B, Hq or Nq zero) returns FFPA_OK without launching; Nkv
 * = 0 writes O = 0 and LSE = -inf.
 */
ffpa_status ffpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                     const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                     const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                     const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                     ffpa_stream_t stream);
ffpa_status ffpa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                        ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                        const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                        const int64_t mask_str[4], const float* scale, int is_causal,
                        int enable_gqa, ffpa_stream_t stream, const ffpa_options* options);

/*
 * Packed variable-length attention forward (FFPA API reference,
 * "ffpa_attn.ffpa_attn_varlen_func").
 *
 *   q [Tq, Hq, D], k and v [Tk, Hkv, D] with strides (t, h, d); o like q.
 *   cu_seqlens_q: int32 device array [nseq+1], cu[0] = 0, cu[nseq] = Tq,
 *   non-decreasing; sequence s owns rows cu[s] .. cu[s+1]-1.
 *   cu_seqlens_k: same for keys, or NULL to reuse cu_seqlens_q.
 *   max_seqlen_q / max_seqlen_k: upper bounds of the per-sequence lengths
 *   (a caller precondition: rows beyond max_seqlen_q are not computed).
 *   lse: [Hq, Tq] fp32 contiguous, or NULL.
 *   causal: lower-right (tail) alignment within each sequence.
 *
 * cu_seqlens live on the device and are not read by the host: a malformed
 * array is a caller precondition (the Python binding checks it on the host).
 * Other checks and error codes as for ffpa_fwd, except that D must be a
 * multiple of 64 (the varlen API takes head dims aligned to 64; else FFPA_ERR_UNSUPPORTED);
 * nseq < 1 or max_seqlen_* < 0 is FFPA_ERR_INVALID.
 */
ffpa_status ffpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                            const int64_t q_str[3], const int64_t k_str[3],
                            const int64_t v_str[3], const int64_t o_str[3],
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                            int enable_gqa, ffpa_stream_t stream);
ffpa_status ffpa_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, ffpa_stream_t stream, const ffpa_options* options);

/*
 * FP8 forward (FFPA README, "Backends" and "Latest News": FP8 attention
 * kernels for large head dims that take bf16/fp16 tensors and return the
 * input type, with the quantisation scales folded into the computation).
 * Same arguments, layouts and checks as ffpa_fwd, plus a caller workspace;
 * the result approximates ffpa_fwd's within the e4m3 error bound.
 *
 * Computation (the pages give no quantisation formula; this is the
 * library's reading): Q, K and V are quantised per (batch, head, block of
 * 128 rows) to e4m3 with scale s = amax / 448 (codes = e4m3(x * 448 / amax),
 * nearest-even, saturated; a zero block gets s = 1), written into the
 * workspace; the attention then runs on the e4m3 tensor cores with s_q s_k
 * folded into each score tile's scale and the V block scale folded into P,
 * which is itself rounded to e4m3.  LSE is that of the scores of the
 * dequantised Q and K.
 *
 *   D: 128..1024, a multiple of 128 (else FFPA_ERR_UNSUPPORTED).
 *   workspace: device memory on q's GPU, 256-byte aligned, at least
 *     ffpa_fwd_fp8_workspace_bytes(...) bytes (else FFPA_ERR_INVALID),
 *     owned by the caller and not read before it is written.  Layout, with
 *     Nqp, Nkp = Nq, Nkv rounded up to 128 and each part starting at the
 *     next multiple of 256 bytes: e4m3 Q [B,Hq,Nqp,D], e4m3 K [B,Hkv,Nkp,D],
 *     e4m3 V transposed [B,Hkv,D,Nkp], then fp32 scales of Q [B,Hq,Nqp/128],
 *     of K and of V [B,Hkv,Nkp/128].  Rows past N are zero.
 *   Inputs must be finite.  Two launches on `stream` (quantisation,
 *   attention); no allocation, no synchronisation.
 *   Kernels (ffpa_options.kernel of ffpa_fwd_fp8_ex): the column split (two
 *   SMs per 128-row tile, each owning D/2 output columns) by default at
 *   D = 384 and 512, and at D = 256 with FFPA_VARIANT_SPLIT; the single-CTA
 *   FP8 kernel otherwise or with FFPA_VARIANT_SINGLE.  Both compute the same
 *   quantised attention (the row maximum, and so the e4m3 rounding of P,
 *   may differ between them).
 */
size_t ffpa_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D);
ffpa_status ffpa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                         ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                         const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                         const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                         const int64_t mask_str[4], const float* scale, int is_causal,
                         int enable_gqa, void* workspace, size_t workspace_bytes,
                         ffpa_stream_t stream);
ffpa_status ffpa_fwd_fp8_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                            ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                            const int64_t q_str[4], const int64_t k_str[4],
                            const int64_t v_str[4], const int64_t o_str[4], const void* mask,
                            ffpa_mask_kind mask_kind, const int64_t mask_str[4],
                            const float* scale, int is_causal, int enable_gqa, void* workspace,
                            size_t workspace_bytes, ffpa_stream_t stream,
                            const ffpa_options* options);

/*
 * Backward of ffpa_fwd (dense layout): the gradients dq, dk, dv
 * of sum(O * dout) with respect to q, k and v (FFPA API reference,
 * "ffpa_attn.ffpa_attn_func": backward through FFPAAttnFunc; the Triton
 * backend's `split_launch` option: separate dKdV and dQ launches).  With
 * P = exp(scale * q k^T - lse) the forward's softmax:
 *   delta = rowsum(dout * o),  dv = P^T dout,  dS = P * (dout v^T - delta),
 *   dq = scale * dS k,  dk = scale * dS^T q,
 * summed over the query heads of a group for dk and dv.
 *
 *   q, o, dout, dq: [B, Hq, Nq, D] (strides q_str, o_str, do_str, dq_str).
 *   k, v, dk, dv: [B, Hkv, Nkv, D] (strides k_str, v_str, dk_str, dv_str).
 *   lse: [B, Hq, Nq] fp32 contiguous, the natural-log LSE that ffpa_fwd
 *     returned for the same q, k, v, scale and is_causal.
 *   delta: [B, Hq, Nq] fp32 contiguous OUTPUT (rowsum(dout * o), the
 *     FlashAttention "softmax_d"); written first and read by the gradient
 *     kernels, so it must not alias any input.
 *   o, dout, dq, dk, dv: the 16-bit type of q; outputs must not alias inputs.
 *   mask, mask_kind, mask_str, scale, is_causal, enable_gqa: as for ffpa_fwd
 *     (the same values as the forward that produced o and lse).  The mask
 *     enters the recomputed scores only: no gradient is formed for it.
 *
 * Strides follow the ffpa_fwd rules (last stride 1, others multiples of 16
 * bytes, 16-byte aligned bases) for every tensor.  Errors as for ffpa_fwd,
 * except that D must be a multiple of 64 (else FFPA_ERR_UNSUPPORTED); a NULL
 * lse or delta is FFPA_ERR_INVALID.  B == 0 writes nothing; Nq == 0 with
 * Nkv > 0 writes zero dk and dv; Nkv == 0 writes zero dq.  Three (D <= 128) or
 * four launches on `stream`; no allocation, no synchronisation.
 */
ffpa_status ffpa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, float* delta, ffpa_dtype dt,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int D, const int64_t q_str[4],
                     const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4],
                     const int64_t do_str[4], const int64_t dq_str[4], const int64_t dk_str[4],
                     const int64_t dv_str[4], const void* mask, ffpa_mask_kind mask_kind,
                     const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                     ffpa_stream_t stream);
ffpa_status ffpa_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        float* delta, ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                        const int64_t o_str[4], const int64_t do_str[4], const int64_t dq_str[4],
                        const int64_t dk_str[4], const int64_t dv_str[4], const void* mask,
                        ffpa_mask_kind mask_kind, const int64_t mask_str[4], const float* scale,
                        int is_causal, int enable_gqa, ffpa_stream_t stream,
                        const ffpa_options* options);

/*
 * ffpa_bwd with a caller-owned workspace for the stored-tile backward: the
 * same arguments, checks and results, plus
 *
 *   workspace, workspace_bytes: device memory of q's device, 16-byte
 *     aligned, owned by the caller, of at least
 *     ffpa_bwd_workspace_bytes(B, Hq, Hkv, Nq, Nkv, D, is_causal) bytes; its
 *     contents on entry do not matter and on return are unspecified.
 *
 * When ffpa_bwd_workspace_bytes() is non-zero (dense layout, D = 128, 256,
 * 384 or 512, Nq > 0, Nkv > 0) and the workspace is large enough, each
 * (128-query, 128-key) tile's softmax P and dS (times scale) are formed
 * once, as 16-bit values, into the workspace, and dq, dv, dk are
 * contractions over the stored tiles: no product of the definition is
 * computed twice (the ffpa_bwd kernels recompute S and dP for every
 * 256-column output slice).  Workspace layout: a 32 KB block of zeros, then
 * P, then dS, each one 32 KB block per (b, hq, query tile, key tile) in that
 * order, where with is_causal only the key tiles that some row of the query
 * tile sees are stored (about half the blocks when Nq = Nkv); inside a block
 * the 8 keys 8u .. 8u+7 of tile row r are the 16 bytes at 2048 u + 16 r.  Three launches on `stream` (delta,
 * scores, contraction).  Otherwise (workspace NULL or too small, or a shape
 * the path does not take) this is ffpa_bwd and the workspace is not
 * touched.  A workspace on another device, or not 16-byte aligned when it
 * would be used, is FFPA_ERR_INVALID.  No allocation, no synchronisation.
 */
size_t ffpa_bwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int is_causal);
ffpa_status ffpa_bwd_ws(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, float* delta, ffpa_dtype dt,
                        int B, int Hq, int Hkv, int Nq, int Nkv, int D, const int64_t q_str[4],
                        const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4],
                        const int64_t do_str[4], const int64_t dq_str[4], const int64_t dk_str[4],
                        const int64_t dv_str[4], const void* mask, ffpa_mask_kind mask_kind,
                        const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                        void* workspace, size_t workspace_bytes, ffpa_stream_t stream);
ffpa_status ffpa_bwd_ws_ex(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           float* delta, ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                           const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                           const int64_t o_str[4], const int64_t do_str[4], const int64_t dq_str[4],
                           const int64_t dk_str[4], const int64_t dv_str[4], const void* mask,
                           ffpa_mask_kind mask_kind, const int64_t mask_str[4], const float* scale,
                           int is_causal, int enable_gqa, void* workspace, size_t workspace_bytes,
                           ffpa_stream_t stream, const ffpa_options* options);

/*
 * Backward of ffpa_fwd_varlen (packed THD layout; FFPA API reference,
 * "ffpa_attn.ffpa_attn_varlen_func"): dq, dk, dv of sum(O * dout), each
 * sequence differentiated as its own dense problem (causal: lower right).
 *
 *   q, o, dout, dq: [Tq, Hq, D]; k, v, dk, dv: [Tk, Hkv, D] (strides over
 *     T, H, D).
 *   lse: [Hq, Tq] fp32 contiguous, the forward's; delta: [Hq, Tq] fp32
 *     contiguous OUTPUT (rowsum(dout * o)).
 *   cu_seqlens_q / cu_seqlens_k / nseq / max_seqlen_*: as for
 *     ffpa_fwd_varlen (device arrays, caller precondition).
 *
 * Checks and error codes as for ffpa_fwd_varlen, plus a NULL lse or delta
 * (FFPA_ERR_INVALID).  Three (D <= 128) or four launches on `stream`; no allocation, no
 * synchronisation.
 */
ffpa_status ffpa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                            const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                            const int64_t o_str[3], const int64_t do_str[3], const int64_t dq_str[3],
                            const int64_t dk_str[3], const int64_t dv_str[3],
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                            int enable_gqa, ffpa_stream_t stream);
ffpa_status ffpa_bwd_varlen_ex(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int64_t do_str[3], const int64_t dq_str[3],
                               const int64_t dk_str[3], const int64_t dv_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, ffpa_stream_t stream, const ffpa_options* options);

/*
 * ffpa_bwd_varlen with a caller-owned workspace for the stored-tile backward
 * (as ffpa_bwd_ws for the dense layout): the same arguments, checks and
 * results, plus
 *
 *   workspace, workspace_bytes: device memory of q's device, 16-byte
 *     aligned, owned by the caller.  The stored-tile path runs when D is
 *     128, 256, 384 or 512, Tq, Tk > 0, and workspace_bytes is at least
 *     ffpa_bwd_varlen_workspace_bytes() of the same sequences (computed on
 *     the host from host copies of cu_seqlens_q / cu_seqlens_k, which the
 *     library cannot read there); a smaller workspace that still holds the
 *     1 KB-rounded header of nseq + 1 int64 and three 32 KB blocks also takes
 *     the path, and a block the sequences need past its end is neither
 *     written nor read: the call's status word then records
 *     FFPA_ERR_INVALID and the gradients are wrong.  Otherwise this is
 *     ffpa_bwd_varlen and the workspace is not touched.
 *
 * Layout: the first stored block of every sequence (nseq + 1 int64, written
 * by the call), a 32 KB block of zeros, then P and dS blocks as for
 * ffpa_bwd_ws, per sequence, query head, query tile and stored key tile
 * (causal: lower right within each sequence).  Four launches on `stream`
 * (delta, block bases, scores, contraction); no allocation, no
 * synchronisation.
 */
size_t ffpa_bwd_varlen_workspace_bytes(const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_k_host,
                                       int nseq, int Hq, int Hkv, int D, int is_causal);
ffpa_status ffpa_bwd_varlen_ws(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int64_t do_str[3], const int64_t dq_str[3],
                               const int64_t dk_str[3], const int64_t dv_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, void* workspace, size_t workspace_bytes,
                               ffpa_stream_t stream);
ffpa_status ffpa_bwd_varlen_ws_ex(const void* q, const void* k, const void* v, const void* o,
                                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                  float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                                  const int64_t q_str[3], const int64_t k_str[3],
                                  const int64_t v_str[3], const int64_t o_str[3],
                                  const int64_t do_str[3], const int64_t dq_str[3],
                                  const int64_t dk_str[3], const int64_t dv_str[3],
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                                  int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                                  int enable_gqa, void* workspace, size_t workspace_bytes,
                                  ffpa_stream_t stream, const ffpa_options* options);

/*
 * Backward for callers that cannot allocate device memory.  The pages have
 * no counterpart: this entry point exists for callers such as plugins that
 * receive only their tensors' pointers from a host framework, runtimes that
 * reserve all device memory up front, and latency-bound paths where a
 * cudaMalloc (which may synchronise the device, or fail once memory is
 * exhausted) is not acceptable.
 *
 * Same arguments, checks and results as ffpa_bwd without `delta`: the
 * per-row values rowsum(dout * o) that the backward keeps between its first
 * kernel and the gradient kernels live in a fixed array inside the library
 * (FFPA_BWD_NOALLOC_MAX_ROWS fp32 values, 4 MiB, held by every GPU that
 * loads the library until the process exits).  The caller still passes
 * every input and the dq, dk, dv outputs; nothing is allocated or freed.
 *  - B * Hq * Nq above FFPA_BWD_NOALLOC_MAX_ROWS: FFPA_ERR_INVALID, nothing
 *    is enqueued (use ffpa_bwd with a caller-owned delta instead).
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    values; nothing in it needs to start at zero (each call writes every
 *    entry it reads).  Calls whose work overlaps on the GPU (on different
 *    streams, or from different threads) race on it: serialise them.
 */
#define FFPA_BWD_NOALLOC_MAX_ROWS 1048576
ffpa_status ffpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                             const int64_t q_str[4], const int64_t k_str[4],
                             const int64_t v_str[4], const int64_t o_str[4],
                             const int64_t do_str[4], const int64_t dq_str[4],
                             const int64_t dk_str[4], const int64_t dv_str[4], const void* mask,
                             ffpa_mask_kind mask_kind, const int64_t mask_str[4],
                             const float* scale, int is_causal, int enable_gqa,
                             ffpa_stream_t stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* ffpa_status_string(ffpa_status status);

/*
 * Checked mode for calls made without an options status word: synchronises
 * `stream`, then reads and clears the FALLBACK status word of the stream's
 * device (see "Thread safety and shared state" above: the word is shared
 * by every such call on that device, on every stream).  Returns FFPA_OK,
 * FFPA_ERR_DEVICE_TIMEOUT, or FFPA_ERR_CUDA if the synchronisation or the
 * read failed.
 */
ffpa_status ffpa_last_device_error(ffpa_stream_t stream);

/*
 * The forward kernel (FFPA_VARIANT_SINGLE, _PAIR, _SPLIT or _DUAL) that a call
 * with ffpa_options.kernel = `kernel` would run for head dimension D on a
 * dense (varlen = 0) or packed varlen (varlen != 0) batch.  Host only;
 * returns -1 for a head dimension or kernel value the library does not take.
 */
int ffpa_selected_kernel(int D, int varlen, int kernel);

#ifdef __cplusplus
}
#endif

#endif /* FFPA_H_ */
