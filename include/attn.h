/*
 * attn.h - C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The library computes exact attention
 *     O = softmax(scale * Q K^T [+ causal mask]) V,   LSE = ln sum exp(scale * Q K^T)
 * with a tiled, streaming softmax on tcgen05 tensor cores, never writing the
 * score matrix to HBM.  Sources of the definition:
 *   - "FlashAttention（V3）深度解析" (dtcms.com), section 2: S = Q K^T,
 *     P = softmax(S), O = P V; section 11 standard_attention: the scores are
 *     scaled by 1/sqrt(d) (here: the caller's `scale`); section 11
 *     _apply_causal_mask: key j is visible to query i iff i >= j, indices
 *     from 0 (top-left alignment, also when Nq != Nk); section 4.2: the
 *     streaming max/denominator merge rule used to process key blocks one
 *     at a time.
 *   - LSE is not defined on the pages; it is the natural-log log-sum-exp of
 *     the scaled, masked logits of each query row.
 *   - FP8: section 4.3 of the same page (per-block scale, dequantisation
 *     fused into the pipeline) and the Together AI summary card
 *     "FlashAttention-3——利用异步与低精度加速注意力机制" (Hadamard transform
 *     with random signs applied per head before FP8 quantisation).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout   Q, O: [B, Nq, Hq, d]; K, V: [B, Nk, Hkv, d] ("BSHD": contiguous,
 *          d innermost), as in the pages' V layout [seqlen, heads, dim]
 *          (section 7.4, TransposeVLayout).  LSE: [B, Hq, Nq] float32.
 * GQA      query head h reads key/value head h / (Hq / Hkv); Hq % Hkv == 0.
 * Pointers are DEVICE pointers owned by the caller; the library never frees
 *          or keeps them.  q, k, v, o (and the FP8 tensors) must be 128-byte
 *          aligned (the TMA alignment pitfall on the gsyq.cn page, section 四);
 *          lse and the descale arrays 16-byte aligned.
 * Streams  `stream` is a cudaStream_t (NULL = legacy default stream).  Calls
 *          enqueue work and return without synchronising; results are valid
 *          once the stream has reached that point.
 * Memory   The library allocates nothing per call.  A status word and the
 *          device properties are set up once per device on first use and
 *          kept until the process exits.
 * Errors   0 on success.  On a negative return nothing was launched (except
 *          ATTN_ERR_CUDA, which reports a failed launch).  Argument errors
 *          are detected on the host before any CUDA call.
 * Empty    B == 0 or Nq == 0 is a valid empty problem: returns 0, launches
 *          nothing.
 * Threads  Entry points may be called from several host threads; the first
 *          call on a device performs the one-time set-up.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of Q/K/V/O for attn_fwd */
#define ATTN_F16 0  /* IEEE binary16 */
#define ATTN_BF16 1 /* bfloat16 */

/* return codes */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG (-1) /* null pointer, negative size, Hq % Hkv != 0,
                                     Nk == 0 with Nq > 0, scale not finite and > 0,
                                     flag not 0/1, size over 2^31-1 rows */
#define ATTN_ERR_UNSUPPORTED (-2) /* head dim or dtype the kernels do not cover,
                                     or no sm_103-class device */
#define ATTN_ERR_MISALIGNED (-3)  /* a pointer violates the alignment rule above */
#define ATTN_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed; see attn_strerror */
#define ATTN_ERR_TIMEOUT (-5)     /* a kernel reported a bounded wait that expired */
#define ATTN_ERR_DEVICE (-6)      /* a kernel reported an internal consistency error */
#define ATTN_ERR_SCRATCH (-7)     /* attn_fwd_splitkv_noalloc: the problem needs more
                                     scratch than its fixed array holds */

/*
 * attn_fwd - fused attention forward, FP16 or BF16.
 *
 *   q     [B, Nq, Hq, d]   dtype      (read)
 *   k, v  [B, Nk, Hkv, d]  dtype      (read)
 *   o     [B, Nq, Hq, d]   dtype      (written: softmax(scale Q K^T [mask]) V,
 *                                      rounded to nearest-even)
 *   lse   [B, Hq, Nq]      float32    (written: natural-log log-sum-exp of the
 *                                      scaled, masked logits of each row)
 *   d     64, 128 or 256
 *   causal 0 or 1 (top-left aligned: key j visible to query i iff j <= i)
 *   scale  > 0 and finite (the workloads use 1/sqrt(d))
 *   dtype  ATTN_F16 or ATTN_BF16
 * Arithmetic: products accumulate in FP32 (tensor memory); the softmax state
 * (row max, row sum) is FP32; the probabilities are rounded to dtype before
 * the P V product.  Non-causal calls whose query rows of a GQA group fit two
 * 128-row tiles (one for d = 256) run with that group's heads packed into
 * the tiles' rows (same results, one K/V stream per group).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int64_t Nq, int64_t Nk, int d, int causal, float scale, int dtype,
             void* stream);

/*
 * attn_prep_fp8 - per-block FP8 E4M3 quantisation with optional incoherent
 * processing (Hadamard transform with random signs), one tensor per call.
 *
 *   x        [B, N, H, d] bfloat16 (read)
 *   x8       written E4M3FN codes:
 *              transpose_out == 0: [B, N, H, d]          (BSHD, like x)
 *              transpose_out == 1: [B, H, d, Npad], Npad = N rounded up to a
 *                                  multiple of 16; positions n >= N are zero.
 *                                  This is the key-contiguous V layout the
 *                                  FP8 P V product reads (the pages' V
 *                                  transpose, section 7.4).
 *   descale  [B, H, ceil(N/128)] float32 (written): one scale per block of
 *            128 tokens x d of one (b, head); descale = amax / 448 rounded
 *            to float32, or 1 for an all-zero block.
 *            code = E4M3 of y / descale, round-to-nearest-even, saturated to
 *            +-448.  Without the transform (y = x) the code is that of the
 *            exact quotient, ties included.  With the transform, y is formed
 *            in float32 and scaled by r = 448 / amax (float32, once per
 *            block) times 1 / sqrt(d): a code may then differ by one step
 *            where y / descale lies within float32 rounding of a midpoint.
 *   signs    NULL (no transform) or [sign_heads, d] int8 of +1/-1 (device,
 *            8-byte aligned).
 *            With signs, every row is replaced, before quantisation, by
 *            y = (x * sigma) H_d / sqrt(d) in float32, H_d the Sylvester
 *            Hadamard matrix and sigma the row of head h / (H / sign_heads).
 *            Apply it to Q and K with the same signs per key/value head
 *            (Q's sign_heads = Hkv); never to V.
 *   d        64, 128 or 256
 * Every prep entry point (this one, attn_prep_fp8_per_tensor,
 * attn_prep_fp8_rope, attn_prep_fp8_qkv) hands its launch's tiles out
 * through one of 64 device counters that the library takes in turn and each
 * launch leaves at zero: at most 64 prep launches may run at the same time
 * (on different streams). A launch holds fewer than 2^31 tiles of 128 tokens
 * (B x ceil(N/128) x H summed over its tensors); larger ones return
 * ATTN_ERR_UNSUPPORTED.
 */
int attn_prep_fp8(const void* x, void* x8, float* descale, int B, int H, int64_t N, int d,
                  const int8_t* signs, int sign_heads, int transpose_out, void* stream);

/*
 * attn_prep_fp8_per_tensor - the baseline FP8 scheme: one scale for the
 * whole tensor instead of one per block, optional Hadamard transform.
 *
 * The summary card (FlashAttention-3 summary, low-precision section) says
 * incoherent processing makes the FP8 error 2.6 times lower than "baseline
 * FP8" without defining it; this is the reading taken for that baseline.
 *
 *   x, x8, signs, sign_heads, transpose_out, d: as attn_prep_fp8.
 *   descale  [B, H, ceil(N/128)] float32 (written): every entry equals
 *            amax / 448 with amax over the whole tensor after the transform
 *            (1 for an all-zero tensor), so attn_fwd_fp8 consumes it
 *            unchanged.  Codes as attn_prep_fp8 with that one descale.
 *            descale[0] serves as the amax
 *            accumulator while the call runs (three kernels and a 4-byte
 *            memset on `stream`).
 *   Returns as attn_prep_fp8.
 */
int attn_prep_fp8_per_tensor(const void* x, void* x8, float* descale, int B, int H, int64_t N,
                             int d, const int8_t* signs, int sign_heads, int transpose_out,
                             void* stream);

/*
 * attn_rope_table - cos and sin tables of the rotary embedding, for
 * attn_prep_fp8_rope.
 *
 * The pages name no rotary variant; the one taken is the rotate-half form:
 * channel c < d/2 pairs with c + d/2 and both turn by the angle
 * (pos0 + n) * base^(-2c/d) at token n.
 *
 *   rope_cos, rope_sin  [N, d/2] float32 (device, written, caller-owned):
 *            cos and sin of the angle, evaluated in double precision and
 *            rounded once to float32.
 *   N        positions (0 returns ATTN_OK with nothing written)
 *   d        even, 2..256
 *   base     > 1 (10000 in most models)
 *   pos0     position of the first row, 0..2^40
 *   Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_MISALIGNED (tables not
 *   4-byte aligned) or ATTN_ERR_CUDA.
 */
int attn_rope_table(float* rope_cos, float* rope_sin, int64_t N, int d, double base,
                    int64_t pos0, void* stream);

/*
 * attn_prep_fp8_rope - rotary embedding, optional Hadamard transform and
 * per-block FP8 quantisation in one pass over a Q or K tensor.
 *
 * The summary card (FlashAttention-3 summary, low-precision section) notes
 * that the Hadamard transform can be fused with the rotary embedding, a
 * bandwidth-bound step, at no extra cost.  Each row is rotated (rotate-half
 * form, see attn_rope_table) in float32, then transformed as in
 * attn_prep_fp8 (when signs is not NULL), then quantised per block.  The
 * rotation is applied before the transform so that the scores are those of
 * the rotated Q and K.
 *
 *   x        [B, N, H, d] bfloat16 (read)
 *   x8       [B, N, H, d] E4M3 codes (written; BSHD only - V takes no rotation)
 *   descale  [B, H, ceil(N/128)] float32 (written), as attn_prep_fp8
 *   rope_cos, rope_sin  [N, d/2] float32 (read; attn_rope_table), row n
 *            for token n of every batch; 16-byte aligned
 *   signs, sign_heads, d: as attn_prep_fp8
 *   Returns as attn_prep_fp8; ATTN_ERR_INVALID_ARG for a NULL table.
 */
int attn_prep_fp8_rope(const void* x, void* x8, float* descale, int B, int H, int64_t N, int d,
                       const float* rope_cos, const float* rope_sin, const int8_t* signs,
                       int sign_heads, void* stream);

/*
 * attn_prep_fp8_qkv - the FP8 preparation of one attention call in one
 * launch: Q and K as attn_prep_fp8 (per-block codes, BSHD) or, with rotary
 * tables, as attn_prep_fp8_rope; V as attn_prep_fp8 with transpose_out = 1.
 * The results are those of the three separate calls, bit for bit; one
 * launch pays the ramp-up and tail of a persistent kernel once instead of
 * three times.  This entry point is an addition of this library, not a step
 * of the pages' method.
 *
 *   q [B, Nq, Hq, d], k, v [B, Nk, Hkv, d]  bfloat16 (read)
 *   q8 [B, Nq, Hq, d], k8 [B, Nk, Hkv, d]   E4M3 codes (written)
 *   v8t [B, Hkv, d, Nkpad]                   E4M3 codes, Nkpad = Nk rounded up to 16
 *   q_descale [B, Hq, ceil(Nq/128)], k_descale, v_descale [B, Hkv, ceil(Nk/128)]
 *   signs     NULL or [Hkv, d] int8 +1/-1 (8-byte aligned): Q and K take the
 *             transform, query head h using row h / (Hq / Hkv)
 *   rope_cos, rope_sin  both NULL or both [max(Nq, Nk), d/2] float32
 *             (attn_rope_table, 16-byte aligned): Q and K are rotated first
 *   d         64, 128 or 256
 * Returns as attn_prep_fp8.
 */
int attn_prep_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8t,
                      float* q_descale, float* k_descale, float* v_descale, int B, int Hq,
                      int Hkv, int64_t Nq, int64_t Nk, int d, const int8_t* signs,
                      const float* rope_cos, const float* rope_sin, void* stream);

/*
 * attn_fwd_fp8 - fused attention forward on FP8 E4M3 inputs.
 *
 *   q8        [B, Nq, Hq, d]     E4M3 codes       q_descale [B, Hq, ceil(Nq/128)]
 *   k8        [B, Nk, Hkv, d]    E4M3 codes       k_descale [B, Hkv, ceil(Nk/128)]
 *   v8t       [B, Hkv, d, Nkpad] E4M3 codes, Nkpad = Nk rounded up to 16, padding
 *             zero (attn_prep_fp8 with transpose_out = 1)
 *                                                 v_descale [B, Hkv, ceil(Nk/128)]
 *   o         [B, Nq, Hq, d] bfloat16 (written)   lse [B, Hq, Nq] float32 (written)
 *   d         64, 128 or 256
 *   hadamard  0 or 1: states whether Q and K went through the transform; the
 *             arithmetic does not change (Q M (K M)^T = Q K^T), the flag is
 *             validated and kept for the caller's bookkeeping.
 * Dequantisation is fused: logits use q_descale * k_descale per 128 x 128
 * tile; the probabilities are quantised to E4M3 for the P V product with the
 * value block's scale folded in; sums and the output stay FP32 until the
 * final bfloat16 rounding.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_descale,
                 const float* k_descale, const float* v_descale, void* o, float* lse, int B,
                 int Hq, int Hkv, int64_t Nq, int64_t Nk, int d, int causal, float scale,
                 int hadamard, void* stream);

/*
 * attn_fwd_splitkv - attn_fwd for long key sequences and few query rows
 * (decode-like shapes), non-causal, FP16/BF16.  The key range of every query
 * block is cut into `num_splits` consecutive ranges processed by different
 * CTAs; each leaves its O / l and LSE in FP32 in `workspace`, and a second
 * kernel combines them with the streaming-softmax merge rule of
 * "FlashAttention（V3）深度解析" section 4.2 (m = max(m_a, m_b),
 * z = z_a e^(m_a - m) + z_b e^(m_b - m)).  When Hq / Hkv divides 128, the
 * query heads of a GQA group share the rows of one query tile, so each
 * key/value head is read once per split.  Same tensors, layouts and results
 * as attn_fwd with causal = 0 (up to FP32 rounding of the merge).
 *   num_splits  >= 1; more splits than 128-key tiles are reduced to one per
 *               tile; with an effective count of 1 the kernel writes O and
 *               LSE itself (GQA group still packed when Nq x Hq/Hkv fits two
 *               query tiles, 128 rows for d = 256)
 *   workspace   device buffer, 256-byte aligned, owned by the caller, at least
 *               attn_splitkv_workspace_bytes(B, Hq, Nq, d, num_splits) bytes;
 *               unused (may be NULL) when the effective count is 1.  Its
 *               contents are scratch: overwritten by every call.
 * Errors as attn_fwd; ATTN_ERR_INVALID_ARG also for num_splits < 1 or a
 * workspace that is missing or too small.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int64_t Nq, int64_t Nk, int d, int num_splits, float scale,
                     int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* attn_splitkv_workspace_bytes - workspace attn_fwd_splitkv needs for these
 * sizes (num_splits x B x Hq x Nq rows of d + 1 floats, plus alignment);
 * 0 for invalid sizes.  No CUDA call. */
size_t attn_splitkv_workspace_bytes(int B, int Hq, int64_t Nq, int d, int num_splits);

/* attn_splitkv_default_splits - a split count that gives one wave of CTAs on
 * the current device for these sizes (at least 1, at most one per key tile,
 * at most 256).  Performs the one-time device set-up if needed. */
int attn_splitkv_default_splits(int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d);

/*
 * attn_fwd_splitkv_noalloc - attn_fwd_splitkv for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * interface for a kind of caller, not part of the method.
 *
 * Who needs it: programs whose device memory is owned by their own pool or
 * arena (a library allocation would compete with it, or fail once the pool
 * holds the device), and services that forbid allocation on the request path
 * (an allocation can block, synchronise the device or fail under memory
 * pressure, breaking their latency and memory bounds).  attn_fwd_splitkv
 * needs a workspace and the other entry points allocate a status word on
 * their first call on a device; this one allocates nothing.  Its per-split partial results and its
 * status word live in a fixed device array of 16 MiB that is part of the
 * library (every GPU that loads the library holds it until the process
 * exits).  The caller passes inputs and outputs exactly as for
 * attn_fwd_splitkv, without a workspace.
 *
 * Limit: num_splits x B x Hq x Nq x (d + 1) x 4 bytes, the first part padded to
 * 256 bytes, must fit in 16 MiB - 256 bytes (e.g. 256 splits of one query per
 * head at Hq = 64, d = 128); otherwise ATTN_ERR_SCRATCH and nothing runs.
 * With an effective split count of 1 (Nk <= 128 keys, or num_splits = 1) the
 * scratch is not used.
 * Set-up: the first call on a device reads device attributes, resolves the
 * tensor-map encoder, looks up the array's device address
 * (cudaGetSymbolAddress) and zeroes the status word with a synchronous
 * cudaMemset; make that first call before any stream capture.
 * Sharing: every call on a device uses the same array and it keeps the last
 * call's contents; calls whose kernels overlap on the GPU (for example on two
 * streams) race on it.  A bounded-wait timeout inside its kernels is recorded
 * in the array's status word; attn_get_status reads and clears it (and
 * allocates nothing).
 * Errors as attn_fwd_splitkv, plus ATTN_ERR_SCRATCH.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d, int num_splits,
                             float scale, int dtype, void* stream);

/*
 * attn_get_status - synchronise `stream`, then read and clear the status
 * words of the current device that kernels set when a bounded wait expires
 * (ATTN_ERR_TIMEOUT) or an internal check fails (ATTN_ERR_DEVICE): the word
 * of the allocating entry points and the one inside the fixed array of
 * attn_fwd_splitkv_noalloc (each only if set up on this device).  Allocates
 * nothing.  Returns 0 if no kernel reported a problem since the last call,
 * ATTN_ERR_CUDA if the synchronisation or a copy failed.
 */
int attn_get_status(void* stream);

/* attn_strerror - static text for a return code; for ATTN_ERR_CUDA the text
 * of the last CUDA failure seen by this thread. */
const char* attn_strerror(int code);

/* attn_launch_count - number of kernels this library has launched in the
 * process so far (monotonic; used to count launches in a timed region). */
int64_t attn_launch_count(void);

/*
 * attn_selftest_bounded_wait - exercises the failure path of the kernels'
 * waits: launches one warp on `stream` that waits, with the same bounded wait
 * every kernel of the library uses, on an mbarrier that nothing arrives on.
 * The wait gives up after its budget (about 2 s of GPU clock), sets the
 * timeout bit of the device status word and the kernel returns; the next
 * attn_get_status reports ATTN_ERR_TIMEOUT and clears the word.  No fault,
 * trap or hang is involved and the context stays usable.  For tests.
 *   Returns ATTN_OK once launched, ATTN_ERR_CUDA if the launch failed.
 */
int attn_selftest_bounded_wait(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
