/*
 * gbattn.h -- C ABI of libgbattn.so: exact tiled attention on GB300 (sm_103a).
 *
 * The library computes exact attention (no approximation):
 *
 *     O = softmax(scale * Q K^T + mask) V,      LSE = log sum_j exp(scale * q.k_j)
 *
 * as defined in M4.3 "IO-Aware Attention and FlashAttention-1" 0x02A (scores, mask before the row
 * normalisation, P V) and 0x09E (LSE = m + log l), with the grouped-query
 * head map of M4.4 "FlashAttention-2 Work Partitioning and the Decode Boundary" 0x06A
 * (kv_head = q_head / (H / Hkv)) and the causal predicate of M4.4 0x05.1A
 * (key k visible to query q iff k <= q + (Sk - Sq), the bottom-right
 * alignment of 0x05.1F).  The forward pass is a tiled online-softmax
 * reduction over the key axis (M4.3 0x07-0x09; M4.4 0x03 Algorithm 1): the
 * per-row (m, l, unnormalised O) state stays on chip and the [Sq, Sk] score
 * and probability matrices never reach device memory.  Decode (one query per
 * sequence) splits the key axis into chunks whose partial states are merged
 * by rescale-and-add (M4.4 0x01 work-axis ledger, Flash-Decoding; M4.3 0x08B
 * merge; M4.3 0x09E (LSE, O) form).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory in any call, never frees caller memory, never
 *    modifies inputs and never synchronises the stream: work is enqueued on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and the call
 *    returns immediately.
 *  - Layout: every tensor is contiguous row-major [batch, heads, seq, d]
 *    ("BHSD"); LSE is contiguous fp32 [batch, heads, seq].
 *  - Pointers must be 16-byte aligned.  Element type of q/k/v/o is given by
 *    `dtype` (GBATTN_F16 or GBATTN_BF16); arithmetic is fp32 with fp16/bf16
 *    tensor-core operands; O is rounded to `dtype` (round-to-nearest-even).
 *  - LSE is the natural-log sum of exp(scale * score) over the visible keys.
 *    A query row with no visible key (only possible when causal and Sq > Sk)
 *    gets O = 0 and LSE = -inf.
 *  - Return value: GBATTN_OK or a negative GBATTN_E* code.  Argument errors
 *    are detected on the host before anything is enqueued.  Asynchronous
 *    device-side failures (a bounded wait inside a kernel that timed out, or
 *    a dynamic shared-memory base without the 1024-byte alignment a kernel
 *    relies on, in which case that kernel writes nothing) are reported by
 *    gbattn_device_status() after the caller synchronises.
 */
#ifndef GBATTN_H_
#define GBATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GBATTN_OK 0
#define GBATTN_EBADSHAPE (-1)       /* B, H, Hkv, Sq, Sk (or Sk_max) < 1, or a size overflows */
#define GBATTN_EHEADS (-2)          /* H % Hkv != 0 (M4.4 0x06A admissibility) */
#define GBATTN_EHEADDIM (-3)        /* d not in {64, 128} */
#define GBATTN_EDTYPE (-4)          /* dtype is neither GBATTN_F16 nor GBATTN_BF16 */
#define GBATTN_EPOINTER (-5)        /* a required pointer is NULL or not 16-byte aligned */
#define GBATTN_EWORKSPACE (-6)      /* workspace smaller than the matching *_workspace_bytes() */
#define GBATTN_ELAUNCH (-7)         /* the CUDA runtime rejected a launch or a tensor map */
#define GBATTN_EDEVICE_TIMEOUT (-8) /* a kernel gave up on device: a bounded wait timed out, or its
                                       shared-memory base was not 1024-byte aligned (gbattn_device_status) */
#define GBATTN_ESPLIT (-9)          /* decode n_split < 1 or > 256 */
#define GBATTN_EUNSUPPORTED (-10)   /* no sm_103a device, or the current device is not sm_103 */

/* Element types of q/k/v/o. */
#define GBATTN_F16 0
#define GBATTN_BF16 1

/*
 * attn_fwd -- exact attention forward (prefill), tiled online softmax.
 *
 *   q     [B, H,   Sq, d]  dtype, input
 *   k, v  [B, Hkv, Sk, d]  dtype, input (query head h reads KV head h / (H / Hkv))
 *   o     [B, H,   Sq, d]  dtype, output
 *   lse   [B, H,   Sq]     fp32, output; may be NULL (then not written)
 *   scale multiplies the fp32 dot product before masking (usually 1/sqrt(d))
 *   causal 0: every key visible; 1: key j visible to query i iff
 *          j <= i + (Sk - Sq)
 *
 * Passages: M4.3 0x02A (definition), M4.3 0x09C-0x09E (unnormalised state,
 * divide once, LSE), M4.4 0x03 Algorithm 1 (query-tile owner streams every
 * visible key tile), M4.4 0x05.1B/0x05.1D (whole-future tiles skipped before
 * Q K^T, partial tiles masked before the row maximum), M4.6 "FlashAttention-3/4
 * Hardware Pipelines" 0x08-0x09 (two query tiles per CTA, TMEM score and
 * output slots, conditional rescaling with threshold 8 in base-2 units).
 *
 * Errors: GBATTN_EBADSHAPE, EHEADS, EHEADDIM, EDTYPE, EPOINTER (q, k, v, o
 * must be non-NULL; lse may be NULL), EUNSUPPORTED, ELAUNCH.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int Hkv, int Sq, int Sk, int d, float scale, int causal,
             int dtype, void *stream);

/*
 * attn_fwd_pair -- the non-causal attn_fwd with d = 128, computed by pairs of
 * CTAs that act as one tcgen05 CTA pair (cta_group::2): each pair owns four
 * 128-row query tiles of one (batch, head), and each of its two CTAs loads
 * half of every K/V tile.  Same arguments, layout, ownership and outputs as
 * attn_fwd with causal = 0 (no causal argument); the result is the same
 * definition (fp32 arithmetic, P rounded to the input dtype for P.V).
 *
 * Passages: as attn_fwd, and M4.6 "FlashAttention-3/4 Hardware Pipelines"
 * 0x08 (the 2-CTA mode of the non-causal d = 128 forward: an M = 256 product
 * over the pair, each CTA supplying its own rows of A and half of B).
 *
 * Errors: GBATTN_EBADSHAPE, EHEADS, EHEADDIM (d != 128), EDTYPE, EPOINTER,
 * EUNSUPPORTED, ELAUNCH.
 */
int attn_fwd_pair(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                  int dtype, void *stream);

/*
 * attn_fwd_fp8_workspace_bytes -- bytes of device workspace attn_fwd_fp8
 * needs: the 8-bit transposed V, B * Hkv * d * Sk_pad with Sk_pad = Sk
 * rounded up to a multiple of 128.  Returns 0 for invalid sizes.
 */
size_t attn_fwd_fp8_workspace_bytes(int B, int Hkv, int Sk, int d);

/*
 * attn_fwd_fp8 -- exact attention forward with E4M3 (FP8) inputs.
 *
 *   q     [B, H,   Sq, d]  E4M3FN codes, input
 *   k, v  [B, Hkv, Sk, d]  E4M3FN codes, input
 *   q_descale, k_descale, v_descale  [B, Hkv] fp32 device arrays or NULL
 *         (NULL = 1): the real values are code * descale of the (batch, KV
 *         head); a query head h uses the descale of KV head h / (H / Hkv)
 *   o     [B, H,   Sq, d]  bf16, output
 *   lse   [B, H,   Sq]     fp32, output (may be NULL): natural-log sum of
 *         exp(scale * q.k) over the visible keys, with the dequantized q, k
 *   scale, causal: as for attn_fwd (d must be 128)
 *   workspace: caller-owned device scratch of at least
 *         attn_fwd_fp8_workspace_bytes(B, Hkv, Sk, d) bytes, 16-byte aligned;
 *         it receives V transposed to [B, Hkv, d, Sk_pad] (the K-major P.V
 *         operand), contents on entry do not matter
 *
 * Definition and passages: the FP8 forward of M4.6 "FlashAttention-3/4
 * Hardware Pipelines" 0x06 -- scores (scale dQ dK) Q8 K8^T in fp32, row
 * state in fp32, probabilities u = 2^4 exp(S - r) rounded to E4M3 for the
 * P V product while the row sum accumulates the fp32 u, O = dV (P8 V8) / l
 * in bf16 (0x06 "Derive Where Every Scale Must Enter", "Why The Source Raises
 * Softmax Probabilities"); probability offset 4 and conditional-rescale
 * threshold 4 (log2 units) keep every u <= 256 < 448 (M4.6 0x09 range
 * contract, E4M3FN row).  The per-(batch, KV head) descale granularity is
 * that of the pinned public API described in 0x06.
 *
 * Errors: GBATTN_EBADSHAPE (also B*Hkv > 65535), EHEADS, EHEADDIM (d != 128),
 * EPOINTER, EWORKSPACE, EUNSUPPORTED, ELAUNCH.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *v, const float *q_descale,
                 const float *k_descale, const float *v_descale, void *o, float *lse,
                 int B, int H, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_decode_workspace_bytes -- bytes of device workspace attn_decode_splitkv
 * needs: one fp32 partial state (m, l, o[d]) per (batch, query head, chunk),
 * i.e. B * Hq * n_split * (d + 2) * 4.  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int n_split, int d);

/*
 * attn_decode_splitkv -- one-query decode over a padded KV cache, split-KV.
 *
 *   q        [B, Hq, 1, d]        dtype, input
 *   k_cache, v_cache [B, Hkv, Sk_max, d] dtype, input; rows >= seqlens[b] are
 *            padding and are never read into the result (they may hold NaN)
 *   seqlens  [B] int32 DEVICE array, 1 <= seqlens[b] <= Sk_max (values
 *            outside that range are clamped into it on the device)
 *   o        [B, Hq, 1, d]        dtype, output
 *   lse      [B, Hq]              fp32, output; may be NULL
 *   n_split  number of key chunks per sequence (1 .. 256); chunk c of
 *            sequence b covers keys [floor(c*L_b/n_split), floor((c+1)*L_b/n_split))
 *   workspace, workspace_bytes: caller-owned device scratch of at least
 *            attn_decode_workspace_bytes(B, Hq, n_split, d) bytes, 16-byte
 *            aligned; it receives the per-chunk partial states, in
 *            natural-log units, as two consecutive fp32 arrays:
 *              o_part [B, Hq, n_split, d]  unnormalised o (o / l is the
 *                                          chunk's attention output)
 *              ml_part[B, Hq, n_split, 2]  (m, l)
 *            an empty chunk is stored as the merge identity
 *            (m = -inf, l = 0, o = 0).
 *
 * Two kernels run in stream order: the partial kernel (one CTA per
 * (chunk, KV head, batch) covering the H/Hkv query heads of that KV head,
 * each K/V row read once) and the merge kernel (M4.3 0x08B common-maximum
 * merge; final O = o / l, LSE = M + log l).
 *
 * Errors: GBATTN_EBADSHAPE, EHEADS, EHEADDIM, EDTYPE, EPOINTER, ESPLIT,
 * EWORKSPACE, EUNSUPPORTED, ELAUNCH.
 */
int attn_decode_splitkv(const void *q, const void *k_cache, const void *v_cache,
                        const int *seqlens, void *o, float *lse,
                        int B, int Hq, int Hkv, int Sk_max, int d, float scale,
                        int n_split, void *workspace, size_t workspace_bytes,
                        int dtype, void *stream);

/*
 * Choosing a backward.  Two entry points compute the same gradients:
 *   attn_bwd_atomic -- the default choice: faster in every measured case
 *       (five 128 x 128 products per (query block, key tile) pair; dQ is
 *       summed by fp32 atomic reductions, so its last bits may differ from
 *       call to call; dK and dV repeat bitwise);
 *   attn_bwd -- when dQ must repeat bitwise (one owner per output element,
 *       seven products per pair).
 */

/*
 * attn_bwd_workspace_bytes -- bytes of device workspace attn_bwd needs: the
 * fp32 row scalars D [B, H, Sq] (rounded up to 256 bytes).  For B=1, H=32,
 * Sq=4096 this is the 0.5 MiB D entry of the scratch ledger in M4.4 0x06.1J;
 * the ledger's fp32 dQ accumulator and expanded per-query-head dK/dV buffers
 * are not needed (see attn_bwd).  Returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int Sq, int d);

/*
 * attn_bwd -- exact attention backward (gradients of attn_fwd).
 *
 *   q, o, dout [B, H,   Sq, d]  dtype, inputs (o is attn_fwd's output for q, k, v)
 *   k, v       [B, Hkv, Sk, d]  dtype, inputs
 *   lse        [B, H,   Sq]     fp32, input: attn_fwd's LSE (natural log)
 *   dq         [B, H,   Sq, d]  dtype, output
 *   dk, dv     [B, Hkv, Sk, d]  dtype, output: summed over the H/Hkv query
 *              heads that read each KV head
 *   scale, causal: as passed to attn_fwd
 *   workspace, workspace_bytes: caller-owned device scratch of at least
 *              attn_bwd_workspace_bytes(B, H, Sq, d) bytes, 16-byte aligned;
 *              its contents on entry do not matter
 *
 * Definition (M4.4 0x06.1A): with P_ij = exp(scale q_i.k_j - LSE_i) over the
 * visible keys, dP = dO V^T, D_i = dO_i . O_i, dS = P o (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.  Three kernels run in
 * stream order: D; one CTA per (128-key tile, batch, KV head) that keeps the
 * tile's dK, dV in tensor memory over every visible query block of every
 * query head in the group (the column owner of 0x06.1B; the GQA sum of
 * 0x06.1H happens in the accumulator); one CTA per (128-row query block,
 * batch, query head) that keeps the block's dQ in tensor memory over every
 * visible key tile (the row owner of 0x06.1I).  Each owner recomputes the
 * scores it needs, so every output element has a single writer and a fixed
 * summation order: results are bitwise repeatable (no atomics, 0x06.1F).
 *
 * Errors: GBATTN_EBADSHAPE, EHEADS, EHEADDIM, EDTYPE,
 * EPOINTER (every pointer required; lse 4-byte aligned), EWORKSPACE,
 * EUNSUPPORTED, ELAUNCH.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, void *dq, void *dk, void *dv,
             int B, int H, int Hkv, int Sq, int Sk, int d, float scale, int causal,
             void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * attn_bwd_atomic_workspace_bytes -- bytes of device workspace attn_bwd_atomic
 * needs: attn_bwd_workspace_bytes(B, H, Sq, d) for the fp32 row scalars D,
 * then the fp32 dQ accumulator [B, H, Sq, d] (the dQaccum entry of the
 * scratch ledger in M4.4 0x06.1J).  Returns 0 for invalid sizes.
 */
size_t attn_bwd_atomic_workspace_bytes(int B, int H, int Sq, int d);

/*
 * attn_bwd_atomic -- exact attention backward on the schedule of M4.4
 * 0x06.1D: one CTA per (128-key tile, batch, KV head) owns dK and dV (summed
 * over the H/Hkv query heads of the group in its accumulators, 0x06.1H) and
 * adds every query block's contribution dS_ij K_j into the fp32 dQ
 * accumulator with atomic adds; a last kernel writes dQ = scale * accumulator
 * in the input dtype.  Same arguments, layouts and definition as attn_bwd
 * (d = 64 or 128); workspace is caller-owned device scratch of at least
 * attn_bwd_atomic_workspace_bytes(B, H, Sq, d) bytes, 16-byte aligned, its
 * contents on entry irrelevant (the call zeroes the accumulator).
 *
 * Atomic adds reach every contribution but not in a fixed order (0x06.1F),
 * so dQ may differ in its last bits between calls; dK and dV are bitwise
 * repeatable.  Five 128 x 128 products per (query block, key tile) pair
 * against attn_bwd's seven.
 *
 * Errors: as attn_bwd.
 */
int attn_bwd_atomic(const void *q, const void *k, const void *v, const void *o, const float *lse,
                    const void *dout, void *dq, void *dk, void *dv,
                    int B, int H, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                    void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv for callers that cannot
 * allocate device memory (a host framework that owns every allocation and
 * forbids plugins from calling cudaMalloc, memory-capped or real-time
 * services that must not enter the allocator, C callers that only receive
 * their input and output pointers).  The pages have no counterpart: this is
 * a packaging variant of the split-KV decode above, not part of the method.
 *
 * Arguments and results are those of attn_decode_splitkv without the
 * workspace pair: the partial states go to a fixed array inside the library
 * (attn_decode_noalloc_scratch_bytes() = 32 MiB, held by every GPU that loads
 * the library until the process exits).  Problems whose
 * attn_decode_workspace_bytes(B, Hq, n_split, d) exceeds that size return
 * GBATTN_EWORKSPACE before any device work.  The call allocates nothing.
 *
 * The first call on each device looks up the array's device address with
 * that device current.  CUDA loads device code lazily by default, so that
 * first call is also the one that loads this part of the library onto the
 * device, the 32 MiB array included, which may allocate and synchronise
 * inside the CUDA runtime.  A caller that must never reach the allocator
 * therefore makes one call (any valid problem) at initialisation, outside
 * any stream capture; later calls allocate nothing.  The address is cached
 * per device with the id of its CUDA context and looked up again if the
 * context changes (after cudaDeviceReset), in which case that call is again
 * a first call.  Every call shares the array (nothing in it needs clearing:
 * each call overwrites the states it reads), so two calls whose kernels may
 * overlap on the GPU race and must be ordered by the caller.
 *
 * Errors: the argument checks and codes of attn_decode_splitkv (EBADSHAPE,
 * EHEADS, EHEADDIM, EDTYPE, EPOINTER, ESPLIT) come first; then
 * GBATTN_EWORKSPACE for a problem too large for the array; EUNSUPPORTED,
 * ELAUNCH.
 */
int attn_decode_splitkv_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                const int *seqlens, void *o, float *lse,
                                int B, int Hq, int Hkv, int Sk_max, int d, float scale,
                                int n_split, int dtype, void *stream);

/* Bytes of the fixed scratch array used by attn_decode_splitkv_noalloc. */
size_t attn_decode_noalloc_scratch_bytes(void);

/*
 * gbattn_causal_tile_counts -- host-only planning helper (no device work).
 * Classifies the (ceil(Sq/Br) x ceil(Sk/Bc)) tile grid with the half-open
 * ranges of M4.4 0x05.1A-B and delta = Sk - Sq:
 *   skipped  : k0 > (q1 - 1) + delta        (whole tile in the future)
 *   full     : (k1 - 1) <= q0 + delta       (no element mask needed)
 *   partial  : otherwise                    (mask cells before the row max)
 * Also returns the number of causally allowed cells and of cells inside
 * visited (full + partial) tiles.  Any output pointer may be NULL.
 * Returns GBATTN_OK or GBATTN_EBADSHAPE.
 */
int gbattn_causal_tile_counts(int Sq, int Sk, int Br, int Bc,
                              long long *full, long long *partial, long long *skipped,
                              long long *allowed_cells, long long *visited_cells);

/*
 * gbattn_exp2_paths -- diagnostic: evaluates the two base-2 exponentials the
 * kernels can use on n (even) device fp32 values x, writing
 *   y_poly[i]: the FMA-pipe software path (range reduction 2^x = 2^n p(f),
 *              degree-3 polynomial p on [0, 1), inputs clamped to
 *              [-126, 127]) -- the software exp2 of M4.6 0x09;
 *   y_hw[i]:   the hardware MUFU approximation (ex2.approx.ftz).
 * All pointers are 8-byte aligned device pointers; work is enqueued on
 * `stream`.  It exists so that tests can pin the software path's accuracy
 * (M4.6 0x09 states a degree-3 maximum relative error near 9e-5); the method
 * has no counterpart.  Errors: GBATTN_EBADSHAPE (n < 0 or odd),
 * GBATTN_EPOINTER, GBATTN_EUNSUPPORTED, GBATTN_ELAUNCH.
 */
int gbattn_exp2_paths(const float *x, float *y_poly, float *y_hw, long long n, void *stream);

/*
 * gbattn_selftest_bounded_wait -- diagnostic of the kernels' failure path:
 * launches one warp whose thread 0 performs the bounded mbarrier wait every
 * kernel role uses on its producer (about 2 s limit).  With arrive != 0 the
 * barrier is satisfied first and nothing is reported; with arrive = 0
 * nothing ever arrives, the wait gives up without faulting or hanging the
 * GPU, and the next gbattn_device_status() returns GBATTN_EDEVICE_TIMEOUT.
 * This is the "consumer waits for a commit the producer never issues" case
 * of the ring's liveness proof in M4.6 "FlashAttention-3/4 Hardware
 * Pipelines" 0x03.  Errors: GBATTN_EUNSUPPORTED, GBATTN_ELAUNCH.
 */
int gbattn_selftest_bounded_wait(int arrive, void *stream);

/*
 * gbattn_device_status -- read and clear the library's device status word.
 * Returns GBATTN_OK, or GBATTN_EDEVICE_TIMEOUT if a kernel gave up since the
 * last call (a bounded wait timed out, or a shared-memory alignment check
 * failed), or GBATTN_ELAUNCH if the device reported an error.
 *
 * Scope: the call synchronises the whole current device
 * (cudaDeviceSynchronize, every stream), and the word is one per device,
 * shared by all streams and host threads that use the library there.  A
 * failure raised by a kernel on one stream is therefore reported to
 * whichever caller polls first, and that call clears it; callers that share
 * a device and need to attribute a failure must poll from one place.
 */
int gbattn_device_status(void);

/*
 * gbattn_timeline_set -- per-CTA timeline of forward launches (attn_fwd,
 * attn_fwd_pair, attn_fwd_fp8; a profiling aid, the method has no
 * counterpart).  While set, every such launch whose grid has at most
 * `capacity` CTAs writes, for CTA i, four unsigned 64-bit values at
 * records[4 i .. 4 i + 3]:
 *   [0] start and [1] end of the CTA, in %globaltimer nanoseconds,
 *   [2] the SM it ran on,
 *   [3] its work unit, (b * H + h) << 32 | u: for attn_fwd and attn_fwd_fp8
 *       u is the query pair (rows 256 u .. 256 u + 255), one CTA each, grid
 *       B * H * ceil(Sq / 256); for attn_fwd_pair u is the 512-row query
 *       block of the CTA's cluster (CTAs 2 c and 2 c + 1), grid
 *       2 * B * H * ceil(Sq / 512).
 * A launch with more CTAs than `capacity` writes nothing.  records is a device pointer owned
 * by the caller, 8-byte aligned, at least 32 * capacity bytes, and must stay
 * valid until the launches that write it have completed.  records = NULL
 * turns the timeline off (capacity is then ignored).  The setting is
 * process-wide and is read when a launch is enqueued.
 * Errors: GBATTN_EPOINTER (records not 8-byte aligned), GBATTN_EBADSHAPE
 * (records != NULL and capacity < 1).
 */
int gbattn_timeline_set(unsigned long long *records, long long capacity);

/* Text for a status code (static storage; never NULL). */
const char *gbattn_error_string(int code);

/* Library version string, e.g. "gbattn 0.1.0 sm_103a". */
const char *gbattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H_ */
