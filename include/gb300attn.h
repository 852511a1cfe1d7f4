/*
 * gb300attn.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention library (libgb300attn.so).
 *
 * The operation, as the tutorial pages define it:
 *
 *   Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + M) V
 *     "04. Self-Attention：Transformer 的核心计算", section 四 (scores,
 *     scale, row softmax, weighted sum) and section 七 (the mask M is added
 *     before the softmax: 0 where a key may be seen, -inf where it may not).
 *   Causal mask: key j is hidden from query i when j > i ("attention-mechanism"
 *     page, section "掩码：因果与 padding").  Padding mask: keys at or past
 *     the sequence's valid length are hidden (same section).
 *   Multi-head layer: Y = Concat(head_1..head_h) W_O with
 *     head_i = Attention(X W_Q^i, X W_K^i, X W_V^i), the three projections
 *     fused into one GEMM with W_QKV = [W_Q | W_K | W_V] ("Self-Attention 机制",
 *     sections "五步计算" and "维度全程跟踪").
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, in DEVICE memory, and owned by the
 *     caller; the library keeps no pointer after a call returns.
 *   - Element types: bf16 (bfloat16) for Q, K, V, O, X, weights and Y; float
 *     for LSE; int32 for kv_lens.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous: errors found on the host are returned before anything
 *     is launched; errors found on the device are reported later by
 *     attn_check_device_status().
 *   - The library allocates no device memory per call.  It keeps, per device
 *     and for the life of the process, a 4-byte device status word (a file-
 *     scope __device__ variable) and cached kernel attributes.
 *   - Thread safety: calls may be made from several host threads; calls on
 *     one stream execute in order.
 */
#ifndef GB300ATTN_H
#define GB300ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* bad size, null pointer, kv_len out of range */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement  */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned            */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed            */
  ATTN_ERR_TIMEOUT = 5,      /* a device-side pipeline wait gave up          */
  ATTN_ERR_TOO_LARGE = 6,    /* problem exceeds the fixed scratch of
                                mha_layer_fwd_noalloc                       */
  ATTN_ERR_SELF_CHECK = 7    /* the self-checking build found a TMA or TMEM
                                access that broke its rules (skipped, not
                                executed); never returned by the normal
                                build                                       */
} attn_status_t;

/*
 * mask_kind bit flags.  PADDING combines with either causal flag; the two
 * causal flags are exclusive.
 *   ATTN_MASK_CAUSAL: key j is hidden from query i when j > i (the look-ahead
 *     mask, aligned to the first key).
 *   ATTN_MASK_CAUSAL_BOTTOM_RIGHT: the same look-ahead mask aligned to the
 *     last key of each sequence, for Lq queries that are the last Lq tokens
 *     of a sequence whose keys include them (decoding against a KV cache,
 *     "Self-Attention 机制", sections "Causal Mask" and "MHA -> MQA -> GQA ->
 *     MLA").  Sequence b holds n_b keys: kv_lens[b] with ATTN_MASK_PADDING,
 *     else Lk.  Query i sits at position p_i = n_b - Lq + i and sees the keys
 *     j <= p_i, so a new token never sees a later new token.  A query with
 *     p_i < 0 sees no key and gets O = 0, LSE = -inf; with this mask no query
 *     row is padding by its index alone.  Without padding it is the shift by
 *     Lk - Lq, equal to ATTN_MASK_CAUSAL when Lq == Lk.
 */
enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_PADDING = 2,
  ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 4
};

/*
 * attn_fwd -- multi-head attention forward over [B, h, L, d] heads.
 *
 *   Q  bf16 [B, h, Lq, d_k]     K  bf16 [B, h, Lk, d_k]     V  bf16 [B, h, Lk, d_v]
 *   O  bf16 [B, h, Lq, d_v]     (written)
 *   LSE float [B, h, Lq]        (written when non-NULL) natural-log
 *                               log-sum-exp of the row's scaled, masked scores
 *   kv_lens int32 [B] device array, required iff mask_kind has the PADDING
 *     bit: sequence b's valid length.  Keys j >= kv_lens[b] are masked; query
 *     rows i >= kv_lens[b] are padding and get O = 0, LSE = -inf (except
 *     with ATTN_MASK_CAUSAL_BOTTOM_RIGHT, whose queries end at the sequence's
 *     end: see above).
 *   mask_kind: ATTN_MASK_* flags (see above).
 *   scale: multiplier of Q K^T; scale <= 0 selects 1 / sqrt(d_k).
 *   A row with no visible key (kv_lens[b] == 0, or Lk == 0) gets O = 0 and
 *   LSE = -inf.  The attention matrix itself is never formed or returned.
 *
 * Supported: d_k == d_v in {64, 128}; B, h, Lq, Lk >= 0 with B*h*ceil(Lq/256)
 * < 2^31 and Lq, Lk < 2^31.  Q, K, V, O must be 16-byte aligned, LSE 4-byte
 * aligned.  Empty problems (B, h or Lq == 0) return ATTN_OK without a launch.
 * A kv_lens entry outside [0, Lk] is clamped on the device and reported as
 * ATTN_ERR_INVALID_ARG by attn_check_device_status().
 */
attn_status_t attn_fwd(const void* Q, const void* K, const void* V, int B, int h, int Lq, int Lk,
                       int d_k, int d_v, int mask_kind, const int32_t* kv_lens, float scale,
                       void* O, float* LSE, void* stream);

/*
 * attn_fwd_gqa -- attn_fwd with grouped-query attention ("Self-Attention 机制",
 * section "MHA -> MQA -> GQA -> MLA"): h query heads share h_kv key/value
 * heads, each run of h/h_kv consecutive query heads reading one K/V head
 * (query head i reads K/V head i / (h/h_kv)).  h_kv == h is attn_fwd (multi-
 * head), h_kv == 1 is multi-query attention.
 *
 *   Q bf16 [B, h, Lq, d_k]; K bf16 [B, h_kv, Lk, d_k]; V bf16 [B, h_kv, Lk, d_v];
 *   O, LSE, kv_lens, mask_kind, scale, alignment and errors as for attn_fwd;
 *   h must be a multiple of h_kv (else ATTN_ERR_INVALID_ARG).
 */
attn_status_t attn_fwd_gqa(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                           int Lq, int Lk, int d_k, int d_v, int mask_kind,
                           const int32_t* kv_lens, float scale, void* O, float* LSE,
                           void* stream);

/*
 * attn_fwd_host -- attn_fwd_gqa with Q, K, V, O, LSE and kv_lens in HOST
 * memory.  The call copies the inputs to the device, runs the attention
 * kernels and copies the results back, overlapping the three.  The work is
 * cut into up to 16 chunks of at least 8 MB, each either whole batch
 * elements or a group of K/V heads of one element with their query heads, so
 * each chunk's Q, K, V, O and LSE are contiguous and the chunks carry equal
 * work.  A chunk's inputs are copied while earlier chunks compute, and its O
 * and LSE are copied back as soon as it is done.  Each (b, head) runs the
 * work items of attn_fwd_gqa: with ATTN_SCHEDULE_TWO_QTILES every element is
 * bit-identical to it.  ATTN_SCHEDULE_SPLIT_KEYS deals an item's key tiles
 * to its two softmax groups by the CTA's running tile count, so there a row
 * may be summed in the other order (a difference of rounding).
 *
 *   Q, K, V, O, LSE, kv_lens   host pointers, layouts as for attn_fwd_gqa;
 *               page-locked memory (cudaHostAlloc / cudaHostRegister) lets
 *               the copies run asynchronously and overlap; pageable memory
 *               works but is copied synchronously.  LSE may be NULL.
 *   workspace   device scratch of at least attn_fwd_host_workspace_bytes(...)
 *               bytes, 256-byte aligned, owned by the caller; it receives
 *               device copies of Q, K, V, O, LSE and kv_lens.  Calls that
 *               share it must not overlap.
 *   stream      the call's work runs on internal streams of the library that
 *               start after the work already queued on `stream`; `stream`
 *               is made to wait for all of it.  The host buffers must stay
 *               valid, and O / LSE must not be read, until `stream` has been
 *               synchronised.
 *
 * Errors as for attn_fwd_gqa, plus ATTN_ERR_INVALID_ARG for a missing or
 * too-small workspace and ATTN_ERR_MISALIGNED for a workspace not 256-byte
 * aligned.
 */
attn_status_t attn_fwd_host(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                            int Lq, int Lk, int d_k, int d_v, int mask_kind,
                            const int32_t* kv_lens, float scale, void* O, float* LSE,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_host_workspace_bytes -- device scratch attn_fwd_host needs for
 * these sizes; 0 for unsupported sizes.
 */
size_t attn_fwd_host_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d_k, int d_v);

/*
 * attn_decode -- attn_fwd_gqa for few query rows against a long key/value
 * cache (decoding: the Lq new tokens are the last Lq of each sequence, so the
 * usual mask is ATTN_MASK_CAUSAL_BOTTOM_RIGHT, with kv_lens for caches of
 * different lengths).  It computes exactly what attn_fwd_gqa computes.
 *
 * How it differs: work is split over the keys.  Each (b, K/V head, chunk of
 * keys) is one work item whose Q tile holds the Lq rows of all h/h_kv query
 * heads that share the K/V head, so every key/value row is read once per K/V
 * head; a second kernel merges the chunks' partial softmaxes by the online
 * softmax identity ("Self-Attention 机制", section "Softmax 的数值稳定性与
 * Online Softmax").
 *
 *   Arguments as for attn_fwd_gqa with d = d_k = d_v, plus
 *   workspace   device scratch of at least attn_decode_workspace_bytes(...)
 *               bytes, 256-byte aligned, owned by the caller; not read
 *               before it is written.  Calls that share it must not overlap.
 *
 * Supported: d in {64, 128}; (h / h_kv) * Lq <= 128 (else
 * ATTN_ERR_UNSUPPORTED: use attn_fwd_gqa).  A workspace smaller than needed
 * returns ATTN_ERR_INVALID_ARG.  Other errors as for attn_fwd_gqa.
 */
attn_status_t attn_decode(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                          int Lq, int Lk, int d, int mask_kind, const int32_t* kv_lens,
                          float scale, void* O, float* LSE, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * attn_decode_workspace_bytes -- scratch size attn_decode needs for these
 * sizes on the current device (it depends on the device's SM count); 0 for
 * empty or unsupported sizes.
 */
size_t attn_decode_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d);

/*
 * attn_decode_host -- one decode step with host buffers for the step's own
 * data and a key/value cache that stays on the device: it copies the Lq new
 * query rows and the new tokens' key and value rows in, writes those rows
 * into the cache, runs attn_decode over the cache and copies O and LSE out,
 * all in order on `stream`.
 *
 *   Q        host bf16 [B, h, Lq, d]: the new tokens' query rows.
 *   K_new, V_new  host bf16 [B, h_kv, Lq, d]: their key and value rows.
 *   K_cache, V_cache  device bf16 [B, h_kv, Lk, d], 16-byte aligned; the
 *            call writes row kv_len_b - Lq + i of (b, K/V head) with new row
 *            i (rows whose position would be negative are dropped) and
 *            reads the cache as attn_decode does.  That row is the position
 *            ATTN_MASK_CAUSAL_BOTTOM_RIGHT gives query i, so each new token
 *            sees the cache up to and including its own key, and no later
 *            new token.
 *   kv_lens  host int32 [B] (required with ATTN_MASK_PADDING): valid keys
 *            of each sequence after the new ones are appended, clamped to
 *            [0, Lk].  Without padding every sequence holds Lk keys and the
 *            new rows are the last Lq.
 *   O, LSE   host bf16 [B, h, Lq, d] and float [B, h, Lq] (LSE may be NULL),
 *            written when the stream reaches the end of the call.
 *   workspace  device scratch of at least attn_decode_host_workspace_bytes()
 *            bytes, 256-byte aligned: staging for the new rows, kv_lens, O,
 *            LSE and attn_decode's own scratch.  Calls that share it must not
 *            overlap.
 *   mask_kind, scale, h_kv, d as for attn_decode.
 *
 * Host buffers may be pinned (the copies then run asynchronously) or
 * pageable.  Lk = 0 returns ATTN_ERR_INVALID_ARG (no cache to append to).
 * Other errors as for attn_decode.
 */
attn_status_t attn_decode_host(const void* Q, const void* K_new, const void* V_new, void* K_cache,
                               void* V_cache, int B, int h, int h_kv, int Lq, int Lk, int d,
                               int mask_kind, const int32_t* kv_lens, float scale, void* O,
                               float* LSE, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * attn_decode_host_workspace_bytes -- device scratch attn_decode_host needs
 * for these sizes on the current device; 0 for empty or unsupported sizes.
 */
size_t attn_decode_host_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d);

/*
 * attn_weights -- the attention matrix A for inspection of small problems.
 * The pages' reference snippets return A = softmax(Q K^T / sqrt(d_k) + M) next
 * to the output ("attention-mechanism" page, section "最小实现";
 * "多模态大模型学习笔记（十四）", section 2.3); attn_fwd never forms it.  This
 * call rebuilds it from the LSE that attn_fwd / attn_fwd_gqa returned for the
 * same Q, K, mask and scale: A_ij = exp(scale * q_i . k_j - LSE_i) for a
 * visible key j and 0 for a masked one (rows with LSE = -inf are all 0).
 *
 *   Q bf16 [B, h, Lq, d_k]; K bf16 [B, h_kv, Lk, d_k]; LSE float [B, h, Lq];
 *   A float [B, h, Lq, Lk] (written).  mask_kind, kv_lens, scale as for
 *   attn_fwd.  d_k <= 256.  It is a plain CUDA-core kernel (one thread per
 *   entry, no tensor cores), meant for shapes small enough to inspect.
 */
attn_status_t attn_weights(const void* Q, const void* K, const float* LSE, int B, int h,
                           int h_kv, int Lq, int Lk, int d_k, int mask_kind,
                           const int32_t* kv_lens, float scale, float* A, void* stream);

/*
 * mha_layer_workspace_bytes -- device workspace mha_layer_fwd needs for this
 * shape: the fused projection QKV bf16 [B, L, 3, h, d_k] plus the concatenated
 * heads bf16 [B, L, d_model].  Returns 0 for an unsupported shape.
 */
size_t mha_layer_workspace_bytes(int B, int L, int d_model, int h);

/*
 * mha_layer_fwd -- the five-step multi-head self-attention layer:
 *   QKV = X W_QKV               (one GEMM; W_QKV columns are [Q | K | V], head
 *                                i owning columns i*d_k .. i*d_k+d_k-1 of each)
 *   O_i = Attention(Q_i, K_i, V_i) with the given mask, d_k = d_model / h
 *   Y   = Concat(O_1 .. O_h) W_O
 *
 *   X bf16 [B, L, d_model];  W_QKV bf16 [d_model, 3*d_model];
 *   W_O bf16 [d_model, d_model];  Y bf16 [B, L, d_model] (written).
 *   The weights multiply from the right (X W, W stored [in, out]); there are
 *   no biases.  kv_lens / mask_kind / scale as for attn_fwd.  Padded query
 *   rows produce Y = 0.
 *   workspace: device buffer of at least mha_layer_workspace_bytes(), 256-byte
 *   aligned; it is scratch, overwritten by the call.
 *
 * Supported: d_model / h in {64, 128}, d_model a multiple of 128, B*L a
 * multiple of 128; all pointers 16-byte aligned.
 */
attn_status_t mha_layer_fwd(const void* X, const void* W_QKV, const void* W_O, int B, int L,
                            int d_model, int h, int mask_kind, const int32_t* kv_lens,
                            float scale, void* Y, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * mha_layer_fwd_host -- mha_layer_fwd with the activations X and Y (and
 * kv_lens) in HOST memory and the weights W_QKV, W_O on the device, as a
 * model's parameters are.  The call copies X to the device, runs the layer
 * and copies Y back, overlapping the three over chunks of whole batch
 * elements of at least 4096 tokens (at most 8 chunks): a chunk's X is copied
 * in while the previous chunk computes, and its Y is copied out as soon as it
 * is done.  Each chunk runs the kernels of mha_layer_fwd on its batch
 * elements, so with the same attention schedule Y is bit-identical to
 * mha_layer_fwd's.
 *
 *   X, Y, kv_lens   host pointers (page-locked memory lets the copies overlap)
 *   W_QKV, W_O      device pointers, 16-byte aligned
 *   workspace       device scratch of at least mha_layer_host_workspace_bytes()
 *                   bytes, 256-byte aligned: device copies of X, Y, kv_lens and
 *                   two layer scratch buffers.  Calls that share it must not
 *                   overlap.
 *   stream          as for attn_fwd_host: the work runs on internal streams
 *                   after the work queued on `stream`, and `stream` waits for
 *                   all of it; Y must not be read before `stream` is
 *                   synchronised.
 * Supported shapes and errors as for mha_layer_fwd.
 */
attn_status_t mha_layer_fwd_host(const void* X, const void* W_QKV, const void* W_O, int B, int L,
                                 int d_model, int h, int mask_kind, const int32_t* kv_lens,
                                 float scale, void* Y, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* mha_layer_host_workspace_bytes -- workspace of mha_layer_fwd_host; 0 for an
 * unsupported shape. */
size_t mha_layer_host_workspace_bytes(int B, int L, int d_model, int h);

/*
 * mha_layer_fwd_noalloc -- the same five-step layer as mha_layer_fwd, for
 * callers that may not allocate device memory: for example a plugin inside a
 * host framework that owns every device buffer through its own pool and does
 * not let plugins call cudaMalloc, or a runtime whose memory plan is fixed at
 * start-up (cudaMalloc can stall the whole device and can fail under memory
 * pressure, which such a runtime cannot afford in the middle of a run).  The
 * tutorial pages have no counterpart to this entry point; it only changes
 * where the layer's scratch lives.
 *
 * The caller still passes X, W_QKV, W_O, Y (and kv_lens) exactly as for
 * mha_layer_fwd.  The scratch (the QKV projection and the concatenated heads,
 * mha_layer_workspace_bytes() bytes) comes from one fixed array of
 * ATTN_NOALLOC_SCRATCH_BYTES (32 MiB) compiled into the library: every GPU on
 * which the library is loaded holds that array until the process exits.
 * Nothing is allocated or freed by the call.
 *   - A shape whose workspace exceeds ATTN_NOALLOC_SCRATCH_BYTES is rejected
 *     with ATTN_ERR_TOO_LARGE before anything is launched (for d_model = 1024
 *     the limit is B*L <= 4096 tokens).
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress on the current device); make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array, which keeps whatever the
 *     last call left in it; the layer overwrites all of the scratch it reads,
 *     so nothing needs clearing.  Calls whose execution overlaps on the GPU
 *     (e.g. on two streams without ordering between them) race on the array
 *     and give wrong results: order them.
 * Returns and validation otherwise as for mha_layer_fwd.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
attn_status_t mha_layer_fwd_noalloc(const void* X, const void* W_QKV, const void* W_O, int B,
                                    int L, int d_model, int h, int mask_kind,
                                    const int32_t* kv_lens, float scale, void* Y, void* stream);

/*
 * attn_gemm_bf16 -- C = A B with bf16 inputs, fp32 accumulation and bf16
 * output: the projection step of the layer, exposed for direct use.
 *   A bf16 [M, K], B bf16 [K, N], C bf16 [M, N], all row-major.
 * Supported: M multiple of 128, N multiple of 256, K multiple of 64;
 * pointers 16-byte aligned.  A 32-byte aligned C is written in whole 32-byte
 * sectors (faster); a C aligned to 16 bytes only, in 16-byte pieces.
 */
attn_status_t attn_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K,
                             void* stream);

/*
 * attn_check_device_status -- synchronize `stream`, then read and clear the
 * current device's status word.  Returns ATTN_ERR_TIMEOUT if a kernel's
 * bounded pipeline wait gave up since the last check, ATTN_ERR_INVALID_ARG if
 * a kv_lens entry was out of range, ATTN_ERR_CUDA if the stream reports a
 * CUDA error, else ATTN_OK.
 */
attn_status_t attn_check_device_status(void* stream);

/*
 * attn_is_checked_build -- 1 for the self-checking build of this library
 * (libgb300attn_checked.so), 0 otherwise.  The self-checking build tests,
 * before every TMA copy and TMEM load or store, the preconditions that the
 * hardware does not check by itself: the innermost TMA coordinate on a
 * 16-byte boundary (and no store below coordinate 0), tile and barrier
 * addresses aligned, and each warp's TMEM access inside its 32-lane quarter
 * and the 512 columns; and it checks that every attention work item decodes
 * to a batch element, head and row block in range.  A violation skips the
 * access (an out-of-range item ends the CTA's work) and makes the next
 * attn_check_device_status return ATTN_ERR_SELF_CHECK.  Results are
 * otherwise identical to the normal build's.
 */
int attn_is_checked_build(void);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * attn_set_wait_limit_ns -- time limit of every device-side pipeline wait
 * (default 2e9 ns).  After it, the kernel stops, records ATTN_ERR_TIMEOUT in
 * the status word and returns instead of waiting forever.  0 restores the
 * default.  Affects launches made after the call.
 */
void attn_set_wait_limit_ns(uint64_t ns);

/*
 * Work schedules of the attention kernel.  Both compute the same function
 * (online softmax over 128-key tiles, fp32 accumulation, bf16 P); they differ
 * in how a CTA's work is laid out on the SM:
 *   ATTN_SCHEDULE_TWO_QTILES  256 query rows per work item, two 128-row Q
 *                             tiles with one softmax warpgroup and one MMA
 *                             issuer warp each (at d = 128 the two issuers
 *                             submit their MMAs to the tensor core in turn)
 *   ATTN_SCHEDULE_SPLIT_KEYS  128 query rows per work item, its key tiles
 *                             dealt alternately to two softmax warpgroups
 *                             with separate accumulators, merged at the end
 *                             of the item; twice as many work items, for
 *                             shapes with too few 256-row items to fill the GPU
 *   ATTN_SCHEDULE_AUTO        SPLIT_KEYS when B * h * ceil(Lq / 256) is below
 *                             the number of SMs, else TWO_QTILES (the default)
 */
typedef enum {
  ATTN_SCHEDULE_AUTO = 0,
  ATTN_SCHEDULE_TWO_QTILES = 1,
  ATTN_SCHEDULE_SPLIT_KEYS = 2
} attn_schedule_t;

/*
 * attn_set_schedule -- schedule of later attention launches (attn_fwd,
 * attn_fwd_gqa and the attention step of mha_layer_fwd / _noalloc); process-
 * wide, like attn_set_wait_limit_ns.  Returns ATTN_ERR_INVALID_ARG (and keeps
 * the current setting) for a value outside attn_schedule_t.
 */
attn_status_t attn_set_schedule(int schedule);

/*
 * attn_debug_skip_kv_load -- testing hook: the next attn_fwd launches skip
 * the K-tile load with this running index in every CTA, so that a pipeline
 * wait runs out and the timeout path is exercised (-1 disables; the default).
 */
void attn_debug_skip_kv_load(long long index);

/*
 * attn_probe_ex2 -- diagnostic: measures the throughput of the special-
 * function unit's exp2 (ex2.approx.ftz.f32), the one transcendental the
 * softmax issues per unmasked score, so that the exp term of the attention
 * roofline (exp count / exp rate) uses a measured rate.
 *
 * Launches `blocks` CTAs of `threads` threads on `stream`; every thread runs
 * `iters` iterations of ATTN_PROBE_EX2_PER_THREAD_ITER (= 32) ex2 in 8
 * independent chains, so one launch performs
 * blocks * threads * iters * 32 exp2.  The caller times the launch with
 * events on `stream`.
 *   timing_out  device, uint64 [blocks][2]: for each CTA, the SM clock
 *               cycles (clock64) and the nanoseconds (globaltimer) it spent
 *               in its loop, both between the same two CTA barriers; their
 *               ratio is the SM clock during the probe
 *   sink        device, one float: never written in practice (it keeps the
 *               chains' results live)
 * Errors: ATTN_ERR_INVALID_ARG for blocks < 1, iters < 1, threads not a
 * multiple of 32 in [32, 1024], or a NULL pointer; ATTN_ERR_CUDA if the launch
 * fails.  Asynchronous, like the other entry points.
 */
#define ATTN_PROBE_EX2_PER_THREAD_ITER 32
attn_status_t attn_probe_ex2(int blocks, int threads, int iters,
                             unsigned long long* timing_out, float* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300ATTN_H */
