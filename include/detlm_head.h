/*
 * detlm_head.h -- batch-invariant LLM output head (lm_head) for GB300 (sm_103a).
 *
 * The output head maps final hidden rows h [B, d] to vocabulary logits
 * z = h . W^T [B, V] and decides the next token ("Greedy Decoding Has a
 * Precision Clause", section "Token-ranking margins explain why numerical
 * error sometimes matters": the lm_head converts the final transformer
 * representation into vocabulary scores). Each call fuses the decision into
 * the projection: greedy argmax with ties to the lowest token id, the gap
 * between the two best logits in bf16 ulps, or the log-probability of a
 * target token.
 *
 * Row invariance: every output of a row is bit-identical whatever the batch
 * size B and whatever other rows share the call, because every reduction
 * order is fixed by the weight's shape (V, d) and never by the row count
 * ("TandemLLM docs, 12 Exactness", section 12.2: matrix-product kernels fix
 * their reduction order by the weight's shape, never by the row count).
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers (or managed memory); pointers
 *    named *_host are host pointers. The library never frees caller memory.
 *    On unified-addressing systems an OUTPUT *_dev pointer may also be
 *    page-locked host memory the device can address (cudaHostAlloc,
 *    cudaHostRegister): the kernels then write the results straight into
 *    it, and they are in host memory once the stream reaches that point.
 *    Inputs (W, h, targets, drafts, seeds) must be device memory.
 *  - Layouts are row-major with d (the reduction axis) contiguous: W is
 *    [V, d] as a linear layer stores its weight, h is [B, d], logits [B, V].
 *  - Element types: DETLM_BF16 and DETLM_FP16 heads take 16-bit inputs and
 *    accumulate in fp32; the DETLM_INT8 head takes int8 inputs and computes
 *    int32 logits exactly.
 *  - Calls that take a stream are asynchronous on that stream; outputs are
 *    ready when the stream reaches that point. One handle serves one stream
 *    at a time (a handle owns one workspace); handles are not thread-safe.
 *  - Errors: every call returns a detlm_status_t and never aborts the
 *    process. Argument errors are found on the host before any GPU work
 *    (DETLM_EINVAL). Device-side conditions (a bounded wait that ran out, an
 *    out-of-range target id) set the handle's device error word; they are
 *    reported by detlm_head_check() and by the *_host calls.
 */
#ifndef DETLM_HEAD_H
#define DETLM_HEAD_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct detlm_head detlm_head_t;     /* opaque handle */

typedef enum {
  DETLM_BF16 = 0,   /* bf16 W and h, fp32 accumulation, fp32 logits        */
  DETLM_FP16 = 1,   /* IEEE fp16 W and h, fp32 accumulation, fp32 logits   */
  DETLM_INT8 = 2,   /* int8 W and h, exact int32 accumulation and logits   */
  DETLM_FP32 = 3    /* fp32 rows: input of the integer front end only      */
} detlm_dtype_t;

typedef enum {
  DETLM_OK = 0,
  DETLM_EINVAL = -1,        /* bad argument (null, size, alignment, dtype)  */
  DETLM_EUNSUPPORTED = -2,  /* operation not defined for this head's dtype  */
  DETLM_ECUDA = -3,         /* a CUDA runtime call failed (no GPU, launch)  */
  DETLM_ETIMEOUT = -4,      /* a device-side bounded wait ran out           */
  DETLM_ENOMEM = -5,        /* device or host allocation failed             */
  DETLM_ETARGET = -6        /* a target id was outside [0, V); logp = NaN  */
} detlm_status_t;

/* Create a head over the weight W_dev [V, d] of the given dtype.
 *
 * "Greedy Decoding Has a Precision Clause", section "Token-ranking margins
 * ...": the weight of the lm_head projection. W is BORROWED: the caller keeps
 * it alive and unchanged until detlm_head_destroy. The handle owns its TMA
 * descriptors, its workspace and a device error word, all made on the
 * current device.
 * Requirements: 1 <= V < 2^31; d >= 1; for BF16/FP16 d % 8 == 0 and for INT8
 * d % 16 == 0 (rows start on 16-byte boundaries); W_dev 16-byte aligned.
 * Returns DETLM_EINVAL on a bad argument, DETLM_ECUDA when no usable GPU. */
int detlm_head_create(detlm_head_t** out, const void* W_dev, int64_t V,
                      int64_t d, int dtype);

/* Grow the workspace so that calls with up to max_B rows allocate nothing.
 * Optional: calls grow it on demand (a synchronous allocation). Call it
 * before capturing calls into a CUDA graph. For an INT8 head, max_B >= 256
 * also makes what its calls of 256 rows or more run on: an fp16 copy of W
 * (2 * V * d bytes, converted once, exactly, and kept until destroy) and an
 * fp16 staging buffer for max_B hidden rows (2 * max_B * d bytes). */
int detlm_head_reserve(detlm_head_t* head, int64_t max_B);

/* Greedy decision for B hidden rows h_dev [B, d].
 *
 * token_dev  int32 [B]: lowest index v attaining max_v z[n, v]
 *            ("Eliminating Nondeterminism in LLM Inference with Integer-Only
 *            Arithmetic", section "DetLLM": argmax breaks ties toward the
 *            lowest token id).
 * gap_dev    BF16/FP16 heads: float [B], (m - s) / ulp_bf16(m), m the best
 *            logit, s the runner-up value of the multiset (s == m on a tie),
 *            ulp_bf16(m) = 2^(max(floor(log2|m|), -126) - 7), computed from
 *            the fp32 logits and rounded once to float ("TandemLLM docs, 12
 *            Exactness", section 12.2: the top-two gap in bf16 ulps). V == 1
 *            gives +inf.
 *            INT8 head: int32 [B], the exact m - s (INT32_MAX when V == 1).
 * logits_dev optional (NULL to skip): float [B, V] fp32 logits (int32 for
 *            INT8) ("TandemLLM docs, 12 Exactness", 12.2: the head returns
 *            fp32 logits).
 * B == 0 is a no-op. h_dev must be 16-byte aligned; outputs 4-byte aligned. */
int detlm_head_greedy(detlm_head_t* head, const void* h_dev, int64_t B,
                      int32_t* token_dev, void* gap_dev, void* logits_dev,
                      cudaStream_t stream);

/* Log-probability of one target token per row (BF16/FP16 heads only).
 *
 * logp_dev[n] = z[n, targets[n]] - log sum_v exp(z[n, v]) in fp32
 * ("batch-logprob-gap": the trainer's per-token log-probability;
 * "Inference and Decoding", section 3, Temperature: softmax at tau = 1).
 * A target outside [0, V) gives NaN and sets DETLM_ETARGET in the error word.
 * targets_dev: int32 [B]; logp_dev: float [B]. B == 0 is a no-op. h_dev must
 * be 16-byte aligned; targets_dev and logp_dev 4-byte aligned. The log-sum-
 * exp runs in a fixed order per row (exact maximum and sum of exp(z - max)
 * per 256-entry vocabulary tile, tiles merged in an order set by V alone:
 * 128 leaves of contiguous tiles, each folded in ascending order, combined
 * in a balanced binary tree), so logp_dev[n] is the same bits for any B and
 * any co-rows.
 * INT8 heads return DETLM_EUNSUPPORTED. */
int detlm_head_logprob(detlm_head_t* head, const void* h_dev,
                       const int32_t* targets_dev, int64_t B, float* logp_dev,
                       cudaStream_t stream);

/* Margin-gated greedy call ("Greedy Decoding Has a Precision Clause",
 * section "Correct the vulnerable token decisions, not every calculation"):
 * an ordinary 16-bit head returns its logits rounded to its storage format
 * and picks their argmax; where the top-two margin of those rounded logits
 * is below tau, the output projection is redone in FP32 and the token is
 * taken from it. Here the FP32 logits are what the projection computes in
 * the first place, so one pass yields both decisions and the gate costs no
 * second projection.
 *
 * Float heads only (INT8: DETLM_EUNSUPPORTED). Per row n:
 *   z16 = each fp32 logit rounded once (nearest, ties to even) to bf16 for
 *         a BF16 head, to fp16 for an FP16 head;
 *   base_token[n] = lowest index of max z16 (the ordinary head's token);
 *   margin[n]     = fp32(max z16 - runner-up of the multiset z16), +inf if
 *                   V == 1;
 *   token[n]      = the fp32 argmax (lowest index, as detlm_head_greedy)
 *                   where margin[n] < tau, else base_token[n];
 *   gap[n], logits: as detlm_head_greedy.
 * tau: any non-NaN float (0.001 in the page's experiments; tau <= 0 never
 * fires and returns the ordinary head's tokens); NaN gives DETLM_EINVAL.
 * base_token_dev and margin_dev may be NULL. */
int detlm_head_greedy_gated(detlm_head_t* head, const void* h_dev, int64_t B,
                            float tau, int32_t* token_dev, float* gap_dev,
                            float* logits_dev, int32_t* base_token_dev,
                            float* margin_dev, cudaStream_t stream);

/* Seeded sampling ("TandemLLM docs, 12 Exactness", 12.5; "Inference and
 * Decoding", section 3): the token of row n is an exact sample of
 * softmax(z_n / T), drawn as the argmax over v of z[n, v] / T + G_v with
 * Gumbel noise G keyed by (seeds[n], positions[n]) alone, so a row draws the
 * same token whatever B, its place in the batch or the other rows.
 *
 * Generator: Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy
 * as 1, 2, 3", SC'11), key = (seed low 32 bits, seed high 32 bits); entry v
 * takes word (v mod 4) of the block with counter (v div 4, t low, t high, 0);
 * word x gives U = (2 * (x >> 9) + 1) * 2^-24 in (0, 1) and G = -log(-log U).
 * Scores in fp32: z / T correctly rounded, logf, one rounded add; the lowest
 * index wins an exact tie of scores.
 *
 * Float heads only (INT8: DETLM_EUNSUPPORTED). temperature: finite and > 0
 * (the greedy call is the T -> 0 limit), else DETLM_EINVAL.
 * seeds_dev, positions_dev: uint64 [B], device, 8-byte aligned.
 * token_dev int32 [B]; score_gap_dev (may be NULL) f32 [B]: the best minus
 * the runner-up score, +inf if V == 1 (how close the draw came to another
 * token); logits_dev (may be NULL): the unperturbed fp32 logits [B, V]. */
int detlm_head_sample(detlm_head_t* head, const void* h_dev, int64_t B,
                      float temperature, const uint64_t* seeds_dev,
                      const uint64_t* positions_dev, int32_t* token_dev,
                      float* score_gap_dev, float* logits_dev,
                      cudaStream_t stream);

/* Integer front end ("Eliminating Nondeterminism in LLM Inference with
 * Integer-Only Arithmetic", section DetLLM: dyadic scales, an integer
 * multiplier and a shift with one fixed rounding rule; each token quantized
 * from its own values). Row n of x (dtype BF16, FP16 or FP32; [B, d],
 * row-major) becomes int8 q[n, :] with, from that row alone,
 *   amax = max_k |x[n, k]|, E = floor(log2 amax), S = E + 8,
 *   M = floor(127 * 2^S / amax)   (in [16256, 32512]),
 *   q = round-half-to-even(x * M / 2^S)   (in [-127, 127]; amax -> +-127),
 * all in exact integer arithmetic on the inputs' significands and
 * exponents; x ~ q * 2^S / M. An all-zero row gives q = 0, M = 0, S = 0.
 * Non-finite inputs give unspecified q (no error is raised).
 * mult_dev / shift_dev: int32 [B] receive M and S. Requirements: B >= 0,
 * 1 <= d < 2^31, x aligned to its element size. */
int detlm_quantize_rows(const void* x_dev, int dtype, int64_t B, int64_t d,
                        int8_t* q_dev, int32_t* mult_dev, int32_t* shift_dev,
                        cudaStream_t stream);

/* The int8 head fed by float rows: detlm_quantize_rows into a buffer the
 * handle owns (grown on demand; growth synchronizes the stream), then the
 * greedy call on the quantized rows. Exact int32 logits of q . W; the
 * row's dequantized logits are logits * 2^S / M (times W's own scale), so
 * the token is the same. INT8 heads only (else DETLM_EUNSUPPORTED);
 * x_dtype BF16, FP16 or FP32. mult_dev / shift_dev may be NULL. */
int detlm_head_greedy_from_float(detlm_head_t* head, const void* x_dev,
                                 int x_dtype, int64_t B, int32_t* token_dev,
                                 int32_t* gap_dev, int32_t* logits_dev,
                                 int32_t* mult_dev, int32_t* shift_dev,
                                 cudaStream_t stream);

/* Greedy speculative verify: the greedy call on n_req * P hidden rows (the P
 * verified positions of each request, request-major) that also returns the
 * accepted draft length of each request. The acceptance is folded into the
 * split-V merge kernel (no extra launch); the handle keeps 8 bytes of
 * per-request workspace, grown on demand (growth synchronizes the stream).
 *
 * "Inference and Decoding", section 6 (Speculative decoding): the target
 * scores every drafted position in one forward pass and keeps the drafted
 * tokens while they agree with it; "TandemLLM docs, 12 Exactness", 12.1: at
 * temperature 0 that is equality with the target's greedy token.
 * drafts_dev int32 [n_req, P]: the token proposed for each position.
 * accepted_dev int32 [n_req]: number of leading positions whose draft equals
 * the greedy token (0 .. P); the caller keeps those drafts and takes
 * token[r, accepted[r]] as the next token when accepted[r] < P.
 * token_dev, gap_dev, logits_dev: as in detlm_head_greedy for B = n_req * P.
 * Requirements: n_req >= 0, P >= 1, n_req * P < 2^31. */
int detlm_head_verify(detlm_head_t* head, const void* h_dev, int64_t n_req,
                      int64_t P, const int32_t* drafts_dev, int32_t* token_dev,
                      void* gap_dev, void* logits_dev, int32_t* accepted_dev,
                      cudaStream_t stream);

/* Host-buffer forms of the two calls: copy h (and targets) from host memory,
 * run the call, copy the results back, wait for the stream, and report the
 * error word. Host buffers may be pageable; pinned buffers copy faster.
 * Device staging buffers are owned by the handle and grow on demand. */
int detlm_head_greedy_host(detlm_head_t* head, const void* h_host, int64_t B,
                           int32_t* token_host, void* gap_host,
                           void* logits_host, cudaStream_t stream);
int detlm_head_logprob_host(detlm_head_t* head, const void* h_host,
                            const int32_t* targets_host, int64_t B,
                            float* logp_host, cudaStream_t stream);

/* Asynchronous forms of the two host-buffer calls, for a caller that issues
 * many calls and reads the results once: they enqueue the copy of h (and
 * targets) to the device, the call, and the copies of the results back to
 * the given host buffers, and return without waiting. Results are in the
 * host buffers after detlm_head_check returns; until then the caller keeps
 * every buffer of every pending call alive and unchanged. The kernels run on
 * `stream`. Result buffers the device can address (pinned host memory from
 * cudaHostAlloc or cudaHostRegister, which is mapped on unified-addressing
 * systems) are written by the kernels directly; otherwise the results go to
 * two alternating device slots and are copied back on a stream of the
 * handle's own, so one call's copy overlaps the next call's kernels. Copies
 * from or to pageable memory make the call wait for them. Device staging is
 * owned by the handle and grows on demand (growth waits for the pending
 * calls). */
int detlm_head_greedy_host_async(detlm_head_t* head, const void* h_host,
                                 int64_t B, int32_t* token_host, void* gap_host,
                                 void* logits_host, cudaStream_t stream);
int detlm_head_logprob_host_async(detlm_head_t* head, const void* h_host,
                                  const int32_t* targets_host, int64_t B,
                                  float* logp_host, cudaStream_t stream);

/* Wait for the stream and for the copies of the handle's pending
 * asynchronous host-buffer calls, read and clear the handle's device error
 * word. DETLM_ETIMEOUT if a kernel's bounded wait ran out (its outputs are
 * then undefined), else DETLM_ETARGET if a target id was out of range, else
 * OK. */
int detlm_head_check(detlm_head_t* head, cudaStream_t stream);

/* Record start/stop around the projection kernel of the NEXT call only (one
 * shot), for timing that kernel with CUDA events on the call's stream. */
int detlm_head_time_next(detlm_head_t* head, cudaEvent_t start,
                         cudaEvent_t stop);

/* Test hook for failure detection. flags = DETLM_DEBUG_STALL makes the next
 * calls' MMA issuer wait on a barrier nothing arrives on, so the kernel's
 * bounded wait runs out after timeout_ns and the call reports
 * DETLM_ETIMEOUT; flags = 0 restores normal operation. timeout_ns = 0 keeps
 * the default limit (2 s). */
#define DETLM_DEBUG_STALL 1
int detlm_head_debug(detlm_head_t* head, int flags, uint64_t timeout_ns);

/* Shape queries: number of 128-row vocabulary tiles, and the column tile
 * (padded rows of h per MMA) a call with B rows uses. */
int detlm_head_tiles(const detlm_head_t* head, int64_t B, int32_t* n_vtiles,
                     int32_t* n_cols);

/* ------------------------------------------------------------------------
 * Vocabulary-parallel heads: W split by rows over P devices (or P heads on
 * one device), one 16-byte record per hidden row exchanged between them.
 *
 * "TandemLLM docs, 12 Exactness", section 12.2: the head's reduction order is
 * fixed by the weight's shape, never by the row count; here it is also fixed
 * independently of P. The greedy records merge exactly (value desc, index
 * asc), and the log-sum-exp tree of detlm_head_logprob (128 leaves of
 * contiguous 256-entry tiles, folded in ascending order, combined in a
 * balanced binary tree) is cut on leaf boundaries, so shards + merge give the
 * single head's token, gap and log-probability bit for bit for P = 1, 2, 4,
 * ..., 128.
 *
 * A caller on P devices: each rank r creates its shard over its own rows
 * W[v_begin:v_end] (detlm_shard_range), runs the *_shard call on the same
 * hidden rows, all-gathers the B records of every rank in rank order into
 * recs [P][B] (a P * B * 16-byte exchange instead of B * V logits), and runs
 * the merge call (every rank gets the same result).
 * ------------------------------------------------------------------------ */

/* One hidden row's record from one shard (16 bytes, 16-byte aligned arrays).
 *   greedy, BF16/FP16 head: m = the shard's best logit, i = the lowest global
 *     vocabulary index attaining it, s = the runner-up value (s == m on a tie);
 *   greedy, INT8 head: the same, with m and s int32 (m_i32, s_i32);
 *   log-prob: m = the shard's largest logit, s = sum over the shard of
 *     exp(z - m) (the root of the shard's subtree of the log-sum-exp tree),
 *     i = 1 when the row's target lies in the shard (then zt is its logit),
 *     else 0. */
typedef struct {
  union { float m; int32_t m_i32; };
  int32_t i;
  union { float s; int32_t s_i32; };
  float zt;
} detlm_shard_rec_t;

/* Rows [*v_begin, *v_end) of a vocabulary of V that shard `rank` of P holds:
 * with n = ceil(V / 256), the 256-entry tiles [floor(rank n / P),
 * floor((rank + 1) n / P)) (the last clipped at V). P: a power of two,
 * 1 <= P <= 128; 0 <= rank < P. A host computation (no GPU needed). A shard
 * is empty when n < P; such a split is refused by detlm_head_create_shard. */
int detlm_shard_range(int64_t V, int P, int rank, int64_t* v_begin,
                      int64_t* v_end);

/* A head over one shard: W_shard_dev [v_end - v_begin, d] holds rows
 * [v_begin, v_end) of the full W (borrowed, as in detlm_head_create; same
 * dtype and alignment rules). V is the full vocabulary. The shard head
 * serves the *_shard calls only (the whole-head calls return
 * DETLM_EUNSUPPORTED); detlm_head_reserve, detlm_head_check,
 * detlm_head_time_next, detlm_head_debug and detlm_head_destroy apply. */
int detlm_head_create_shard(detlm_head_t** out, const void* W_shard_dev,
                            int64_t V, int64_t d, int dtype, int P, int rank);

/* Greedy records of this shard for B hidden rows h_dev [B, d]:
 * rec_dev [B] (device, 16-byte aligned). logits_dev (NULL to skip): the
 * shard's fp32 (int32 for INT8) logits [B, v_end - v_begin], columns in the
 * shard's own order. */
int detlm_head_greedy_shard(detlm_head_t* head, const void* h_dev, int64_t B,
                            detlm_shard_rec_t* rec_dev, void* logits_dev,
                            cudaStream_t stream);

/* Log-prob records of this shard (BF16/FP16 heads; INT8: DETLM_EUNSUPPORTED).
 * targets_dev int32 [B]: global vocabulary ids. rec_dev [B]. */
int detlm_head_logprob_shard(detlm_head_t* head, const void* h_dev,
                             const int32_t* targets_dev, int64_t B,
                             detlm_shard_rec_t* rec_dev, cudaStream_t stream);

/* Token and gap from the P shards' greedy records recs_dev [P][B] (shard
 * r's B records at recs_dev + r * B). dtype: the heads' dtype. token_dev
 * int32 [B]; gap_dev float [B] in bf16 ulps (INT8: int32 [B], m - s), as
 * detlm_head_greedy returns them. No handle: the call allocates nothing. */
int detlm_merge_greedy_shards(const detlm_shard_rec_t* recs_dev, int P,
                              int64_t B, int dtype, int32_t* token_dev,
                              void* gap_dev, cudaStream_t stream);

/* Log-probabilities from the P shards' log-prob records recs_dev [P][B]:
 * logp = zt - (M + log S) with (M, S) the balanced-tree merge of the shards'
 * (m, s), zt from the shard holding the target. V: the full vocabulary. A
 * target outside [0, V) gives NaN and, when err_dev is not NULL, sets
 * DETLM_ETARGET's bit (2) in *err_dev. */
int detlm_merge_logprob_shards(const detlm_shard_rec_t* recs_dev, int P,
                               int64_t B, int64_t V, const int32_t* targets_dev,
                               float* logp_dev, int* err_dev,
                               cudaStream_t stream);

/* Greedy call that allocates no device memory at all (no counterpart in the
 * source pages; this is a deployment convenience).
 *
 * Meant for callers that may not call cudaMalloc or any other allocator:
 * code living inside a framework that has already reserved all of the GPU's
 * memory for itself (an inference server that pre-reserves HBM for its KV
 * cache), plugin interfaces whose execute step must not allocate, and hot
 * paths that cannot afford the device-wide synchronisation an allocation
 * implies. It needs no handle: pass the weight directly.
 *
 * Same computation and outputs as detlm_head_greedy on a BF16 or FP16 head
 * (same kernels, bit-identical results); INT8 returns DETLM_EUNSUPPORTED.
 * The split-V records live in one static device array of
 * DETLM_NOALLOC_SCRATCH_BYTES bytes, compiled into this library: every GPU
 * that loads the library holds it until the process exits. A call needs
 * 256 + 3 * 4 * ceil(V / 128) * B bytes of it (rounded up to 256-byte
 * parts); larger B returns DETLM_EINVAL before any GPU work.
 * err_dev: optional int on the device, set to 0 by the call and then to a
 * non-zero error bit if a bounded wait in the kernel ran out (the outputs
 * are then undefined). NULL: the error word lives in the static array and is
 * not reported.
 * The first call on each device looks up the array's device address with
 * that device current (a one-time runtime query, no allocation; repeated
 * once after a device reset, which gives the device a new context); make
 * that first call before capturing any stream. All calls share the array and it
 * keeps the last call's contents (each call clears what must start at zero):
 * calls that may run at the same time on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller. */
#define DETLM_NOALLOC_SCRATCH_BYTES (8u << 20)
int detlm_greedy_noalloc(const void* W_dev, int64_t V, int64_t d, int dtype,
                         const void* h_dev, int64_t B, int32_t* token_dev,
                         float* gap_dev, float* logits_dev, int* err_dev,
                         cudaStream_t stream);

/* Release the handle: waits for the device (the handle's work may still run
 * on any stream), then frees everything the handle owns. W is not freed. */
void detlm_head_destroy(detlm_head_t* head);

const char* detlm_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* DETLM_HEAD_H */
