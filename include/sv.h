/*
 * sv.h - C ABI of the GB300 speculative-decoding verification library (libsv.so).
 *
 * The verification step of speculative decoding: for each of B sequences a
 * drafter proposed K_b tokens t_0..t_{K_b-1}, and the target produced K_b + 1
 * rows over the vocabulary; row i is the target's distribution after the
 * committed prefix and t_0..t_{i-1}, so it scores t_i, and row K_b is the bonus
 * row.  Each call returns per sequence the accepted prefix length n and one
 * more token (the correction at the first rejection, or the bonus).  The
 * caller keeps t_0..t_{n-1} and appends next_token.
 *   - spec-verify model card, sections "API" and "Usage": verify_greedy(
 *     target_probs [K+1, V], draft_tokens [K]) and accept(target_probs,
 *     draft_probs [K, V], draft_tokens, generator), both returning
 *     (n_accepted, next_token).
 *   - TensorSharp speculative_decoding.md, "The shared runtime", step 2: the
 *     verify batch is [last, d1..dK]; row m's token is the correction or bonus.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every array argument is a DEVICE pointer (cudaMalloc'd, managed,
 *   or device-accessible) owned by the caller.  The library allocates nothing
 *   and keeps no state between calls.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Each call enqueues exactly one kernel launch on it and returns
 *   without synchronising; results are valid once the stream reaches that
 *   point.  Two calls may run concurrently only on distinct output buffers.
 * Layout.  Rows are row-major with `row_stride` ELEMENTS between consecutive
 *   rows (row_stride >= V).  Sequence b owns:
 *     target rows   cu_k[b] + b .. cu_k[b+1] + b      (K_b + 1 rows)
 *     draft rows    cu_k[b]     .. cu_k[b+1] - 1      (K_b rows)
 *     draft tokens  cu_k[b]     .. cu_k[b+1] - 1      (int32 ids in [0, V))
 *     uniforms      cu_k[b] + b .. cu_k[b+1] + b      (K_b + 1 floats)
 *   where K_b = cu_k[b+1] - cu_k[b].  With cu_k == NULL every K_b = K and
 *   cu_k[b] = b*K.  `sum_k` is the number of draft tokens the arrays hold
 *   (sum of K_b; B*K when cu_k is NULL): ragged offsets outside [0, sum_k] or
 *   K_b outside [0, K] are reported per sequence (SV_SEQ_BAD_LAYOUT), never
 *   read.  Draft-length gates that pick K_b per sequence are the source of the
 *   ragged layout (PocketLLM dspark.md, draft-length gate).
 * Outputs.  n_accepted[b] in [0, K_b]; next_token[b] in [0, V), or -1 when the
 *   sequence's inputs are invalid; status[b] is an OR of SV_SEQ_* bits.
 * Return value.  Host-detectable problems only (bad sizes, NULL pointers,
 *   unsupported shapes, launch failure).  On a non-OK return nothing was
 *   enqueued; sv_last_error() describes the problem.  Data-dependent problems
 *   are reported per sequence in status[b].
 * Determinism.  Results are a pure function of the inputs (no atomics decide
 *   anything; reductions have a fixed order), so repeated calls agree bit for
 *   bit.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SV_F32 = 0, SV_BF16 = 1, SV_F16 = 2 } sv_dtype;

typedef enum {
  SV_OK = 0,
  SV_ERR_ARG = 1,         /* invalid argument (NULL pointer, size out of range) */
  SV_ERR_CUDA = 2,        /* a CUDA runtime call failed (launch, attribute) */
  SV_ERR_UNSUPPORTED = 3  /* valid but unsupported shape (e.g. V too large) */
} sv_status;

/* Per-sequence status bits written to status[b]. */
#define SV_SEQ_BAD_TOKEN 1u      /* a draft id outside [0, V) was reached */
#define SV_SEQ_BAD_VALUE 2u      /* NaN/Inf/negative probability, NaN/+Inf logit,
                                    uniform outside [0,1), or bad temperature */
#define SV_SEQ_ZERO_MASS 4u      /* a needed row has zero mass (next = -1), or the
                                    residual was empty and the draw fell back to p */
#define SV_SEQ_NEAR_BOUNDARY 8u  /* the inverse-CDF draw u*R landed within 1e-5*R
                                    of a CDF step (the id may differ from another
                                    implementation's rounding) */
#define SV_SEQ_EXACT_PATH 16u    /* an accept decision needed the exact-mass path */
#define SV_SEQ_TIMEOUT 32u       /* a bounded device wait gave up; outputs invalid */
#define SV_SEQ_BAD_LAYOUT 64u    /* ragged offsets out of range (n = 0, next = -1) */

/* Flags (bit OR) accepted by every entry point. */
#define SV_FLAG_FORCE_EXACT 1u   /* decide every accept test on exact masses
                                    (testing aid; same results, slower) */
#define SV_FLAG_EXPIRE_EXCHANGE 2u /* testing aid: every wait for the records
                                    of the sequence's cluster gives up at once,
                                    as a wait on a stalled peer would, so each
                                    sequence that exchanges ends with
                                    SV_SEQ_TIMEOUT, n = 0, next_token = -1; the
                                    kernel still drains its own copies and
                                    returns normally */
#define SV_FLAG_PLAN_ROWS 4u     /* take the row-parallel plan where the shape
                                    allows it (same results; for comparisons) */
#define SV_FLAG_PLAN_CHAIN 8u    /* take the chain plan (one cluster per
                                    sequence walking its rows); wins over
                                    SV_FLAG_PLAN_ROWS */

/*
 * Greedy verification (temperature 0).
 *   spec-verify model card, section "Method", first bullet: accept t_i while it
 *   equals argmax(target_i); at the first miss emit argmax(target_i); if all
 *   K_b match emit argmax(target_{K_b}).  llmstudio.ru "Как работает
 *   speculative decoding и MTP", section 13 (left-to-right, stop at the first
 *   mismatch).
 * target: B*(K+1) (ragged: sum_k + B) rows of `dtype` (probabilities or raw
 *   logits; only the argmax is read).  Ties resolve to the lowest index.  NaN
 *   never wins (it ranks below -Inf) and sets SV_SEQ_BAD_VALUE; an all-NaN row
 *   yields index 0.  A draft id outside [0, V) counts as a mismatch and sets
 *   SV_SEQ_BAD_TOKEN.  Rows past the first mismatch are not needed (early exit).
 */
sv_status sv_verify_greedy(const void* target, sv_dtype dtype, int64_t row_stride,
                           const int32_t* draft_tokens, const int32_t* cu_k,
                           int32_t batch, int32_t k, int32_t sum_k, int32_t vocab,
                           int32_t* n_accepted, int32_t* next_token, uint32_t* status,
                           uint32_t flags, void* stream);

/*
 * Speculative (rejection) sampling from f32 probability rows.
 *   spec-verify model card, section "Method", second bullet: accept t_i with
 *   probability min(1, p_i(t_i)/q_i(t_i)); on rejection resample from
 *   norm(max(0, p_i - q_i)); if all are accepted sample the bonus from p_K;
 *   randomness enters only through explicit uniforms.  Section "Correctness":
 *   probabilities need not be normalised and masses are summed exactly.
 *   llmstudio.ru sections 15-17 (accept rule, residual), 47-48 (order).
 * target_probs: target rows; draft_probs: draft rows (same row_stride), both
 *   f32, non-negative and finite, warped identically by the caller.
 * uniforms: per sequence K_b + 1 floats in [0, 1): u_0..u_{K_b-1} drive the
 *   accept tests; u_{K_b} is the single draw for the resample or the bonus.
 * Decision: accept t_i iff  u_i * q_i(t_i) * Zp_i  <  p_i(t_i) * Zq_i  in exact
 *   real arithmetic, Z being the exact sums of the f32 rows (equivalently
 *   u_i < min(1, phat/qhat)); decisions are therefore independent of any
 *   summation order.  Draws: next = min{v : C_v > u*R} over the running sum C
 *   of the normalised residual (or of p_K), computed in 64-bit fixed point.
 * Errors stop the sequence at that row with next_token = -1: SV_SEQ_BAD_TOKEN,
 *   SV_SEQ_BAD_VALUE, SV_SEQ_ZERO_MASS (checked in that order).
 */
sv_status sv_accept(const float* target_probs, const float* draft_probs, int64_t row_stride,
                    const int32_t* draft_tokens, const float* uniforms, const int32_t* cu_k,
                    int32_t batch, int32_t k, int32_t sum_k, int32_t vocab,
                    int32_t* n_accepted, int32_t* next_token, uint32_t* status,
                    uint32_t flags, void* stream);

/*
 * Mixed greedy / sampled verification from logits with a fused softmax.
 *   llmstudio.ru section 38: p and q are the distributions after the sampling
 *   transforms (here: temperature), applied identically to target and draft;
 *   section 13 / 37: temperature 0 is greedy.  spec-verify card, "Requirements
 *   and limits": distribution preservation needs identical warping.
 * temperature[b] (f32, device): 0 selects greedy for sequence b (raw-logit
 *   argmax, draft rows unread); T > 0 warps both rows to the weights
 *   w_v = 2^((l_v - m) * log2(e)/T)  (m = row max; 16-bit inputs: one fp32
 *   subtract and multiply, f32 inputs: a double-float argument; exp2 on the
 *   special-function unit, subnormal results flushed to 0) and runs the
 *   sampling rule above on those weights with their exact masses.  NaN or +Inf
 *   logits, or a negative / NaN / infinite temperature, set SV_SEQ_BAD_VALUE;
 *   a row of all -Inf has zero mass.
 * warped_target_out / warped_draft_out (optional, may be NULL; f32, row stride
 *   V, same row numbering as the inputs): receive the weights w_v of every row
 *   the kernel warped, for testing.  Rows it did not reach are left untouched.
 */
sv_status sv_accept_from_logits(const void* target_logits, const void* draft_logits,
                                sv_dtype dtype, int64_t row_stride, const float* temperature,
                                const int32_t* draft_tokens, const float* uniforms,
                                const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                uint32_t* status, float* warped_target_out,
                                float* warped_draft_out, uint32_t flags, void* stream);

/*
 * Bytes of device workspace a verification call of this size needs.  The
 * verification calls take no workspace: the chain plan combines a sequence's
 * per-row partials (masses, maxima, argmax candidates, draw totals) inside its
 * thread-block cluster through distributed shared memory, and the
 * row-parallel plan (taken for long drafts, K >= 8) counts its per-row records
 * into the library's own static device arrays (one slot per stream, back at
 * zero when each launch ends).  The query exists so that a caller written
 * against a workspace interface sizes nothing; it returns 0 for every argument.
 *   batch  B (>= 0), k  the largest K_b, vocab  V,
 *   mode   SV_MODE_GREEDY (sv_verify_greedy), SV_MODE_PROBS (sv_accept) or
 *          SV_MODE_LOGITS (sv_accept_from_logits).
 * spec-verify model card, section "API": the verification calls of the card
 * take rows and tokens only; a batched library of this kind commonly asks the
 * caller for scratch, and this one needs none.
 */
#define SV_MODE_GREEDY 0
#define SV_MODE_PROBS 1
#define SV_MODE_LOGITS 2
size_t sv_workspace_size(int32_t batch, int32_t k, int32_t vocab, int32_t mode);

/* Static string for a status code. */
const char* sv_status_string(sv_status s);

/* Message describing the last non-OK return on the calling thread ("" if none). */
const char* sv_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
