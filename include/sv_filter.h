/*
 * sv_filter.h - top-k / top-p sampler filters of libsv.so, applied alike to
 * the target's and the draft's rows before verification.
 *
 * llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
 * section 38: the sampling pipeline turns raw logits into the effective
 * distribution in the order penalties, temperature, top-k, top-p, other
 * filters, normalisation, and speculative sampling compares the target's and
 * the draft's distributions after that pipeline.  So a sampled sequence's
 * filters cut every target row and every draft row the same way.
 *
 * Both filters keep {v : l_v >= floor} for one logit floor per row, so the
 * work splits into two calls:
 *   sv_sampler_floors              one kernel: the floor of every row;
 *   sv_accept_from_logits_floored  the verification of sv.h's
 *                                  sv_accept_from_logits with the floors
 *                                  applied (weight 0 below the floor) in every
 *                                  pass: the masses, p(t) and q(t), the
 *                                  residual and bonus draws, and the warped
 *                                  rows it may write.
 *
 * Definitions (per sequence b with temperature T_b > 0; greedy sequences,
 * T_b = 0, get floor -inf and are unaffected):
 *   top-k: keep every token whose logit is >= the k-th largest logit of the
 *     row (ties at the boundary all kept); k <= 0, or k >= the row's non-NaN
 *     count, keeps everything.
 *   top-p: on the tokens top-k kept, with weights w_v = 2^((l_v - m) log2(e)/T)
 *     (m the row maximum), keep token v iff the weight of the kept tokens with
 *     a strictly larger logit is < p * (their total weight): the smallest prefix
 *     of the ranking whose mass reaches p, equal logits kept or dropped
 *     together.  p >= 1 keeps everything; p NaN or <= 0 is invalid.
 *   The floor is the lowest kept logit (exact: a value of the row).  NaN
 *   logits take no part in the ranking; a row whose maximum is +Inf, NaN-only
 *   or -Inf gets floor -inf (the verification reports it).
 * Arithmetic of top-p.  The weights are those the verification kernel uses
 *   (fp32, the same exponent); each is truncated to a multiple of 2^-40 and
 *   summed as a 64-bit integer, so the sums are exact and independent of
 *   order; the boundary test compares them in fp64.  The kept set can
 *   therefore differ from an exact-arithmetic one only where the mass above
 *   a logit is within about 1e-6 of p times the total.
 *
 * Conventions are those of sv.h: DEVICE pointers owned by the caller, one
 * kernel launch per call on `stream` (a cudaStream_t, NULL = legacy default),
 * no synchronisation, host-detectable errors return SV_ERR_* with a message
 * in sv_last_error().
 */
#ifndef SV_FILTER_H
#define SV_FILTER_H

#include <stdint.h>

#include "sv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Floors of every target row and every draft row.
 *   target_logits [sum(K_b + 1), V], draft_logits [sum K_b, V] in `dtype`,
 *     rows `row_stride` elements apart, laid out as for sv_accept_from_logits
 *     (cu_k NULL: K_b = k for every sequence; else the exclusive prefix sum
 *     [batch + 1] with sum_k = cu_k[batch]).
 *   temperature [batch] f32; top_k [batch] int32 (NULL: no top-k);
 *   top_p [batch] f32 (NULL: no top-p).
 * Outputs: floor_target [sum(K_b + 1)] and floor_draft [sum K_b] f32 (either may
 * be NULL to skip those rows).  A sequence with an invalid top-p gets NaN
 * floors, which sv_accept_from_logits_floored reports as SV_SEQ_BAD_VALUE; a
 * sequence with a bad temperature or ragged offsets gets -inf floors (the
 * verification reports those itself).  Errors: SV_ERR_ARG for a bad dtype,
 * shape, stride or NULL required pointer (as sv_accept_from_logits checks them);
 * SV_ERR_CUDA for a launch failure.  With batch = 0, or with both top_k and
 * top_p NULL, nothing is launched and the floors are not written. */
sv_status sv_sampler_floors(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                            int64_t row_stride, const float* temperature, const int32_t* top_k,
                            const float* top_p, const int32_t* cu_k, int32_t batch, int32_t k,
                            int32_t sum_k, int32_t vocab, float* floor_target, float* floor_draft,
                            void* stream);

/* sv_accept_from_logits (sv.h, same arguments and results) with per-row
 * floors: a logit below its row's floor has weight 0 everywhere.
 * floor_target [sum(K_b + 1)] and floor_draft [sum K_b] f32, either NULL for no
 * floor on those rows; -inf is no floor.  A NaN floor on a row the walk reads
 * is SV_SEQ_BAD_VALUE at that row (next_token -1).  Greedy sequences ignore
 * the floors (the argmax is always kept). */
sv_status sv_accept_from_logits_floored(const void* target_logits, const void* draft_logits,
                                        sv_dtype dtype, int64_t row_stride, const float* temperature,
                                        const int32_t* draft_tokens, const float* uniforms,
                                        const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                        int32_t vocab, const float* floor_target,
                                        const float* floor_draft, int32_t* n_accepted,
                                        int32_t* next_token, uint32_t* status,
                                        float* warped_target_out, float* warped_draft_out,
                                        uint32_t flags, void* stream);

/* The filtered verification in one call: sv_sampler_floors and then
 * sv_accept_from_logits_floored on the same arguments, with the floors held
 * in the library's own scratch (results identical to those two calls, up to
 * the draws' boundary band and the SV_SEQ_EXACT_PATH / SV_SEQ_NEAR_BOUNDARY
 * bits).  top_k / top_p as sv_sampler_floors (both NULL: sv_accept_from_logits).
 * For 16-bit logits with top_k set, a fused plan decides every sequence
 * whose top-k is in [1, 64] and whose kept tokens its per-CTA candidate lists
 * hold (the keys at or above each row slice's k-th largest contain every key
 * the filters keep), without a floors pass over the rows; the floors kernel
 * and the floored verification then run for the remaining sequences only.
 * The library takes it for every such batch whose rows are long enough to
 * hold its candidate lists in their slices' shared memory (about 3700
 * logits); SV_FLAG_PLAN_CHAIN refuses it (the two steps on every sequence)
 * and SV_FLAG_PLAN_ROWS is accepted.  Up to
 * three kernel launches on `stream`; the scratch is one slot per stream (a
 * stream beyond the library's four slots gets SV_ERR_UNSUPPORTED), so calls
 * on one stream are ordered and calls on different streams do not share it. */
sv_status sv_accept_from_logits_filtered(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                                         int64_t row_stride, const float* temperature, const int32_t* top_k,
                                         const float* top_p, const int32_t* draft_tokens, const float* uniforms,
                                         const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                         int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                         uint32_t* status, uint32_t flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_FILTER_H */
