/*
 * sv_penalties.h - repetition, frequency and presence penalties ahead of
 * verification (part of libsv.so).
 *
 * llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
 * section 38: the sampling pipeline applies penalties to the raw logits
 * before the temperature and the top-k / top-p filters, for the target's p
 * and alike for the draft's q, and speculative sampling verifies those
 * effective distributions.  Section 39: a stateful sampler keeps the
 * guarantee only when its state follows the speculative branch; here the
 * state that scores row i of a sequence is its history plus the drafted
 * tokens t_0..t_{i-1} that row i assumes accepted.
 *
 * The call rewrites, in place, only the logits of tokens the state has seen
 * (at most history + K_b ids per row): call it on the raw rows, then
 * sv_accept_from_logits / sv_sampler_floors on the same rows.
 *
 * Per touched logit x, with c = occurrences of the token in the history and
 * in t_0..t_{i-1} (c > 0): in f32, one rounding per operation,
 *   x = x < 0 ? x * repetition : x / repetition;
 *   x = x - frequency * c;
 *   x = x - presence;
 * then rounded to the row's storage type (nearest, ties to even).
 * repetition = 1, frequency = 0, presence = 0 leave a sequence untouched.
 */
#ifndef SV_PENALTIES_H
#define SV_PENALTIES_H

#include <stdint.h>

#include "sv.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SV_PENALTY_MAX_DISTINCT 8192 /* distinct token ids per sequence (history + drafts) */
#define SV_PENALTY_MAX_K 1024        /* largest K_b */

/*
 * target_logits, draft_logits: the rows of sv_accept_from_logits (same layout,
 *   `row_stride` elements apart, `dtype`), modified in place.
 * hist_offsets [batch + 1], hist_tokens [hist_total]: sequence b's history
 *   is hist_tokens[hist_offsets[b] .. hist_offsets[b+1]); both NULL (and
 *   hist_total 0) for no history.  Ids outside [0, vocab) are skipped;
 *   offsets outside [0, hist_total] are the sequence's SV_SEQ_BAD_LAYOUT.
 * draft_tokens, cu_k, batch, k, sum_k, vocab: as the verification calls.
 * repetition, frequency, presence [batch]: per-sequence parameters.
 * status [batch] out: 0, or SV_SEQ_BAD_LAYOUT (offsets out of range, or more
 *   than SV_PENALTY_MAX_DISTINCT distinct ids), or SV_SEQ_BAD_VALUE
 *   (repetition not a positive finite number, frequency or presence not
 *   finite); the rows of such a sequence are left as they are.
 * One launch on `stream` (one CTA per sequence); k <= SV_PENALTY_MAX_K.
 */
sv_status sv_apply_penalties(void* target_logits, void* draft_logits, sv_dtype dtype, int64_t row_stride,
                             const int32_t* hist_offsets, const int32_t* hist_tokens, int32_t hist_total,
                             const int32_t* draft_tokens, const int32_t* cu_k, int32_t batch, int32_t k,
                             int32_t sum_k, int32_t vocab, const float* repetition, const float* frequency,
                             const float* presence, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_PENALTIES_H */
