/*
 * sv_gate.h - the draft-length gate of libsv.so: how many of the drafted
 * tokens each sequence submits to verification (the source of the ragged
 * cu_k that sv_accept / sv_accept_from_logits / sv_verify_greedy take), and
 * the online calibration it learns from verified rounds.
 *
 * PocketLLM docs/dspark.md, the draft-length gate section: the drafter emits
 * a confidence per drafted position; a calibration table gives P(draft token
 * matches | confidence bucket) = p; a round that submits n drafts yields
 *     E(n) = 1 + sum_{i<n} prod_{j<=i} p_j      expected tokens, and costs
 *     cost(0) = plain_ms,  cost(n) = draft_ms + verify_base_ms + verify_slope_ms * n,
 * and the gate takes n* = argmax E(n)/cost(n) only when E(n*)/cost(n*) >=
 * margin * E(K_b)/cost(K_b) (else the full draft K_b), never fewer than
 * min_draft drafts, and n = 0 when the committed token's logit margin
 * (top1 - top2) is below margin_threshold (> 0 enables that pre-draft skip).
 * The table is learned online: a round that submitted K_b drafts of which n
 * were accepted records a hit for positions 0..n-1 and a miss at position n
 * when n < K_b (later positions are censored, never recorded); counts decay
 * by `decay` per round before the new ones are added.
 *
 * Conventions are those of sv.h: every array is a DEVICE pointer owned by the
 * caller; each call enqueues exactly one kernel on `stream` (a cudaStream_t,
 * NULL = legacy default) and does not synchronise; host-detectable errors
 * return SV_ERR_* with a message in sv_last_error().
 *
 * Buckets.  n_buckets (1..32) half-open intervals of the confidence,
 *   [edges[i-1], edges[i]), with edges[-1] = -inf and edges[n_buckets-1] = +inf;
 *   `edges` holds the n_buckets - 1 increasing inner edges (f32).  A NaN
 *   confidence falls in bucket 0.  hits[k] / total[k] (f64) are bucket k's
 *   decayed counts; a bucket with total 0 has p = 1 (a cold gate keeps the
 *   full draft).
 * Arithmetic.  The rule above is defined on exact values (p = hits / total,
 *   the double parameters as given).  The kernel evaluates it in fp32, one
 *   rounding per operation: p as an fp64 quotient rounded to fp32, the
 *   parameters rounded to fp32 once, E by running product and sum, cost as
 *   (draft_ms + verify_base_ms) + verify_slope_ms * n, the ratio E / cost, the
 *   margin test against margin * ratio(K_b), ties to the smaller n.  Each
 *   ratio is then within (3n + 6) * 2^-24 of its exact value, so the chosen n
 *   is the exact rule's except where two compared quantities lie within
 *   those bounds of each other (near-ties, where either choice is within the
 *   fp32 evaluation's rounding).  The counts stay fp64.
 */
#ifndef SV_GATE_H
#define SV_GATE_H

#include <stdint.h>

#include "sv.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SV_GATE_MAX_K 64        /* drafted positions per sequence */
#define SV_GATE_MAX_BUCKETS 32

typedef struct {
  double margin;           /* truncation must win by this factor (>= 0; the page: 1.15) */
  double draft_ms;         /* cost of drafting (>= 0; 196) */
  double verify_base_ms;   /* fixed cost of a verify (>= 0; 300) */
  double verify_slope_ms;  /* per-token cost of a verify (>= 0; 109) */
  double plain_ms;         /* one plain decode step (> 0; 303) */
  float margin_threshold;  /* pre-draft skip below this logit margin; <= 0 disables (0) */
  int32_t min_draft;       /* never fewer drafts than this, capped at K_b (>= 0; 0) */
} sv_gate_params;

/* Per-sequence submitted draft lengths and their exclusive prefix sum.
 *   confidence   [B, K] f32, row b = sequence b's drafted positions 0..K-1
 *   k_drafted    [B] int32, drafts made for b (NULL: all K); clamped to [0, K]
 *   logit_margin [B] f32, committed-token top1 - top2 logit (NULL: no skip)
 *   edges [n_buckets-1] f32; hits, total [n_buckets] f64 (read only)
 *   params       HOST pointer, checked on the host
 * Outputs: n_out [B] int32 in [0, K_b]; cu_k_out [B+1] int32 with cu_k_out[0] = 0
 * and cu_k_out[b+1] = cu_k_out[b] + n_out[b] (ready for the verify calls; the
 * caller compacts its draft tokens accordingly).  B may be 0 (cu_k_out[0] is
 * still written).  Errors: SV_ERR_ARG for B < 0, K outside [0, SV_GATE_MAX_K],
 * n_buckets outside [1, SV_GATE_MAX_BUCKETS], a NULL required pointer, or
 * params outside the ranges above (B*K must fit int32); SV_ERR_CUDA for a
 * launch failure. */
sv_status sv_gate_draft_lengths(const float* confidence, const int32_t* k_drafted,
                                const float* logit_margin, const float* edges,
                                const double* hits, const double* total, int n_buckets, int B,
                                int K, const sv_gate_params* params, int32_t* n_out,
                                int32_t* cu_k_out, void* stream);

/* One round of calibration, in place on hits / total:
 *   hits[k]  <- decay * hits[k]  + (hits recorded in bucket k this round)
 *   total[k] <- decay * total[k] + (hits and misses recorded in bucket k)
 * with, for each sequence b, n_submitted[b] (clamped to [0, K]) the drafts it
 * submitted and n_accepted[b] (clamped to [0, n_submitted[b]]) the accepted
 * prefix: positions 0..n_accepted[b]-1 are hits, position n_accepted[b] is a
 * miss when n_accepted[b] < n_submitted[b].  decay in [0, 1].  Same errors
 * as above. */
sv_status sv_gate_update(const float* confidence, const int32_t* n_submitted,
                         const int32_t* n_accepted, const float* edges, double* hits,
                         double* total, int n_buckets, int B, int K, double decay,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_GATE_H */
