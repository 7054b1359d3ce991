/*
 * sv_lm_head.h - the LM head in front of verification (part of libsv.so).
 *
 * llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
 * section 21: the verified positions' logits are their hidden states times
 * the vocabulary projection, computed for every position of a verification
 * batch at once; section 22: greedy verification needs each row's argmax,
 * sampled verification the whole distribution.  TensorSharp
 * speculative_decoding.md, "DFlash and DFlash2": the drafter borrows the
 * target's LM head, so target and draft positions use one projection W.
 *
 * The product is a dense contraction (2 * rows * V * d FLOP on a V x d
 * projection), so it runs on the tensor cores: bf16 operands staged by TMA,
 * fp32 accumulators in tensor memory.  The conventions of sv.h apply
 * (device pointers owned by the caller, stream-ordered, no host sync,
 * host-detectable errors as sv_status with sv_last_error()).
 *
 * Layouts (all row-major, bf16 = 16-bit bfloat16):
 *   states  [rows, dim] bf16, consecutive rows `dim` elements apart;
 *   proj    [vocab, dim] bf16, row v = token v's output embedding;
 *   logits  [rows, ld] f32, ld >= vocab.
 * Requirements: dim a multiple of 8 (16-byte rows), every base pointer
 * 16-byte aligned, ld a multiple of 4; otherwise SV_ERR_ARG.
 */
#ifndef SV_LM_HEAD_H
#define SV_LM_HEAD_H

#include <stddef.h>
#include <stdint.h>

#include "sv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * logits = states . proj^T in fp32 (one launch).  `err`, optional device
 * word: bit 0 is OR-ed in if a bounded device wait of the kernel gave up
 * (the logits are then invalid); the caller zeroes it.
 * llmstudio.ru section 21 (logits of all verified positions in one product).
 */
sv_status sv_lm_head_logits(const void* states, const void* proj, int32_t rows, int32_t vocab,
                            int32_t dim, float* logits, int64_t ld, uint32_t* err, void* stream);

/*
 * Bytes of workspace sv_lm_head_verify needs: 256 bytes of flags, then the
 * fp32 logits of the sum_k + batch target rows and the sum_k draft rows,
 * rows ldv = vocab rounded up to a multiple of 4 apart.
 */
size_t sv_lm_head_workspace_size(int32_t batch, int32_t sum_k, int32_t vocab);

/*
 * Verification from hidden states: the target and draft rows' logits through
 * the one projection, then the mixed greedy / sampled verification of
 * sv_accept_from_logits on them (per-sequence temperature, 0 = greedy).
 *   target_states [sum_k + batch, dim] bf16 (sequence b: rows cu_k[b] + b ..
 *                 cu_k[b+1] + b, as the target rows of sv.h);
 *   draft_states  [sum_k, dim] bf16 (sequence b: rows cu_k[b] .. cu_k[b+1] - 1);
 *   temperature, draft_tokens, uniforms, cu_k, batch, k, sum_k, outputs and
 *   flags as sv_accept_from_logits (include/sv.h);
 *   workspace     device buffer of sv_lm_head_workspace_size() bytes,
 *                 16-byte aligned, no initial contents needed; after the call
 *                 (once the stream reaches it) it holds the logits the
 *                 verification read: target rows at byte offset 256, draft
 *                 rows after them, each ldv floats.  Calls that share a
 *                 workspace must not overlap on the GPU.
 * Enqueues a 4-byte memset of the workspace flags and two kernel launches
 * (the product, then the verification).  A bounded wait that gave up in the
 * product marks every sequence SV_SEQ_TIMEOUT with n = 0, next_token = -1.
 */
sv_status sv_lm_head_verify(const void* target_states, const void* draft_states, const void* proj,
                            int32_t dim, const float* temperature, const int32_t* draft_tokens,
                            const float* uniforms, const int32_t* cu_k, int32_t batch, int32_t k,
                            int32_t sum_k, int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                            uint32_t* status, void* workspace, size_t workspace_bytes, uint32_t flags,
                            void* stream);

/*
 * sv_lm_head_verify without a workspace: the library's own scratch, a device
 * array of SV_STATIC_SCRATCH_BYTES reserved once per device when libsv.so's
 * module loads there, takes the workspace's place.  The pages have no
 * counterpart to this call; it is this library's, for callers that cannot
 * allocate device memory per call or keep a workspace: code that runs where
 * no allocator is reachable (a plugin whose host framework owns every
 * allocation) or that must not call cudaMalloc on the decode path (it
 * synchronises the device).
 *   Arguments, results and launches as sv_lm_head_verify (no workspace
 *   arguments).  A call whose sv_lm_head_workspace_size() exceeds
 *   SV_STATIC_SCRATCH_BYTES returns SV_ERR_UNSUPPORTED and enqueues nothing
 *   (64 MiB hold, for example, B = 8, K = 5 at V = 128256).
 *   Every call on a device uses the same scratch: calls that overlap on the
 *   GPU (different streams, or different host threads with no ordering
 *   between them) race on it and their results are undefined.  Issue them on
 *   one stream.
 *   The first call on each device looks up the scratch's address (a host-side
 *   runtime query); make that first call before any stream capture.
 */
#define SV_STATIC_SCRATCH_BYTES (64u << 20)
sv_status sv_lm_head_verify_static(const void* target_states, const void* draft_states, const void* proj,
                                   int32_t dim, const float* temperature, const int32_t* draft_tokens,
                                   const float* uniforms, const int32_t* cu_k, int32_t batch, int32_t k,
                                   int32_t sum_k, int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                   uint32_t* status, uint32_t flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_LM_HEAD_H */
