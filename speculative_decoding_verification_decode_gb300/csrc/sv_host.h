// Host helpers shared by the library's translation units (not part of the ABI).
#pragma once
#include "../../include/sv.h"

namespace svh {

// Records a printf-style message for sv_last_error() and returns `s`.
sv_status fail(sv_status s, const char* fmt, ...);
// Clears the message at the start of an entry point.
void clear_error();

// sv_accept_from_logits (with the optional sampler-filter floors of
// sv_filter.h), plus `ext_err`: a device word that, when nonzero at the
// kernel's start, marks every sequence SV_SEQ_TIMEOUT (the kernel that wrote
// the rows gave up); NULL for none.
sv_status accept_logits(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                        int64_t row_stride, const float* temperature, const int32_t* draft_tokens,
                        const float* uniforms, const int32_t* cu_k, int32_t batch, int32_t k,
                        int32_t sum_k, int32_t vocab, const float* floor_target,
                        const float* floor_draft, int32_t* n_accepted, int32_t* next_token,
                        uint32_t* status, float* warped_target_out, float* warped_draft_out,
                        const uint32_t* ext_err, uint32_t flags, void* stream);

}  // namespace svh
