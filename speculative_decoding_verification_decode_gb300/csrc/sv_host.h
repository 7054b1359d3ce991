// Host helpers shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda_runtime.h>

#include "../../include/sv.h"

namespace svk {
struct Params;
}

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
                        const uint32_t* ext_err, uint32_t flags, void* stream, const int* gate = nullptr);

// sv_sampler_floors with a per-sequence gate (device int [batch]; 0 skips the
// sequence, NULL computes every one).
sv_status sampler_floors_gated(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                               int64_t row_stride, const float* temperature, const int32_t* top_k,
                               const float* top_p, const int32_t* cu_k, int32_t batch, int32_t k,
                               int32_t sum_k, int32_t vocab, float* floor_target, float* floor_draft,
                               const int* gate, void* stream);

// The row-parallel plan (sv_rows.cu): the cluster size it would launch a
// call of this shape with (0: the shape cannot take it), and its launch
// (SV_ERR_UNSUPPORTED when no scratch slot is free for the stream, or the
// shape does not fit; the caller then takes the chain plan).  `p` carries the
// call's arguments as the chain kernel's parameters do.
int rows_cluster_size(int mode, int elem, const svk::Params& p);
sv_status launch_rows(int mode, sv_dtype dtype, const svk::Params& p, bool filtered, cudaStream_t stream);

// The filtered verification's scratch on this stream (the row-parallel
// plan's slot): a per-sequence fallback flag and the floors of the target
// and draft rows.  False when no slot is free or the call is larger than one.
bool rows_filter_scratch(cudaStream_t stream, int batch, int t_rows, int** flag, float** floor_t,
                         float** floor_d);
// The fused top-k / top-p plan (16-bit logits): decides every sequence whose
// rows its candidate lists can decide and flags the rest in the slot's
// fallback flags.  SV_ERR_UNSUPPORTED when the shape cannot take it.
sv_status launch_rows_topk(sv_dtype dtype, const svk::Params& p, const int32_t* top_k, const float* top_p,
                           cudaStream_t stream);

}  // namespace svh
