// sv_lm_head_verify_static: verification from hidden states with the
// library's own fixed scratch instead of a caller workspace.
//
// For callers that cannot hand the library device memory per call: code that
// runs where no allocator is reachable (a plugin whose host framework owns
// every allocation, a decode loop that must not call cudaMalloc because it
// synchronises the device), or that cannot keep a workspace alive between
// calls.  The scratch is a file-scope device array, reserved once when the
// library's module is loaded on a device; no call allocates anything.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sv_lm_head.h"
#include "sv_host.h"

namespace {

// The scratch every call on a device uses (logits of the verified rows and
// the product's error word, laid out as sv_lm_head_verify's workspace).
static __device__ __align__(256) unsigned char g_scratch[SV_STATIC_SCRATCH_BYTES];

std::mutex g_lookup_mutex;
void* g_scratch_addr[64] = {nullptr};

// Address of g_scratch on the current device, looked up once per device
// (with that device current); a non-OK status with sv_last_error() set on
// failure.
sv_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64)
    return svh::fail(SV_ERR_UNSUPPORTED, "device index %d beyond the 64 this library tracks", dev);
  std::lock_guard<std::mutex> lock(g_lookup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return svh::fail(SV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_lm_head_verify_static(const void* target_states, const void* draft_states,
                                              const void* proj, int32_t dim, const float* temperature,
                                              const int32_t* draft_tokens, const float* uniforms,
                                              const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                              int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                              uint32_t* status, uint32_t flags, void* stream) {
  svh::clear_error();
  if (batch < 0 || sum_k < 0 || vocab < 1) return svh::fail(SV_ERR_ARG, "size out of range");
  const size_t need = sv_lm_head_workspace_size(batch, sum_k, vocab);
  if (need > static_cast<size_t>(SV_STATIC_SCRATCH_BYTES))
    return svh::fail(SV_ERR_UNSUPPORTED,
                     "the call needs %zu bytes of scratch; the static scratch holds %zu (use sv_lm_head_verify "
                     "with a workspace)",
                     need, static_cast<size_t>(SV_STATIC_SCRATCH_BYTES));
  if (batch == 0) return SV_OK;
  void* scratch = nullptr;
  const sv_status s = scratch_address(&scratch);
  if (s != SV_OK) return s;
  // the workspace entry point zeroes the error word it needs and checks
  // every other argument
  return sv_lm_head_verify(target_states, draft_states, proj, dim, temperature, draft_tokens, uniforms, cu_k,
                           batch, k, sum_k, vocab, n_accepted, next_token, status, scratch,
                           static_cast<size_t>(SV_STATIC_SCRATCH_BYTES), flags, stream);
}
