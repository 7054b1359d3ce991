// Repetition / frequency / presence penalties ahead of verification
// (llmstudio.ru sections 38-39), in place on the raw logits rows.
//
// One CTA per sequence.  Its threads count the sequence's history ids in a
// shared-memory hash table (open addressing, 16384 slots, at most 8192
// distinct ids, so the load stays at or below one half), add the drafted ids
// with count 0, then walk the table: the thread owning id v rewrites v's
// logit in target row i and draft row i for every row i whose state (the
// history plus t_0..t_{i-1}) has seen v.  Only those logits are read and
// written: a few thousand elements per sequence against rows of V.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/sv_penalties.h"
#include "sv_host.h"

namespace svp {

constexpr int kThreads = 256;
constexpr int kSlots = 2 * SV_PENALTY_MAX_DISTINCT;  // power of two
constexpr int kSlotBits = 14;
static_assert((1 << kSlotBits) == kSlots, "slot count");
constexpr uint32_t ST_BAD_VALUE = 2u, ST_BAD_LAYOUT = 64u;

struct Params {
  void* tgt;
  void* drf;
  long long stride;
  const int* hoff;
  const int* htok;
  const int* tok;
  const int* cu_k;
  const float* rep;
  const float* freq;
  const float* pres;
  unsigned* st;
  int B, K, V, sum_k, htotal;
};

template <typename T>
struct Cvt;
template <>
struct Cvt<float> {
  static __device__ float load(const float* p) { return *p; }
  static __device__ void store(float* p, float v) { *p = v; }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <>
struct Cvt<__half> {
  static __device__ float load(const __half* p) { return __half2float(*p); }
  static __device__ void store(__half* p, float v) { *p = __float2half_rn(v); }
};

__device__ __forceinline__ uint32_t slot_of(int v) {
  return (static_cast<uint32_t>(v) * 2654435761u) >> (32 - kSlotBits);
}

// Inserts id v (adding `add` to its count); false when the table is full.
__device__ bool insert(int* keys, int* counts, int v, int add) {
  uint32_t s = slot_of(v);
  for (int probe = 0; probe < kSlots; ++probe, s = (s + 1) & (kSlots - 1)) {
    const int k = keys[s];
    if (k == v) {
      if (add) atomicAdd(&counts[s], add);
      return true;
    }
    if (k == -1) {
      const int prev = atomicCAS(&keys[s], -1, v);
      if (prev == -1 || prev == v) {
        if (add) atomicAdd(&counts[s], add);
        return true;
      }
    }
  }
  return false;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) penalties_kernel(Params P) {
  extern __shared__ int sh[];
  int* keys = sh;                 // kSlots
  int* counts = sh + kSlots;      // kSlots
  int* drafts = sh + 2 * kSlots;  // K
  __shared__ int s_bad, s_distinct;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;

  int kb = P.K, t0 = b * (P.K + 1), d0 = b * P.K;
  bool layout_ok = true;
  if (P.cu_k) {
    const int lo = P.cu_k[b], hi = P.cu_k[b + 1];
    if (lo < 0 || hi < lo || hi > P.sum_k || hi - lo > P.K) {
      layout_ok = false;
    } else {
      kb = hi - lo;
      t0 = lo + b;
      d0 = lo;
    }
  }
  int h0 = 0, h1 = 0;
  if (layout_ok && P.hoff) {
    h0 = P.hoff[b];
    h1 = P.hoff[b + 1];
    if (h0 < 0 || h1 < h0 || h1 > P.htotal) layout_ok = false;
  }
  if (!layout_ok) {
    if (tid == 0) P.st[b] = ST_BAD_LAYOUT;
    return;
  }
  const float r = P.rep[b], fr = P.freq[b], pr = P.pres[b];
  if (!(r > 0.f && r <= 3.402823466e38f) || !isfinite(fr) || !isfinite(pr)) {
    if (tid == 0) P.st[b] = ST_BAD_VALUE;
    return;
  }
  for (int s = tid; s < kSlots; s += kThreads) {
    keys[s] = -1;
    counts[s] = 0;
  }
  for (int i = tid; i < kb; i += kThreads) drafts[i] = P.tok[d0 + i];
  if (tid == 0) {
    s_bad = 0;
    s_distinct = 0;
  }
  __syncthreads();
  // history ids with their counts, then the drafted ids (count 0)
  bool full = false;
  for (int h = h0 + tid; h < h1; h += kThreads) {
    const int v = P.htok[h];
    if (v >= 0 && v < P.V && !insert(keys, counts, v, 1)) full = true;
  }
  for (int i = tid; i < kb; i += kThreads) {
    const int v = drafts[i];
    if (v >= 0 && v < P.V && !insert(keys, counts, v, 0)) full = true;
  }
  if (full) atomicOr(&s_bad, 1);
  __syncthreads();
  int mine = 0;
  for (int s = tid; s < kSlots; s += kThreads) mine += keys[s] != -1;
  atomicAdd(&s_distinct, mine);
  __syncthreads();
  if (s_bad || s_distinct > SV_PENALTY_MAX_DISTINCT) {
    if (tid == 0) P.st[b] = ST_BAD_LAYOUT;
    return;
  }
  if (r == 1.f && fr == 0.f && pr == 0.f) {  // neutral: the rows stay bit for bit
    if (tid == 0) P.st[b] = 0u;
    return;
  }

  T* tg = static_cast<T*>(P.tgt);
  T* dr = static_cast<T*>(P.drf);
  for (int s = tid; s < kSlots; s += kThreads) {
    const int v = keys[s];
    if (v == -1) continue;
    int c = counts[s];
    for (int i = 0; i <= kb; ++i) {
      if (i > 0 && drafts[i - 1] == v) ++c;  // row i's state has appended t_{i-1}
      if (c == 0) continue;
      const float cf = static_cast<float>(c);
      const int nrows = i < kb ? 2 : 1;
      for (int part = 0; part < nrows; ++part) {
        T* e = (part == 0 ? tg + (t0 + i) * P.stride : dr + (d0 + i) * P.stride) + v;
        float x = Cvt<T>::load(e);
        x = x < 0.f ? __fmul_rn(x, r) : __fdiv_rn(x, r);
        x = __fsub_rn(x, __fmul_rn(fr, cf));
        x = __fsub_rn(x, pr);
        Cvt<T>::store(e, x);
      }
    }
  }
  if (tid == 0) P.st[b] = 0u;
}

}  // namespace svp

extern "C" sv_status sv_apply_penalties(void* target_logits, void* draft_logits, sv_dtype dtype, int64_t row_stride,
                                        const int32_t* hist_offsets, const int32_t* hist_tokens,
                                        int32_t hist_total, const int32_t* draft_tokens, const int32_t* cu_k, int32_t batch, int32_t k,
                                        int32_t sum_k, int32_t vocab, const float* repetition,
                                        const float* frequency, const float* presence, uint32_t* status,
                                        void* stream) {
  svh::clear_error();
  if (batch < 0 || k < 0 || sum_k < 0 || vocab < 1) return svh::fail(SV_ERR_ARG, "size out of range");
  if (k > SV_PENALTY_MAX_K) return svh::fail(SV_ERR_UNSUPPORTED, "k (%d) > %d", k, SV_PENALTY_MAX_K);
  if (row_stride < vocab) return svh::fail(SV_ERR_ARG, "row_stride < vocab");
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return svh::fail(SV_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (!cu_k && static_cast<long long>(batch) * k != sum_k)
    return svh::fail(SV_ERR_ARG, "without cu_k, sum_k must equal batch * k");
  if ((hist_offsets == nullptr) != (hist_tokens == nullptr) || hist_total < 0 || (!hist_tokens && hist_total))
    return svh::fail(SV_ERR_ARG, "hist_offsets and hist_tokens are both NULL (hist_total 0) or both set");
  if (batch == 0) return SV_OK;
  if (!target_logits || (sum_k > 0 && (!draft_logits || !draft_tokens)) || !repetition || !frequency ||
      !presence || !status)
    return svh::fail(SV_ERR_ARG, "a pointer is NULL");
  svp::Params p;
  p.tgt = target_logits;
  p.drf = draft_logits;
  p.stride = row_stride;
  p.hoff = hist_offsets;
  p.htok = hist_tokens;
  p.tok = draft_tokens;
  p.cu_k = cu_k;
  p.rep = repetition;
  p.freq = frequency;
  p.pres = presence;
  p.st = status;
  p.B = batch;
  p.K = k;
  p.V = vocab;
  p.sum_k = sum_k;
  p.htotal = hist_total;
  const size_t smem = (2 * static_cast<size_t>(svp::kSlots) + k) * sizeof(int);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the shared-memory opt-in, once per (device, element type)
  static bool attr_set[64][3] = {};
  auto go = [&](void (*kern)(svp::Params)) -> sv_status {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!attr_set[dev][dtype]) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>((2 * svp::kSlots + SV_PENALTY_MAX_K) * sizeof(int)));
      if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      attr_set[dev][dtype] = true;
    }
    kern<<<static_cast<unsigned>(batch), svp::kThreads, smem, st>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return SV_OK;
  };
  switch (dtype) {
    case SV_F32: return go(svp::penalties_kernel<float>);
    case SV_BF16: return go(svp::penalties_kernel<__nv_bfloat16>);
    default: return go(svp::penalties_kernel<__half>);
  }
}
