// Host side of libsv.so: argument checks, launch planning, the C ABI.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/sv.h"
#include "../../include/sv_filter.h"
#include "sv_host.h"
#include "sv_verify.cuh"

namespace svh {

thread_local char g_err[512] = "";

sv_status fail(sv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

void clear_error() { g_err[0] = '\0'; }

}  // namespace svh

namespace {

using svh::fail;
using svh::g_err;

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

int bit_length(unsigned long long v) {
  int n = 0;
  while (v) {
    ++n;
    v >>= 1;
  }
  return n;
}

struct Plan {
  int C, slice, slot_bytes, nck, S;
  int vsum_off, tail_off;
  size_t smem;
};

constexpr size_t kSmemPerSM = 227 * 1024;  // usable shared memory per SM (bytes)
constexpr size_t kSmemTwoCtas = kSmemPerSM / 2 - 1024;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// Ring slots hold 32 KB: a CTA's bulk copies complete roughly one after
// another (about 0.3-0.4 us each whatever their size, measured on GB300), so
// the per-CTA streaming rate grows with the copy size; 16 KB copies held a
// CTA near 50 GB/s, 32 KB ones near 80 GB/s.
constexpr int kSlotBytes = 32768;
constexpr int kSampleSlots = 3;  // ring depth in sampling mode (two CTAs per SM)
constexpr int kGreedySlots = 2;  // ring depth in greedy mode
static_assert(kSlotBytes <= svk::kMaxSlotBytes, "ring slot larger than the kernel allows");

// Layout of one CTA's dynamic shared memory for a given cluster size C and
// ring depth S: [ring S x slot][draw group sums / exact buckets][SmemTail].
void layout(bool sampling, int V, int elem, int C, int ring_slots, Plan& p) {
  const int vec = 16 / elem;
  long long slice = (V + C - 1) / C;
  slice = (slice + vec - 1) / vec * vec;
  p.C = static_cast<int>((V + slice - 1) / slice);
  p.slice = static_cast<int>(slice);
  const long long slice_bytes = slice * elem;
  p.slot_bytes = static_cast<int>(slice_bytes < kSlotBytes ? round_up(slice_bytes, 16) : kSlotBytes);
  p.nck = static_cast<int>((slice_bytes + p.slot_bytes - 1) / p.slot_bytes);
  p.S = ring_slots;
  size_t ring = static_cast<size_t>(p.S) * p.slot_bytes;
  size_t vs = 0;
  if (sampling) {
    // the next row streams in as the consumers free slots of the current one
    p.S = 2 * p.nck + 1 < kSampleSlots ? 2 * p.nck + 1 : kSampleSlots;
    ring = static_cast<size_t>(p.S) * p.slot_bytes;
    // one u64 per group of kGroupVecs 16-byte vectors, or the exact-sum buckets
    const long long nvt = (slice + vec - 1) / vec;
    vs = static_cast<size_t>((nvt + svk::kGroupVecs - 1) / svk::kGroupVecs) * 8;
    if (vs < 2 * svk::kBuckets * 8) vs = 2 * svk::kBuckets * 8;
  }
  p.vsum_off = static_cast<int>(round_up(ring, 128));
  p.tail_off = static_cast<int>(round_up(p.vsum_off + vs, 128));
  p.smem = p.tail_off + sizeof(svk::SmemTail);
}

// One cluster of C CTAs per sequence: the smallest C (two CTAs still fitting
// on an SM) that gives the batch at least two CTAs per SM or, when sampling,
// brings the slice down to kSampleSliceEl elements.  A sampling sequence is a
// chain of dependent row passes, so slices past that length lengthen every
// link; smaller ones add cluster exchanges and launch more CTAs than fit at
// once (measured on GB300 at V = 32000 and V = 128256).  A batch too small to
// give half the SMs a CTA at that size keeps splitting its rows (down to
// kMinSampleSliceEl elements, up to 16 CTAs): the SMs are idle otherwise, and
// shorter slices shorten every link of its chains (measured: one sequence at
// V = 32000 f32 23.2 -> 17.1 us, eight at V = 128256 bf16 25.2 -> 21.2 us;
// sixteen at V = 128256 went from 29.3 to 35.5 us at 16 CTAs, hence the half).
constexpr long long kSampleSliceEl = 16384;
constexpr long long kMinSampleSliceEl = 2048;

bool make_plan(bool sampling, int B, int V, int elem, Plan& out) {
  const int vec = 16 / elem;
  const long long nvec = (V + vec - 1) / vec;
  const long long want = 2LL * sm_count();
  bool found = false;
  for (int C = 1; C <= svk::kMaxCluster; C *= 2) {
    if (C > 1 && C > nvec) break;
    Plan p;
    layout(sampling, V, elem, C, kGreedySlots, p);
    if (p.smem > kSmemPerSM || p.S > svk::kMaxSlots) continue;
    out = p;
    found = true;
    if (p.smem <= kSmemTwoCtas &&
        (static_cast<long long>(B) * p.C >= want ||
         (sampling && p.slice <= kSampleSliceEl &&
          (2LL * B * p.C >= sm_count() || p.slice <= kMinSampleSliceEl))))
      break;
  }
  return found;
}

// Per device and kernel: the largest dynamic shared memory opted in so far,
// whether the non-portable cluster size is allowed, and the cluster sizes
// (with their shared memory) already checked to fit.  The attribute and
// occupancy queries run once per combination instead of on every call.
struct KernelCache {
  size_t smem_set;
  bool cluster16;
  unsigned fits_mask;       // bit c: clusters of c CTAs checked at smem_fit[c]
  size_t smem_fit[svk::kMaxCluster + 1];
};

template <int MODE, typename T, bool FL>
KernelCache& kernel_cache(int dev) {
  static KernelCache cache[64] = {};
  return cache[dev >= 0 && dev < 64 ? dev : 0];
}

template <int MODE, typename T, bool FL>
sv_status launch_k(svk::Params prm, const Plan& pl, cudaStream_t stream) {
  auto kern = svk::sv_verify_kernel<MODE, T, FL>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  KernelCache& kc = kernel_cache<MODE, T, FL>(dev);
  cudaError_t e;
  if (kc.smem_set < pl.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.smem));
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "cudaFuncSetAttribute(smem): %s", cudaGetErrorString(e));
    kc.smem_set = pl.smem;
  }
  if (pl.C > 8 && !kc.cluster16) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
      return fail(SV_ERR_CUDA, "cudaFuncSetAttribute(cluster): %s", cudaGetErrorString(e));
    kc.cluster16 = true;
  }
  prm.slice = pl.slice;
  prm.slot_bytes = pl.slot_bytes;
  prm.S = pl.S;
  prm.vsum_off = pl.vsum_off;
  prm.tail_off = pl.tail_off;
  prm.look = 1;  // stream the next row while the current one is decided
  const unsigned gy = static_cast<unsigned>(prm.B < 65535 ? prm.B : 65535);
  const unsigned gz = static_cast<unsigned>((prm.B + gy - 1) / gy);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.C), gy, gz);
  cfg.blockDim = dim3(svk::threads_of(MODE), 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned bit = 1u << pl.C;
  if (!(kc.fits_mask & bit) || kc.smem_fit[pl.C] < pl.smem) {
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
    if (clusters < 1)
      return fail(SV_ERR_UNSUPPORTED, "no cluster of %d CTAs with %zu B shared memory fits", pl.C, pl.smem);
    kc.fits_mask |= bit;
    kc.smem_fit[pl.C] = pl.smem;
  }
  e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

template <int MODE, typename T>
sv_status launch(svk::Params prm, const Plan& pl, cudaStream_t stream) {
  if constexpr (MODE == svk::MODE_LOGITS) {
    if (prm.flo_t || prm.flo_d) return launch_k<MODE, T, true>(prm, pl, stream);
  }
  return launch_k<MODE, T, false>(prm, pl, stream);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sv_status check_common(const void* target, int64_t row_stride, const int32_t* tokens,
                       const int32_t* cu_k, int32_t B, int32_t K, int32_t sum_k, int32_t V,
                       const int32_t* n_out, const int32_t* next_out, const uint32_t* st_out,
                       uint32_t flags) {
  g_err[0] = '\0';
  if (B < 0) return fail(SV_ERR_ARG, "batch must be >= 0 (got %d)", B);
  if (K < 0) return fail(SV_ERR_ARG, "k must be >= 0 (got %d)", K);
  if (V < 1) return fail(SV_ERR_ARG, "vocab must be >= 1 (got %d)", V);
  if (sum_k < 0) return fail(SV_ERR_ARG, "sum_k must be >= 0 (got %d)", sum_k);
  if (row_stride < V) return fail(SV_ERR_ARG, "row_stride (%lld) < vocab (%d)", (long long)row_stride, V);
  if (!cu_k && static_cast<long long>(B) * K != sum_k)
    return fail(SV_ERR_ARG, "without cu_k, sum_k must equal batch * k (%lld), got %d",
                static_cast<long long>(B) * K, sum_k);
  if (static_cast<long long>(sum_k) + B > 0x7FFFFFFFLL)
    return fail(SV_ERR_ARG, "too many rows (sum_k + batch > 2^31 - 1)");
  if (flags & ~static_cast<uint32_t>(SV_FLAG_FORCE_EXACT | SV_FLAG_EXPIRE_EXCHANGE | SV_FLAG_PLAN_ROWS |
                                     SV_FLAG_PLAN_CHAIN))
    return fail(SV_ERR_ARG, "unknown flag bits 0x%x", flags);
  if (B == 0) return SV_OK;
  if (!target) return fail(SV_ERR_ARG, "target pointer is NULL");
  if (sum_k > 0 && !tokens) return fail(SV_ERR_ARG, "draft_tokens is NULL");
  if (!n_out || !next_out || !st_out) return fail(SV_ERR_ARG, "an output pointer is NULL");
  return SV_OK;
}

svk::Params base_params(const void* tgt, const void* drf, int64_t stride, const int32_t* tok,
                        const float* uni, const int32_t* cu_k, const float* temp, int B, int K,
                        int V, int sum_k, int32_t* n_out, int32_t* next_out, uint32_t* st_out,
                        uint32_t flags) {
  svk::Params p;
  std::memset(&p, 0, sizeof(p));
  p.tgt = tgt;
  p.drf = drf;
  p.stride = stride;
  p.tok = tok;
  p.uni = uni;
  p.cu_k = cu_k;
  p.temp = temp;
  p.B = B;
  p.K = K;
  p.V = V;
  p.sum_k = sum_k;
  p.n_out = n_out;
  p.next_out = next_out;
  p.st_out = st_out;
  p.flags = flags;
  p.fixed_shift = 62 - bit_length(static_cast<unsigned long long>(V));
  return p;
}

// The plan of a call: the row-parallel kernel (sv_rows.cuh) or the chain
// kernel (sv_verify.cuh).  The chain walks a sequence's rows one dependent
// link after another; the row-parallel plan decides every row at once but
// pays a whole item per wave of clusters.  So it takes long drafts (K >= 8,
// where accepted chains can be long) whose items fit in about two and a half
// waves of three CTAs per SM (eight CTAs per SM).  Measured on GB300
// (row-parallel against chain): sampling, K = 40 at acceptance 0.995, twelve
// sequences of V = 3001, 28 us against 521 us; K = 16, four sequences of
// V = 32000, 21 against 50 us; K = 16, eight sequences of V = 128256 bf16,
// 40 against 44 us; K = 8, sixteen of them, 46 against 48 us; greedy with
// every draft accepted, K = 40, 15 against 95 us; while B = 64, K = 5 at
// V = 128256 (3072 CTAs) takes 66 against 60 us.
bool choose_rows(uint32_t flags, int mode, int elem, const svk::Params& p) {
  if (flags & SV_FLAG_PLAN_CHAIN) return false;
  const int C = svh::rows_cluster_size(mode, elem, p);
  if (C == 0) return false;
  if (flags & SV_FLAG_PLAN_ROWS) return true;
  const long long ctas = static_cast<long long>(C) * p.B * (p.K + 1LL);
  return p.K >= 8 && ctas <= 8LL * sm_count();
}

// Launches the row-parallel plan; false (error message cleared) when it
// declined the call (no scratch slot for the stream), so the chain plan runs.
bool try_rows(int mode, sv_dtype dtype, const svk::Params& p, bool filtered, cudaStream_t st, sv_status& out) {
  out = svh::launch_rows(mode, dtype, p, filtered, st);
  if (out == SV_ERR_UNSUPPORTED) {
    g_err[0] = '\0';
    return false;
  }
  return true;
}

}  // namespace

extern "C" {

sv_status sv_verify_greedy(const void* target, sv_dtype dtype, int64_t row_stride,
                           const int32_t* draft_tokens, const int32_t* cu_k, int32_t batch,
                           int32_t k, int32_t sum_k, int32_t vocab, int32_t* n_accepted,
                           int32_t* next_token, uint32_t* status, uint32_t flags, void* stream) {
  sv_status s = check_common(target, row_stride, draft_tokens, cu_k, batch, k, sum_k, vocab,
                             n_accepted, next_token, status, flags);
  if (s != SV_OK || batch == 0) return s;
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return fail(SV_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
  const int elem = dtype == SV_F32 ? 4 : 2;
  Plan pl;
  if (!make_plan(false, batch, vocab, elem, pl)) return fail(SV_ERR_UNSUPPORTED, "vocab %d too large", vocab);
  svk::Params p = base_params(target, nullptr, row_stride, draft_tokens, nullptr, cu_k, nullptr,
                              batch, k, vocab, sum_k, n_accepted, next_token, status, flags);
  p.use_tma = aligned16(target) && (row_stride * elem) % 16 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  sv_status rs;
  if (choose_rows(flags, svk::MODE_GREEDY, elem, p) && try_rows(svk::MODE_GREEDY, dtype, p, false, st, rs)) return rs;
  switch (dtype) {
    case SV_F32: return launch<svk::MODE_GREEDY, float>(p, pl, st);
    case SV_BF16: return launch<svk::MODE_GREEDY, __nv_bfloat16>(p, pl, st);
    default: return launch<svk::MODE_GREEDY, __half>(p, pl, st);
  }
}

sv_status sv_accept(const float* target_probs, const float* draft_probs, int64_t row_stride,
                    const int32_t* draft_tokens, const float* uniforms, const int32_t* cu_k,
                    int32_t batch, int32_t k, int32_t sum_k, int32_t vocab, int32_t* n_accepted,
                    int32_t* next_token, uint32_t* status, uint32_t flags, void* stream) {
  sv_status s = check_common(target_probs, row_stride, draft_tokens, cu_k, batch, k, sum_k, vocab,
                             n_accepted, next_token, status, flags);
  if (s != SV_OK || batch == 0) return s;
  if (sum_k > 0 && !draft_probs) return fail(SV_ERR_ARG, "draft_probs is NULL");
  if (!uniforms) return fail(SV_ERR_ARG, "uniforms is NULL");
  Plan pl;
  if (!make_plan(true, batch, vocab, 4, pl))
    return fail(SV_ERR_UNSUPPORTED, "vocab %d too large", vocab);
  svk::Params p = base_params(target_probs, draft_probs, row_stride, draft_tokens, uniforms, cu_k,
                              nullptr, batch, k, vocab, sum_k, n_accepted, next_token, status, flags);
  p.use_tma = aligned16(target_probs) && (!draft_probs || aligned16(draft_probs)) &&
              (row_stride * 4) % 16 == 0;
  sv_status rs;
  if (choose_rows(flags, svk::MODE_PROBS, 4, p) &&
      try_rows(svk::MODE_PROBS, SV_F32, p, false, static_cast<cudaStream_t>(stream), rs))
    return rs;
  return launch<svk::MODE_PROBS, float>(p, pl, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

sv_status svh::accept_logits(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                             int64_t row_stride, const float* temperature, const int32_t* draft_tokens,
                             const float* uniforms, const int32_t* cu_k, int32_t batch, int32_t k,
                             int32_t sum_k, int32_t vocab, const float* floor_target,
                             const float* floor_draft, int32_t* n_accepted, int32_t* next_token,
                             uint32_t* status, float* warped_target_out, float* warped_draft_out,
                             const uint32_t* ext_err, uint32_t flags, void* stream, const int* gate) {
  sv_status s = check_common(target_logits, row_stride, draft_tokens, cu_k, batch, k, sum_k, vocab,
                             n_accepted, next_token, status, flags);
  if (s != SV_OK || batch == 0) return s;
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return fail(SV_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (sum_k > 0 && !draft_logits) return fail(SV_ERR_ARG, "draft_logits is NULL");
  if (!uniforms) return fail(SV_ERR_ARG, "uniforms is NULL");
  if (!temperature) return fail(SV_ERR_ARG, "temperature is NULL");
  const int elem = dtype == SV_F32 ? 4 : 2;
  Plan pl;
  if (!make_plan(true, batch, vocab, elem, pl))
    return fail(SV_ERR_UNSUPPORTED, "vocab %d too large", vocab);
  svk::Params p = base_params(target_logits, draft_logits, row_stride, draft_tokens, uniforms, cu_k,
                              temperature, batch, k, vocab, sum_k, n_accepted, next_token, status,
                              flags);
  p.wt_out = warped_target_out;
  p.wd_out = warped_draft_out;
  p.flo_t = floor_target;
  p.flo_d = floor_draft;
  p.ext_err = ext_err;
  p.gate = gate;
  p.use_tma = aligned16(target_logits) && (!draft_logits || aligned16(draft_logits)) &&
              (row_stride * elem) % 16 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  sv_status rs;
  if (choose_rows(flags, svk::MODE_LOGITS, elem, p) &&
      try_rows(svk::MODE_LOGITS, dtype, p, floor_target || floor_draft, st, rs))
    return rs;
  switch (dtype) {
    case SV_F32: return launch<svk::MODE_LOGITS, float>(p, pl, st);
    case SV_BF16: return launch<svk::MODE_LOGITS, __nv_bfloat16>(p, pl, st);
    default: return launch<svk::MODE_LOGITS, __half>(p, pl, st);
  }
}

extern "C" {

sv_status sv_accept_from_logits(const void* target_logits, const void* draft_logits,
                                sv_dtype dtype, int64_t row_stride, const float* temperature,
                                const int32_t* draft_tokens, const float* uniforms,
                                const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                uint32_t* status, float* warped_target_out,
                                float* warped_draft_out, uint32_t flags, void* stream) {
  return svh::accept_logits(target_logits, draft_logits, dtype, row_stride, temperature, draft_tokens,
                            uniforms, cu_k, batch, k, sum_k, vocab, nullptr, nullptr, n_accepted,
                            next_token, status, warped_target_out, warped_draft_out, nullptr, flags,
                            stream);
}

sv_status sv_accept_from_logits_floored(const void* target_logits, const void* draft_logits,
                                        sv_dtype dtype, int64_t row_stride, const float* temperature,
                                        const int32_t* draft_tokens, const float* uniforms,
                                        const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                        int32_t vocab, const float* floor_target,
                                        const float* floor_draft, int32_t* n_accepted,
                                        int32_t* next_token, uint32_t* status,
                                        float* warped_target_out, float* warped_draft_out,
                                        uint32_t flags, void* stream) {
  return svh::accept_logits(target_logits, draft_logits, dtype, row_stride, temperature, draft_tokens,
                            uniforms, cu_k, batch, k, sum_k, vocab, floor_target, floor_draft, n_accepted,
                            next_token, status, warped_target_out, warped_draft_out, nullptr, flags,
                            stream);
}

sv_status sv_accept_from_logits_filtered(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                                         int64_t row_stride, const float* temperature, const int32_t* top_k,
                                         const float* top_p, const int32_t* draft_tokens, const float* uniforms,
                                         const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k,
                                         int32_t vocab, int32_t* n_accepted, int32_t* next_token,
                                         uint32_t* status, uint32_t flags, void* stream) {
  if (!top_k && !top_p)
    return svh::accept_logits(target_logits, draft_logits, dtype, row_stride, temperature, draft_tokens, uniforms,
                              cu_k, batch, k, sum_k, vocab, nullptr, nullptr, n_accepted, next_token, status,
                              nullptr, nullptr, nullptr, flags, stream);
  // every host check of the verification and of the floors before anything is enqueued
  sv_status s = check_common(target_logits, row_stride, draft_tokens, cu_k, batch, k, sum_k, vocab, n_accepted,
                             next_token, status, flags);
  if (s != SV_OK || batch == 0) return s;
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return fail(SV_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (sum_k > 0 && !draft_logits) return fail(SV_ERR_ARG, "draft_logits is NULL");
  if (!uniforms) return fail(SV_ERR_ARG, "uniforms is NULL");
  if (!temperature) return fail(SV_ERR_ARG, "temperature is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* gate = nullptr;
  float *ft = nullptr, *fd = nullptr;
  if (!svh::rows_filter_scratch(st, batch, sum_k + batch, &gate, &ft, &fd))
    return fail(SV_ERR_UNSUPPORTED, "no scratch slot for the floors on this stream (or a call beyond one)");
  const int elem = dtype == SV_F32 ? 4 : 2;
  bool fused = false;
  // The fused plan decides the sequences its candidate lists can decide; the
  // floors and the floored verification then run for the rest only.  It is
  // taken for every 16-bit batch with top-k: measured on GB300 at V = 128256
  // bf16, top-k 50 / top-p 0.9, B = 256 K = 5 197 against 527 us, B = 64
  // K = 5 95 against 189 us, B = 16 K = 5 62 against 83 us, B = 8 K = 5 47
  // against 71 us, B = 8 K = 16 72 against 85 us, B = 1 K = 5 46 against 76
  // us (one A/B call).
  if (dtype != SV_F32 && top_k && !(flags & SV_FLAG_PLAN_CHAIN)) {
    svk::Params p = base_params(target_logits, draft_logits, row_stride, draft_tokens, uniforms, cu_k,
                                temperature, batch, k, vocab, sum_k, n_accepted, next_token, status, flags);
    p.use_tma = aligned16(target_logits) && (!draft_logits || aligned16(draft_logits)) &&
                (row_stride * elem) % 16 == 0;
    s = svh::launch_rows_topk(dtype, p, top_k, top_p, st);
    if (s == SV_OK) fused = true;
    else if (s != SV_ERR_UNSUPPORTED) return s;
    else g_err[0] = '\0';
  }
  s = svh::sampler_floors_gated(target_logits, draft_logits, dtype, row_stride, temperature, top_k, top_p, cu_k,
                                batch, k, sum_k, vocab, ft, fd, fused ? gate : nullptr, stream);
  if (s != SV_OK) return s;
  return svh::accept_logits(target_logits, draft_logits, dtype, row_stride, temperature, draft_tokens, uniforms, cu_k,
                            batch, k, sum_k, vocab, ft, fd, n_accepted, next_token, status, nullptr, nullptr,
                            nullptr, flags, stream, fused ? gate : nullptr);
}

size_t sv_workspace_size(int32_t batch, int32_t k, int32_t vocab, int32_t mode) {
  (void)batch;
  (void)k;
  (void)vocab;
  (void)mode;
  return 0;  // partials are exchanged through distributed shared memory
}

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_ARG: return "SV_ERR_ARG: invalid argument";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: CUDA runtime error";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: unsupported shape";
  }
  return "unknown sv_status";
}

const char* sv_last_error(void) { return g_err; }

int32_t sv_version(void) { return 100; }

}  // extern "C"
