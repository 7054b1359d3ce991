// The draft-length gate (PocketLLM docs/dspark.md, the draft-length gate
// section): per sequence, how many drafted tokens to submit to verification,
// and the online calibration of P(match | confidence bucket).  The formulas
// and the order of every operation are those of include/sv_gate.h.
//
// Both kernels are one CTA: the work is a few dozen flops per drafted
// position, so the launch and the latency of reading the small inputs are
// the cost.  Each walks the batch in tiles of kThreads sequences: the CTA
// first reads the tile's confidences with coalesced loads and keeps their
// bucket ids in shared memory (one memory latency per tile, not one per
// position), then one thread handles one sequence.  The gate scans the
// tile's lengths into cu_k with a running carry; the update tallies the
// round's observations with shared-memory integer atomics (exact, so the
// result does not depend on their order) and then decays and adds them per
// bucket.
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/sv_gate.h"
#include "sv_host.h"

namespace svg {

constexpr int kThreads = 512;  // sequences per tile; kThreads * K bucket ids in shared memory
constexpr int kMaxBuckets = SV_GATE_MAX_BUCKETS;
constexpr int kMaxK = SV_GATE_MAX_K;

struct GateArgs {
  const float* conf;
  const int32_t* k_drafted;
  const float* logit_margin;
  const float* edges;
  const double* hits;
  const double* total;
  int32_t* n_out;
  int32_t* cu_out;
  float margin, draft_ms, verify_base_ms, verify_slope_ms, plain_ms;  // rounded to fp32 once
  float margin_threshold;
  int min_draft;
  int nb, B, K;
};

struct UpdateArgs {
  const float* conf;
  const int32_t* n_sub;
  const int32_t* n_acc;
  const float* edges;
  double* hits;
  double* total;
  double decay;
  int nb, B, K;
};

// Index of the half-open bucket holding c (NaN -> 0).
__device__ __forceinline__ int bucket_of(float c, const float* edges, int nb) {
  if (c != c) return 0;
  int b = 0;
  for (int e = 0; e < nb - 1; ++e) b += c >= edges[e] ? 1 : 0;
  return b;
}

__device__ __forceinline__ int clamp_i(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// The decision runs in fp32 (it only picks an integer; fp64 is a small
// fraction of fp32's rate on this part), one rounding per operation: every
// ratio is within (3n + 6) * 2^-24 of the exact E(n)/cost(n), so the length
// is the exact rule's wherever no two compared ratios are that close.
__device__ int gate_one(const GateArgs& a, int kb, float lm, const uint8_t* bk, const float* p) {
  if (a.margin_threshold > 0.f && a.logit_margin && lm < a.margin_threshold) return 0;
  const int n_lo = a.min_draft < kb ? a.min_draft : kb;
  const float fixed = __fadd_rn(a.draft_ms, a.verify_base_ms);
  int best_n = n_lo;
  float best_r = 0.f, full_r = 0.f, e = 1.f, prod = 1.f;
  for (int n = 0; n <= kb; ++n) {
    if (n > 0) {
      prod = __fmul_rn(prod, p[bk[n - 1]]);
      e = __fadd_rn(e, prod);
    }
    const float cost = n == 0 ? a.plain_ms : __fadd_rn(fixed, __fmul_rn(a.verify_slope_ms, static_cast<float>(n)));
    const float r = __fdiv_rn(e, cost);
    if (n == n_lo || (n > n_lo && r > best_r)) {
      if (n > n_lo) best_n = n;
      best_r = r;
    }
    if (n == kb) full_r = r;
  }
  if (best_n < kb && best_r >= __fmul_rn(a.margin, full_r)) return best_n;
  return kb;
}

// Bucket ids of the tile's confidences (positions 0..K-1 of sequences
// base .. base + kThreads - 1), read with coalesced loads.
__device__ __forceinline__ void tile_buckets(const float* conf, int base, int B, int K, const float* edges, int nb,
                                             uint8_t* bk) {
  const int n = (min(B, base + kThreads) - base) * K;
  const float* src = conf + static_cast<long long>(base) * K;
  for (int e = threadIdx.x; e < n; e += kThreads) bk[e] = static_cast<uint8_t>(bucket_of(src[e], edges, nb));
}

__global__ void __launch_bounds__(kThreads) gate_kernel(const GateArgs a) {
  extern __shared__ uint8_t s_bk[];  // [kThreads * K] bucket ids of the tile
  __shared__ float s_edges[kMaxBuckets];
  __shared__ float s_p[kMaxBuckets];
  __shared__ int s_warp[kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (t < a.nb - 1) s_edges[t] = a.edges[t];
  if (t < a.nb) {  // p = hits / total as an fp64 quotient, rounded to fp32
    const double h = a.hits[t], tot = a.total[t];
    s_p[t] = tot > 0.0 ? static_cast<float>(__ddiv_rn(h, tot)) : 1.f;
  }
  __syncthreads();
  int carry = 0;  // lengths of the sequences before this tile
  for (int base = 0; base < a.B; base += kThreads) {
    const int b = base + t;
    const int kb = b < a.B ? (a.k_drafted ? clamp_i(a.k_drafted[b], 0, a.K) : a.K) : 0;
    const float lm = (b < a.B && a.logit_margin) ? a.logit_margin[b] : 0.f;
    tile_buckets(a.conf, base, a.B, a.K, s_edges, a.nb, s_bk);
    __syncthreads();
    const int n = b < a.B ? gate_one(a, kb, lm, s_bk + t * a.K, s_p) : 0;
    if (b < a.B) a.n_out[b] = n;
    // exclusive scan of n over the tile (warp scans, then the warp totals)
    int inc = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    int before = 0, tile = 0;
#pragma unroll
    for (int k = 0; k < kThreads / 32; ++k) {
      before += k < w ? s_warp[k] : 0;
      tile += s_warp[k];
    }
    if (b < a.B) a.cu_out[b] = carry + before + inc - n;
    carry += tile;
    __syncthreads();  // s_warp and s_bk are rewritten by the next tile
  }
  if (t == 0) a.cu_out[a.B] = carry;
}

__global__ void __launch_bounds__(kThreads) update_kernel(const UpdateArgs a) {
  extern __shared__ uint8_t s_bk[];  // [kThreads * K] bucket ids of the tile
  __shared__ float s_edges[kMaxBuckets];
  __shared__ unsigned s_h[kMaxBuckets], s_t[kMaxBuckets];
  const int t = threadIdx.x;
  if (t < a.nb - 1) s_edges[t] = a.edges[t];
  if (t < kMaxBuckets) s_h[t] = s_t[t] = 0u;
  __syncthreads();
  for (int base = 0; base < a.B; base += kThreads) {
    const int b = base + t;
    const int ks = b < a.B ? clamp_i(a.n_sub[b], 0, a.K) : 0;
    const int na = b < a.B ? clamp_i(a.n_acc[b], 0, ks) : 0;
    tile_buckets(a.conf, base, a.B, a.K, s_edges, a.nb, s_bk);
    __syncthreads();
    const uint8_t* bk = s_bk + t * a.K;
    for (int i = 0; i < na; ++i) {
      atomicAdd(&s_h[bk[i]], 1u);
      atomicAdd(&s_t[bk[i]], 1u);
    }
    if (na < ks) atomicAdd(&s_t[bk[na]], 1u);
    __syncthreads();  // s_bk is rewritten by the next tile
  }
  if (t < a.nb) {
    a.hits[t] = __dadd_rn(__dmul_rn(a.decay, a.hits[t]), static_cast<double>(s_h[t]));
    a.total[t] = __dadd_rn(__dmul_rn(a.decay, a.total[t]), static_cast<double>(s_t[t]));
  }
}

bool finite_nonneg(double v) { return std::isfinite(v) && v >= 0.0; }

sv_status check_common(const float* conf, const float* edges, const void* hits, const void* total,
                       int n_buckets, int B, int K) {
  if (B < 0) return svh::fail(SV_ERR_ARG, "batch must be >= 0 (got %d)", B);
  if (K < 0 || K > kMaxK) return svh::fail(SV_ERR_ARG, "k must be in [0, %d] (got %d)", kMaxK, K);
  if (static_cast<long long>(B) * K > 0x7FFFFFFFLL) return svh::fail(SV_ERR_ARG, "batch * k exceeds 2^31 - 1");
  if (n_buckets < 1 || n_buckets > kMaxBuckets)
    return svh::fail(SV_ERR_ARG, "n_buckets must be in [1, %d] (got %d)", kMaxBuckets, n_buckets);
  if (!conf && static_cast<long long>(B) * K > 0) return svh::fail(SV_ERR_ARG, "confidence pointer is NULL");
  if (!edges && n_buckets > 1) return svh::fail(SV_ERR_ARG, "edges pointer is NULL");
  if (!hits || !total) return svh::fail(SV_ERR_ARG, "hits / total pointer is NULL");
  return SV_OK;
}

}  // namespace svg

extern "C" sv_status sv_gate_draft_lengths(const float* confidence, const int32_t* k_drafted,
                                           const float* logit_margin, const float* edges,
                                           const double* hits, const double* total, int n_buckets,
                                           int B, int K, const sv_gate_params* params, int32_t* n_out,
                                           int32_t* cu_k_out, void* stream) {
  svh::clear_error();
  sv_status st = svg::check_common(confidence, edges, hits, total, n_buckets, B, K);
  if (st != SV_OK) return st;
  if (!params) return svh::fail(SV_ERR_ARG, "params pointer is NULL");
  if (!cu_k_out || (!n_out && B > 0)) return svh::fail(SV_ERR_ARG, "output pointer is NULL");
  const sv_gate_params& q = *params;
  if (!svg::finite_nonneg(q.margin) || !svg::finite_nonneg(q.draft_ms) || !svg::finite_nonneg(q.verify_base_ms) ||
      !svg::finite_nonneg(q.verify_slope_ms) || !(std::isfinite(q.plain_ms) && q.plain_ms > 0.0) ||
      !(q.draft_ms + q.verify_base_ms + q.verify_slope_ms > 0.0) || !(q.margin_threshold == q.margin_threshold) ||
      q.min_draft < 0)
    return svh::fail(SV_ERR_ARG, "gate params out of range (costs >= 0 with a positive verify and plain cost, "
                                 "margin >= 0, min_draft >= 0)");
  svg::GateArgs a;
  a.conf = confidence;
  a.k_drafted = k_drafted;
  a.logit_margin = logit_margin;
  a.edges = edges;
  a.hits = hits;
  a.total = total;
  a.n_out = n_out;
  a.cu_out = cu_k_out;
  a.margin = static_cast<float>(q.margin);
  a.draft_ms = static_cast<float>(q.draft_ms);
  a.verify_base_ms = static_cast<float>(q.verify_base_ms);
  a.verify_slope_ms = static_cast<float>(q.verify_slope_ms);
  a.plain_ms = static_cast<float>(q.plain_ms);
  a.margin_threshold = q.margin_threshold;
  a.min_draft = q.min_draft;
  a.nb = n_buckets;
  a.B = B;
  a.K = K;
  svg::gate_kernel<<<1, svg::kThreads, static_cast<size_t>(svg::kThreads) * K, static_cast<cudaStream_t>(stream)>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "gate kernel launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

extern "C" sv_status sv_gate_update(const float* confidence, const int32_t* n_submitted,
                                    const int32_t* n_accepted, const float* edges, double* hits,
                                    double* total, int n_buckets, int B, int K, double decay, void* stream) {
  svh::clear_error();
  sv_status st = svg::check_common(confidence, edges, hits, total, n_buckets, B, K);
  if (st != SV_OK) return st;
  if (B > 0 && (!n_submitted || !n_accepted)) return svh::fail(SV_ERR_ARG, "length pointer is NULL");
  if (!(decay >= 0.0 && decay <= 1.0)) return svh::fail(SV_ERR_ARG, "decay must be in [0, 1] (got %g)", decay);
  svg::UpdateArgs a;
  a.conf = confidence;
  a.n_sub = n_submitted;
  a.n_acc = n_accepted;
  a.edges = edges;
  a.hits = hits;
  a.total = total;
  a.decay = decay;
  a.nb = n_buckets;
  a.B = B;
  a.K = K;
  svg::update_kernel<<<1, svg::kThreads, static_cast<size_t>(svg::kThreads) * K, static_cast<cudaStream_t>(stream)>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "gate update launch: %s", cudaGetErrorString(e));
  return SV_OK;
}
