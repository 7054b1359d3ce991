// The draft-length gate (PocketLLM docs/dspark.md, the draft-length gate
// section): per sequence, how many drafted tokens to submit to verification,
// and the online calibration of P(match | confidence bucket).  The formulas
// and the order of every fp64 operation are those of include/sv_gate.h.
//
// Both kernels are one CTA: the work is a few dozen flops per drafted
// position, so the launch and one pass over the small inputs are the cost.
// The gate walks the batch in tiles of kThreads sequences, one thread per
// sequence, and scans the tile's lengths into cu_k with a running carry; the
// update tallies the round's observations with shared-memory integer
// atomics (exact, so the result does not depend on their order) and then
// decays and adds them per bucket.
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/sv_gate.h"
#include "sv_host.h"

namespace svg {

constexpr int kThreads = 256;
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
  double margin, draft_ms, verify_base_ms, verify_slope_ms, plain_ms;
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

__device__ int gate_one(const GateArgs& a, int b, const float* edges, const double* p) {
  const int kb = a.k_drafted ? clamp_i(a.k_drafted[b], 0, a.K) : a.K;
  if (a.margin_threshold > 0.f && a.logit_margin && a.logit_margin[b] < a.margin_threshold) return 0;
  const int n_lo = a.min_draft < kb ? a.min_draft : kb;
  const float* conf = a.conf + static_cast<long long>(b) * a.K;
  const double fixed = __dadd_rn(a.draft_ms, a.verify_base_ms);
  int best_n = -1;
  double best_r = 0.0, full_r = 0.0, e = 1.0, prod = 1.0;
  for (int n = 0; n <= kb; ++n) {
    if (n > 0) {
      prod = __dmul_rn(prod, p[bucket_of(conf[n - 1], edges, a.nb)]);
      e = __dadd_rn(e, prod);
    }
    const double cost = n == 0 ? a.plain_ms : __dadd_rn(fixed, __dmul_rn(a.verify_slope_ms, static_cast<double>(n)));
    const double r = __ddiv_rn(e, cost);
    if (n >= n_lo && (best_n < 0 || r > best_r)) {
      best_n = n;
      best_r = r;
    }
    if (n == kb) full_r = r;
  }
  if (best_n < kb && best_r >= __dmul_rn(a.margin, full_r)) return best_n;
  return kb;
}

__global__ void __launch_bounds__(kThreads) gate_kernel(const GateArgs a) {
  __shared__ float s_edges[kMaxBuckets];
  __shared__ double s_p[kMaxBuckets];
  __shared__ int s_warp[kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (t < a.nb - 1) s_edges[t] = a.edges[t];
  if (t < a.nb) {
    const double h = a.hits[t], tot = a.total[t];
    s_p[t] = tot > 0.0 ? __ddiv_rn(h, tot) : 1.0;
  }
  __syncthreads();
  int carry = 0;  // lengths of the sequences before this tile
  for (int base = 0; base < a.B; base += kThreads) {
    const int b = base + t;
    const int n = b < a.B ? gate_one(a, b, s_edges, s_p) : 0;
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
    __syncthreads();  // s_warp is rewritten by the next tile
  }
  if (t == 0) a.cu_out[a.B] = carry;
}

__global__ void __launch_bounds__(kThreads) update_kernel(const UpdateArgs a) {
  __shared__ float s_edges[kMaxBuckets];
  __shared__ unsigned s_h[kMaxBuckets], s_t[kMaxBuckets];
  const int t = threadIdx.x;
  if (t < a.nb - 1) s_edges[t] = a.edges[t];
  if (t < kMaxBuckets) s_h[t] = s_t[t] = 0u;
  __syncthreads();
  for (int b = t; b < a.B; b += kThreads) {
    const int ks = clamp_i(a.n_sub[b], 0, a.K);
    const int na = clamp_i(a.n_acc[b], 0, ks);
    const float* conf = a.conf + static_cast<long long>(b) * a.K;
    for (int i = 0; i < na; ++i) {
      const int k = bucket_of(conf[i], s_edges, a.nb);
      atomicAdd(&s_h[k], 1u);
      atomicAdd(&s_t[k], 1u);
    }
    if (na < ks) atomicAdd(&s_t[bucket_of(conf[na], s_edges, a.nb)], 1u);
  }
  __syncthreads();
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
  a.margin = q.margin;
  a.draft_ms = q.draft_ms;
  a.verify_base_ms = q.verify_base_ms;
  a.verify_slope_ms = q.verify_slope_ms;
  a.plain_ms = q.plain_ms;
  a.margin_threshold = q.margin_threshold;
  a.min_draft = q.min_draft;
  a.nb = n_buckets;
  a.B = B;
  a.K = K;
  svg::gate_kernel<<<1, svg::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
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
  svg::update_kernel<<<1, svg::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "gate update launch: %s", cudaGetErrorString(e));
  return SV_OK;
}
