// Top-k / top-p floors of logit rows (llmstudio.ru, "Как работает speculative
// decoding и MTP при инференсе LLM", section 38: temperature, then top-k,
// then top-p, alike for the target's and the draft's rows).  The definitions
// are those of include/sv_filter.h.
//
// One CTA per row.  Each logit gets an order-preserving integer key (the
// sign-flipped bit pattern: 32 bits for f32, the raw 16 bits for bf16 / f16;
// -0 keyed as +0, NaN skipped), and each floor is found by a radix select over
// those keys: per level, a shared-memory histogram of the keys that share the
// prefix chosen so far, then one warp scans the bins from the top to find the
// lowest bin whose "mass above" still passes the test (count above < k for
// top-k; weight above < p * Z for top-p).  The first level is 11 bits wide
// (sign, exponent and two mantissa bits of an f32), so the logits of a row
// spread over many bins and the shared-memory atomics rarely collide.
//
// The first pass over the row also keeps each thread's 8 largest keys in
// registers (4096 candidates per row, then in shared memory).  A floor among
// the top few thousand logits (the usual top-k, and top-p of a peaked row) is
// then selected from the candidates alone, with a check that proves the
// answer is the row's own; otherwise the select runs over the whole row.  So
// top-k reads the row once and top-p twice (the second pass sums the kept
// weight, without atomics).
//
// Counts are 32-bit integers and weights 64-bit fixed point (2^-40 units,
// truncated), so every sum is exact and independent of the order of the
// atomics: the result is deterministic.
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "../../include/sv_filter.h"
#include "sv_host.h"
#include "sv_kernel.cuh"

namespace svf {

constexpr int kThreads = 512;
constexpr int kWarpsF = kThreads / 32;
constexpr int kMaxBins = 2048;
constexpr int kCand = 8;  // largest keys each thread keeps from the first pass

struct Args {
  const void* tgt;
  const void* drf;
  long long stride;
  const float* temp;
  const int32_t* top_k;
  const float* top_p;
  const int32_t* cu_k;
  int B, K, V, sum_k;
  float* ft;
  float* fd;
};

// Order-preserving keys and the radix levels over them (widths 11 + 11 + 10
// for 32-bit keys, 11 + 5 for 16-bit ones).
template <typename T>
struct KeyOf;
template <>
struct KeyOf<float> {
  static constexpr int kLevels = 3;
  __device__ static int shift(int l) { return l == 0 ? 21 : (l == 1 ? 10 : 0); }
  __device__ static int width(int l) { return l == 2 ? 10 : 11; }
  __device__ static bool key(uint32_t raw, uint32_t& k) {
    if ((raw & 0x7FFFFFFFu) > 0x7F800000u) return false;  // NaN
    if ((raw & 0x7FFFFFFFu) == 0u) raw = 0u;              // -0 ranks as +0
    k = (raw & 0x80000000u) ? ~raw : (raw | 0x80000000u);
    return true;
  }
  __device__ static float value_raw(uint32_t raw) { return __uint_as_float(raw); }
  __device__ static float value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
};
template <typename T>
struct Key16 {
  static constexpr int kLevels = 2;
  __device__ static int shift(int l) { return l == 0 ? 5 : 0; }
  __device__ static int width(int l) { return l == 0 ? 11 : 5; }
  static constexpr uint32_t kInfBits = std::is_same<T, __nv_bfloat16>::value ? 0x7F80u : 0x7C00u;
  __device__ static bool key(uint32_t raw, uint32_t& k) {
    if ((raw & 0x7FFFu) > kInfBits) return false;  // NaN
    if ((raw & 0x7FFFu) == 0u) raw = 0u;
    k = (raw & 0x8000u) ? (~raw & 0xFFFFu) : (raw | 0x8000u);
    return true;
  }
  __device__ static float value_raw(uint32_t raw) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(raw << 16);
    else return __half2float(__ushort_as_half(static_cast<unsigned short>(raw)));
  }
  __device__ static float value(uint32_t k) {
    return value_raw((k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu));
  }
};
template <>
struct KeyOf<__nv_bfloat16> : Key16<__nv_bfloat16> {};
template <>
struct KeyOf<__half> : Key16<__half> {};

// f(raw bits) for every element of a row: 16-byte loads where the row is
// aligned (kLoads of them in flight per thread), element loads for the rest.
// The order of the calls is immaterial (every use is an exact integer
// reduction).
template <typename T, typename F>
__device__ __forceinline__ void vec_elems(const uint4 v, F& f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if constexpr (sizeof(T) == 4) {
      f(w[j]);
    } else {
      f(w[j] & 0xFFFFu);
      f(w[j] >> 16);
    }
  }
}

template <typename T, typename F>
__device__ __forceinline__ void for_each_raw(const T* row, int V, F&& f) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  constexpr int kLoads = 4;
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) {
    const int nv = V / VEC;
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    int vi = threadIdx.x;
    for (; vi + (kLoads - 1) * kThreads < nv; vi += kLoads * kThreads) {
      uint4 v[kLoads];
#pragma unroll
      for (int u = 0; u < kLoads; ++u) v[u] = __ldg(r4 + vi + u * kThreads);
#pragma unroll
      for (int u = 0; u < kLoads; ++u) vec_elems<T>(v[u], f);
    }
    for (; vi < nv; vi += kThreads) vec_elems<T>(__ldg(r4 + vi), f);
    done = nv * VEC;
  }
  for (int e = done + static_cast<int>(threadIdx.x); e < V; e += kThreads) {
    if constexpr (sizeof(T) == 4) f(__ldg(reinterpret_cast<const uint32_t*>(row) + e));
    else f(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)));
  }
}

// Selection state shared by the CTA: the key prefix chosen so far and the
// count / weight of the keys above it.
struct Sel {
  uint32_t prefix;
  int ok;
  unsigned long long c_above, m_above;  // keys above the chosen prefix
  unsigned long long c_grp, m_grp;      // keys in the chosen bin
};

// Does a bin whose higher keys hold (c, m) still pass the test?
struct Crit {
  bool by_count;
  unsigned long long k_lim;  // top-k: count above < k
  double m_lim;              // top-p: weight above < p * Z
  __device__ __forceinline__ bool within(unsigned long long c, unsigned long long m) const {
    return by_count ? c < k_lim : static_cast<double>(m) < m_lim;
  }
};

// Warp: among 32 lanes holding (c, m) for consecutive ranges (lane 31 the
// highest keys), the lowest lane that passes the test with its exclusive
// "above" (plus the carry) and holds at least one key; -1 if none.
__device__ __forceinline__ int warp_pick(unsigned long long c, unsigned long long m, unsigned long long carry_c,
                                         unsigned long long carry_m, const Crit& cr, unsigned long long& out_c,
                                         unsigned long long& out_m) {
  const int lane = threadIdx.x & 31;
  unsigned long long sc = c, sm = m;  // inclusive sums over lanes >= this one
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tc = __shfl_down_sync(0xFFFFFFFFu, sc, o);
    const unsigned long long tm = __shfl_down_sync(0xFFFFFFFFu, sm, o);
    if (lane + o < 32) {
      sc += tc;
      sm += tm;
    }
  }
  const unsigned long long ac = carry_c + (sc - c), am = carry_m + (sm - m);
  const unsigned cand = __ballot_sync(0xFFFFFFFFu, c > 0ull && cr.within(ac, am));
  if (cand == 0u) return -1;
  const int l = __ffs(cand) - 1;
  out_c = __shfl_sync(0xFFFFFFFFu, ac, l);
  out_m = __shfl_sync(0xFFFFFFFFu, am, l);
  return l;
}

// Warp 0: the lowest non-empty bin of hc / hm (nb bins, a multiple of 32)
// whose keys above pass the test; updates s (prefix extended by `width` bits,
// the carry by the bins above the chosen one).
__device__ __forceinline__ void scan_bins(const unsigned* hc, const unsigned long long* hm, int nb, int width,
                                          const Crit& cr, Sel& s) {
  const int lane = threadIdx.x & 31;
  const int per = nb / 32;
  unsigned long long c = 0, m = 0;
  for (int j = 0; j < per; ++j) {
    c += hc[lane * per + j];
    m += hm[lane * per + j];
  }
  unsigned long long ac, am;
  const int l1 = warp_pick(c, m, s.c_above, s.m_above, cr, ac, am);
  if (l1 < 0) {  // unreachable while the carry passes the test (the top key always does)
    if (lane == 0) s.ok = 0;
    return;
  }
  // lanes split the chosen range of `per` bins, q bins each
  const int q = per >= 32 ? per / 32 : 1;
  const int base = l1 * per;
  c = m = 0;
  if (lane * q < per) {
    for (int j = 0; j < q; ++j) {
      c += hc[base + lane * q + j];
      m += hm[base + lane * q + j];
    }
  }
  const int l2 = warp_pick(c, m, ac, am, cr, ac, am);
  if (l2 < 0) {
    if (lane == 0) s.ok = 0;
    return;
  }
  if (lane == l2) {  // at most two bins left: walk them from the top
    int bin = -1;
    unsigned long long bc = 0, bm = 0;
    for (int j = q - 1; j >= 0; --j) {
      const int b = base + lane * q + j;
      if (hc[b] == 0u) continue;
      if (!cr.within(ac, am)) break;
      bin = b;
      bc = ac;
      bm = am;
      ac += hc[b];
      am += hm[b];
    }
    if (bin < 0) {
      s.ok = 0;
    } else {
      s.prefix = (s.prefix << width) | static_cast<uint32_t>(bin);
      s.c_above = bc;
      s.m_above = bm;
      s.c_grp = hc[bin];
      s.m_grp = hm[bin];
    }
  }
}

// Radix select over the keys a source yields (src(f) calls f(key) for each),
// skipping keys below `lower`: leaves in `sel` the lowest key whose keys above
// pass the test, their count and weight, and the count and weight of the
// keys equal to it.  Collective (every thread of the CTA).
template <typename KT, typename Src, typename WFn>
__device__ __forceinline__ void radix_select(const Src& src, const WFn& weight, bool use_mass, uint32_t lower,
                                             const Crit& cr, unsigned* h_cnt, unsigned long long* h_mass,
                                             Sel& sel) {
  const int tid = threadIdx.x;
  __syncthreads();  // earlier readers of `sel` and of the histograms are done
  if (tid == 0) sel = Sel{0u, 1, 0ull, 0ull, 0ull, 0ull};
  for (int l = 0; l < KT::kLevels; ++l) {
    const int nb = 1 << KT::width(l);
    const int sh = KT::shift(l);
    const int hs = sh + KT::width(l);
    for (int j = tid; j < nb; j += kThreads) {
      h_cnt[j] = 0u;
      h_mass[j] = 0ull;
    }
    __syncthreads();  // also publishes the previous level's choice
    const uint32_t pre = sel.prefix;
    const bool ok = sel.ok != 0;
    if (ok) {
      src([&](uint32_t k) {
        if (k < lower || (l > 0 && (k >> hs) != pre)) return;
        const int bin = static_cast<int>((k >> sh) & static_cast<uint32_t>(nb - 1));
        atomicAdd(&h_cnt[bin], 1u);
        if (use_mass) {
          const unsigned long long w = weight(k);
          if (w) atomicAdd(&h_mass[bin], w);
        }
      });
    }
    __syncthreads();
    if (tid < 32 && ok) scan_bins(h_cnt, h_mass, nb, KT::width(l), cr, sel);
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) floors_kernel(const __grid_constant__ Args a) {
  using KT = KeyOf<T>;
  using WarpT = typename svk::WarpOf<T>::type;
  __shared__ unsigned h_cnt[kMaxBins];
  __shared__ unsigned long long h_mass[kMaxBins];
  __shared__ uint32_t cand[kThreads * kCand];
  __shared__ unsigned r_max[kWarpsF], r_cnt[kWarpsF], r_g[kWarpsF];
  __shared__ unsigned long long r_z[kWarpsF];
  __shared__ Sel sel;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const long long b = blockIdx.y + static_cast<long long>(blockIdx.z) * gridDim.y;
  if (b >= a.B) return;
  int kb = a.K;
  long long t0 = b * (a.K + 1LL), d0 = b * static_cast<long long>(a.K);
  if (a.cu_k) {
    const int lo = a.cu_k[b], hi = a.cu_k[b + 1];
    if (lo < 0 || hi < lo || hi > a.sum_k || hi - lo > a.K) return;  // no rows of its own
    kb = hi - lo;
    t0 = lo + b;
    d0 = lo;
  }
  const int r = blockIdx.x;
  if (r > 2 * kb) return;
  const bool is_d = r > kb;
  const int i = is_d ? r - kb - 1 : r;
  float* out = is_d ? a.fd : a.ft;
  if (!out) return;
  out += (is_d ? d0 : t0) + i;
  const T* row = static_cast<const T*>(is_d ? a.drf : a.tgt) + ((is_d ? d0 : t0) + i) * a.stride;

  // ---- the sequence's parameters
  const float temp = a.temp[b];
  const int kk = a.top_k ? a.top_k[b] : 0;
  const float p = a.top_p ? a.top_p[b] : 1.f;
  if (!(temp > 0.f && temp <= FLT_MAX)) {  // greedy, or a temperature the verification rejects
    if (tid == 0) *out = -kInfF;
    return;
  }
  if (!(p > 0.f)) {  // NaN or <= 0: invalid
    if (tid == 0) *out = __uint_as_float(0x7FC00000u);
    return;
  }
  bool use_k = kk > 0 && kk < a.V;
  const bool use_p = p < 1.f;
  if (!use_k && !use_p) {
    if (tid == 0) *out = -kInfF;
    return;
  }

  // ---- pass 1: the row maximum, the non-NaN count, and each thread's kCand
  // largest keys (candidates; 0 = none).  Every key above G, the largest of
  // the threads' smallest candidates, is a candidate.
  uint32_t kmax = 0u, nn = 0u;
  uint32_t c[kCand];
#pragma unroll
  for (int j = 0; j < kCand; ++j) c[j] = 0u;
  for_each_raw<T>(row, a.V, [&](uint32_t raw) {
    uint32_t k;
    if (!KT::key(raw, k)) return;
    kmax = max(kmax, k);
    ++nn;
    if (k > c[kCand - 1]) {
      c[kCand - 1] = k;
#pragma unroll
      for (int j = kCand - 1; j > 0; --j) {
        if (c[j] > c[j - 1]) {
          const uint32_t t = c[j];
          c[j] = c[j - 1];
          c[j - 1] = t;
        }
      }
    }
  });
#pragma unroll
  for (int j = 0; j < kCand; ++j) cand[tid * kCand + j] = c[j];
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  nn = __reduce_add_sync(0xFFFFFFFFu, nn);
  const uint32_t gl = __reduce_max_sync(0xFFFFFFFFu, c[kCand - 1]);
  if (lane == 0) {
    r_max[warp] = kmax;
    r_cnt[warp] = nn;
    r_g[warp] = gl;
  }
  __syncthreads();
  kmax = 0u;
  nn = 0u;
  uint32_t G = 0u;
  for (int w = 0; w < kWarpsF; ++w) {
    kmax = max(kmax, r_max[w]);
    nn += r_cnt[w];
    G = max(G, r_g[w]);
  }
  const float m = KT::value(kmax);
  if (nn == 0u || !(m > -kInfF && m < kInfF)) {  // no finite maximum: no filter
    if (tid == 0) *out = -kInfF;
    return;
  }
  if (use_k && static_cast<uint32_t>(kk) >= nn) use_k = false;  // k covers the row

  auto cand_src = [&](auto f) {
    for (int j = tid; j < kThreads * kCand; j += kThreads) {
      const uint32_t k = cand[j];
      if (k) f(k);
    }
  };
  auto row_src = [&](auto f) {
    for_each_raw<T>(row, a.V, [&](uint32_t raw) {
      uint32_t k;
      if (KT::key(raw, k)) f(k);
    });
  };
  // A selection among the candidates is the row's own when the chosen key is
  // above G (so every key at or above it is a candidate: the counts and
  // weights above it and at it are complete) and the test already fails once
  // its own group is added (so no lower key can pass).

  // ---- top-k: the k-th largest key
  uint32_t key_k = 0u;  // below every key: keeps all
  if (use_k) {
    const Crit cr{true, static_cast<unsigned long long>(kk), 0.0};
    auto none = [](uint32_t) { return 0ull; };
    radix_select<KT>(cand_src, none, false, 0u, cr, h_cnt, h_mass, sel);
    const bool exact = sel.ok && sel.prefix > G && !cr.within(sel.c_above + sel.c_grp, 0ull);
    if (!exact) radix_select<KT>(row_src, none, false, 0u, cr, h_cnt, h_mass, sel);
    key_k = sel.ok ? sel.prefix : 0u;
  }

  // ---- top-p on what top-k kept: the lowest key whose kept weight above is < p Z
  uint32_t key_p = key_k;
  if (use_p && key_k < kmax) {
    float khi, klo;
    svk::log2e_over(temp, khi, klo);
    WarpT wf;
    if constexpr (sizeof(T) == 4) {
      wf.m = m;
      wf.khi = khi;
      wf.klo = klo;
    } else {
      wf.m = m;
      wf.k = khi;
    }
    wf.lo = -kInfF;
    auto weight = [&](uint32_t k) -> unsigned long long {
      return __float2ull_rz(__fmul_rn(wf(KT::value(k)), 0x1p40f));
    };
    // Z: the kept weight (a pass over the row without atomics)
    unsigned long long z = 0ull;
    row_src([&](uint32_t k) {
      if (k >= key_k) z += weight(k);
    });
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    if (lane == 0) r_z[warp] = z;
    __syncthreads();
    z = 0ull;
    for (int w = 0; w < kWarpsF; ++w) z += r_z[w];
    const Crit cr{false, 0ull, static_cast<double>(p) * static_cast<double>(z)};
    radix_select<KT>(cand_src, weight, true, key_k, cr, h_cnt, h_mass, sel);
    const bool exact = sel.ok && sel.prefix > G && !cr.within(0ull, sel.m_above + sel.m_grp);
    if (!exact) radix_select<KT>(row_src, weight, true, key_k, cr, h_cnt, h_mass, sel);
    if (sel.ok) key_p = sel.prefix;
  }
  if (tid == 0) *out = key_p == 0u ? -kInfF : KT::value(key_p);
}

template <typename T>
sv_status launch(const Args& a, cudaStream_t st) {
  const int gy = a.B < 65535 ? a.B : 65535;
  const int gz = (a.B + gy - 1) / gy;
  floors_kernel<T><<<dim3(2 * a.K + 1, gy, gz), kThreads, 0, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "floors kernel launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

}  // namespace svf

extern "C" sv_status sv_sampler_floors(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                                       int64_t row_stride, const float* temperature, const int32_t* top_k,
                                       const float* top_p, const int32_t* cu_k, int32_t batch, int32_t k,
                                       int32_t sum_k, int32_t vocab, float* floor_target, float* floor_draft,
                                       void* stream) {
  svh::clear_error();
  if (batch < 0) return svh::fail(SV_ERR_ARG, "batch must be >= 0 (got %d)", batch);
  if (k < 0) return svh::fail(SV_ERR_ARG, "k must be >= 0 (got %d)", k);
  if (vocab < 1) return svh::fail(SV_ERR_ARG, "vocab must be >= 1 (got %d)", vocab);
  if (sum_k < 0) return svh::fail(SV_ERR_ARG, "sum_k must be >= 0 (got %d)", sum_k);
  if (row_stride < vocab)
    return svh::fail(SV_ERR_ARG, "row_stride (%lld) < vocab (%d)", static_cast<long long>(row_stride), vocab);
  if (!cu_k && static_cast<long long>(batch) * k != sum_k)
    return svh::fail(SV_ERR_ARG, "without cu_k, sum_k must equal batch * k (%lld), got %d",
                     static_cast<long long>(batch) * k, sum_k);
  if (static_cast<long long>(sum_k) + batch > 0x7FFFFFFFLL)
    return svh::fail(SV_ERR_ARG, "too many rows (sum_k + batch > 2^31 - 1)");
  if (2LL * k + 1 > 0x7FFFFFFFLL) return svh::fail(SV_ERR_ARG, "k too large");
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return svh::fail(SV_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (batch == 0 || (!top_k && !top_p)) return SV_OK;
  if (!target_logits) return svh::fail(SV_ERR_ARG, "target pointer is NULL");
  if (sum_k > 0 && !draft_logits && floor_draft) return svh::fail(SV_ERR_ARG, "draft_logits is NULL");
  if (!temperature) return svh::fail(SV_ERR_ARG, "temperature is NULL");
  if (!floor_target && !floor_draft) return SV_OK;
  svf::Args a;
  a.tgt = target_logits;
  a.drf = draft_logits;
  a.stride = row_stride;
  a.temp = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.cu_k = cu_k;
  a.B = batch;
  a.K = k;
  a.V = vocab;
  a.sum_k = sum_k;
  a.ft = floor_target;
  a.fd = floor_draft;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case SV_F32: return svf::launch<float>(a, st);
    case SV_BF16: return svf::launch<__nv_bfloat16>(a, st);
    default: return svf::launch<__half>(a, st);
  }
}
