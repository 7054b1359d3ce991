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
// A sample of 4096 logits (64 runs of consecutive logits spread over the
// row, one round trip) gives a lower bound L of the floor.  Top-k: the lowest
// key of the first-level bin holding the sample's rank of 2k logits plus a
// margin; one pass over the row then takes the maximum and the non-NaN count
// and appends every logit >= L to a shared-memory list.  Top-p alone: a first
// pass takes the maximum (the weights need it), L is the sample's rank of
// about 2500 logits, and a second pass appends every logit >= L and sums the
// row's weight Z.  The exact selects then run on the list: its counts and
// weights are complete for every key >= L, so a floor found there is the
// row's own when (top-k) the list holds at least k keys, or (top-p alone)
// the test already fails once the chosen key's own group is added.  When a
// check fails or the list overflows, the same selects run over the whole row
// instead (a few more passes; correct, only slower).
//
// Counts are 32-bit integers and weights 64-bit fixed point (2^-40 units,
// truncated, converted with integer operations), so every sum is exact and
// independent of the order of the atomics: the result is deterministic.  The
// first pass takes the maximum element by element in f32: a version on packed
// bf16x2 words measured the fp64 pipe (which is slow on this part) 60-70 %
// busy.
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>
#include <type_traits>

#include "../../include/sv_filter.h"
#include "sv_host.h"
#include "sv_kernel.cuh"

namespace svf {

constexpr int kThreads = 512;
constexpr int kWarpsF = kThreads / 32;
constexpr int kMaxBins = 2048;
constexpr int kCap = 4096;  // sampled keys, then collected keys, in shared memory
constexpr int kSampleRuns = 64;  // runs of consecutive logits the sample takes
constexpr int kTopSet = 64;      // a top-k set this small takes top-p by ranking

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
  const int* gate;  // per sequence: 0 = skip (NULL: every sequence)
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
  __device__ static uint32_t raw_of(float x) { return __float_as_uint(x); }
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
  // the raw bits of a value of this type (exact: x came from value_raw)
  __device__ static uint32_t raw_of(float x) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return __float_as_uint(x) >> 16;
    else return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
  }
};
template <>
struct KeyOf<__nv_bfloat16> : Key16<__nv_bfloat16> {};
template <>
struct KeyOf<__half> : Key16<__half> {};

// Every element of a row: fw(32-bit word) for the 16-byte aligned part (one
// f32 or two packed 16-bit values per word; kLoads vectors in flight per
// thread), fe(raw bits) for single elements elsewhere.  The order of the
// calls is immaterial (every use is an exact integer reduction or a max).
template <typename T, typename FW, typename FE>
__device__ __forceinline__ void for_each_word(const T* row, int V, FW&& fw, FE&& fe) {
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
      for (int u = 0; u < kLoads; ++u) {
        fw(v[u].x);
        fw(v[u].y);
        fw(v[u].z);
        fw(v[u].w);
      }
    }
    for (; vi < nv; vi += kThreads) {
      const uint4 v = __ldg(r4 + vi);
      fw(v.x);
      fw(v.y);
      fw(v.z);
      fw(v.w);
    }
    done = nv * VEC;
  }
  for (int e = done + static_cast<int>(threadIdx.x); e < V; e += kThreads) {
    if constexpr (sizeof(T) == 4) fe(__ldg(reinterpret_cast<const uint32_t*>(row) + e));
    else fe(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)));
  }
}

// f(raw bits) for every element of a row.
template <typename T, typename F>
__device__ __forceinline__ void for_each_raw(const T* row, int V, F&& f) {
  for_each_word<T>(
      row, V,
      [&](uint32_t w) {
        if constexpr (sizeof(T) == 4) {
          f(w);
        } else {
          f(w & 0xFFFFu);
          f(w >> 16);
        }
      },
      f);
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

// Warp 0: the lowest non-empty bin of hc / hm (32 * PER bins) whose keys
// above pass the test; updates s (prefix extended by `width` bits, the carry
// by the bins above the chosen one, the group by the chosen bin).  PER is a
// compile-time count so each lane's loads are unrolled and overlap.
template <int PER>
__device__ __forceinline__ void scan_bins(const unsigned* hc, const unsigned long long* hm, int width,
                                          const Crit& cr, Sel& s) {
  const int lane = threadIdx.x & 31;
  unsigned long long c = 0, m = 0;
  // each lane sums its own PER bins, starting at a lane-dependent offset so
  // the 32 lanes read 32 different banks at every step
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int b = lane * PER + ((j + lane) & (PER - 1));
    c += hc[b];
    m += hm[b];
  }
  unsigned long long ac, am;
  const int l1 = warp_pick(c, m, s.c_above, s.m_above, cr, ac, am);
  if (l1 < 0) {  // unreachable while the carry passes the test (the top key always does)
    if (lane == 0) s.ok = 0;
    return;
  }
  // lanes split the chosen range of PER bins, Q bins each
  constexpr int Q = PER >= 32 ? PER / 32 : 1;
  const int base = l1 * PER;
  c = m = 0;
  if (lane * Q < PER) {
#pragma unroll
    for (int j = 0; j < Q; ++j) {
      c += hc[base + lane * Q + j];
      m += hm[base + lane * Q + j];
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
#pragma unroll
    for (int j = Q - 1; j >= 0; --j) {
      const int b = base + lane * Q + j;
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
// LEVELS < KT::kLevels stops early: the prefix then names the bin (a range
// of keys) that holds the answer.
template <typename KT, int LEVELS = KT::kLevels, typename Src, typename WFn>
__device__ __forceinline__ void radix_select(const Src& src, const WFn& weight, bool use_mass, uint32_t lower,
                                             const Crit& cr, unsigned* h_cnt, unsigned long long* h_mass,
                                             Sel& sel) {
  const int tid = threadIdx.x;
  __syncthreads();  // earlier readers of `sel` and of the histograms are done
  if (tid == 0) sel = Sel{0u, 1, 0ull, 0ull, 0ull, 0ull};
  for (int l = 0; l < LEVELS; ++l) {
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
    if (tid < 32 && ok) {
      if (nb == 2048) scan_bins<64>(h_cnt, h_mass, KT::width(l), cr, sel);
      else if (nb == 1024) scan_bins<32>(h_cnt, h_mass, KT::width(l), cr, sel);
      else scan_bins<1>(h_cnt, h_mass, KT::width(l), cr, sel);
    }
    __syncthreads();
  }
}

// Warp: the top-p floor of a top-k set of n <= kTopSet keys (tk[0..n)):
// the lowest key whose higher-ranked weight (the keys strictly above it)
// passes the test.  Each lane ranks its two keys against all n (ties: by
// position) and places them in descending order in `ord`; lane 0 then walks
// the ranking once, group by group.  Returns the key on every lane.
template <typename WFn>
__device__ __forceinline__ uint32_t top_p_small(uint32_t* tk, int n, const WFn& weight, const Crit& cr) {
  const int lane = threadIdx.x & 31;
  __shared__ uint32_t ord[kTopSet];
  for (int h = 0; h < kTopSet / 32; ++h) {
    const int j = lane + 32 * h;
    if (j >= n) continue;
    const uint32_t kj = tk[j];
    int rank = 0;
    for (int m = 0; m < n; ++m) {
      const uint32_t km = tk[m];
      rank += (km > kj || (km == kj && m < j)) ? 1 : 0;
    }
    ord[rank] = kj;
  }
  __syncwarp();
  uint32_t ans = 0u;
  if (lane == 0) {
    unsigned long long above = 0ull;  // weight of the keys strictly above the current group
    int j = 0;
    while (j < n) {
      const uint32_t g = ord[j];
      if (!cr.within(0ull, above)) break;
      ans = g;
      unsigned long long w = 0ull;
      while (j < n && ord[j] == g) {
        w += weight(g);
        ++j;
      }
      above += w;
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ans, 0);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) floors_kernel(const __grid_constant__ Args a) {
  using KT = KeyOf<T>;
  using WarpT = typename svk::WarpOf<T>::type;
  __shared__ unsigned h_cnt[kMaxBins];
  __shared__ unsigned long long h_mass[kMaxBins];
  __shared__ uint32_t col[kCap];  // the sample, then the collected keys
  __shared__ unsigned r_cnt[kWarpsF];
  __shared__ float r_max[kWarpsF];
  __shared__ unsigned long long r_z[kWarpsF];
  __shared__ Sel sel;
  __shared__ int n_col;
  __shared__ uint32_t tk[kTopSet];  // the top-k set, when small
  __shared__ int n_tk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const long long b = blockIdx.y + static_cast<long long>(blockIdx.z) * gridDim.y;
  if (b >= a.B) return;
  if (a.gate && !a.gate[b]) return;
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

  // ---- a sample of kCap keys (0: NaN) into `col`: kSampleRuns runs of
  // consecutive logits spread evenly over the row (a few sectors each, so
  // the sample costs one round trip and a few KB, not one sector per key)
  {
    constexpr int kRun = kCap / kSampleRuns;
    constexpr int kPer = kCap / kThreads;  // consecutive sampled logits per thread
    static_assert(kRun % kPer == 0, "runs split evenly over threads");
    const int e0 = tid * kPer;  // this thread's first sample slot
    const long long span = a.V > kRun ? static_cast<long long>(a.V - kRun) : 0;
    const long long base = span * (e0 / kRun) / (kSampleRuns - 1);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const long long e = (base + (e0 % kRun) + j) % a.V;
      uint32_t raw;
      if constexpr (sizeof(T) == 4) raw = __ldg(reinterpret_cast<const uint32_t*>(row) + e);
      else raw = static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e));
      uint32_t k;
      col[e0 + j] = KT::key(raw, k) ? k : 0u;
    }
  }
  if (tid == 0) n_col = 0;
  auto none = [](uint32_t) { return 0ull; };
  auto samp_src = [&](auto f) {
    for (int j = tid; j < kCap; j += kThreads) {
      const uint32_t k = col[j];
      if (k) f(k);
    }
  };
  // a lower bound L of the floor from the sample: the sample's rank of `j`
  // logits, or with `coarse` the lowest key of the first-level bin that holds
  // it (one radix level instead of all; a rank beyond the sample collects
  // every logit); every logit >= L is collected below
  auto lower_bound = [&](unsigned long long j, bool coarse) -> uint32_t {
    uint32_t Lk = 1u;  // every key is >= 1
    if (j >= 1ull && j < static_cast<unsigned long long>(kCap)) {
      if (coarse) {
        radix_select<KT, 1>(samp_src, none, false, 0u, Crit{true, j, 0.0}, h_cnt, h_mass, sel);
        if (sel.ok) Lk = sel.prefix << KT::shift(0);
      } else {
        radix_select<KT>(samp_src, none, false, 0u, Crit{true, j, 0.0}, h_cnt, h_mass, sel);
        if (sel.ok) Lk = sel.prefix;
      }
      if (Lk == 0u) Lk = 1u;
    }
    __syncthreads();  // the sample is no longer read
    return Lk;
  };
  // every key >= L into `col` (its count is exact), the row maximum and its
  // non-NaN count, and with `need_z` the total weight (the maximum known)
  float mx = -kInfF;
  uint32_t nan_n = 0u;
  unsigned long long z = 0ull;
  // need_max / need_z: std::true_type or std::false_type (each pass is
  // compiled with exactly the work it does per element)
  auto collect = [&](uint32_t L, auto need_max, auto need_z, const auto& wfz) {
    // compared as values (NaN never passes; -0 and +0 compare equal, as
    // their keys are equal); keys only for the logits collected
    const float Lf = L == 1u ? -kInfF : KT::value(L);
    for_each_raw<T>(row, a.V, [&](uint32_t raw) {
      const float x = KT::value_raw(raw);
      if constexpr (decltype(need_max)::value) {
        mx = fmaxf(mx, x);  // NaN never wins
        nan_n += x != x ? 1u : 0u;
      }
      if constexpr (decltype(need_z)::value) {
        if (x == x) z += svk::floor_u64(__fmul_rn(wfz(x), 0x1p40f));
      }
      if (x >= Lf) {
        uint32_t k;
        KT::key(raw, k);
        const int at = atomicAdd(&n_col, 1);
        if (at < kCap) col[at] = k;
      }
    });
  };
  auto reduce_max = [&]() -> uint32_t {  // the CTA's maximum into mx; returns the non-NaN count
    float wm = svk::warp_max_f(mx);
    uint32_t wn = __reduce_add_sync(0xFFFFFFFFu, nan_n);
    if (lane == 0) {
      r_max[warp] = wm;
      r_cnt[warp] = wn;
    }
    __syncthreads();
    mx = -kInfF;
    wn = 0u;
    for (int w = 0; w < kWarpsF; ++w) {
      mx = fmaxf(mx, r_max[w]);
      wn += r_cnt[w];
    }
    return static_cast<uint32_t>(a.V) - wn;
  };
  auto no_wf = [](float) { return 0.f; };

  uint32_t nn;
  if (use_k) {
    // top-k: one pass over the row collects every key >= L (the sample's
    // rank of 2k logits, taking every logit as non-NaN, plus a margin) and
    // takes the maximum and the non-NaN count on the way
    const uint32_t L = lower_bound(2ull * static_cast<unsigned long long>(kk) * kCap / a.V + 16ull, true);
    collect(L, std::true_type{}, std::false_type{}, no_wf);
    nn = reduce_max();
  } else {
    // top-p alone: the maximum first (the weights need it), then a pass that
    // collects every key >= L (the sample's rank of about 0.6 kCap logits:
    // a nucleus of up to a couple of thousand logits is then complete) and
    // sums the row's weight Z
    for_each_raw<T>(row, a.V, [&](uint32_t raw) {
      const float x = KT::value_raw(raw);
      mx = fmaxf(mx, x);
      nan_n += x != x ? 1u : 0u;
    });
    nn = reduce_max();
  }
  if (nn == 0u || !(mx > -kInfF && mx < kInfF)) {  // no finite maximum: no filter
    if (tid == 0) *out = -kInfF;
    return;
  }
  uint32_t kmax;
  KT::key(KT::raw_of(mx), kmax);
  const float m = KT::value(kmax);
  bool k_covers = use_k && static_cast<uint32_t>(kk) >= nn;  // k covers the row
  if (k_covers) use_k = false;
  if (!use_k && !use_p) {
    if (tid == 0) *out = -kInfF;
    return;
  }

  float khi = 0.f, klo = 0.f;
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
    return svk::floor_u64(__fmul_rn(wf(KT::value(k)), 0x1p40f));
  };
  auto col_src = [&](auto f) {
    const int n = min(n_col, kCap);
    for (int j = tid; j < n; j += kThreads) f(col[j]);
  };

  if (!use_k && !k_covers) {  // top-p alone: the collecting pass with Z
    const uint32_t L = lower_bound((6ull * kCap / 10ull) * kCap / nn, false);
    collect(L, std::false_type{}, std::true_type{}, wf);
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    if (lane == 0) r_z[warp] = z;
    __syncthreads();
    z = 0ull;
    for (int w = 0; w < kWarpsF; ++w) z += r_z[w];
  }
  __syncthreads();
  const int nc = n_col;
  // the collection holds every key >= L unless it overflowed; for top-k it
  // must also reach k keys (else the k-th largest lies below L).  A top-k
  // that covers the row leaves top-p alone without its Z: the full-row path.
  bool fast = !k_covers && nc <= kCap && (!use_k || nc >= kk);

  uint32_t key_k = 0u, key_p = 0u;
  if (fast) {
    if (use_k) {
      radix_select<KT>(col_src, none, false, 0u, Crit{true, static_cast<unsigned long long>(kk), 0.0}, h_cnt,
                       h_mass, sel);
      fast = sel.ok != 0;
      key_k = sel.prefix;
      key_p = key_k;
    }
    if (fast && use_p && key_k < kmax) {
      if (use_k) {  // Z over the top-k set, all of it collected; the set itself into tk
        if (tid == 0) n_tk = 0;
        __syncthreads();
        unsigned long long zk = 0ull;
        col_src([&](uint32_t k) {
          if (k < key_k) return;
          zk += weight(k);
          const int at = atomicAdd(&n_tk, 1);
          if (at < kTopSet) tk[at] = k;
        });
#pragma unroll
        for (int o = 16; o; o >>= 1) zk += __shfl_xor_sync(0xFFFFFFFFu, zk, o);
        __syncthreads();
        if (lane == 0) r_z[warp] = zk;
        __syncthreads();
        z = 0ull;
        for (int w = 0; w < kWarpsF; ++w) z += r_z[w];
      }
      const Crit cr{false, 0ull, static_cast<double>(p) * static_cast<double>(z)};
      if (use_k && n_tk <= kTopSet) {
        // a top-k set of at most kTopSet keys: warp 0 ranks them, sums the
        // weights in descending order and keeps the groups of equal keys
        // whose higher-ranked weight passes the test (the radix select's
        // rule, key by key)
        if (warp == 0) key_p = top_p_small(tk, n_tk, weight, cr);
        if (tid == 0) sel.prefix = key_p;
        __syncthreads();
        key_p = sel.prefix;
      } else {
        radix_select<KT>(col_src, weight, true, key_k, cr, h_cnt, h_mass, sel);
        // with top-k every key above the answer is collected; with top-p alone
        // the answer is the row's own once the test fails with its own group
        fast = sel.ok && (use_k || !cr.within(0ull, sel.m_above + sel.m_grp));
        key_p = sel.prefix;
      }
    }
  }
  if (!fast) {  // full-row radix selects
    auto row_src = [&](auto f) {
      for_each_raw<T>(row, a.V, [&](uint32_t raw) {
        uint32_t k;
        if (KT::key(raw, k)) f(k);
      });
    };
    key_k = 0u;
    if (use_k) {
      radix_select<KT>(row_src, none, false, 0u, Crit{true, static_cast<unsigned long long>(kk), 0.0}, h_cnt,
                       h_mass, sel);
      key_k = sel.ok ? sel.prefix : 0u;
    }
    key_p = key_k;
    if (use_p && key_k < kmax) {
      unsigned long long zr = 0ull;
      row_src([&](uint32_t k) {
        if (k >= key_k) zr += weight(k);
      });
#pragma unroll
      for (int o = 16; o; o >>= 1) zr += __shfl_xor_sync(0xFFFFFFFFu, zr, o);
      __syncthreads();
      if (lane == 0) r_z[warp] = zr;
      __syncthreads();
      zr = 0ull;
      for (int w = 0; w < kWarpsF; ++w) zr += r_z[w];
      radix_select<KT>(row_src, weight, true, key_k,
                       Crit{false, 0ull, static_cast<double>(p) * static_cast<double>(zr)}, h_cnt, h_mass, sel);
      if (sel.ok) key_p = sel.prefix;
    }
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
  return svh::sampler_floors_gated(target_logits, draft_logits, dtype, row_stride, temperature, top_k, top_p, cu_k,
                                   batch, k, sum_k, vocab, floor_target, floor_draft, nullptr, stream);
}

sv_status svh::sampler_floors_gated(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                                    int64_t row_stride, const float* temperature, const int32_t* top_k,
                                    const float* top_p, const int32_t* cu_k, int32_t batch, int32_t k,
                                    int32_t sum_k, int32_t vocab, float* floor_target, float* floor_draft,
                                    const int* gate, void* stream) {
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
  a.gate = gate;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case SV_F32: return svf::launch<float>(a, st);
    case SV_BF16: return svf::launch<__nv_bfloat16>(a, st);
    default: return svf::launch<__half>(a, st);
  }
}
