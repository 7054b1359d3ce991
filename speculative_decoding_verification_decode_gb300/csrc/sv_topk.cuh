// Helpers of the row-parallel kernel's fused top-k / top-p path (16-bit
// logits): order-preserving keys, selects over small key sets, packed scans
// of shared-memory slices, and the top-p walk.  The definitions are those of
// include/sv_filter.h and the floors kernel (sv_filter.cu): the top-k floor is the k-th largest
// logit (ties kept); the top-p floor is, among the top-k tokens, the lowest
// logit whose higher-ranked weight (fp32 weights truncated to multiples of
// 2^-40, summed exactly as integers) is still below p times the set's total,
// compared in fp64.
#pragma once
#include "sv_kernel.cuh"

namespace svk {

constexpr int kTopKMax = 64;    // top-k sizes the fused path takes
constexpr int kListCap = 256;   // candidates a CTA may contribute per row
constexpr int kKeptCap = 256;   // kept tokens per row the fused decision and draw take
// rank 0's work space beyond its receive area: kept sets [2][kKeptCap] (8 B),
// two index orders [kKeptCap] (4 B), two 256-bin histograms, the top-k sets,
// their orders, weights and entries [2][kTopKMax] (4 + 4 + 8 + 8 B), 32 scalars
constexpr int kTopkScratch = 2 * kKeptCap * 8 + 2 * kKeptCap * 4 + 2 * 256 * 4 + 2 * kTopKMax * 24 + 32 * 4;

// Order-preserving 16-bit keys of bf16 / f16 bits: negative values flipped,
// positive ones with the sign bit set, -0 keyed as +0.  NaN has no key.
template <typename T>
struct Key16x {
  static constexpr uint32_t kInfBits = std::is_same<T, __nv_bfloat16>::value ? 0x7F80u : 0x7C00u;
  __device__ __forceinline__ static bool key(uint32_t raw, uint32_t& k) {
    if ((raw & 0x7FFFu) > kInfBits) return false;
    if ((raw & 0x7FFFu) == 0u) raw = 0u;
    k = (raw & 0x8000u) ? (~raw & 0xFFFFu) : (raw | 0x8000u);
    return true;
  }
  __device__ __forceinline__ static uint32_t raw(uint32_t k) {  // the bits of a key's value
    return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    const uint32_t raw = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(raw << 16);
    else return __half2float(__ushort_as_half(static_cast<unsigned short>(raw)));
  }
};

// Warp: the lowest non-empty bin of hist[0..256) whose count of keys in
// higher bins, plus `above`, is below `lim` (the bin holding the lim-th
// largest key, or the lowest non-empty bin when fewer keys exist).  Lane l
// covers bins 8l..8l+7.  Returns the bin (-1 if every bin is empty) and the
// count above it in `out_above`.
__device__ __forceinline__ int pick_bin_count(const unsigned* hist, unsigned above, unsigned lim,
                                              unsigned& out_above) {
  const int lane = threadIdx.x & 31;
  unsigned h[8];
  unsigned c = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = hist[lane * 8 + j];
    c += h[j];
  }
  unsigned sc = c;  // inclusive sum over lanes >= this one
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_down_sync(0xFFFFFFFFu, sc, o);
    if (lane + o < 32) sc += t;
  }
  unsigned ab = above + (sc - c);  // keys in bins above this lane's range
  int mine = -1;
  unsigned mine_above = 0;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (h[j] && ab < lim) {
      mine = lane * 8 + j;
      mine_above = ab;
    }
    ab += h[j];
  }
  const unsigned has = __ballot_sync(0xFFFFFFFFu, mine >= 0);
  if (!has) return -1;
  const int L = __ffs(has) - 1;
  out_above = __shfl_sync(0xFFFFFFFFu, mine_above, L);
  return __shfl_sync(0xFFFFFFFFu, mine, L);
}

// Warp: the top-p floor key of a set of n <= kTopKMax keys tk[0..n): among
// the distinct keys, the lowest whose higher-ranked weight (the keys strictly
// above it) is below m_lim.  The keys are ranked into descending order
// (`ord`, with their weights in `ordw`), their weights prefix-summed, and the
// test taken at every group's first position at once: the weight above grows
// down the ranking, so the passing groups are a prefix of it and the answer
// is the last of them.  Returns the key on every lane (0 when n = 0).
template <typename WFn>
__device__ __forceinline__ uint32_t top_p_walk(const uint32_t* tk, int n, const WFn& weight, double m_lim,
                                               uint32_t* ord, unsigned long long* ordw) {
  const int lane = threadIdx.x & 31;
  for (int h = 0; h < kTopKMax / 32; ++h) {
    const int j = lane + 32 * h;
    if (j >= n) continue;
    const uint32_t kj = tk[j];
    int rank = 0;
#pragma unroll 8
    for (int m = 0; m < n; ++m) {
      const uint32_t km = tk[m];
      rank += (km > kj || (km == kj && m < j)) ? 1 : 0;
    }
    ord[rank] = kj;
    ordw[rank] = weight(kj);
  }
  __syncwarp();
  // lane l holds ranks 2l and 2l + 1: their exclusive prefix of weight
  static_assert(kTopKMax == 64, "two ranks per lane");
  const int r0 = 2 * lane, r1 = r0 + 1;
  const unsigned long long w0 = r0 < n ? ordw[r0] : 0ull, w1 = r1 < n ? ordw[r1] : 0ull;
  unsigned long long inc = w0 + w1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += t;
  }
  const unsigned long long ex0 = inc - w0 - w1, ex1 = ex0 + w0;
  // a group starts at rank r when r is 0 or its key differs from rank r - 1's
  const bool g0 = r0 < n && (r0 == 0 || ord[r0] != ord[r0 - 1]);
  const bool g1 = r1 < n && ord[r1] != ord[r0];
  const bool p0 = g0 && static_cast<double>(ex0) < m_lim;
  const bool p1 = g1 && static_cast<double>(ex1) < m_lim;
  const unsigned b0 = __ballot_sync(0xFFFFFFFFu, p0), b1 = __ballot_sync(0xFFFFFFFFu, p1);
  // the last passing group start in rank order
  int best = -1;
  if (b0 | b1) {
    const int l0 = b0 ? 31 - __clz(b0) : -1, l1 = b1 ? 31 - __clz(b1) : -1;
    best = max(l0 >= 0 ? 2 * l0 : -1, l1 >= 0 ? 2 * l1 + 1 : -1);
  }
  __syncwarp();
  return best >= 0 ? ord[best] : 0u;
}

// NaN-propagating maximum of a 16-bit shared-memory slice (+-Inf count as
// values): the thread's partial over 16-byte vectors and the tail.
template <typename T>
__device__ __forceinline__ float slice_max_nan16(const T* s, int n) {
  constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
  const int nv = n / 8;
  uint32_t h = kBf ? 0xFF80FF80u : 0xFC00FC00u;
  for (int vi = threadIdx.x; vi < nv; vi += 256) {
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    if constexpr (kBf) h = bf16x2_max_nan(h, bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w)));
    else h = f16x2_max_nan(h, f16x2_max_nan(f16x2_max_nan(v.x, v.y), f16x2_max_nan(v.z, v.w)));
  }
  float m = kBf ? fmax_nan(bf_lo(h), bf_hi(h)) : fmax_nan(h_lo(h), h_hi(h));
  for (int e = nv * 8 + static_cast<int>(threadIdx.x); e < n; e += 256) m = fmax_nan(m, ElemTraits<T>::to_f(s[e]));
  return m;
}

// 0xFFFF in each 16-bit half of a packed pair a that is >= the same half of
// t (an ordered compare: NaN gives 0).
template <typename T>
__device__ __forceinline__ uint32_t ge_mask2(uint32_t a, uint32_t t) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value)
    return __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&t));
  else
    return __hge2_mask(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&t));
}

// The elements of a 16-bit shared-memory slice (no NaN) whose value is at
// least that of key `lo_key`, as seen by one thread of 256.  count() counts
// this thread's share with one packed compare per pair of elements and
// remembers up to kMarks of the 16-byte vectors that hold one; visit(f) then
// calls f(key, e) for each of those elements, in vector order, looking only
// into the remembered vectors (into all of them when there were more).
template <typename T>
struct KeysAtLeast16 {
  static constexpr int kMarks = 4;
  const T* s;
  int n;
  uint32_t t2;  // the floor's bits in both halves
  int nm = 0;   // vectors of this thread that hold an element
  int vm[kMarks] = {0, 0, 0, 0};
  __device__ __forceinline__ KeysAtLeast16(const T* s_, int n_, uint32_t lo_key) : s(s_), n(n_) {
    const uint32_t r = Key16x<T>::raw(lo_key);
    t2 = r | (r << 16);
  }
  __device__ __forceinline__ unsigned count() {
    const int nv = n / 8;
    unsigned c = 0u;
    for (int vi = threadIdx.x; vi < nv; vi += 256) {
      const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
      const unsigned cv = __popc(ge_mask2<T>(v.x, t2)) + __popc(ge_mask2<T>(v.y, t2)) +
                          __popc(ge_mask2<T>(v.z, t2)) + __popc(ge_mask2<T>(v.w, t2));
      if (cv) {
#pragma unroll
        for (int j = 0; j < kMarks; ++j)
          if (nm == j) vm[j] = vi;
        ++nm;
      }
      c += cv;
    }
    c >>= 4;  // 16 mask bits per element
    for (int e = nv * 8 + static_cast<int>(threadIdx.x); e < n; e += 256)
      c += ge_mask2<T>(reinterpret_cast<const unsigned short*>(s)[e], t2) & 1u;
    return c;
  }
  template <typename F>
  __device__ __forceinline__ void emit(int vi, F& f) const {
    using KY = Key16x<T>;
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t m = ge_mask2<T>(w[q], t2);
      uint32_t k = 0u;
      if (m & 0xFFFFu) {
        KY::key(w[q] & 0xFFFFu, k);
        f(k, vi * 8 + 2 * q);
      }
      if (m >> 16) {
        KY::key(w[q] >> 16, k);
        f(k, vi * 8 + 2 * q + 1);
      }
    }
  }
  template <typename F>
  __device__ __forceinline__ void visit(F&& f) const {
    const int nv = n / 8;
    if (nm <= kMarks) {
#pragma unroll
      for (int j = 0; j < kMarks; ++j)
        if (j < nm) emit(vm[j], f);
    } else {
      for (int vi = threadIdx.x; vi < nv; vi += 256) {
        const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
        if ((ge_mask2<T>(v.x, t2) | ge_mask2<T>(v.y, t2) | ge_mask2<T>(v.z, t2) | ge_mask2<T>(v.w, t2)) != 0u)
          emit(vi, f);
      }
    }
    for (int e = nv * 8 + static_cast<int>(threadIdx.x); e < n; e += 256) {
      const uint32_t raw = reinterpret_cast<const unsigned short*>(s)[e];
      if (ge_mask2<T>(raw, t2) & 1u) {
        uint32_t k = 0u;
        Key16x<T>::key(raw, k);
        f(k, e);
      }
    }
  }
};

// Warp: the lim-th largest of 256 keys keys[0..256) (lim in [1, 256]): the
// largest L with at least lim keys >= L, by bisection between the smallest
// and the largest key.
__device__ __forceinline__ uint32_t kth_of_256(const uint32_t* keys, unsigned lim) {
  const int lane = threadIdx.x & 31;
  uint32_t v[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = keys[q * 32 + lane];
  uint32_t lo = v[0], hi = v[0];
#pragma unroll
  for (int q = 1; q < 8; ++q) {
    lo = min(lo, v[q]);
    hi = max(hi, v[q]);
  }
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);  // every key is >= lo: the answer is in [lo, hi]
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
#pragma unroll 1
  while (lo < hi) {
    const uint32_t c = lo + (hi - lo + 1u) / 2u;
    unsigned cnt = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) cnt += v[q] >= c ? 1u : 0u;
    if (__reduce_add_sync(0xFFFFFFFFu, cnt) >= lim) lo = c;
    else hi = c - 1u;
  }
  return lo;
}

// Warp: appends the lanes whose `pred` holds to list[*n..] in lane order
// (the count in *n, a register every lane holds; entries past cap are
// dropped but counted).
template <typename E>
__device__ __forceinline__ void warp_compact(bool pred, const E& e, E* list, int cap, int& n) {
  const unsigned b = __ballot_sync(0xFFFFFFFFu, pred);
  const int lane = threadIdx.x & 31;
  const int at = n + __popc(b & ((1u << lane) - 1u));
  if (pred && at < cap) list[at] = e;
  n += __popc(b);
}

}  // namespace svk
