// Helpers of the row-parallel kernel's fused top-k / top-p path (16-bit
// logits): order-preserving keys, radix selects over shared-memory key sets,
// and the top-p walk.  The definitions are those of include/sv_filter.h and
// the floors kernel (sv_filter.cu): the top-k floor is the k-th largest
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
// their orders and weights [2][kTopKMax] (4 + 4 + 8 B), 32 scalars
constexpr int kTopkScratch = 2 * kKeptCap * 8 + 2 * kKeptCap * 4 + 2 * 256 * 4 + 2 * kTopKMax * 16 + 32 * 4;

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

// One count into hist[bin], aggregated over the lanes of the warp that add
// to the same bin at this point (keys of a row crowd into few bins).
__device__ __forceinline__ void hist_add(unsigned* hist, uint32_t bin) {
  const unsigned act = __activemask();
  const unsigned same = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(same) - 1)) atomicAdd(&hist[bin], __popc(same));
}

// A slot in a shared-memory list for every lane whose `pred` holds (one
// atomic per warp); -1 for the other lanes.
__device__ __forceinline__ int warp_append(int* counter, bool pred) {
  const unsigned act = __activemask();
  const unsigned b = __ballot_sync(act, pred);
  if (!b) return -1;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(b) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(b));
  base = __shfl_sync(act, base, leader);
  return pred ? base + __popc(b & ((1u << lane) - 1u)) : -1;
}

// The lim-th largest key of a source when it lies within 255 keys of the
// largest key kmax: one histogram of kmax - k over the keys in that window
// (the rest of the row passes without an atomic).  Returns 0 when fewer than
// lim keys lie in the window (the caller then takes kth_largest16).
template <typename Src>
__device__ __forceinline__ uint32_t kth_near_max16(const Src& src, uint32_t kmax, unsigned lim, unsigned* hist,
                                                   int* pick) {
  const int tid = threadIdx.x;
  __syncthreads();  // earlier readers of hist and pick are done
  hist[tid] = 0u;
  __syncthreads();
  src([&](uint32_t k) {
    const uint32_t d = kmax - k;
    if (d < 256u) hist_add(hist, 255u - d);  // bin 255: kmax itself
  });
  __syncthreads();
  if (tid < 32) {
    unsigned tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) tot += hist[tid * 8 + j];
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
    unsigned ab = 0;
    const int bin = tot >= lim ? pick_bin_count(hist, 0u, lim, ab) : -1;
    if (tid == 0) pick[0] = bin;
  }
  __syncthreads();
  const int bin = pick[0];
  return bin < 0 ? 0u : kmax - (255u - static_cast<uint32_t>(bin));
}

// The lim-th largest 16-bit key of a key source (CTA collective, 256
// threads): two radix levels of 8 bits over shared-memory histograms.
// src(f) calls f(key) for every key of the set (each thread its share).
// Returns 0 for an empty set.  `hist` holds 256 counters; `pick` two ints.
template <typename Src>
__device__ __forceinline__ uint32_t kth_largest16(const Src& src, unsigned lim, unsigned* hist, int* pick) {
  const int tid = threadIdx.x;
  uint32_t hi = 0;
  unsigned above = 0;
  for (int level = 0; level < 2; ++level) {
    __syncthreads();  // earlier readers of hist and pick are done
    hist[tid] = 0u;
    __syncthreads();
    src([&](uint32_t k) {
      if (level == 0) hist_add(hist, k >> 8);
      else if ((k >> 8) == hi) hist_add(hist, k & 0xFFu);
    });
    __syncthreads();
    if (tid < 32) {
      unsigned ab = 0;
      const int bin = pick_bin_count(hist, above, lim, ab);
      if (tid == 0) {
        pick[0] = bin;
        pick[1] = static_cast<int>(ab);
      }
    }
    __syncthreads();
    const int bin = pick[0];
    if (bin < 0) return 0u;
    if (level == 0) {
      hi = static_cast<uint32_t>(bin);
      above = static_cast<unsigned>(pick[1]);
    } else {
      return (hi << 8) | static_cast<uint32_t>(bin);
    }
  }
  return 0u;
}

// Warp: the top-p floor key of a set of n <= kTopKMax keys tk[0..n): walking
// the distinct keys from the largest, the lowest key whose higher-ranked
// weight (keys strictly above it) is below m_lim.  `ord` holds kTopKMax
// words and `ordw` kTopKMax weights.  Returns the key on every lane (0 when
// n = 0).
template <typename WFn>
__device__ __forceinline__ uint32_t top_p_walk(const uint32_t* tk, int n, const WFn& weight, double m_lim,
                                               uint32_t* ord, unsigned long long* ordw) {
  const int lane = threadIdx.x & 31;
  for (int h = 0; h < kTopKMax / 32; ++h) {
    const int j = lane + 32 * h;
    if (j >= n) continue;
    const uint32_t kj = tk[j];
    int rank = 0;
    for (int m = 0; m < n; ++m) {
      const uint32_t km = tk[m];
      rank += (km > kj || (km == kj && m < j)) ? 1 : 0;
    }
    ord[rank] = kj;
    ordw[rank] = weight(kj);
  }
  __syncwarp();
  uint32_t ans = 0u;
  if (lane == 0) {
    unsigned long long above = 0ull;  // weight of the keys strictly above the current group
    int j = 0;
    while (j < n) {
      const uint32_t g = ord[j];
      if (!(static_cast<double>(above) < m_lim)) break;
      ans = g;
      unsigned long long w = 0ull;
      while (j < n && ord[j] == g) {
        w += ordw[j];
        ++j;
      }
      above += w;
    }
  }
  __syncwarp();
  return __shfl_sync(0xFFFFFFFFu, ans, 0);
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

// f(key, e) for every non-NaN element e of a 16-bit shared-memory slice
// (each of the CTA's 256 threads its share; 16-byte vectors, then the tail).
template <typename T, typename F>
__device__ __forceinline__ void for_keys16(const T* s, int n, F&& f) {
  using KY = Key16x<T>;
  const int nv = n / 8;
  for (int vi = threadIdx.x; vi < nv; vi += 256) {
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t k;
      if (KY::key(w[q] & 0xFFFFu, k)) f(k, vi * 8 + 2 * q);
      if (KY::key(w[q] >> 16, k)) f(k, vi * 8 + 2 * q + 1);
    }
  }
  for (int e = nv * 8 + static_cast<int>(threadIdx.x); e < n; e += 256) {
    uint32_t k;
    if (KY::key(reinterpret_cast<const unsigned short*>(s)[e], k)) f(k, e);
  }
}

// f(value, e) for every element e of a 16-bit shared-memory slice whose value
// is at least `lo` (a value of the row's type; the row holds no NaN): the
// comparison runs on the unpacked floats, the caller's work only on the few
// elements that pass.
template <typename T, typename F>
__device__ __forceinline__ void for_values_at_least(const T* s, int n, float lo, F&& f) {
  const int nv = n / 8;
  for (int vi = threadIdx.x; vi < nv; vi += 256) {
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float a, c;
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        a = bf_lo(w[q]);
        c = bf_hi(w[q]);
      } else {
        a = h_lo(w[q]);
        c = h_hi(w[q]);
      }
      if (a >= lo) f(w[q] & 0xFFFFu, vi * 8 + 2 * q);
      if (c >= lo) f(w[q] >> 16, vi * 8 + 2 * q + 1);
    }
  }
  for (int e = nv * 8 + static_cast<int>(threadIdx.x); e < n; e += 256) {
    const unsigned short raw = reinterpret_cast<const unsigned short*>(s)[e];
    if (ElemTraits<T>::to_f(s[e]) >= lo) f(static_cast<uint32_t>(raw), e);
  }
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
