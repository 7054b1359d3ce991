// Verification kernel: one thread-block cluster per sequence, one V-slice per CTA.
//
// Work of one sequence b (K_b drafts, rows 0..K_b):
//   * a producer warp streams this CTA's slice of every needed row into a
//     shared-memory ring with 1-D bulk copies (cp.async.bulk, full/empty
//     mbarriers), running ahead of the consumers by up to S chunks;
//   * eight consumer warps reduce each chunk (argmax, row mass, or an online
//     softmax with a tracked error bound);
//   * per row the CTAs combine their partial statistics through distributed
//     shared memory: each CTA pushes a small record into every peer and
//     arrives on the peer's mbarrier; every CTA then takes the same decision
//     from the same records in the same order (no global-memory scratch);
//   * greedy chunks are released as soon as they are reduced; in sampling mode
//     the current row pair stays resident until its decision, so the exact
//     fallback, the residual and the inverse-CDF scan read shared memory only;
//   * the walk stops at the first miss / rejection; later rows are not read
//     (chunks already in flight are drained before exit).
//
// Decisions in sampling mode are the exact real predicate
//     u * q(t) * Zp  <  p(t) * Zq
// on the exact sums Zp, Zq of the f32 row weights: an approximate sum with a
// rigorous error bound decides whenever the bound allows, otherwise the CTAs
// sum the resident rows exactly (integer significand buckets, 32-bit limbs)
// and compare big integers.  Inverse-CDF draws run in 64-bit fixed point so
// every level (vector, thread, block, cluster) of the scan is consistent.
#pragma once
#include <cfloat>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "sv_ptx.cuh"

namespace svk {

constexpr int kConsumers = 256;  // consumer threads (8 warps)
constexpr int kWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxSlots = 16;
constexpr int kMaxSlotBytes = 32768;
constexpr int kMaxCluster = 16;
constexpr int kRecWords = 32;
constexpr int kBuckets = 254;
constexpr int kLimbs = 12;
constexpr int kBigLimbs = 32;

enum : int { MODE_GREEDY = 0, MODE_PROBS = 1, MODE_LOGITS = 2 };

#define kInfF (__uint_as_float(0x7F800000u))

constexpr uint32_t ST_BAD_TOKEN = 1u, ST_BAD_VALUE = 2u, ST_ZERO_MASS = 4u, ST_NEAR = 8u,
                   ST_EXACT = 16u, ST_TIMEOUT = 32u, ST_BAD_LAYOUT = 64u;
constexpr uint32_t FLAG_FORCE_EXACT = 1u;

constexpr double kU32 = 5.9604644775390625e-8;  // 2^-24, unit roundoff of f32
// Relative error bound used for ex2.approx.ftz.f32 (normal results); the
// measured maximum on GB300 is checked against it by a GPU test.
constexpr double kEx2Rel = 4.76837158203125e-7;  // 2^-21

struct Params {
  const void* tgt;
  const void* drf;
  long long stride;  // row stride in elements
  const int* tok;
  const float* uni;
  const int* cu_k;
  const float* temp;
  int B, K, V, sum_k;
  int* n_out;
  int* next_out;
  unsigned* st_out;
  float* wt_out;
  float* wd_out;
  unsigned flags;
  int slice;       // elements per CTA slice (multiple of the vector width)
  int slot_bytes;  // bytes per ring slot (multiple of 16)
  int S;           // ring slots
  int use_tma;
  int fixed_shift;
  int vsum_off;  // byte offset of the per-vector draw sums (sampling)
  int tail_off;  // byte offset of SmemTail
};

struct __align__(16) SmemTail {
  uint32_t recs[2][kMaxCluster][kRecWords];
  uint32_t myrec[kRecWords];
  double redd[kWarps * 4];
  unsigned long long redu[kWarps];
  float redf[kWarps * 2];
  int redi[kWarps * 2];
  uint64_t xbar[2];
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  double bd[8];    // broadcast of decision inputs from thread 0
  int bi[8];
  volatile int stop;  // consumers -> producer: issue nothing more
};

// ------------------------------------------------------------------ element types

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<float> {
  static constexpr int kVec = 4;
  static constexpr int kFlush = 8;  // vectors per fp32 partial (32 elements)
  __device__ static float to_f(float x) { return x; }
};
template <>
struct ElemTraits<__nv_bfloat16> {
  static constexpr int kVec = 8;
  static constexpr int kFlush = 4;
  __device__ static float to_f(__nv_bfloat16 x) {
    return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(x)) << 16);
  }
};
template <>
struct ElemTraits<__half> {
  static constexpr int kVec = 8;
  static constexpr int kFlush = 4;
  __device__ static float to_f(__half x) { return __half2float(x); }
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float h_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float h_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Load vector `vi` (16 bytes) of a shared-memory chunk as floats.
template <typename T>
__device__ __forceinline__ void load_vec(const T* s, int vi, float* x) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  } else {
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        x[2 * k] = bf_lo(w[k]);
        x[2 * k + 1] = bf_hi(w[k]);
      } else {
        x[2 * k] = h_lo(w[k]);
        x[2 * k + 1] = h_hi(w[k]);
      }
    }
  }
}

// NaN-propagating max of vector `vi` (packed for 16-bit types).
template <typename T>
__device__ __forceinline__ float vec_max_nan(const T* s, int vi) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    return fmax_nan(fmax_nan(v.x, v.y), fmax_nan(v.z, v.w));
  } else {
    const uint4 v = reinterpret_cast<const uint4*>(s)[vi];
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
      const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
      return fmax_nan(bf_lo(m), bf_hi(m));
    } else {
      const uint32_t m = f16x2_max_nan(f16x2_max_nan(v.x, v.y), f16x2_max_nan(v.z, v.w));
      return fmax_nan(h_lo(m), h_hi(m));
    }
  }
}

// Pairwise sum of N floats (depth log2 N).
template <int N>
__device__ __forceinline__ float tree_sum(const float* x) {
  if constexpr (N == 1) {
    return x[0];
  } else {
    return __fadd_rn(tree_sum<N / 2>(x), tree_sum<N / 2>(x + N / 2));
  }
}

// ------------------------------------------------------------------ accumulators

// fp32 partial sums of at most kFlush vectors, folded into an fp64 total.
// Each element passes through at most 3 (vector tree) + 7 (partial) fp32
// roundings, so the total is within 10 * 2^-24 (relative) of the exact sum.
struct Acc {
  double d;
  float f;
  int c;
  __device__ __forceinline__ void init() {
    d = 0.0;
    f = 0.f;
    c = 0;
  }
  template <int kFlush>
  __device__ __forceinline__ void add(float t) {
    f = __fadd_rn(f, t);
    if (++c == kFlush) {
      d += static_cast<double>(f);
      f = 0.f;
      c = 0;
    }
  }
  __device__ __forceinline__ double total() const { return d + static_cast<double>(f); }
};

// ------------------------------------------------------------------ logits -> weights

// The defined weights of a warped row (the values whose exact sum is the
// row mass): w = 2^((l - m) * k) with m the row maximum and k = log2(e)/T.
// 16-bit logits: one fp32 subtract and multiply, then ex2.approx.ftz.
struct Warp16 {
  float m, k;
  __device__ __forceinline__ float operator()(float l) const {
    return ex2_ftz(__fmul_rn(__fsub_rn(l, m), k));
  }
};

// f32 logits: l - m as an exact two-term sum, the product with the
// double-float k = khi + klo kept to about 2^-40, and the low part applied as
// a first-order correction to 2^hi.
struct Warp32 {
  float m, khi, klo;
  __device__ __forceinline__ float operator()(float l) const {
    const float s = __fsub_rn(l, m);
    const float bb = __fsub_rn(s, l);
    const float err = __fadd_rn(__fsub_rn(l, __fsub_rn(s, bb)), __fsub_rn(-m, bb));
    const float xh = __fmul_rn(s, khi);
    const float xl = __fadd_rn(__fmaf_rn(s, khi, -xh), __fmaf_rn(s, klo, __fmul_rn(err, khi)));
    const float e0 = ex2_ftz(xh);
    return e0 == 0.f ? 0.f : __fmaf_rn(e0, __fmul_rn(xl, 0.6931471805599453f), e0);
  }
};

template <typename T>
struct WarpOf {
  using type = Warp16;
};
template <>
struct WarpOf<float> {
  using type = Warp32;
};

struct NoWarp {
  __device__ __forceinline__ float operator()(float x) const { return x; }
};

// Online softmax of one thread's elements: running maximum m, and
//   s = sum 2^(-nx),  w = sum 2^(-nx) * nx,   nx = (m - l) * k >= 0,
// rescaled when m grows.  It approximates the row mass Z = sum w_v of the
// defined weights; the error bound is
//   |S - Z| <= S * ((R + 2)(e + u) + 2e + 16u) + W * 4 ln2 u   (times 2)
// with e the ex2 bound, u = 2^-24 and R the number of rescale steps.
struct Online {
  float m;
  float s32, w32;
  double s64, w64;
  int nv, r;
  __device__ __forceinline__ void init() {
    m = -kInfF;
    s32 = w32 = 0.f;
    s64 = w64 = 0.0;
    nv = 0;
    r = 0;
  }
  __device__ __forceinline__ void rescale_to(float mnew, float k) {
    const float d = __fmul_rn(__fsub_rn(mnew, m), k);
    const float f = ex2_ftz(-d);
    w64 = (w64 + static_cast<double>(d) * s64) * static_cast<double>(f);
    s64 *= static_cast<double>(f);
    w32 = __fmul_rn(__fmaf_rn(d, s32, w32), f);
    s32 = __fmul_rn(s32, f);
    m = mnew;
    ++r;
  }
  template <int VEC, int FL>
  __device__ __forceinline__ void add_vec(const float* x, float vm, float k) {
    if (!(vm <= m)) {
      if (!(vm > -kInfF)) return;  // NaN (flagged by the caller) or all -Inf
      if (m == -kInfF) m = vm;
      else rescale_to(vm, k);
    }
    if (m == -kInfF) return;
    float e[VEC];
    float wa = 0.f, wb = 0.f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const float nx = fminf(__fmul_rn(__fsub_rn(m, x[j]), k), 3.0e38f);
      e[j] = ex2_ftz(-nx);
      if (j & 1) wb = __fmaf_rn(e[j], nx, wb);
      else wa = __fmaf_rn(e[j], nx, wa);
    }
    s32 = __fadd_rn(s32, tree_sum<VEC>(e));
    w32 = __fadd_rn(w32, __fadd_rn(wa, wb));
    if (++nv == FL) {
      s64 += static_cast<double>(s32);
      w64 += static_cast<double>(w32);
      s32 = w32 = 0.f;
      nv = 0;
    }
  }
  __device__ __forceinline__ double S() const { return s64 + static_cast<double>(s32); }
  __device__ __forceinline__ double W() const { return w64 + static_cast<double>(w32); }
};

__device__ __forceinline__ double online_bound(double S, double W, int R) {
  const double cs = (R + 2) * (kEx2Rel + kU32) + 2.0 * kEx2Rel + 16.0 * kU32;
  const double cw = 4.0 * 0.6931471805599453 * kU32;
  return 2.0 * (S * cs + W * cw) + 1e-30;
}

// ------------------------------------------------------------------ block reductions (consumers)

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Sums of up to four doubles across the consumer threads (fixed order).
template <int N>
__device__ __forceinline__ void block_sum_dn(double* v, double* red) {
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = warp_sum_d(v[j]);
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int j = 0; j < N; ++j) red[j * kWarps + (threadIdx.x >> 5)] = v[j];
  bar_consumers<kConsumers>();
#pragma unroll
  for (int j = 0; j < N; ++j) {
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[j * kWarps + w];
    v[j] = s;
  }
  bar_consumers<kConsumers>();
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  bar_consumers<kConsumers>();
  unsigned long long s = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) s += red[w];
  bar_consumers<kConsumers>();
  return s;
}

// kOp 0: NaN-propagating max, 1: NaN-propagating min, of two floats at once.
template <int kOp>
__device__ __forceinline__ void block_ext_f2(float& a, float& b, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float x = __shfl_xor_sync(0xFFFFFFFFu, a, o);
    const float y = __shfl_xor_sync(0xFFFFFFFFu, b, o);
    a = kOp == 0 ? fmax_nan(a, x) : fmin_nan(a, x);
    b = kOp == 0 ? fmax_nan(b, y) : fmin_nan(b, y);
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = a;
    red[kWarps + (threadIdx.x >> 5)] = b;
  }
  bar_consumers<kConsumers>();
  a = red[0];
  b = red[kWarps];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    a = kOp == 0 ? fmax_nan(a, red[w]) : fmin_nan(a, red[w]);
    b = kOp == 0 ? fmax_nan(b, red[kWarps + w]) : fmin_nan(b, red[kWarps + w]);
  }
  bar_consumers<kConsumers>();
}

__device__ __forceinline__ int block_max_i(int v, int* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  bar_consumers<kConsumers>();
  int s = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) s = max(s, red[w]);
  bar_consumers<kConsumers>();
  return s;
}

// Argmax candidate ordering: a valid index beats "none" (INT_MAX); larger value
// wins; equal values go to the lower index.  NaN never enters a candidate.
__device__ __forceinline__ bool arg_better(float va, int ia, float vb, int ib) {
  if (ia == INT_MAX) return false;
  if (ib == INT_MAX) return true;
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void block_argmax(float& v, int& i, float* redf, int* redi) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int j = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (arg_better(w, j, v, i)) {
      v = w;
      i = j;
    }
  }
  if ((threadIdx.x & 31) == 0) {
    redf[threadIdx.x >> 5] = v;
    redi[threadIdx.x >> 5] = i;
  }
  bar_consumers<kConsumers>();
  v = redf[0];
  i = redi[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w)
    if (arg_better(redf[w], redi[w], v, i)) {
      v = redf[w];
      i = redi[w];
    }
  bar_consumers<kConsumers>();
}

__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v,
                                                                  unsigned long long* red,
                                                                  unsigned long long& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) red[w] = inc;
  bar_consumers<kConsumers>();
  unsigned long long before = 0, tot = 0;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) {
    if (k < w) before += red[k];
    tot += red[k];
  }
  bar_consumers<kConsumers>();
  total = tot;
  return before + inc - v;
}

// ------------------------------------------------------------------ exact arithmetic

__device__ __forceinline__ void f32_parts(float x, uint32_t& M, int& s) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t e = (b >> 23) & 0xFFu, f = b & 0x7FFFFFu;
  M = e ? (f | 0x800000u) : f;
  s = e ? static_cast<int>(e) - 1 : 0;  // x = M * 2^(s - 149)
}

__device__ __forceinline__ void bucket_add(unsigned long long* bk, float x) {
  uint32_t M;
  int s;
  f32_parts(x, M, s);
  if (M) atomicAdd(&bk[s], static_cast<unsigned long long>(M));
}

// sum_s bk[s] * 2^s  ->  kLimbs little-endian 32-bit limbs.
__device__ __noinline__ void buckets_to_limbs(const unsigned long long* bk, uint32_t* limbs) {
  unsigned long long acc[kLimbs];
  for (int i = 0; i < kLimbs; ++i) acc[i] = 0;
  for (int s = 0; s < kBuckets; ++s) {
    const unsigned long long v = bk[s];
    if (!v) continue;
    const int w = s >> 5, off = s & 31;
    const unsigned long long lo = v << off;
    const unsigned long long hi = off ? (v >> (64 - off)) : 0ull;
    acc[w] += lo & 0xFFFFFFFFull;
    acc[w + 1] += lo >> 32;
    acc[w + 2] += hi;
  }
  unsigned long long carry = 0;
  for (int i = 0; i < kLimbs; ++i) {
    const unsigned long long t = acc[i] + carry;
    limbs[i] = static_cast<uint32_t>(t);
    carry = t >> 32;
  }
}

struct Big {
  uint32_t w[kBigLimbs];
};

__device__ __forceinline__ void big_set(Big& a, const uint32_t* limbs) {
  for (int i = 0; i < kBigLimbs; ++i) a.w[i] = i < kLimbs ? limbs[i] : 0u;
}

__device__ __forceinline__ void big_mul_u32(Big& a, uint32_t m) {
  unsigned long long carry = 0;
  for (int i = 0; i < kBigLimbs; ++i) {
    const unsigned long long t = static_cast<unsigned long long>(a.w[i]) * m + carry;
    a.w[i] = static_cast<uint32_t>(t);
    carry = t >> 32;
  }
}

__device__ __forceinline__ void big_shl(Big& a, int bits) {
  const int q = bits >> 5, r = bits & 31;
  for (int i = kBigLimbs - 1; i >= 0; --i) {
    const int src = i - q;
    uint32_t v = 0;
    if (src >= 0) {
      v = a.w[src] << r;
      if (r && src - 1 >= 0) v |= a.w[src - 1] >> (32 - r);
    }
    a.w[i] = v;
  }
}

__device__ __forceinline__ int big_cmp(const Big& a, const Big& b) {
  for (int i = kBigLimbs - 1; i >= 0; --i)
    if (a.w[i] != b.w[i]) return a.w[i] < b.w[i] ? -1 : 1;
  return 0;
}

// Exact  u * q_t * Sp  <  p_t * Sq  (both sides scaled by 2^447; see f32_parts).
__device__ __noinline__ bool exact_accept(float u, float pt, float qt, const uint32_t* sp,
                                          const uint32_t* sq) {
  uint32_t Mu, Mq, Mp;
  int su, sq_, sp_;
  f32_parts(u, Mu, su);
  f32_parts(qt, Mq, sq_);
  f32_parts(pt, Mp, sp_);
  Big L, R;
  big_set(L, sp);
  big_mul_u32(L, Mu);
  big_mul_u32(L, Mq);
  big_set(R, sq);
  big_mul_u32(R, Mp);
  const int el = su + sq_, er = sp_ + 149;
  const int m = el < er ? el : er;
  big_shl(L, el - m);
  big_shl(R, er - m);
  return big_cmp(L, R) < 0;
}

__device__ __forceinline__ double limbs_to_double(const uint32_t* l) {
  double z = 0.0;
  for (int i = kLimbs - 1; i >= 0; --i) z = z * 4294967296.0 + static_cast<double>(l[i]);
  return ldexp(z, -149);
}

// 1: certain accept, 0: certain reject, -1: inside the error band.  Zp, Zq
// are approximate masses with |Zp - exact| <= Bp and |Zq - exact| <= Bq.
__device__ __forceinline__ int filter_decide(float u, float pt, float qt, double Zp, double Bp,
                                             double Zq, double Bq) {
  const double a = static_cast<double>(u) * static_cast<double>(qt);  // exact
  const double bp = static_cast<double>(pt);
  if (bp == 0.0) return 0;  // rhs = 0 <= lhs
  if (a == 0.0) return 1;   // lhs = 0 < rhs  (pt > 0, Zq > 0 checked earlier)
  const double L = a * Zp, R = bp * Zq;
  const double E = a * Bp + bp * Bq + (L + R) * 4.5e-16;
  if (R - L > E) return 1;
  if (L - R > E) return 0;
  return -1;
}

// floor(u * R) for u in [0, 1) exactly.
__device__ __forceinline__ unsigned long long tau_of(float u, unsigned long long R) {
  uint32_t M;
  int s;
  f32_parts(u, M, s);
  if (!M) return 0ull;
  const int sh = 149 - s;  // u = M * 2^-sh, sh >= 24 for u < 1
  const unsigned long long lo = static_cast<unsigned long long>(M) * R;
  const unsigned long long hi = __umul64hi(static_cast<unsigned long long>(M), R);
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (lo >> sh) | (hi << (64 - sh));
}

// Normalised draw weights: residual max(0, phat - qhat) or phat alone.
struct DrawW {
  float sp, ap, sq, aq, scale;
  int resid;
  __device__ __forceinline__ float operator()(float p, float q) const {
    const float a = __fmul_rn(__fmul_rn(p, sp), ap);
    if (!resid) return a;
    return fmaxf(__fsub_rn(a, __fmul_rn(__fmul_rn(q, sq), aq)), 0.f);
  }
  // fixed point of a (partial) vector sum
  __device__ __forceinline__ unsigned long long fix(float v) const {
    return __float2ull_rz(__fmul_rn(v, scale));
  }
};

// Power-of-two pre-scale and reciprocal of a row mass so that p * sp * ap is
// the normalised weight without leaving the fp32 range.
__device__ __forceinline__ void norm_factors(double Z, float& s, float& a) {
  double ss = 1.0;
  if (Z > 0x1p100) ss = 0x1p-64;
  if (Z < 0x1p-100) ss = 0x1p64;
  s = static_cast<float>(ss);
  a = static_cast<float>(1.0 / (Z * ss));
}

}  // namespace svk
