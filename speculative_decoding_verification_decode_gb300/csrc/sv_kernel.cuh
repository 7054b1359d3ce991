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
//   * chunks are released as soon as they are reduced, so the producer streams
//     the next row while the current one is being decided (one row of
//     lookahead); the exact fallback, the residual and the inverse-CDF walk
//     read the decided row again from global memory (mostly L2);
//   * the walk stops at the first miss / rejection; rows past the next one
//     are never read (chunks already in flight are drained before exit).
//
// Decisions in sampling mode are the exact real predicate
//     u * q(t) * Zp  <  p(t) * Zq
// on the exact sums Zp, Zq of the f32 row weights: an approximate sum with a
// rigorous error bound decides whenever the bound allows, otherwise the CTAs
// sum the row exactly (integer significand buckets, 32-bit limbs)
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
constexpr int kDecideWarp = kWarps + 1;    // warp 9 (sampling): combines and decides rows
constexpr int kThreads = kConsumers + 64;  // + the producer warp and the decision warp
constexpr int kMaxSlots = 16;
constexpr int kMaxSlotBytes = 32768;
constexpr int kMaxCluster = 16;
constexpr int kRecWords = 32;
constexpr int kBuckets = 254;
constexpr int kLimbs = 12;
constexpr int kBigLimbs = 32;
constexpr int kMaxGather = 32;  // rows whose decision inputs are prefetched at start
constexpr int kGroupVecs = 32;  // 16-byte vectors per fixed-point group sum of the draw

enum : int { MODE_GREEDY = 0, MODE_PROBS = 1, MODE_LOGITS = 2 };

// Threads of a CTA: greedy verification has no decision warp.
constexpr int threads_of(int mode) { return mode == MODE_GREEDY ? kThreads - 32 : kThreads; }

#define kInfF (__uint_as_float(0x7F800000u))

constexpr uint32_t ST_BAD_TOKEN = 1u, ST_BAD_VALUE = 2u, ST_ZERO_MASS = 4u, ST_NEAR = 8u,
                   ST_EXACT = 16u, ST_TIMEOUT = 32u, ST_BAD_LAYOUT = 64u;
constexpr uint32_t FLAG_FORCE_EXACT = 1u;
constexpr uint32_t FLAG_EXPIRE_EXCHANGE = 2u;  // exchange waits give up without polling (tests)

constexpr double kU32 = 5.9604644775390625e-8;  // 2^-24, unit roundoff of f32
// Relative error bound used for ex2.approx.ftz.f32 (normal results); the
// measured maximum on GB300 is checked against it by a GPU test.
constexpr double kEx2Rel = 4.76837158203125e-7;  // 2^-21
static_assert(kEx2Rel == 8.0 * kU32, "online_bound() writes e as 8u");

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
  const float* flo_t;  // per-row floors of the sampler filters (NULL: none)
  const float* flo_d;
  const unsigned* ext_err;  // nonzero word: the kernel that wrote the rows gave up (NULL: none)
  const int* gate;          // per sequence: 0 = leave the sequence to another launch (NULL: every one)
  unsigned flags;
  int slice;       // elements per CTA slice (multiple of the vector width)
  int slot_bytes;  // bytes per ring slot (multiple of 16)
  int S;           // ring slots
  int use_tma;
  int fixed_shift;
  int vsum_off;  // byte offset of the draw's group sums / exact buckets (sampling)
  int look;      // rows the producer may stream past the last accepted row
  int tail_off;  // byte offset of SmemTail
};

// A row's outcome, from the decision warp to the consumer warps.
struct Dec {
  int act;
  uint32_t st;   // status bits so far
  float mp, mq;  // row maxima (logits: the weights' m)
  float u_draw;  // the draw's uniform (ACT_DRAW)
};

struct __align__(16) SmemTail {
  uint32_t recs[2][kMaxCluster][kRecWords];  // records pushed by the cluster's CTAs
  uint32_t myrec[kRecWords];                 // this CTA's outgoing record
  float wf[kWarps][8];                       // per-warp partial results (greedy)
  int wi[kWarps][4];
  float wf2[2][kWarps][8];  // per-warp partials of rows i, i + 1 (sampling)
  int wi2[2][kWarps][4];
  Dec dec[2];               // outcomes of rows i, i + 1
  uint32_t lp[kLimbs], lq[kLimbs], infl;  // exact masses of the row (limbs) and +Inf flags
  int xc;                   // exchanges done (slot and parity of the next one)
  unsigned long long wu[kWarps];
  int bi[8];
  float dpar[4];  // draw weight parameters (computed once by thread 0)
  // decision inputs of rows 0..kMaxGather-1, loaded at the start
  int g_t[kMaxGather];
  float g_u[kMaxGather], g_p[kMaxGather], g_q[kMaxGather];
  uint64_t xbar[2];
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  volatile int stop;           // consumers -> producer: issue nothing more
  volatile int go_row;         // consumers -> producer: rows decided so far
  volatile int cut_row;        // consumers -> producer: the row they cut short (-1: none)
  uint64_t pfull[2];           // consumers -> decision warp: partials of row i ready
  uint64_t dfull[2];           // decision warp -> consumers: outcome of row i ready
  uint64_t xfull, xdec;        // exact pass: limbs ready / final outcome ready
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

// One 16-byte vector of a shared-memory chunk: unpacked floats and their
// NaN-propagating maximum (packed compare for 16-bit types), from one load.
template <typename T>
__device__ __forceinline__ float load_vec_max(const T* s, int vi, float* x) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
    return fmax_nan(fmax_nan(v.x, v.y), fmax_nan(v.z, v.w));
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
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
      const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
      return fmax_nan(bf_lo(m), bf_hi(m));
    } else {
      const uint32_t m = f16x2_max_nan(f16x2_max_nan(v.x, v.y), f16x2_max_nan(v.z, v.w));
      return fmax_nan(h_lo(m), h_hi(m));
    }
  }
}

// U vectors of a shared-memory chunk, vectors base + u * kConsumers (those
// at or past nv are absent and read as -Inf): unpacked floats, their
// NaN-propagating maximum, and their minimum over the present vectors (a
// lower bound for every present element), each from one packed tree.
template <typename T, int U, int VEC>
__device__ __forceinline__ void load_block(const T* s, int base, int nv, float (&x)[U][VEC], bool (&have)[U],
                                           float& vmax, float& vmin) {
  if constexpr (sizeof(T) == 4) {
    float hi = -kInfF, lo = kInfF;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = base + u * kConsumers;
      have[u] = vi < nv;
      const float4 v = have[u] ? reinterpret_cast<const float4*>(s)[vi] : make_float4(-kInfF, -kInfF, -kInfF, -kInfF);
      x[u][0] = v.x;
      x[u][1] = v.y;
      x[u][2] = v.z;
      x[u][3] = v.w;
      hi = fmax_nan(hi, fmax_nan(fmax_nan(v.x, v.y), fmax_nan(v.z, v.w)));
      if (have[u]) lo = fminf(lo, fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
    }
    vmax = hi;
    vmin = lo;
  } else {
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kNegInf2 = kBf ? 0xFF80FF80u : 0xFC00FC00u;
    constexpr uint32_t kPosInf2 = kBf ? 0x7F807F80u : 0x7C007C00u;
    uint32_t w[U][4];
    uint32_t hi2 = kNegInf2, lo2 = kPosInf2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = base + u * kConsumers;
      have[u] = vi < nv;
      const uint4 v = have[u] ? reinterpret_cast<const uint4*>(s)[vi] : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
      w[u][0] = v.x;
      w[u][1] = v.y;
      w[u][2] = v.z;
      w[u][3] = v.w;
      if constexpr (kBf) {
        hi2 = bf16x2_max_nan(hi2, bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w)));
        if (have[u]) lo2 = bf16x2_min(lo2, bf16x2_min(bf16x2_min(v.x, v.y), bf16x2_min(v.z, v.w)));
      } else {
        hi2 = f16x2_max_nan(hi2, f16x2_max_nan(f16x2_max_nan(v.x, v.y), f16x2_max_nan(v.z, v.w)));
        if (have[u]) lo2 = f16x2_min(lo2, f16x2_min(f16x2_min(v.x, v.y), f16x2_min(v.z, v.w)));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        x[u][2 * q] = kBf ? bf_lo(w[u][q]) : h_lo(w[u][q]);
        x[u][2 * q + 1] = kBf ? bf_hi(w[u][q]) : h_hi(w[u][q]);
      }
    vmax = kBf ? fmax_nan(bf_lo(hi2), bf_hi(hi2)) : fmax_nan(h_lo(hi2), h_hi(hi2));
    vmin = kBf ? fminf(bf_lo(lo2), bf_hi(lo2)) : fminf(h_lo(lo2), h_hi(lo2));
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

// ------------------------------------------------------------------ double-float (fp32 pairs)
// hi + lo with |lo| <= ulp(hi)/2; relative error of each operation ~2^-44.
// Used by thread 0 instead of fp64 (GB300's fp64 rate is a small fraction of
// its fp32 rate and would sit on the per-row critical path).
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ DF fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  const DF s = two_sum(x.hi, y.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ DF df_mul_f(DF x, float y) {
  DF p = two_prod(x.hi, y);
  p.lo = __fmaf_rn(x.lo, y, p.lo);
  return fast_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ DF df_mul(DF x, DF y) {
  DF p = two_prod(x.hi, y.hi);
  p.lo = __fmaf_rn(x.hi, y.lo, __fmaf_rn(x.lo, y.hi, p.lo));
  return fast_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ DF df_neg(DF x) { return {-x.hi, -x.lo}; }

// Butterfly sum across a warp (the addition is commutative bit for bit, so
// every lane ends with the same pair).
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const DF w = {__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
    v = df_add(v, w);
  }
  return v;
}

// ------------------------------------------------------------------ accumulators

// Per-thread fp32 sum of vector sums.  A thread that adds n_v vector sums
// (each a pairwise tree of VEC elements) is within (n_v + log2 VEC) * 2^-24 of
// its exact sum; the warp, CTA and cluster levels add 12 more roundings (fp32
// trees of 5, 3 and 4 levels).  sum_bound() states the total bound.
struct Acc {
  float f;
  __device__ __forceinline__ void init() { f = 0.f; }
  __device__ __forceinline__ void add(float t) { f = __fadd_rn(f, t); }
};

__device__ __forceinline__ float sum_bound(float Z, int nadd) {
  return 2.02f * Z * (static_cast<float>(nadd + 12) * 0x1p-24f);
}

// ------------------------------------------------------------------ logits -> weights

// The defined weights of a warped row (the values whose exact sum is the
// row mass): w = 2^((l - m) * k) with m the row maximum and k = log2(e)/T.
// 16-bit logits: one fp32 subtract and multiply, then ex2.approx.ftz.
// Both weigh a logit below the row's floor `lo` (the sampler filters' cut;
// -Inf: none) as 0.
struct Warp16 {
  float m, k, lo;
  __device__ __forceinline__ float operator()(float l) const {
    return l < lo ? 0.f : ex2_ftz(__fmul_rn(__fsub_rn(l, m), k));
  }
};

// f32 logits: l - m as an exact two-term sum, the product with the
// double-float k = khi + klo kept to about 2^-40, and the low part applied as
// a first-order correction to 2^hi.
struct Warp32 {
  float m, khi, klo, lo;
  __device__ __forceinline__ float operator()(float l) const {
    if (l < lo) return 0.f;
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

// Probability rows are used as they are (`lo` stays -Inf: no floors there).
struct NoWarp {
  float lo;
  __device__ __forceinline__ float operator()(float x) const { return x; }
};

// Online softmax of one thread's elements: running maximum m, and
//   s = sum 2^(-nx),  w = sum 2^(-nx) * nx,   nx = (m - l) * k >= 0,
// rescaled when m grows (all in fp32).  It approximates the row mass
// Z = sum w_v of the defined weights within
//   |S - Z| <= 2 * (S * ((R + 3)(e + u) + 2e + (n + 12) u + ln2 |m k| u) + W * 5 ln2 u)
// with e the ex2 bound, u = 2^-24, R the rescale steps of any element and n
// the fp32 additions of any element inside its thread (the 12 are the
// warp, CTA and cluster trees).
struct Online {
  float m, s, w;
  int r;
  __device__ __forceinline__ void init() {
    m = -kInfF;
    s = w = 0.f;
    r = 0;
  }
  __device__ __forceinline__ void rescale_to(float mnew, float k) {
    const float d = __fmul_rn(__fsub_rn(mnew, m), k);
    const float f = ex2_ftz(-d);
    w = __fmul_rn(__fmaf_rn(d, s, w), f);
    s = __fmul_rn(s, f);
    m = mnew;
    ++r;
  }
  template <int VEC>
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
    s = __fadd_rn(s, tree_sum<VEC>(e));
    w = __fadd_rn(w, __fadd_rn(wa, wb));
  }
  // U vectors at once (vectors u with have[u] false are absent, their
  // elements -Inf): one max test and rescale for the block, then U * VEC
  // independent exps.  Each element still goes through one vector tree and
  // one addition into s.  w takes an upper bound of the block's share: every
  // element has nx <= (m - vmin) k, and ex2 flushes to 0 past nx = 126, so
  // sum(e nx) <= sum(e) * min((m - vmin) k, 128).
  template <int U, int VEC>
  __device__ __forceinline__ void add_block(const float (&x)[U][VEC], const bool (&have)[U], float vm,
                                            float vmin, float k) {
    if (!(vm <= m)) {
      if (!(vm > -kInfF)) return;  // NaN (flagged by the caller) or all -Inf
      if (m == -kInfF) m = vm;
      else rescale_to(vm, k);
    }
    if (m == -kInfF) return;
    float t[U];
    const float mk = __fmul_rn(m, k);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float e[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) e[j] = ex2_ftz(__fmaf_rn(x[u][j], k, -mk));
      t[u] = tree_sum<VEC>(e);
    }
    float tb = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (have[u]) {
        s = __fadd_rn(s, t[u]);
        tb = __fadd_rn(tb, t[u]);
      }
    }
    const float nxm = fminf(__fmul_rn(__fsub_rn(m, vmin), k), 128.f);
    w = __fmaf_rn(tb, nxm, w);
  }
};

// The pass forms each exponent as x k - m k with one FMA (m k rounded once
// per block), which moves every argument by at most (|m k| + nx) u / 2 from
// (x - m) k: a relative weight error of ln2 (|m k| + nx) u / 2, which adds
// ln2 |m k| u to the S coefficient and ln2 u to the W one.
__device__ __forceinline__ float online_bound(float S, float W, int R, int nadd, float mk_abs) {
  // (R + 3)(e + u) + 2e + (nadd + 12)u with e = 8u: an integer times u, exact
  // in fp32 (no fp64 on this path)
  const float cs = static_cast<float>(9 * (R + 3) + 16 + nadd + 12) * 0x1p-24f + 0.6932f * 0x1p-24f * mk_abs;
  constexpr float cw = 3.4657360f * 0x1p-24f;  // 5 ln2 u, rounded up
  return 2.02f * (S * cs + W * cw);
}

// k = log2(e) / T as an fp32 pair (hi, lo) without fp64, whose rate on this
// part is a small fraction of fp32's: the correctly rounded quotient, its
// remainder by one FMA (exact), and a correction quotient.  k is clamped to
// FLT_MAX (a temperature so small that 1/T overflows).
__device__ __forceinline__ void log2e_over(float T, float& khi, float& klo) {
  constexpr float kL2eHi = 1.44269502162933349609375f;  // fp32 nearest to log2(e)
  constexpr float kL2eLo = 1.925963033500011e-08f;      // log2(e) - kL2eHi
  const float q = __fdiv_rn(kL2eHi, T);
  if (!(q < FLT_MAX)) {
    khi = FLT_MAX;
    klo = 0.f;
    return;
  }
  const float r = __fmaf_rn(-q, T, kL2eHi);
  const DF k = fast_two_sum(q, __fdiv_rn(__fadd_rn(r, kL2eLo), T));
  khi = k.hi;
  klo = k.lo;
}

// ------------------------------------------------------------------ warp reductions
// Butterflies over groups of W lanes (W a power of two, at most 32): every
// lane ends with the result of its own group.  The decision warp combines 8
// warp partials (W = 8) and at most 16 CTA records (W = 16), so it takes 3 and
// 4 levels where a whole-warp butterfly would take 5.

template <int W = 32>
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <int W = 32>
__device__ __forceinline__ float warp_max_nan_f(float v) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <int W = 32>
__device__ __forceinline__ float warp_min_nan_f(float v) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v = fmin_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <int W = 32>
__device__ __forceinline__ float warp_max_f(float v) {  // inputs never NaN
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <int W = 32>
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Argmax candidate ordering: a valid index beats "none" (INT_MAX); larger value
// wins; equal values go to the lower index.  NaN never enters a candidate.
__device__ __forceinline__ bool arg_better(float va, int ia, float vb, int ib) {
  if (ia == INT_MAX) return false;
  if (ib == INT_MAX) return true;
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int j = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (arg_better(w, j, v, i)) {
      v = w;
      i = j;
    }
  }
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
static __device__ __noinline__ void buckets_to_limbs(const unsigned long long* bk, uint32_t* limbs) {
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
static __device__ __noinline__ bool exact_accept(float u, float pt, float qt, const uint32_t* sp,
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

// 1: certain accept, 0: certain reject, -1: inside the error band (or a scale
// where fp32 pairs could lose accuracy).  Zp, Zq are approximate masses with
// |Zp - exact| <= Bp and |Zq - exact| <= Bq.
__device__ __forceinline__ int filter_decide(float u, float pt, float qt, DF Zp, float Bp, DF Zq,
                                             float Bq) {
  if (pt == 0.f) return 0;  // rhs = 0 <= lhs
  if (u == 0.f || qt == 0.f) return 1;  // lhs = 0 < rhs  (pt > 0, Zq > 0 checked earlier)
  const DF a = two_prod(u, qt);  // exact unless tiny
  const float lo = 0x1p-90f, hi = 0x1p90f;
  if (!(a.hi >= lo && pt >= lo && Zp.hi >= lo && Zp.hi <= hi && Zq.hi >= lo && Zq.hi <= hi))
    return -1;
  const DF L = df_mul(a, Zp), R = df_mul_f(Zq, pt);
  const DF D = df_add(R, df_neg(L));
  const float E = 1.01f * (a.hi * Bp + pt * Bq + (L.hi + R.hi) * 0x1p-40f);
  if (D.hi > E) return 1;
  if (D.hi < -E) return 0;
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

// floor(y) for 0 <= y < 2^63 from the fp32 bits (integer pipe; truncation).
__device__ __forceinline__ unsigned long long floor_u64(float y) {
  const uint32_t b = __float_as_uint(y);
  const int e = static_cast<int>(b >> 23) - 127;
  if (e < 0) return 0ull;
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;
  return e >= 23 ? (m << (e - 23)) : (m >> (23 - e));
}

// Normalised draw weights of f32 probabilities: max(0, phat - qhat), or phat.
struct DrawProbs {
  float sp, ap, sq, aq, scale;
  int resid;
  __device__ __forceinline__ float operator()(float p, float q) const {
    const float a = __fmul_rn(__fmul_rn(p, sp), ap);
    if (!resid) return a;
    return fmaxf(__fsub_rn(a, __fmul_rn(__fmul_rn(q, sq), aq)), 0.f);
  }
  __device__ __forceinline__ unsigned long long fix(float v) const {
    return floor_u64(__fmul_rn(v, scale));
  }
};

// Normalised draw weights of logits: the normalisation is folded into the
// exponent, 2^(l k + c) with c = -m k - log2 Z (one FMA and one ex2 per row).
// Only the draw uses these (they need not equal the defined weights bit for
// bit; both passes of the draw use the same function).
// FL: the rows carry sampler-filter floors (logits below weigh 0).
template <bool FL>
struct DrawLogits {
  float k, cp, cq, scale;
  float lo_p, lo_q;  // the rows' floors (FL only)
  int resid;
  __device__ __forceinline__ float operator()(float lp, float lq) const {
    float a = ex2_ftz(__fmaf_rn(lp, k, cp));
    if constexpr (FL) a = lp < lo_p ? 0.f : a;
    if (!resid) return a;
    float b = ex2_ftz(__fmaf_rn(lq, k, cq));
    if constexpr (FL) b = lq < lo_q ? 0.f : b;
    return fmaxf(__fsub_rn(a, b), 0.f);
  }
  __device__ __forceinline__ unsigned long long fix(float v) const {
    return floor_u64(__fmul_rn(v, scale));
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
