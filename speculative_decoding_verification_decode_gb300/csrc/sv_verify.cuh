// The verification kernel (design notes in sv_kernel.cuh).
#pragma once
#include <type_traits>

#include "sv_kernel.cuh"

namespace svk {

// ------------------------------------------------------------------ chunk passes
// `s` points at a shared-memory chunk of `n` consecutive row elements whose
// first element is column `e0` of the row.  Consumer thread `c` handles the
// 16-byte vectors c, c + 256, ... (conflict-free, coalesced).

template <typename T>
__device__ __forceinline__ void chunk_argmax(const T* s, int n, int e0, float& bv, int& bi,
                                             uint32_t& nanf) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kConsumers) {
    const float m = vec_max_nan(s, vi);
    if (!(m <= bv)) {  // a new maximum, a NaN, or no candidate yet
      float x[VEC];
      load_vec(s, vi, x);
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        if (x[k] != x[k]) {
          nanf = 1u;
        } else if (bv != bv || x[k] > bv) {
          bv = x[k];
          bi = e0 + vi * VEC + k;
        }
      }
    }
  }
  for (int e = nv * VEC + threadIdx.x; e < n; e += kConsumers) {
    const float x = ElemTraits<T>::to_f(s[e]);
    if (x != x) {
      nanf = 1u;
    } else if (bv != bv || x > bv) {
      bv = x;
      bi = e0 + e;
    }
  }
}

__device__ __forceinline__ void chunk_mass_f32(const float* s, int n, Acc& a, float& mn) {
  const int nv = n >> 2;
  int vi = threadIdx.x;
  for (; vi + kConsumers < nv; vi += 2 * kConsumers) {
    const float4 v0 = reinterpret_cast<const float4*>(s)[vi];
    const float4 v1 = reinterpret_cast<const float4*>(s)[vi + kConsumers];
    const float x0[4] = {v0.x, v0.y, v0.z, v0.w};
    const float x1[4] = {v1.x, v1.y, v1.z, v1.w};
    a.add<8>(tree_sum<4>(x0));
    a.add<8>(tree_sum<4>(x1));
    mn = fmin_nan(mn, fmin_nan(fmin_nan(fmin_nan(v0.x, v0.y), fmin_nan(v0.z, v0.w)),
                               fmin_nan(fmin_nan(v1.x, v1.y), fmin_nan(v1.z, v1.w))));
  }
  if (vi < nv) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    const float x[4] = {v.x, v.y, v.z, v.w};
    a.add<8>(tree_sum<4>(x));
    mn = fmin_nan(mn, fmin_nan(fmin_nan(v.x, v.y), fmin_nan(v.z, v.w)));
  }
  for (int e = (nv << 2) + threadIdx.x; e < n; e += kConsumers) {
    a.add<8>(s[e]);
    mn = fmin_nan(mn, s[e]);
  }
}

// Online softmax over a chunk of logits; `mx` tracks the NaN-propagating max
// (for validity), `o` the running max and sums (for the mass).
template <typename T>
__device__ __forceinline__ void chunk_online(const T* s, int n, float k, Online& o, float& mx) {
  constexpr int VEC = ElemTraits<T>::kVec;
  constexpr int FL = ElemTraits<T>::kFlush;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kConsumers) {
    const float vm = vec_max_nan(s, vi);
    mx = fmax_nan(mx, vm);
    float x[VEC];
    load_vec(s, vi, x);
    o.add_vec<VEC, FL>(x, vm, k);
  }
  for (int e = nv * VEC + threadIdx.x; e < n; e += kConsumers) {
    const float x = ElemTraits<T>::to_f(s[e]);
    mx = fmax_nan(mx, x);
    o.add_vec<1, FL>(&x, x, k);
  }
}

template <typename T, typename W>
__device__ __forceinline__ void chunk_write_weights(const T* s, int n, int e0, const W& wf,
                                                    float* out) {
  for (int e = threadIdx.x; e < n; e += kConsumers) out[e0 + e] = wf(ElemTraits<T>::to_f(s[e]));
}

template <typename T, typename W>
__device__ __forceinline__ void chunk_exact(const T* s, int n, const W& wf, unsigned long long* bk,
                                            uint32_t& bad) {
  for (int e = threadIdx.x; e < n; e += kConsumers) {
    const float x = wf(ElemTraits<T>::to_f(s[e]));
    if (!(x <= FLT_MAX)) bad = 1u;  // +Inf (NaN and negatives were rejected before)
    else bucket_add(bk, x);
  }
}

// Draw weights of vector `vi` of a chunk pair (`sq` may be null): writes up to
// VEC weights and returns how many elements the vector holds.
template <typename T, typename W>
__device__ __forceinline__ int vec_draw_weights(const T* sp, const T* sq, int n, int vi,
                                                const W& wfp, const W& wfq, const DrawW& dw,
                                                float* r) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int e0 = vi * VEC;
  if (e0 + VEC <= n) {
    float xp[VEC], xq[VEC];
    load_vec(sp, vi, xp);
    if (sq) load_vec(sq, vi, xq);
#pragma unroll
    for (int k = 0; k < VEC; ++k) r[k] = dw(wfp(xp[k]), sq ? wfq(xq[k]) : 0.f);
    return VEC;
  }
  const int cnt = n - e0;
  for (int k = 0; k < cnt; ++k) {
    const float p = wfp(ElemTraits<T>::to_f(sp[e0 + k]));
    const float q = sq ? wfq(ElemTraits<T>::to_f(sq[e0 + k])) : 0.f;
    r[k] = dw(p, q);
  }
  return cnt;
}

// Left-to-right fp32 sum of r[0..cnt) (the order the owner's walk repeats).
__device__ __forceinline__ float seq_sum_n(const float* r, int cnt) {
  float t = r[0];
  for (int k = 1; k < cnt; ++k) t = __fadd_rn(t, r[k]);
  return t;
}

// ------------------------------------------------------------------ the kernel

enum : int { ACT_CONTINUE = 0, ACT_STOP = 1, ACT_EXACT = 2, ACT_DRAW = 3, ACT_ABORT = 4 };

template <int MODE, typename T>
__global__ void __launch_bounds__(kThreads, 2) sv_verify_kernel(const __grid_constant__ Params P) {
  using TR = ElemTraits<T>;
  constexpr int VEC = TR::kVec;
  constexpr int ELEM = static_cast<int>(sizeof(T));
  using WarpT =
      typename std::conditional<MODE == MODE_LOGITS, typename WarpOf<T>::type, NoWarp>::type;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  unsigned long long* vsum = reinterpret_cast<unsigned long long*>(smem + P.vsum_off);
  SmemTail& sm = *reinterpret_cast<SmemTail*>(smem + P.tail_off);
  const int tid = threadIdx.x;

  const long long b = blockIdx.y + static_cast<long long>(blockIdx.z) * gridDim.y;
  if (b >= P.B) return;  // the whole cluster shares b
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();

  // ---------------------------------------------------------------- sequence layout
  int kb = P.K;
  long long t0 = b * (P.K + 1LL), d0 = b * static_cast<long long>(P.K);
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
  bool sampling = MODE != MODE_GREEDY;
  float temp = 0.f;
  bool temp_ok = true;
  if (MODE == MODE_LOGITS && layout_ok) {
    temp = P.temp[b];
    temp_ok = temp >= 0.f && temp <= FLT_MAX;
    sampling = temp > 0.f;
  }
  if (!layout_ok || !temp_ok) {
    if (rank == 0 && tid == 0) {
      P.n_out[b] = 0;
      P.next_out[b] = -1;
      P.st_out[b] = layout_ok ? ST_BAD_VALUE : ST_BAD_LAYOUT;
    }
    return;
  }

  const T* tgt = static_cast<const T*>(P.tgt);
  const T* drf = static_cast<const T*>(P.drf);
  const int S = P.S;
  const int ck_el = P.slot_bytes / ELEM;
  const int v_lo = static_cast<int>(rank) * P.slice;
  const int v_hi = min(P.V, v_lo + P.slice);
  const int n_el = max(0, v_hi - v_lo);
  const int nck = (n_el + ck_el - 1) / ck_el;
  const long long total_items = sampling ? static_cast<long long>(kb) * 2 * nck + nck
                                         : static_cast<long long>(kb + 1) * nck;

  // item g of this CTA's load sequence: (row, target/draft, chunk) -> source
  auto item = [&](long long g, const T*& src, int& e0, int& n) {
    long long r;
    int j;
    bool isq = false;
    if (sampling) {
      r = g / (2 * nck);
      const int w = static_cast<int>(g - r * 2 * nck);
      isq = w >= nck;
      j = isq ? w - nck : w;
    } else {
      r = g / nck;
      j = static_cast<int>(g - r * nck);
    }
    e0 = v_lo + j * ck_el;
    n = min(v_hi, e0 + ck_el) - e0;
    const long long row = isq ? d0 + r : t0 + r;
    src = (isq ? drf : tgt) + row * P.stride + e0;
  };
  auto slot_ptr = [&](long long g) {
    return reinterpret_cast<const T*>(ring + static_cast<long long>(g % S) * P.slot_bytes);
  };

  // ---------------------------------------------------------------- barriers
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kWarps);
    }
    mbar_init(&sm.xbar[0], C);
    mbar_init(&sm.xbar[1], C);
    sm.stop = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  cluster_sync_all();  // every peer's barriers exist before the first remote arrive

  // ================================================================ producer warp
  if (tid >= kConsumers) {
    const int lane = tid - kConsumers;
    long long g = 0;
    for (; g < total_items; ++g) {
      const int slot = static_cast<int>(g % S);
      int go = 1;
      if (lane == 0) {
        if (g >= S) {
          const uint32_t par = static_cast<uint32_t>(((g / S) - 1) & 1);
          uint32_t polls = 0;
          while (!mbar_try_wait(&sm.empty[slot], par)) {
            if (sm.stop || ++polls == kWaitPolls) {
              go = 0;
              break;
            }
          }
        }
        if (sm.stop) go = 0;
      }
      go = __shfl_sync(0xFFFFFFFFu, go, 0);
      if (!go) break;
      const T* src;
      int e0, n;
      item(g, src, e0, n);
      const uint32_t bytes = static_cast<uint32_t>(n) * ELEM;
      const uint32_t tma = P.use_tma ? (bytes & ~15u) : 0u;
      T* dst = reinterpret_cast<T*>(ring + static_cast<long long>(slot) * P.slot_bytes);
      for (int e = static_cast<int>(tma / ELEM) + lane; e < n; e += 32) dst[e] = src[e];
      __syncwarp();
      if (lane == 0) {
        if (tma) {
          mbar_arrive_expect_tx(&sm.full[slot], tma);
          bulk_g2s(dst, src, tma, &sm.full[slot]);
        } else {
          mbar_arrive_local(&sm.full[slot]);
        }
      }
    }
    // no bulk copy may still be writing this CTA's shared memory at exit
    if (lane == 0)
      for (long long gg = g > S ? g - S : 0; gg < g; ++gg)
        mbar_wait_bounded(&sm.full[gg % S], static_cast<uint32_t>((gg / S) & 1));
    return;
  }

  // ================================================================ consumers
  const int lane = tid & 31;
  uint32_t tmo = 0;
  auto acquire = [&](long long g) {
    if (!mbar_wait_bounded(&sm.full[g % S], static_cast<uint32_t>((g / S) & 1))) tmo = 1u;
  };
  auto release = [&](long long g) {
    __syncwarp();
    if (lane == 0) mbar_arrive_local(&sm.empty[g % S]);
  };

  int xc = 0, last_slot = 0;
  auto xchg = [&](int words) -> bool {
    bar_consumers<kConsumers>();
    const int slot = xc & 1;
    const uint32_t par = static_cast<uint32_t>((xc >> 1) & 1);
    ++xc;
    last_slot = slot;
    if (tid < static_cast<int>(C)) {
      const uint32_t dst = dsmem_addr(&sm.recs[slot][rank][0], static_cast<uint32_t>(tid));
      for (int w = 0; w < words; w += 4)
        dsmem_st_v4(dst + 4u * w, *reinterpret_cast<const uint4*>(&sm.myrec[w]));
      dsmem_arrive_release(dsmem_addr(&sm.xbar[slot], static_cast<uint32_t>(tid)));
    }
    const bool ok = mbar_wait_cluster_bounded(&sm.xbar[slot], par);
    return bar_consumers_and<kConsumers>(ok) != 0;
  };
  auto rec = [&](uint32_t c, int w) -> uint32_t { return sm.recs[last_slot][c][w]; };
  auto rec_d = [&](uint32_t c, int w) -> double {
    return __hiloint2double(static_cast<int>(rec(c, w + 1)), static_cast<int>(rec(c, w)));
  };
  auto rec_u64 = [&](uint32_t c, int w) -> unsigned long long {
    return static_cast<unsigned long long>(rec(c, w)) |
           (static_cast<unsigned long long>(rec(c, w + 1)) << 32);
  };
  auto put_d = [&](int w, double v) {
    sm.myrec[w] = static_cast<uint32_t>(__double2loint(v));
    sm.myrec[w + 1] = static_cast<uint32_t>(__double2hiint(v));
  };
  auto finish = [&](int n, int nxt, uint32_t s) {  // thread 0 of the writing CTA
    P.n_out[b] = n;
    P.next_out[b] = nxt;
    P.st_out[b] = s;
  };

  uint32_t st = 0;  // status bits (thread 0)
  bool abort = false;

  if (!sampling) {
    // ============================================================== greedy
    for (int i = 0;; ++i) {
      float bv = __int_as_float(0x7FFFFFFF);  // NaN: no candidate yet
      int bi = INT_MAX;
      uint32_t nanf = 0;
      for (int j = 0; j < nck; ++j) {
        const long long g = static_cast<long long>(i) * nck + j;
        acquire(g);
        const T* src;
        int e0, n;
        item(g, src, e0, n);
        chunk_argmax<T>(slot_ptr(g), n, e0, bv, bi, nanf);
        release(g);
      }
      if (bv != bv) bi = INT_MAX;
      block_argmax(bv, bi, sm.redf, sm.redi);
      nanf = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(nanf)));
      tmo = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(tmo)));
      if (tid == 0) {
        sm.myrec[0] = __float_as_uint(bv);
        sm.myrec[1] = static_cast<uint32_t>(bi);
        sm.myrec[2] = nanf | (tmo << 1);
        sm.myrec[3] = 0u;
      }
      if (!xchg(4)) {
        abort = true;
        break;
      }
      float v = 0.f;
      int a = INT_MAX;
      uint32_t fl = 0;
      for (uint32_t c = 0; c < C; ++c) {
        const float vc = __uint_as_float(rec(c, 0));
        const int ic = static_cast<int>(rec(c, 1));
        fl |= rec(c, 2);
        if (arg_better(vc, ic, v, a)) {
          v = vc;
          a = ic;
        }
      }
      if (fl & 2u) {
        abort = true;
        break;
      }
      if (a == INT_MAX) a = 0;  // an all-NaN row
      if (fl & 1u) st |= ST_BAD_VALUE;
      bool stop = false;
      uint32_t extra = 0;
      if (i == kb) {
        stop = true;
      } else {
        const int t = P.tok[d0 + i];
        if (t < 0 || t >= P.V) {
          stop = true;
          extra = ST_BAD_TOKEN;
        } else if (t != a) {
          stop = true;
        }
      }
      if (stop) {
        if (tid == 0) {
          sm.stop = 1;
          if (rank == 0) finish(i, a, st | extra);
        }
        break;
      }
    }
  } else {
    // ============================================================== sampling
    float khi = 0.f, klo = 0.f;
    if (MODE == MODE_LOGITS) {
      double kd = 1.4426950408889634074 / static_cast<double>(temp);
      if (kd > FLT_MAX) kd = FLT_MAX;
      khi = static_cast<float>(kd);
      klo = static_cast<float>(kd - static_cast<double>(khi));
    }
    auto make_warp = [&](float m) {
      WarpT w;
      if constexpr (MODE == MODE_LOGITS) {
        if constexpr (sizeof(T) == 4) {
          w.m = m;
          w.khi = khi;
          w.klo = klo;
        } else {
          w.m = m;
          w.k = khi;
        }
      }
      (void)m;
      return w;
    };
    const bool force_exact = (P.flags & FLAG_FORCE_EXACT) != 0u;
    unsigned long long* buckets = vsum;  // the exact pass and the draw never overlap

    // Exact masses of the resident rows at item `base` (collective).  Thread 0
    // receives the summed limbs in lp / lq and the +Inf flags.
    uint32_t lp[kLimbs], lq[kLimbs];
    auto exact_pass = [&](long long base, bool with_q, const WarpT& wfp, const WarpT& wfq,
                          uint32_t& infl) -> bool {
      for (int k = tid; k < 2 * kBuckets; k += kConsumers) buckets[k] = 0ull;
      bar_consumers<kConsumers>();
      uint32_t bp = 0, bq = 0;
      for (int j = 0; j < nck; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        chunk_exact<T>(slot_ptr(base + j), n, wfp, buckets, bp);
        if (with_q) chunk_exact<T>(slot_ptr(base + nck + j), n, wfq, buckets + kBuckets, bq);
      }
      bp = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(bp)));
      bq = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(bq)));
      if (tid == 0) {
        buckets_to_limbs(buckets, &sm.myrec[0]);
        buckets_to_limbs(buckets + kBuckets, &sm.myrec[kLimbs]);
        sm.myrec[2 * kLimbs] = bp | (bq << 1);
        sm.myrec[2 * kLimbs + 1] = sm.myrec[2 * kLimbs + 2] = sm.myrec[2 * kLimbs + 3] = 0u;
      }
      if (!xchg(2 * kLimbs + 4)) return false;
      if (tid == 0) {
        unsigned long long ap[kLimbs], aq[kLimbs];
        for (int k = 0; k < kLimbs; ++k) ap[k] = aq[k] = 0ull;
        infl = 0;
        for (uint32_t c = 0; c < C; ++c) {
          for (int k = 0; k < kLimbs; ++k) {
            ap[k] += rec(c, k);
            aq[k] += rec(c, kLimbs + k);
          }
          infl |= rec(c, 2 * kLimbs);
        }
        unsigned long long cp = 0, cq = 0;
        for (int k = 0; k < kLimbs; ++k) {
          cp += ap[k];
          cq += aq[k];
          lp[k] = static_cast<uint32_t>(cp);
          lq[k] = static_cast<uint32_t>(cq);
          cp >>= 32;
          cq >>= 32;
        }
      }
      return true;
    };

    // Inverse-CDF draw over the resident row at item `base` (collective).
    // Returns 0 when done (the owning CTA wrote the outputs), 1 when the
    // residual is empty, -1 when a device wait gave up.
    auto draw = [&](long long base, bool resid, const WarpT& wfp, const WarpT& wfq, double Zp,
                    double Zq, int n_acc, uint32_t st_in, float u_draw) -> int {
      DrawW dw;
      norm_factors(Zp, dw.sp, dw.ap);
      norm_factors(resid ? Zq : 1.0, dw.sq, dw.aq);
      dw.scale = __uint_as_float(static_cast<uint32_t>(127 + P.fixed_shift) << 23);
      dw.resid = resid ? 1 : 0;
      const int vpc = ck_el / VEC;  // vectors per full chunk
      unsigned long long mine = 0;
      for (int j = 0; j < nck; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        const T* sp = slot_ptr(base + j);
        const T* sq = resid ? slot_ptr(base + nck + j) : nullptr;
        const int nv = (n + VEC - 1) / VEC;
        for (int vi = tid; vi < nv; vi += kConsumers) {
          float r[VEC];
          const int cnt = vec_draw_weights<T>(sp, sq, n, vi, wfp, wfq, dw, r);
          const unsigned long long f = dw.fix(seq_sum_n(r, cnt));
          vsum[j * vpc + vi] = f;
          mine += f;
        }
      }
      mine = block_sum_u64(mine, sm.redu);
      if (tid == 0) {
        sm.myrec[0] = static_cast<uint32_t>(mine);
        sm.myrec[1] = static_cast<uint32_t>(mine >> 32);
        sm.myrec[2] = sm.myrec[3] = 0u;
      }
      if (!xchg(4)) return -1;
      unsigned long long R = 0;
      for (uint32_t c = 0; c < C; ++c) R += rec_u64(c, 0);
      if (R == 0) {
        if (resid) return 1;
        if (tid == 0 && rank == 0) finish(n_acc, -1, st_in | ST_ZERO_MASS);
        return 0;
      }
      const unsigned long long tau = tau_of(u_draw, R);
      unsigned long long cum = 0, tloc = 0;
      uint32_t owner = C;
      for (uint32_t c = 0; c < C; ++c) {
        const unsigned long long rc = rec_u64(c, 0);
        if (tau < cum + rc) {
          owner = c;
          tloc = tau - cum;
          break;
        }
        cum += rc;
      }
      if (owner == C) {  // cannot happen: tau < R
        if (tid == 0 && rank == 0) finish(n_acc, -1, st_in | ST_TIMEOUT);
        return 0;
      }
      if (rank != owner) return 0;
      // ---- the owner: a scan of its per-vector sums, then one vector's elements
      int nvt = 0;
      for (int j = 0; j < nck; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        nvt = j * vpc + (n + VEC - 1) / VEC;
      }
      const int seg = (nvt + kConsumers - 1) / kConsumers;
      const int lo = min(nvt, tid * seg), hi = min(nvt, lo + seg);
      unsigned long long s = 0;
      for (int q = lo; q < hi; ++q) s += vsum[q];
      unsigned long long tot;
      const unsigned long long ex = block_excl_scan_u64(s, sm.redu, tot);
      if (tid == 0) sm.bi[0] = -1;
      bar_consumers<kConsumers>();
      if (tloc >= ex && tloc < ex + s) {
        unsigned long long c0 = ex;
        int q = lo;
        for (; q < hi - 1; ++q) {
          if (tloc < c0 + vsum[q]) break;
          c0 += vsum[q];
        }
        const int j = q / vpc, vi = q - j * vpc;
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        float r[VEC];
        const int cnt = vec_draw_weights<T>(slot_ptr(base + j),
                                            resid ? slot_ptr(base + nck + j) : nullptr, n, vi,
                                            wfp, wfq, dw, r);
        float acc = 0.f;
        unsigned long long prev = c0;
        for (int k = 0; k < cnt; ++k) {
          acc = k == 0 ? r[0] : __fadd_rn(acc, r[k]);
          const unsigned long long cur = c0 + dw.fix(acc);
          if (tloc < cur || k == cnt - 1) {
            const unsigned long long dlo = tloc - prev, dhi = cur > tloc ? cur - tloc : 0ull;
            const unsigned long long dmin = dlo < dhi ? dlo : dhi;
            sm.bi[0] = e0 + vi * VEC + k;
            sm.bi[1] = static_cast<double>(dmin) <= 1e-5 * static_cast<double>(R) ? 1 : 0;
            break;
          }
          prev = cur;
        }
      }
      bar_consumers<kConsumers>();
      if (tid == 0) {
        const int found = sm.bi[0];
        const uint32_t near = (found >= 0 && sm.bi[1]) ? ST_NEAR : 0u;
        finish(n_acc, found, found >= 0 ? (st_in | near) : (st_in | ST_TIMEOUT));
      }
      return 0;
    };

    for (int i = 0;; ++i) {
      const bool bonus = i == kb;
      const long long base = static_cast<long long>(i) * 2 * nck;
      const int nit = bonus ? nck : 2 * nck;

      // decision inputs gathered early by thread 0 (their latency overlaps the pass)
      int t = -1;
      float gp = 0.f, gq = 0.f, u = 0.f;
      if (tid == 0) {
        u = P.uni[t0 + i];
        if (!bonus) {
          t = P.tok[d0 + i];
          if (t >= 0 && t < P.V) {
            gp = TR::to_f(tgt[(t0 + i) * P.stride + t]);
            gq = TR::to_f(drf[(d0 + i) * P.stride + t]);
          }
        }
      }

      // ---- the pass over this row's chunks, as they arrive
      Acc ap, aq;
      Online op, oq;
      ap.init();
      aq.init();
      op.init();
      oq.init();
      float ep = MODE == MODE_PROBS ? kInfF : -kInfF;  // probs: min; logits: max (validity)
      float eq = ep;
      for (int j = 0; j < nit; ++j) {
        const long long g = base + j;
        acquire(g);
        const T* src;
        int e0, n;
        item(g, src, e0, n);
        const bool isq = j >= nck;
        if constexpr (MODE == MODE_PROBS)
          chunk_mass_f32(reinterpret_cast<const float*>(slot_ptr(g)), n, isq ? aq : ap,
                         isq ? eq : ep);
        else
          chunk_online<T>(slot_ptr(g), n, khi, isq ? oq : op, isq ? eq : ep);
      }

      // ---- CTA partials -> record
      tmo = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(tmo)));
      if constexpr (MODE == MODE_PROBS) {
        double v[2] = {ap.total(), aq.total()};
        block_sum_dn<2>(v, sm.redd);
        block_ext_f2<1>(ep, eq, sm.redf);
        if (tid == 0) {
          put_d(0, v[0]);
          put_d(2, v[1]);
          sm.myrec[4] = __float_as_uint(ep);
          sm.myrec[5] = __float_as_uint(eq);
          sm.myrec[6] = tmo;
          sm.myrec[7] = 0u;
        }
        if (!xchg(8)) {
          abort = true;
          break;
        }
      } else {
        float mcp = op.m, mcq = oq.m;
        block_ext_f2<0>(mcp, mcq, sm.redf);  // CTA running maxima (never NaN)
        block_ext_f2<0>(ep, eq, sm.redf);    // NaN-propagating maxima (validity)
        const int rr = block_max_i(max(op.r, oq.r), sm.redi);
        double v[4] = {0.0, 0.0, 0.0, 0.0};
        if (op.m > -kInfF) {
          const float d = __fmul_rn(__fsub_rn(mcp, op.m), khi);
          const double f = static_cast<double>(ex2_ftz(-d));
          v[0] = op.S() * f;
          v[1] = (op.W() + static_cast<double>(d) * op.S()) * f;
        }
        if (oq.m > -kInfF) {
          const float d = __fmul_rn(__fsub_rn(mcq, oq.m), khi);
          const double f = static_cast<double>(ex2_ftz(-d));
          v[2] = oq.S() * f;
          v[3] = (oq.W() + static_cast<double>(d) * oq.S()) * f;
        }
        block_sum_dn<4>(v, sm.redd);
        if (tid == 0) {
          sm.myrec[0] = __float_as_uint(mcp);
          sm.myrec[1] = __float_as_uint(mcq);
          sm.myrec[2] = __float_as_uint(ep);
          sm.myrec[3] = __float_as_uint(eq);
          put_d(4, v[0]);
          put_d(6, v[1]);
          put_d(8, v[2]);
          put_d(10, v[3]);
          sm.myrec[12] = static_cast<uint32_t>(rr);
          sm.myrec[13] = tmo;
          sm.myrec[14] = sm.myrec[15] = 0u;
        }
        if (!xchg(16)) {
          abort = true;
          break;
        }
      }

      // ---- thread 0 combines the records (same order in every CTA)
      if (tid == 0) {
        double Zp = 0.0, Zq = 0.0, Bp = 0.0, Bq = 0.0;
        float mp, mq, vp, vq;  // logits: row maxima / validity maxima; probs: minima
        uint32_t anytmo = 0;
        if constexpr (MODE == MODE_PROBS) {
          vp = vq = kInfF;
          for (uint32_t c = 0; c < C; ++c) {
            Zp += rec_d(c, 0);
            Zq += rec_d(c, 2);
            vp = fmin_nan(vp, __uint_as_float(rec(c, 4)));
            vq = fmin_nan(vq, __uint_as_float(rec(c, 5)));
            anytmo |= rec(c, 6);
          }
          mp = mq = 0.f;
          Bp = Zp * 16.0 * kU32;
          Bq = Zq * 16.0 * kU32;
        } else {
          mp = mq = -kInfF;
          vp = vq = -kInfF;
          int R = 0;
          for (uint32_t c = 0; c < C; ++c) {
            mp = fmaxf(mp, __uint_as_float(rec(c, 0)));
            mq = fmaxf(mq, __uint_as_float(rec(c, 1)));
            vp = fmax_nan(vp, __uint_as_float(rec(c, 2)));
            vq = fmax_nan(vq, __uint_as_float(rec(c, 3)));
            R = max(R, static_cast<int>(rec(c, 12)));
            anytmo |= rec(c, 13);
          }
          double Wp = 0.0, Wq = 0.0;
          for (uint32_t c = 0; c < C; ++c) {
            const float mcp = __uint_as_float(rec(c, 0)), mcq = __uint_as_float(rec(c, 1));
            if (mcp > -kInfF) {
              const float d = __fmul_rn(__fsub_rn(mp, mcp), khi);
              const double f = exp2(-static_cast<double>(d));
              Zp += rec_d(c, 4) * f;
              Wp += (rec_d(c, 6) + static_cast<double>(d) * rec_d(c, 4)) * f;
            }
            if (mcq > -kInfF) {
              const float d = __fmul_rn(__fsub_rn(mq, mcq), khi);
              const double f = exp2(-static_cast<double>(d));
              Zq += rec_d(c, 8) * f;
              Wq += (rec_d(c, 10) + static_cast<double>(d) * rec_d(c, 8)) * f;
            }
          }
          Bp = online_bound(Zp, Wp, R) + static_cast<double>(P.V) * 1.2e-38;
          Bq = online_bound(Zq, Wq, R) + static_cast<double>(P.V) * 1.2e-38;
        }
        uint32_t err = 0;
        if (!bonus && (t < 0 || t >= P.V)) err = ST_BAD_TOKEN;
        bool p_bad, q_bad;
        if constexpr (MODE == MODE_PROBS) {
          p_bad = !(vp >= 0.f);  // NaN or a negative value
          q_bad = !bonus && !(vq >= 0.f);
        } else {
          p_bad = !(vp < kInfF);  // NaN or +Inf logit
          q_bad = !bonus && !(vq < kInfF);
        }
        // probabilities: a non-finite approximate mass means a +Inf element
        // or an fp32 overflow of the partial sums; the exact pass tells.
        const bool need_inf_check = MODE == MODE_PROBS && !anytmo && !err && !p_bad && !q_bad &&
                                    (!(Zp <= DBL_MAX) || (!bonus && !(Zq <= DBL_MAX)));
        sm.bi[0] = anytmo ? ACT_ABORT : ACT_CONTINUE;
        sm.bi[1] = static_cast<int>(err);
        sm.bi[2] = (p_bad ? 1 : 0) | (q_bad ? 2 : 0) | (need_inf_check ? 4 : 0);
        sm.bd[0] = Zp;
        sm.bd[1] = Zq;
        sm.bd[2] = Bp;
        sm.bd[3] = Bq;
        sm.bd[4] = static_cast<double>(mp);
        sm.bd[5] = static_cast<double>(mq);
      }
      bar_consumers<kConsumers>();
      if (sm.bi[0] == ACT_ABORT) {
        abort = true;
        break;
      }
      const float mp = static_cast<float>(sm.bd[4]), mq = static_cast<float>(sm.bd[5]);
      const WarpT wfp = make_warp(mp), wfq = make_warp(mq);
      bool have_exact = false;
      if (sm.bi[2] & 4) {
        uint32_t infl = 0;
        if (!exact_pass(base, !bonus, wfp, wfq, infl)) {
          abort = true;
          break;
        }
        if (tid == 0) {
          sm.bi[2] = (sm.bi[2] & 3) | (infl & 1u ? 1 : 0) | (infl & 2u ? 2 : 0);
          sm.bd[0] = limbs_to_double(lp);
          sm.bd[1] = bonus ? 0.0 : limbs_to_double(lq);
        }
        have_exact = true;
      }
      // ---- input errors in the oracle's order, then the accept test
      if (tid == 0) {
        const double Zp = sm.bd[0], Zq = sm.bd[1];
        uint32_t err = static_cast<uint32_t>(sm.bi[1]);
        const bool p_bad = sm.bi[2] & 1, q_bad = (sm.bi[2] >> 1) & 1;
        if (!err && p_bad) err = ST_BAD_VALUE;
        if (!err && q_bad) err = ST_BAD_VALUE;
        if (!err && !(u >= 0.f && u < 1.f)) err = ST_BAD_VALUE;
        const bool p_zero = MODE == MODE_PROBS ? Zp == 0.0 : mp == -kInfF;
        const bool q_zero = MODE == MODE_PROBS ? Zq == 0.0 : mq == -kInfF;
        int act;
        if (err) {
          if (rank == 0) finish(i, -1, st | err);
          act = ACT_STOP;
        } else if (p_zero) {
          if (rank == 0) finish(i, -1, st | ST_ZERO_MASS);
          act = ACT_STOP;
        } else if (bonus) {
          act = ACT_DRAW;  // all K_b drafts accepted: the bonus comes from p_K
        } else if (q_zero) {
          if (rank == 0) finish(i, -1, st | ST_ZERO_MASS);
          act = ACT_STOP;
        } else {
          const float pt = wfp(gp), qt = wfq(gq);
          sm.bd[6] = pt;
          sm.bd[7] = qt;
          if (have_exact) {
            act = exact_accept(u, pt, qt, lp, lq) ? ACT_CONTINUE : ACT_DRAW;
            st |= ST_EXACT;
          } else {
            const int dec = filter_decide(u, pt, qt, Zp, sm.bd[2], Zq, sm.bd[3]);
            act = (force_exact || dec < 0) ? ACT_EXACT : (dec ? ACT_CONTINUE : ACT_DRAW);
          }
        }
        if (act == ACT_STOP || act == ACT_DRAW) sm.stop = 1;
        sm.bi[0] = act;
        sm.bi[4] = static_cast<int>(st);
      }
      bar_consumers<kConsumers>();
      int act = sm.bi[0];
      if (act == ACT_EXACT) {
        uint32_t infl = 0;
        if (!exact_pass(base, true, wfp, wfq, infl)) {
          abort = true;
          break;
        }
        if (tid == 0) {
          act = exact_accept(u, static_cast<float>(sm.bd[6]), static_cast<float>(sm.bd[7]), lp, lq)
                    ? ACT_CONTINUE
                    : ACT_DRAW;
          st |= ST_EXACT;
          if (act == ACT_DRAW) sm.stop = 1;
          sm.bi[0] = act;
          sm.bi[4] = static_cast<int>(st);
        }
        bar_consumers<kConsumers>();
        act = sm.bi[0];
      }
      // warped weights of this row for the caller (testing aid)
      if (MODE == MODE_LOGITS && (P.wt_out || P.wd_out) && act != ACT_STOP) {
        for (int j = 0; j < nck; ++j) {
          const T* src;
          int e0, n;
          item(base + j, src, e0, n);
          if (P.wt_out)
            chunk_write_weights<T>(slot_ptr(base + j), n, e0, wfp,
                                   P.wt_out + (t0 + i) * static_cast<long long>(P.V));
          if (P.wd_out && !bonus)
            chunk_write_weights<T>(slot_ptr(base + nck + j), n, e0, wfq,
                                   P.wd_out + (d0 + i) * static_cast<long long>(P.V));
        }
      }
      if (act == ACT_STOP) break;
      if (act == ACT_CONTINUE) {
        for (int j = 0; j < nit; ++j) release(base + j);
        continue;
      }
      // ---- ACT_DRAW: the bonus from p_K, or the residual after the first rejection
      const uint32_t st_now = static_cast<uint32_t>(sm.bi[4]);
      const float u_draw = P.uni[t0 + kb];
      if (!bonus && !(u_draw >= 0.f && u_draw < 1.f)) {
        if (tid == 0 && rank == 0) finish(i, -1, st_now | ST_BAD_VALUE);
        break;
      }
      const double Zp = sm.bd[0], Zq = sm.bd[1];
      int code = draw(base, !bonus, wfp, wfq, Zp, bonus ? 1.0 : Zq, bonus ? kb : i, st_now, u_draw);
      if (code == 1) code = draw(base, false, wfp, wfq, Zp, 1.0, i, st_now | ST_ZERO_MASS, u_draw);
      if (code < 0) abort = true;
      break;
    }
  }

  if (abort && tid == 0) finish(0, -1, ST_TIMEOUT);
  if (tid == 0) sm.stop = 1;  // the producer stops issuing and drains its copies
}

}  // namespace svk
