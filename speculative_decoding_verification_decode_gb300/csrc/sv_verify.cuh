// The verification kernel (see sv_kernel.cuh for the design notes).
#pragma once
#include <type_traits>

#include "sv_kernel.cuh"

namespace svk {

// ------------------------------------------------------------------ chunk passes
// `s` points at a shared-memory chunk of `n` consecutive row elements whose
// first element is column `e0` of the row.

template <typename T>
__device__ __forceinline__ void chunk_argmax(const T* s, int n, int e0, float& bv, int& bi,
                                             uint32_t& nanf) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kThreads) {
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
  for (int e = nv * VEC + threadIdx.x; e < n; e += kThreads) {
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
  for (int vi = threadIdx.x; vi < nv; vi += kThreads) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    const float x[4] = {v.x, v.y, v.z, v.w};
    a.add<8>(seq_sum<4>(x));
    mn = fmin_nan(mn, fmin_nan(fmin_nan(v.x, v.y), fmin_nan(v.z, v.w)));
  }
  for (int e = (nv << 2) + threadIdx.x; e < n; e += kThreads) {
    a.add<8>(s[e]);
    mn = fmin_nan(mn, s[e]);
  }
}

template <typename T>
__device__ __forceinline__ void chunk_max(const T* s, int n, float& mx) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kThreads) mx = fmax_nan(mx, vec_max_nan(s, vi));
  for (int e = nv * VEC + threadIdx.x; e < n; e += kThreads)
    mx = fmax_nan(mx, ElemTraits<T>::to_f(s[e]));
}

template <typename T, typename W>
__device__ __forceinline__ void chunk_wmass(const T* s, int n, int e0, const W& wf, Acc& a,
                                            float* wout) {
  constexpr int VEC = ElemTraits<T>::kVec;
  constexpr int FL = ElemTraits<T>::kFlush;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kThreads) {
    float x[VEC];
    load_vec(s, vi, x);
#pragma unroll
    for (int k = 0; k < VEC; ++k) x[k] = wf(x[k]);
    a.add<FL>(seq_sum<VEC>(x));
    if (wout) {
#pragma unroll
      for (int k = 0; k < VEC; ++k) wout[e0 + vi * VEC + k] = x[k];
    }
  }
  for (int e = nv * VEC + threadIdx.x; e < n; e += kThreads) {
    const float w = wf(ElemTraits<T>::to_f(s[e]));
    a.add<FL>(w);
    if (wout) wout[e0 + e] = w;
  }
}

template <typename T, typename W>
__device__ __forceinline__ void chunk_exact(const T* s, int n, const W& wf, unsigned long long* bk,
                                            uint32_t& bad) {
  for (int e = threadIdx.x; e < n; e += kThreads) {
    const float x = wf(ElemTraits<T>::to_f(s[e]));
    if (!(x <= FLT_MAX)) bad = 1u;  // +Inf (NaN and negatives were rejected before)
    else bucket_add(bk, x);
  }
}

template <typename T, typename W>
__device__ __forceinline__ unsigned long long draw_elem(const T* sp, const T* sq, int e,
                                                        const W& wf_p, const W& wf_q,
                                                        const DrawW& dw) {
  const float p = wf_p(ElemTraits<T>::to_f(sp[e]));
  const float q = sq ? wf_q(ElemTraits<T>::to_f(sq[e])) : 0.f;
  return dw(p, q);
}

template <typename T, typename W>
__device__ __forceinline__ unsigned long long chunk_draw_sum(const T* sp, const T* sq, int n,
                                                             const W& wf_p, const W& wf_q,
                                                             const DrawW& dw) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int nv = n / VEC;
  unsigned long long acc = 0;
  for (int vi = threadIdx.x; vi < nv; vi += kThreads) {
    float xp[VEC], xq[VEC];
    load_vec(sp, vi, xp);
    if (sq) load_vec(sq, vi, xq);
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc += dw(wf_p(xp[k]), sq ? wf_q(xq[k]) : 0.f);
  }
  for (int e = nv * VEC + threadIdx.x; e < n; e += kThreads) acc += draw_elem(sp, sq, e, wf_p, wf_q, dw);
  return acc;
}

// ------------------------------------------------------------------ the kernel

template <int MODE, typename T>
__global__ void __launch_bounds__(kThreads, 2) sv_verify_kernel(const Params P) {
  using TR = ElemTraits<T>;
  constexpr int VEC = TR::kVec;
  constexpr int ELEM = static_cast<int>(sizeof(T));
  using WarpT =
      typename std::conditional<MODE == MODE_LOGITS, typename WarpOf<T>::type, NoWarp>::type;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  SmemTail& sm = *reinterpret_cast<SmemTail*>(smem + P.S * kSlotBytes);
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
  const int v_lo = static_cast<int>(rank) * P.slice;
  const int v_hi = min(P.V, v_lo + P.slice);
  const int n_el = max(0, v_hi - v_lo);
  const int nck = (n_el + P.ck_el - 1) / P.ck_el;
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
    e0 = v_lo + j * P.ck_el;
    n = min(v_hi, e0 + P.ck_el) - e0;
    const long long row = isq ? d0 + r : t0 + r;
    src = (isq ? drf : tgt) + row * P.stride + e0;
  };
  auto slot_ptr = [&](long long g) {
    return reinterpret_cast<const T*>(ring + (g % P.S) * kSlotBytes);
  };

  // ---------------------------------------------------------------- barriers
  if (tid == 0) {
    for (int s = 0; s < P.S; ++s) mbar_init(&sm.full[s], 1);
    mbar_init(&sm.xbar[0], C);
    mbar_init(&sm.xbar[1], C);
    fence_mbar_init_cluster();
  }
  __syncthreads();
  cluster_sync_all();  // every peer's barriers exist before the first remote arrive

  // ---------------------------------------------------------------- producer (thread 0)
  long long issued = 0, released = 0;
  const long long limit = total_items;
  auto issue = [&](long long g) {
    const T* src;
    int e0, n;
    item(g, src, e0, n);
    const int slot = static_cast<int>(g % P.S);
    const uint32_t bytes = static_cast<uint32_t>(n) * ELEM;
    const uint32_t tma = P.use_tma ? (bytes & ~15u) : 0u;
    if (tma) {
      mbar_arrive_expect_tx(&sm.full[slot], tma);
      bulk_g2s(ring + slot * kSlotBytes, src, tma, &sm.full[slot]);
    } else {
      mbar_arrive_local(&sm.full[slot]);
    }
  };
  auto pump = [&]() {
    while (issued < limit && issued < released + P.S) {
      issue(issued);
      ++issued;
    }
  };
  if (tid == 0) pump();

  // ---------------------------------------------------------------- consumer helpers
  long long consumed = 0;
  auto acquire = [&](long long g) -> bool {
    const T* src;
    int e0, n;
    item(g, src, e0, n);
    const int slot = static_cast<int>(g % P.S);
    const bool ok = mbar_wait_bounded(&sm.full[slot], static_cast<uint32_t>((g / P.S) & 1));
    // elements the bulk copy did not move (unaligned rows, or a ragged tail)
    const int done =
        P.use_tma ? static_cast<int>(((static_cast<uint32_t>(n) * ELEM) & ~15u) / ELEM) : 0;
    T* dst = reinterpret_cast<T*>(ring + slot * kSlotBytes);
    for (int e = done + tid; e < n; e += kThreads) dst[e] = src[e];
    return __syncthreads_and(ok) != 0;
  };
  auto release_to = [&](long long g_end) {
    __syncthreads();
    if (tid == 0) {
      released = g_end;
      pump();
    }
  };

  int xc = 0, last_slot = 0;
  auto xchg = [&](int words) -> bool {
    __syncthreads();
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
    return __syncthreads_and(ok) != 0;
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
  auto finish = [&](int n, int nxt, uint32_t s) {
    if (tid == 0) {
      P.n_out[b] = n;
      P.next_out[b] = nxt;
      P.st_out[b] = s;
    }
  };

  uint32_t st = 0;
  bool abort = false;

  if (!sampling) {
    // ============================================================== greedy
    for (int i = 0;; ++i) {
      float bv = __int_as_float(0x7FFFFFFF);  // NaN: no candidate yet
      int bi = INT_MAX;
      uint32_t nanf = 0;
      for (int j = 0; j < nck; ++j) {
        const long long g = static_cast<long long>(i) * nck + j;
        if (!acquire(g)) {
          abort = true;
          break;
        }
        const T* src;
        int e0, n;
        item(g, src, e0, n);
        chunk_argmax<T>(slot_ptr(g), n, e0, bv, bi, nanf);
        consumed = g + 1;
        release_to(g + 1);
      }
      if (abort) break;
      if (bv != bv) bi = INT_MAX;
      block_argmax(bv, bi, sm.redf, sm.redi);
      nanf = static_cast<uint32_t>(__syncthreads_or(static_cast<int>(nanf)));
      if (tid == 0) {
        sm.myrec[0] = __float_as_uint(bv);
        sm.myrec[1] = static_cast<uint32_t>(bi);
        sm.myrec[2] = nanf;
        sm.myrec[3] = 0u;
      }
      if (!xchg(4)) {
        abort = true;
        break;
      }
      float v = 0.f;
      int a = INT_MAX;
      uint32_t nf = 0;
      for (uint32_t c = 0; c < C; ++c) {
        const float vc = __uint_as_float(rec(c, 0));
        const int ic = static_cast<int>(rec(c, 1));
        nf |= rec(c, 2);
        if (arg_better(vc, ic, v, a)) {
          v = vc;
          a = ic;
        }
      }
      if (a == INT_MAX) a = 0;  // an all-NaN row
      if (nf) st |= ST_BAD_VALUE;
      if (i == kb) {
        if (rank == 0) finish(kb, a, st);
        break;
      }
      const int t = P.tok[d0 + i];
      if (t < 0 || t >= P.V) {
        if (rank == 0) finish(i, a, st | ST_BAD_TOKEN);
        break;
      }
      if (t != a) {
        if (rank == 0) finish(i, a, st);
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
    const float u_draw = P.uni[t0 + kb];

    // Exact masses of the resident rows at item `base` (collective).  Fills
    // kLimbs limbs per row (identical in every CTA) and the +Inf flags.
    auto exact_pass = [&](long long base, bool with_q, const WarpT& wfp, const WarpT& wfq,
                          uint32_t* lp, uint32_t* lq, uint32_t& infl) -> bool {
      for (int k = tid; k < 2 * kBuckets; k += kThreads) (&sm.buckets[0][0])[k] = 0ull;
      __syncthreads();
      uint32_t bp = 0, bq = 0;
      for (int j = 0; j < nck; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        chunk_exact<T>(slot_ptr(base + j), n, wfp, sm.buckets[0], bp);
        if (with_q) chunk_exact<T>(slot_ptr(base + nck + j), n, wfq, sm.buckets[1], bq);
      }
      bp = static_cast<uint32_t>(__syncthreads_or(static_cast<int>(bp)));
      bq = static_cast<uint32_t>(__syncthreads_or(static_cast<int>(bq)));
      if (tid == 0) {
        buckets_to_limbs(sm.buckets[0], &sm.myrec[0]);
        buckets_to_limbs(sm.buckets[1], &sm.myrec[kLimbs]);
        sm.myrec[2 * kLimbs] = bp | (bq << 1);
        sm.myrec[2 * kLimbs + 1] = sm.myrec[2 * kLimbs + 2] = sm.myrec[2 * kLimbs + 3] = 0u;
      }
      if (!xchg(2 * kLimbs + 4)) return false;
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
      return true;
    };

    // Inverse-CDF draw over the resident row at item `base` (collective).
    // Returns 0 when done (the owning CTA wrote the outputs), 1 when the
    // residual is empty, -1 when a device wait gave up.
    auto draw = [&](long long base, bool resid, const WarpT& wfp, const WarpT& wfq, double Zp,
                    double Zq, int n_acc, uint32_t st_in) -> int {
      DrawW dw;
      norm_factors(Zp, dw.sp, dw.ap);
      norm_factors(resid ? Zq : 1.0, dw.sq, dw.aq);
      dw.scale = __uint_as_float(static_cast<uint32_t>(127 + P.fixed_shift) << 23);
      dw.resid = resid ? 1 : 0;
      unsigned long long mine = 0;
      for (int j = 0; j < nck; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        mine += chunk_draw_sum<T>(slot_ptr(base + j), resid ? slot_ptr(base + nck + j) : nullptr,
                                  n, wfp, wfq, dw);
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
        if (rank == 0) finish(n_acc, -1, st_in | ST_ZERO_MASS);
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
        if (rank == 0) finish(n_acc, -1, st_in | ST_TIMEOUT);
        return 0;
      }
      if (rank != owner) return 0;
      // ---- the owner walks its slice in element order, one tile per pass
      if (tid == 0) {
        sm.misc[0] = -1;
        sm.misc[1] = 0;
      }
      __syncthreads();
      unsigned long long run = 0;
      bool hit = false;
      for (int j = 0; j < nck && !hit; ++j) {
        const T* src;
        int e0, n;
        item(base + j, src, e0, n);
        const T* sp = slot_ptr(base + j);
        const T* sq = resid ? slot_ptr(base + nck + j) : nullptr;
        const int nv = (n + VEC - 1) / VEC;
        for (int tile = 0; tile < nv; tile += kThreads) {
          const int vi = tile + tid;
          unsigned long long s = 0;
          if (vi < nv) {
            for (int k = 0; k < VEC; ++k) {
              const int e = vi * VEC + k;
              if (e < n) s += draw_elem(sp, sq, e, wfp, wfq, dw);
            }
          }
          unsigned long long tot;
          const unsigned long long ex = block_excl_scan_u64(s, sm.redu, tot);
          if (tloc < run + tot) {
            if (vi < nv && tloc >= run + ex && tloc < run + ex + s) {
              unsigned long long c0 = run + ex;
              for (int k = 0; k < VEC; ++k) {
                const int e = vi * VEC + k;
                if (e >= n) break;
                const unsigned long long w = draw_elem(sp, sq, e, wfp, wfq, dw);
                if (tloc < c0 + w) {
                  const unsigned long long dlo = tloc - c0, dhi = c0 + w - tloc;
                  const unsigned long long dmin = dlo < dhi ? dlo : dhi;
                  sm.misc[0] = e0 + e;
                  sm.misc[1] = static_cast<double>(dmin) <= 1e-5 * static_cast<double>(R) ? 1 : 0;
                  break;
                }
                c0 += w;
              }
            }
            hit = true;
            break;
          }
          run += tot;
        }
      }
      __syncthreads();
      const int found = sm.misc[0];
      const uint32_t near = (found >= 0 && sm.misc[1]) ? ST_NEAR : 0u;
      finish(n_acc, found, found >= 0 ? (st_in | near) : (st_in | ST_TIMEOUT));
      return 0;
    };

    for (int i = 0;; ++i) {
      const bool bonus = i == kb;
      const long long base = static_cast<long long>(i) * 2 * nck;
      const int nit = bonus ? nck : 2 * nck;

      // ---- pass 1: masses (probabilities) or maxima (logits) of the slice
      Acc ap, aq;
      ap.init();
      aq.init();
      float ext_p = MODE == MODE_PROBS ? kInfF : -kInfF;
      float ext_q = ext_p;
      for (int j = 0; j < nit; ++j) {
        const long long g = base + j;
        if (!acquire(g)) {
          abort = true;
          break;
        }
        const T* src;
        int e0, n;
        item(g, src, e0, n);
        const bool isq = j >= nck;
        if constexpr (MODE == MODE_PROBS)
          chunk_mass_f32(reinterpret_cast<const float*>(slot_ptr(g)), n, isq ? aq : ap,
                         isq ? ext_q : ext_p);
        else
          chunk_max<T>(slot_ptr(g), n, isq ? ext_q : ext_p);
      }
      if (abort) break;
      consumed = base + nit;

      double Zp = 0.0, Zq = 0.0;
      float mp, mq;  // probabilities: row minimum; logits: row maximum (NaN-propagating)
      if constexpr (MODE == MODE_PROBS) {
        const double zp = block_sum_d(ap.total(), sm.redd);
        const double zq = block_sum_d(aq.total(), sm.redd);
        const float a1 = block_ext_f<1>(ext_p, sm.redf);
        const float a2 = block_ext_f<1>(ext_q, sm.redf);
        if (tid == 0) {
          put_d(0, zp);
          put_d(2, zq);
          sm.myrec[4] = __float_as_uint(a1);
          sm.myrec[5] = __float_as_uint(a2);
          sm.myrec[6] = sm.myrec[7] = 0u;
        }
        if (!xchg(8)) {
          abort = true;
          break;
        }
        mp = kInfF;
        mq = kInfF;
        for (uint32_t c = 0; c < C; ++c) {
          Zp += rec_d(c, 0);
          Zq += rec_d(c, 2);
          mp = fmin_nan(mp, __uint_as_float(rec(c, 4)));
          mq = fmin_nan(mq, __uint_as_float(rec(c, 5)));
        }
      } else {
        const float a1 = block_ext_f<0>(ext_p, sm.redf);
        const float a2 = block_ext_f<0>(ext_q, sm.redf);
        if (tid == 0) {
          sm.myrec[0] = __float_as_uint(a1);
          sm.myrec[1] = __float_as_uint(a2);
          sm.myrec[2] = sm.myrec[3] = 0u;
        }
        if (!xchg(4)) {
          abort = true;
          break;
        }
        mp = -kInfF;
        mq = -kInfF;
        for (uint32_t c = 0; c < C; ++c) {
          mp = fmax_nan(mp, __uint_as_float(rec(c, 0)));
          mq = fmax_nan(mq, __uint_as_float(rec(c, 1)));
        }
      }

      // ---- input errors, in the order the oracle checks them
      uint32_t err = 0;
      int t = -1;
      if (!bonus) {
        t = P.tok[d0 + i];
        if (t < 0 || t >= P.V) err = ST_BAD_TOKEN;
      }
      bool p_bad, q_bad;
      if constexpr (MODE == MODE_PROBS) {
        p_bad = !(mp >= 0.f);  // NaN or a negative value
        q_bad = !bonus && !(mq >= 0.f);
      } else {
        p_bad = !(mp < kInfF);  // NaN or +Inf logit
        q_bad = !bonus && !(mq < kInfF);
      }
      const WarpT wfp = make_warp(mp), wfq = make_warp(mq);
      bool have_exact = false;
      uint32_t lp[kLimbs], lq[kLimbs];
      if constexpr (MODE == MODE_PROBS) {
        // A non-finite approximate mass means a +Inf element or an fp32
        // overflow of the partial sums: the exact pass tells them apart.
        if (!err && !p_bad && !q_bad && (!(Zp <= DBL_MAX) || (!bonus && !(Zq <= DBL_MAX)))) {
          uint32_t infl = 0;
          if (!exact_pass(base, !bonus, wfp, wfq, lp, lq, infl)) {
            abort = true;
            break;
          }
          if (infl & 1u) p_bad = true;
          if (infl & 2u) q_bad = true;
          Zp = limbs_to_double(lp);
          Zq = bonus ? 0.0 : limbs_to_double(lq);
          have_exact = true;
        }
      }
      if (!err && p_bad) err = ST_BAD_VALUE;
      if (!err && q_bad) err = ST_BAD_VALUE;
      const float u = P.uni[t0 + i];
      if (!err && !(u >= 0.f && u < 1.f)) err = ST_BAD_VALUE;
      if (err) {
        if (rank == 0) finish(i, -1, st | err);
        break;
      }
      const bool p_zero = MODE == MODE_PROBS ? Zp == 0.0 : mp == -kInfF;
      if (p_zero) {
        if (rank == 0) finish(i, -1, st | ST_ZERO_MASS);
        break;
      }
      if constexpr (MODE == MODE_LOGITS) {
        if (!bonus && mq == -kInfF) {
          if (rank == 0) finish(i, -1, st | ST_ZERO_MASS);
          break;
        }
        // ---- pass 2: weights of the resident rows and their masses
        Acc bp, bq;
        bp.init();
        bq.init();
        for (int j = 0; j < nck; ++j) {
          const T* src;
          int e0, n;
          item(base + j, src, e0, n);
          chunk_wmass<T>(slot_ptr(base + j), n, e0, wfp, bp,
                         P.wt_out ? P.wt_out + (t0 + i) * static_cast<long long>(P.V) : nullptr);
          if (!bonus)
            chunk_wmass<T>(slot_ptr(base + nck + j), n, e0, wfq, bq,
                           P.wd_out ? P.wd_out + (d0 + i) * static_cast<long long>(P.V) : nullptr);
        }
        const double zp = block_sum_d(bp.total(), sm.redd);
        const double zq = block_sum_d(bq.total(), sm.redd);
        if (tid == 0) {
          put_d(0, zp);
          put_d(2, zq);
        }
        if (!xchg(4)) {
          abort = true;
          break;
        }
        for (uint32_t c = 0; c < C; ++c) {
          Zp += rec_d(c, 0);
          Zq += rec_d(c, 2);
        }
      }
      if (bonus) {
        // all K_b drafts accepted: the bonus token is drawn from p_K
        if (draw(base, false, wfp, wfq, Zp, 1.0, kb, st) < 0) abort = true;
        break;
      }
      if (MODE == MODE_PROBS && Zq == 0.0) {
        if (rank == 0) finish(i, -1, st | ST_ZERO_MASS);
        break;
      }

      // ---- the accept test  u * q(t) * Zp < p(t) * Zq
      float pt, qt;
      {
        const float lpt = TR::to_f(tgt[(t0 + i) * P.stride + t]);
        const float lqt = TR::to_f(drf[(d0 + i) * P.stride + t]);
        pt = wfp(lpt);
        qt = wfq(lqt);
      }
      int dec = have_exact ? -1 : filter_decide(u, pt, qt, Zp, Zq);
      if (force_exact || dec < 0) {
        if (!have_exact) {
          uint32_t infl = 0;
          if (!exact_pass(base, true, wfp, wfq, lp, lq, infl)) {
            abort = true;
            break;
          }
          have_exact = true;
        }
        dec = exact_accept(u, pt, qt, lp, lq) ? 1 : 0;
        st |= ST_EXACT;
      }
      if (dec) {
        release_to(base + nit);
        continue;
      }
      // ---- first rejection: resample from norm(max(0, phat - qhat)) with u_K
      if (!(u_draw >= 0.f && u_draw < 1.f)) {
        if (rank == 0) finish(i, -1, st | ST_BAD_VALUE);
        break;
      }
      int code = draw(base, true, wfp, wfq, Zp, Zq, i, st);
      if (code == 1) code = draw(base, false, wfp, wfq, Zp, 1.0, i, st | ST_ZERO_MASS);
      if (code < 0) abort = true;
      break;
    }
  }

  if (abort) finish(0, -1, ST_TIMEOUT);
  // no bulk copy may still be writing this CTA's shared memory at exit
  if (tid == 0)
    for (long long g = consumed; g < issued; ++g)
      mbar_wait_bounded(&sm.full[g % P.S], static_cast<uint32_t>((g / P.S) & 1));
}

}  // namespace svk
