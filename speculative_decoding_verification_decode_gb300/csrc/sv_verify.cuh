// The verification kernel (design notes in sv_kernel.cuh).
#pragma once
#include <type_traits>

#include "sv_kernel.cuh"

namespace svk {

// ------------------------------------------------------------------ chunk passes
// `s` points at `n` consecutive row elements (shared memory, or global memory
// for the second looks at a row) whose first element is column `e0`.
// Consumer thread c handles the 16-byte vectors c, c + 256, ...

template <typename T>
__device__ __forceinline__ void chunk_argmax(const T* s, int n, int e0, float& bv, int& bi,
                                             uint32_t& nanf) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int nv = n / VEC;
  for (int vi = threadIdx.x; vi < nv; vi += kConsumers) {
    float x[VEC];
    const float m = load_vec_max(s, vi, x);
    if (!(m <= bv)) {  // a new maximum, a NaN, or no candidate yet
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
    a.add(tree_sum<4>(x0));
    a.add(tree_sum<4>(x1));
    mn = fmin_nan(mn, fmin_nan(fmin_nan(fmin_nan(v0.x, v0.y), fmin_nan(v0.z, v0.w)),
                               fmin_nan(fmin_nan(v1.x, v1.y), fmin_nan(v1.z, v1.w))));
  }
  if (vi < nv) {
    const float4 v = reinterpret_cast<const float4*>(s)[vi];
    const float x[4] = {v.x, v.y, v.z, v.w};
    a.add(tree_sum<4>(x));
    mn = fmin_nan(mn, fmin_nan(fmin_nan(v.x, v.y), fmin_nan(v.z, v.w)));
  }
  for (int e = (nv << 2) + threadIdx.x; e < n; e += kConsumers) {
    a.add(s[e]);
    mn = fmin_nan(mn, s[e]);
  }
}

// Online softmax over a chunk of logits; `mx` tracks the NaN-propagating max
// (for validity), `o` the running max and sums (for the mass).  Logits below
// the row's floor `lo` (the sampler filters; -Inf: none) enter the sums as
// -Inf, i.e. with weight 0; the maximum and the validity check see them as
// they are (the floor never exceeds the row maximum).
template <typename T, bool FL>
__device__ __forceinline__ void chunk_online(const T* s, int n, float k, float lo, Online& o, float& mx) {
  constexpr int VEC = ElemTraits<T>::kVec;
  constexpr int U = 4;  // vectors a thread holds at once (independent exps)
  const int nv = n / VEC;
  for (int base = threadIdx.x; base < nv; base += U * kConsumers) {
    float x[U][VEC];
    bool have[U];
    float vm, vmin;
    load_block<T, U, VEC>(s, base, nv, x, have, vm, vmin);
    mx = fmax_nan(mx, vm);
    if constexpr (FL) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < VEC; ++j) x[u][j] = x[u][j] < lo ? -kInfF : x[u][j];
    }
    o.add_block<U, VEC>(x, have, vm, vmin, k);
  }
  for (int e = nv * VEC + threadIdx.x; e < n; e += kConsumers) {
    const float x = ElemTraits<T>::to_f(s[e]);
    mx = fmax_nan(mx, x);
    const float xm = (FL && x < lo) ? -kInfF : x;
    o.add_vec<1>(&xm, xm, k);
  }
}

// Element e of a row slice in global memory.
template <typename T>
__device__ __forceinline__ float gload(const T* p, int e) {
  if constexpr (sizeof(T) == 4) {
    return __ldg(reinterpret_cast<const float*>(p) + e);
  } else {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p) + e);
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(static_cast<uint32_t>(b) << 16);
    else return __half2float(__ushort_as_half(b));
  }
}

// The floats of one 16-byte vector.
template <typename T>
__device__ __forceinline__ void unpack_vec(const uint4 v, float* x) {
  if constexpr (sizeof(T) == 4) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  } else {
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

// Vector vi (16 bytes) of a 16-byte aligned row slice in global memory.
template <typename T>
__device__ __forceinline__ void gload_vec(const T* p, int vi, float* x) {
  unpack_vec<T>(__ldg(reinterpret_cast<const uint4*>(p) + vi), x);
}

// Draw weights of vector vi of a row slice pair in global memory (`q` may be
// null).  Always fills VEC entries (zero past the slice end); returns the
// number of real elements.
template <typename T, typename D>
__device__ __forceinline__ int vec_draw_weights(const T* p, const T* q, int n, int vi, bool vec_ok,
                                                const D& dw, float* r) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int e0 = vi * VEC;
  float xp[VEC], xq[VEC];
  int cnt = VEC;
  if (vec_ok && e0 + VEC <= n) {
    gload_vec<T>(p, vi, xp);
    if (q) gload_vec<T>(q, vi, xq);
  } else {
    cnt = min(VEC, n - e0);
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      xp[k] = k < cnt ? gload<T>(p, e0 + k) : 0.f;
      xq[k] = (q && k < cnt) ? gload<T>(q, e0 + k) : 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < VEC; ++k) r[k] = k < cnt ? dw(xp[k], q ? xq[k] : 0.f) : 0.f;
  return cnt;
}

// Left-to-right fp32 sum of r[0..VEC) (the order the owner's walk repeats).
template <int VEC>
__device__ __forceinline__ float seq_sum(const float* r) {
  float t = r[0];
#pragma unroll
  for (int k = 1; k < VEC; ++k) t = __fadd_rn(t, r[k]);
  return t;
}

// ------------------------------------------------------------------ the kernel

enum : int { ACT_CONTINUE = 0, ACT_STOP = 1, ACT_EXACT = 2, ACT_DRAW = 3, ACT_ABORT = 4 };

// FL: logits rows with sampler-filter floors (P.flo_t / P.flo_d); a separate
// instantiation, so the unfiltered kernels carry none of its code.
template <int MODE, typename T, bool FL = false>
__global__ void __launch_bounds__(threads_of(MODE), 2) sv_verify_kernel(const __grid_constant__ Params P) {
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
  if (P.gate && !P.gate[b]) return;
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
      P.st_out[b] = (layout_ok ? ST_BAD_VALUE : ST_BAD_LAYOUT) | (P.ext_err && *P.ext_err ? ST_TIMEOUT : 0u);
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
  const int last_n = n_el - (nck - 1) * ck_el;
  // start of this CTA's slice of target row r (draft row r when q)
  auto row_slice = [&](bool q, int r) -> const T* {
    return q ? drf + (d0 + r) * P.stride + v_lo : tgt + (t0 + r) * P.stride + v_lo;
  };
  // the sampler filters' floor of target row r (draft row r when q); -Inf: none
  auto row_floor = [&](bool q, int r) -> float {
    if constexpr (!FL) {
      (void)q;
      (void)r;
      return -kInfF;
    } else {
      const float* f = q ? P.flo_d : P.flo_t;
      return f ? __ldg(f + (q ? d0 : t0) + r) : -kInfF;
    }
  };

  // ---------------------------------------------------------------- barriers
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kWarps);
    }
    mbar_init(&sm.xbar[0], C);
    mbar_init(&sm.xbar[1], C);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&sm.pfull[q], kWarps);
      mbar_init(&sm.dfull[q], 1);
    }
    mbar_init(&sm.xfull, 1);
    mbar_init(&sm.xdec, 1);
    sm.xc = 0;
    sm.cut_row = -1;
    sm.stop = 0;
    sm.go_row = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  cluster_sync_all();  // every peer's barriers exist before the first remote arrive
  // The warp index taken from lane 0 is warp-uniform for the compiler too, so
  // branches on it are not treated as divergent and the warp-collective code
  // inside them compiles to its converged form.
  const int warp = __shfl_sync(0xFFFFFFFFu, tid >> 5, 0);
  const int lane = tid & 31;

  // ================================================================ producer warp
  if (warp == kWarps) {
    int slot = 0;
    uint32_t round = 0;
    bool stopped = false;
    for (int r = 0; r <= kb && !stopped; ++r) {
      const int parts = (sampling && r < kb) ? 2 : 1;
      for (int part = 0; part < parts && !stopped; ++part) {
        const T* rowp = row_slice(part == 1, r);
        for (int j = 0; j < nck; ++j) {
          int go = 1;
          if (lane == 0) {
            // Sampling: the consumers reduce every row up to P.look past the
            // last accepted row (row i + 1 while row i is decided) unless they
            // cut a row short together (sm.cut_row: that row and every later
            // one are never consumed), so exactly those rows are issued; the
            // stop flag is not consulted inside them.  Greedy: the consumers
            // stop at once, so may the producer.
            const bool may_stop = !sampling;
            // sampling: the row gate comes before the wait for a free slot, as
            // that slot may hold a chunk of a cut row that is never released
            if (sampling && j == 0 && part == 0) {
              uint32_t polls = 0;
              while (r > sm.go_row + P.look && !sm.stop) {
                __nanosleep(32);  // the next row is issued within a fraction of a microsecond
                if (++polls == kWaitPolls * 64u) break;
              }
              if (r > sm.go_row + P.look) go = 0;  // stopped, or the wait gave up
            }
            if (go && round > 0) {
              uint32_t polls = 0;  // poll (not suspend): the flags must be seen at once
              while (!mbar_test(&sm.empty[slot], (round - 1) & 1u)) {
                const int cr = sm.cut_row;
                if ((may_stop && sm.stop) || (cr >= 0 && r >= cr) || ++polls == kWaitPolls * 128u) {
                  go = 0;
                  break;
                }
                __nanosleep(32);
              }
            }
            const int cr = sm.cut_row;
            if (cr >= 0 && r >= cr) go = 0;
            if (may_stop && sm.stop) go = 0;
          }
          go = __shfl_sync(0xFFFFFFFFu, go, 0);
          if (!go) {
            stopped = true;
            break;
          }
          const int n = j == nck - 1 ? last_n : ck_el;
          const T* src = rowp + j * ck_el;
          T* dst = reinterpret_cast<T*>(ring + slot * P.slot_bytes);
          const uint32_t bytes = static_cast<uint32_t>(n) * ELEM;
          const uint32_t tma = P.use_tma ? (bytes & ~15u) : 0u;
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
          if (++slot == S) {
            slot = 0;
            ++round;
          }
        }
      }
    }
    // no bulk copy may still be writing this CTA's shared memory at exit
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        if (s < slot) mbar_wait_bounded(&sm.full[s], round & 1u);
        else if (round > 0) mbar_wait_bounded(&sm.full[s], (round - 1) & 1u);
      }
    }
  } else if (warp != kDecideWarp || sampling) {  // greedy rows are decided by consumer warp 0

  // ================================================================ consumers (and the decision warp)
  // The last consumer warp fetches every row's decision inputs (draft token,
  // uniform, p(t), q(t)) now, while the first chunks are still in flight.
  if (warp == kWarps - 1 && lane < kMaxGather && lane <= kb) {
    const int i = lane;
    sm.g_u[i] = (sampling && P.uni) ? ld_issue_f32(P.uni + t0 + i) : 0.f;
    int t = -1;
    float gp = 0.f, gq = 0.f;
    if (i < kb) {
      t = ld_issue_s32(P.tok + d0 + i);
      if (sampling && t >= 0 && t < P.V) {
        if constexpr (sizeof(T) == 4) {
          gp = ld_issue_f32(reinterpret_cast<const float*>(tgt + (t0 + i) * P.stride + t));
          gq = ld_issue_f32(reinterpret_cast<const float*>(drf + (d0 + i) * P.stride + t));
        } else {
          const unsigned short hp =
              ld_issue_u16(reinterpret_cast<const unsigned short*>(tgt + (t0 + i) * P.stride + t));
          const unsigned short hq =
              ld_issue_u16(reinterpret_cast<const unsigned short*>(drf + (d0 + i) * P.stride + t));
          gp = TR::to_f(*reinterpret_cast<const T*>(&hp));
          gq = TR::to_f(*reinterpret_cast<const T*>(&hq));
        }
      }
    }
    sm.g_t[i] = t;
    sm.g_p[i] = gp;
    sm.g_q[i] = gq;
  }
  // row i's inputs (thread 0, after a consumer barrier has passed)
  auto row_token = [&](int i) -> int { return i < kMaxGather ? sm.g_t[i] : P.tok[d0 + i]; };
  uint32_t tmo = 0;
  int cslot = 0, rslot = 0;  // acquire and release cursors (same order)
  uint32_t cround = 0;
  auto acquire = [&]() -> const T* {
    if (!mbar_wait_bounded(&sm.full[cslot], cround & 1u)) tmo = 1u;
    const T* s = reinterpret_cast<const T*>(ring + cslot * P.slot_bytes);
    if (++cslot == S) {
      cslot = 0;
      ++cround;
    }
    return s;
  };
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive_local(&sm.empty[rslot]);
    if (++rslot == S) rslot = 0;
  };

  // Exchange of sm.myrec with every CTA of the cluster: a collective of
  // warp 0 (lane c pushes the record into CTA c, then every lane waits until
  // all C records have arrived here).
  // (The count of exchanges lives in shared memory: the decision warp and
  // consumer warp 0 take turns, handing over through mbarriers.)
  int last_slot = 0;
  auto send_recv = [&](int words) -> bool {
    warp_converged();
    const int x = sm.xc;
    __syncwarp();
    if (lane == 0) sm.xc = x + 1;
    const int slot = x & 1;
    const uint32_t par = static_cast<uint32_t>((x >> 1) & 1);
    last_slot = slot;
    if (lane < static_cast<int>(C)) {
      const uint32_t dst = dsmem_addr(&sm.recs[slot][rank][0], static_cast<uint32_t>(lane));
      for (int w = 0; w < words; w += 4)
        dsmem_st_v4(dst + 4u * w, *reinterpret_cast<const uint4*>(&sm.myrec[w]));
      dsmem_arrive_release(dsmem_addr(&sm.xbar[slot], static_cast<uint32_t>(lane)));
    }
    const bool ok =
        mbar_wait_cluster_bounded(&sm.xbar[slot], par, (P.flags & FLAG_EXPIRE_EXCHANGE) ? 0u : kWaitPolls);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
  };
  auto rec = [&](uint32_t c, int w) -> uint32_t { return sm.recs[last_slot][c][w]; };
  auto recf = [&](uint32_t c, int w) -> float { return __uint_as_float(rec(c, w)); };
  auto rec_u64 = [&](uint32_t c, int w) -> unsigned long long {
    return static_cast<unsigned long long>(rec(c, w)) |
           (static_cast<unsigned long long>(rec(c, w + 1)) << 32);
  };
  auto putf = [&](int w, float v) { sm.myrec[w] = __float_as_uint(v); };
  auto put_u64 = [&](int w, unsigned long long v) {
    sm.myrec[w] = static_cast<uint32_t>(v);
    sm.myrec[w + 1] = static_cast<uint32_t>(v >> 32);
  };
  auto finish = [&](int n, int nxt, uint32_t s) {  // thread 0 of the writing CTA
    if (P.ext_err && *P.ext_err) {  // the producer of the rows gave up: they are invalid
      n = 0;
      nxt = -1;
      s |= ST_TIMEOUT;
    }
    P.n_out[b] = n;
    P.next_out[b] = nxt;
    P.st_out[b] = s;
  };

  bool abort = false;

  if (!sampling) {
    // ============================================================== greedy
    uint32_t st = 0;
    for (int i = 0;; ++i) {
      float bv = __int_as_float(0x7FFFFFFF);  // NaN: no candidate yet
      int bi = INT_MAX;
      uint32_t nanf = 0;
      for (int j = 0; j < nck; ++j) {
        const T* s = acquire();
        chunk_argmax<T>(s, j == nck - 1 ? last_n : ck_el, v_lo + j * ck_el, bv, bi, nanf);
        release();
      }
      if (bv != bv) bi = INT_MAX;
      warp_converged();
      warp_argmax(bv, bi);
      const uint32_t fl = __reduce_or_sync(0xFFFFFFFFu, nanf | (tmo << 1));
      if (lane == 0) {
        sm.wf[warp][0] = bv;
        sm.wi[warp][0] = bi;
        sm.wi[warp][1] = static_cast<int>(fl);
      }
      bar_consumers<kConsumers>();
      if (warp == 0) {
        warp_converged();
        // lanes 0..7: the warps' candidates; then the cluster's records
        float v = lane < kWarps ? sm.wf[lane][0] : 0.f;
        int a = lane < kWarps ? sm.wi[lane][0] : INT_MAX;
        uint32_t f = lane < kWarps ? static_cast<uint32_t>(sm.wi[lane][1]) : 0u;
        warp_argmax(v, a);
        f = __reduce_or_sync(0xFFFFFFFFu, f);
        if (lane == 0) {
          sm.myrec[0] = __float_as_uint(v);
          sm.myrec[1] = static_cast<uint32_t>(a);
          sm.myrec[2] = f;
          sm.myrec[3] = 0u;
        }
        int act = ACT_CONTINUE;
        if (!send_recv(4)) {
          act = ACT_ABORT;
        } else {
          warp_converged();
          const bool mine = lane < static_cast<int>(C);
          v = mine ? recf(lane, 0) : 0.f;
          a = mine ? static_cast<int>(rec(lane, 1)) : INT_MAX;
          f = __reduce_or_sync(0xFFFFFFFFu, mine ? rec(lane, 2) : 0u);
          warp_argmax(v, a);
          if (f & 2u) {
            act = ACT_ABORT;
          } else if (lane == 0) {
            if (a == INT_MAX) a = 0;  // an all-NaN row
            if (f & 1u) st |= ST_BAD_VALUE;
            if (i == kb) {
              act = ACT_STOP;
              if (rank == 0) finish(kb, a, st);
            } else {
              const int t = row_token(i);
              if (t < 0 || t >= P.V) {
                act = ACT_STOP;
                if (rank == 0) finish(i, a, st | ST_BAD_TOKEN);
              } else if (t != a) {
                act = ACT_STOP;
                if (rank == 0) finish(i, a, st);
              }
            }
          }
        }
        if (lane == 0) {
          if (act != ACT_CONTINUE) sm.stop = 1;
          sm.bi[0] = act;
        }
      }
      bar_consumers<kConsumers>();
      const int act = sm.bi[0];
      if (act == ACT_ABORT) abort = true;
      if (act != ACT_CONTINUE) break;
    }
  } else {
    // ============================================================== sampling
    float khi = 0.f, klo = 0.f;
    if (MODE == MODE_LOGITS) log2e_over(temp, khi, klo);
    auto make_warp = [&](float m, float lo) {
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
      w.lo = lo;
      (void)m;
      return w;
    };
    // the weight functors of row i (target, and draft unless i is the bonus row)
    auto warp_p = [&](int i, float m) { return make_warp(m, MODE == MODE_LOGITS ? row_floor(false, i) : -kInfF); };
    auto warp_q = [&](int i, float m, bool bonus) {
      return make_warp(m, (MODE == MODE_LOGITS && !bonus) ? row_floor(true, i) : -kInfF);
    };
    const bool force_exact = (P.flags & FLAG_FORCE_EXACT) != 0u;
    unsigned long long* buckets = vsum;  // the exact pass and the draw never overlap
    // fp32 additions any element goes through inside its thread
    int nadd = 0;
    for (int j = 0; j < nck; ++j) {
      const int n = j == nck - 1 ? last_n : ck_el;
      nadd += (n / VEC + kConsumers - 1) / kConsumers + (n % VEC ? 1 : 0);
    }
    nadd += (VEC == 8 ? 3 : 2);

    // ---- exact masses of row i (consumer collective; reads the row slices
    // from global memory).  Thread 0 leaves the summed limbs and the +Inf
    // flags in shared memory for the decision warp.
    auto exact_pass = [&](int i, bool with_q, const WarpT& wfp, const WarpT& wfq) -> bool {
      for (int k = tid; k < 2 * kBuckets; k += kConsumers) buckets[k] = 0ull;
      bar_consumers<kConsumers>();
      uint32_t bp = 0, bq = 0;
      const T* p = row_slice(false, i);
      const T* q = with_q ? row_slice(true, i) : nullptr;
      for (int e = tid; e < n_el; e += kConsumers) {
        const float x = wfp(gload<T>(p, e));
        if (!(x <= FLT_MAX)) bp = 1u;  // +Inf (NaN and negatives were rejected before)
        else bucket_add(buckets, x);
        if (q) {
          const float y = wfq(gload<T>(q, e));
          if (!(y <= FLT_MAX)) bq = 1u;
          else bucket_add(buckets + kBuckets, y);
        }
      }
      bp = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(bp)));
      bq = static_cast<uint32_t>(bar_consumers_or<kConsumers>(static_cast<int>(bq)));
      if (tid == 0) {
        buckets_to_limbs(buckets, &sm.myrec[0]);
        buckets_to_limbs(buckets + kBuckets, &sm.myrec[kLimbs]);
        sm.myrec[2 * kLimbs] = bp | (bq << 1);
        sm.myrec[2 * kLimbs + 1] = sm.myrec[2 * kLimbs + 2] = sm.myrec[2 * kLimbs + 3] = 0u;
      }
      bool ok = true;
      if (warp == 0) ok = send_recv(2 * kLimbs + 4);
      if (tid == 0) {
        if (ok) {
          unsigned long long ap[kLimbs], aq[kLimbs];
          for (int k = 0; k < kLimbs; ++k) ap[k] = aq[k] = 0ull;
          uint32_t infl = 0;
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
            sm.lp[k] = static_cast<uint32_t>(cp);
            sm.lq[k] = static_cast<uint32_t>(cq);
            cp >>= 32;
            cq >>= 32;
          }
          sm.infl = infl;
        }
        sm.bi[5] = ok ? 1 : 0;
      }
      bar_consumers<kConsumers>();
      return sm.bi[5] != 0;
    };

    // Inverse-CDF draw over row i, read again from global memory (it was just
    // streamed, so mostly from L2; collective).  Returns 0 when done (the
    // owning CTA wrote the outputs), 1 when the residual is empty, -1 when a
    // device wait gave up.
    using DrawT = typename std::conditional<MODE == MODE_LOGITS, DrawLogits<FL>, DrawProbs>::type;
    auto draw = [&](int n_acc_row, bool resid, int n_acc, uint32_t st_in, float u_draw) -> int {
      DrawT dw;
      dw.scale = __uint_as_float(static_cast<uint32_t>(127 + P.fixed_shift) << 23);
      dw.resid = resid ? 1 : 0;
      if constexpr (MODE == MODE_LOGITS) {
        dw.k = khi;  // c = -m k - log2 Z, folded into one FMA per element
        dw.cp = sm.dpar[0];
        dw.cq = sm.dpar[1];
        dw.lo_p = row_floor(false, n_acc_row);
        dw.lo_q = resid ? row_floor(true, n_acc_row) : -kInfF;
      } else {
        dw.sp = sm.dpar[0];
        dw.ap = sm.dpar[1];
        dw.sq = sm.dpar[2];
        dw.aq = sm.dpar[3];
      }
      const T* gp = row_slice(false, n_acc_row);
      const T* gq = resid ? row_slice(true, n_acc_row) : nullptr;
      const bool vec_ok = P.use_tma != 0;  // 16-byte aligned rows (slices start on vectors)
      const int nvt = (n_el + VEC - 1) / VEC;
      const int ng = (nvt + kGroupVecs - 1) / kGroupVecs;
      unsigned long long mine = 0;
      // Each thread takes U consecutive vectors, so kGroupVecs / U neighbouring
      // lanes cover one group of vectors, whose fixed-point sum goes to
      // shared memory (the owner's walk re-reads only the crossing group).
      constexpr int U = 4;
      constexpr int LG = kGroupVecs / U;  // lanes per group
      static_assert(LG == 8, "group sums reduce over 8 lanes");
      const int nfull = vec_ok ? n_el / VEC : 0;  // whole vectors read as 16-byte loads
      for (int it = 0; it * kConsumers * U < nvt; ++it) {  // same trip count for every thread
        const int v0 = (it * kConsumers + tid) * U;
        uint4 rp[U], rq[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int vi = v0 + u;
          if (vi < nfull) {
            rp[u] = __ldg(reinterpret_cast<const uint4*>(gp) + vi);
            rq[u] = gq ? __ldg(reinterpret_cast<const uint4*>(gq) + vi) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
        unsigned long long fs = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int vi = v0 + u;
          if (vi >= nvt) break;
          float r[VEC];
          if (vi < nfull) {
            float xp[VEC], xq[VEC];
            unpack_vec<T>(rp[u], xp);
            unpack_vec<T>(rq[u], xq);
#pragma unroll
            for (int q = 0; q < VEC; ++q) r[q] = dw(xp[q], gq ? xq[q] : 0.f);
          } else {
            vec_draw_weights<T>(gp, gq, n_el, vi, vec_ok, dw, r);
          }
          fs += dw.fix(seq_sum<VEC>(r));
        }
        mine += fs;
        fs += __shfl_xor_sync(0xFFFFFFFFu, fs, 1);
        fs += __shfl_xor_sync(0xFFFFFFFFu, fs, 2);
        fs += __shfl_xor_sync(0xFFFFFFFFu, fs, 4);
        const int g = v0 / kGroupVecs;
        if ((lane & (LG - 1)) == 0 && g < ng) vsum[g] = fs;
      }
      warp_converged();
      mine = warp_sum_u64(mine);
      if (lane == 0) sm.wu[warp] = mine;
      bar_consumers<kConsumers>();
      if (warp == 0) {
        warp_converged();
        const unsigned long long tot = warp_sum_u64(lane < kWarps ? sm.wu[lane] : 0ull);
        if (lane == 0) {
          put_u64(0, tot);
          sm.myrec[2] = sm.myrec[3] = 0u;
        }
        int code = 0;
        if (!send_recv(4)) {
          code = -1;
        } else {
          warp_converged();
          // lanes 0..C-1: the CTAs' totals, an inclusive scan across lanes
          const unsigned long long rc = lane < static_cast<int>(C) ? rec_u64(lane, 0) : 0ull;
          unsigned long long inc = rc;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += n;
          }
          const unsigned long long R = __shfl_sync(0xFFFFFFFFu, inc, 31);
          if (R == 0) {
            code = resid ? 1 : 0;
            if (lane == 0 && !resid && rank == 0) finish(n_acc, -1, st_in | ST_ZERO_MASS);
          } else {
            const unsigned long long tau = tau_of(u_draw, R);
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, lane < static_cast<int>(C) && tau < inc);
            const int owner = hit ? __ffs(hit) - 1 : -1;
            const unsigned long long before = owner >= 0 ? __shfl_sync(0xFFFFFFFFu, inc - rc, owner) : 0ull;
            if (owner < 0) {  // cannot happen: tau < R
              if (lane == 0 && rank == 0) finish(n_acc, -1, st_in | ST_TIMEOUT);
            } else if (owner == static_cast<int>(rank)) {
              code = 2;  // this CTA walks its slice
              if (lane == 0) {
                sm.wu[0] = tau - before;
                sm.wu[1] = R;
              }
            }
          }
        }
        if (lane == 0) sm.bi[0] = code;
      }
      bar_consumers<kConsumers>();
      const int code = sm.bi[0];
      if (code != 2) return code;
      // ---- the owner, warp 0 alone: a scan of the group sums (lane l takes
      // a run of consecutive groups), then the crossing group's vectors, then
      // one vector's elements; the other warps are done.
      if (warp != 0) return 0;
      warp_converged();
      const unsigned long long tloc = sm.wu[0];
      const double Rd = static_cast<double>(sm.wu[1]);
      const int seg = (ng + 31) / 32;
      const int lo = min(ng, lane * seg), hi = min(ng, lo + seg);
      unsigned long long s = 0;
      for (int g = lo; g < hi; ++g) s += vsum[g];
      unsigned long long inc = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += n;
      }
      const unsigned long long ex = inc - s;
      const uint32_t seg_hit = __ballot_sync(0xFFFFFFFFu, tloc >= ex && tloc < inc);
      int g_hit = -1;
      unsigned long long c0 = 0;
      if (seg_hit) {
        const int L = __ffs(seg_hit) - 1;
        if (lane == L) {
          c0 = ex;
          int g = lo;
          for (; g < hi - 1; ++g) {
            if (tloc < c0 + vsum[g]) break;
            c0 += vsum[g];
          }
          g_hit = g;
        }
        g_hit = __shfl_sync(0xFFFFFFFFu, g_hit, L);
        c0 = __shfl_sync(0xFFFFFFFFu, c0, L);
      }
      int found = -1, near_b = 0;
      if (g_hit >= 0) {
        const int v = g_hit * kGroupVecs + lane;
        float r[VEC];
        int cnt = 0;
        unsigned long long f = 0;
        if (v < nvt) {
          cnt = vec_draw_weights<T>(gp, gq, n_el, v, vec_ok, dw, r);
          f = dw.fix(seq_sum<VEC>(r));
        }
        unsigned long long vinc = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, vinc, o);
          if (lane >= o) vinc += n;
        }
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, v < nvt && tloc < c0 + vinc);
        if (hit) {
          const int L = __ffs(hit) - 1;
          if (lane == L) {
            const unsigned long long cv = c0 + vinc - f;  // the CDF before this vector
            float acc = r[0];
            unsigned long long prev = cv;
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
              if (k > 0) acc = __fadd_rn(acc, r[k]);
              const unsigned long long cur = cv + dw.fix(acc);
              if (k < cnt && (tloc < cur || k == cnt - 1)) {
                const unsigned long long dlo = tloc - prev, dhi = cur > tloc ? cur - tloc : 0ull;
                const unsigned long long dmin = dlo < dhi ? dlo : dhi;
                found = v_lo + v * VEC + k;
                near_b = static_cast<double>(dmin) <= 1e-5 * Rd ? 1 : 0;
                break;
              }
              prev = cur;
            }
          }
          found = __shfl_sync(0xFFFFFFFFu, found, L);
          near_b = __shfl_sync(0xFFFFFFFFu, near_b, L);
        }
      }
      if (lane == 0) {
        const uint32_t near = (found >= 0 && near_b) ? ST_NEAR : 0u;
        finish(n_acc, found, found >= 0 ? (st_in | near) : (st_in | ST_TIMEOUT));
      }
      return 0;
    };

    // ---- the pipelined row loop.  The consumer warps reduce row i + 1
    // while the decision warp combines, exchanges and decides row i; a
    // rejection of row i cuts that pass short.
    if (warp == kDecideWarp) {
      // ================================================ decision warp
      uint32_t st = 0;
      int xr = 0;  // exact passes so far
      for (int i = 0;; ++i) {
        const bool bonus = i == kb;
        const int pb = i & 1;
        const bool okp = mbar_wait_bounded(&sm.pfull[pb], static_cast<uint32_t>((i >> 1) & 1));
        warp_converged();
        // lane w < 8 holds warp w's partials, lane c < C will hold CTA c's
        // record; sums are fp32 trees over those lanes (3 and 4 levels).
        // Record flags: bit 0 a wait gave up, bit 1 / 2 a bad target / draft
        // value (probabilities: NaN or negative; logits: NaN or +Inf).
        static_assert(kWarps == 8 && kMaxCluster <= 16, "combine widths");
        const bool wl = lane < kWarps;
        const bool cl = lane < static_cast<int>(C);
        DF Zp = {0.f, 0.f}, Zq = {0.f, 0.f};
        float Bp = 0.f, Bq = 0.f;
        float mp = 0.f, mq = 0.f;
        uint32_t anytmo = okp ? 0u : 1u, badf = 0u;
        const float4 fa = *reinterpret_cast<const float4*>(&sm.wf2[pb][lane & 7][0]);
        const float4 fb = *reinterpret_cast<const float4*>(&sm.wf2[pb][lane & 7][4]);
        const int2 ia = *reinterpret_cast<const int2*>(&sm.wi2[pb][lane & 7][0]);
        const uint32_t tf = __reduce_or_sync(0xFFFFFFFFu, wl ? static_cast<uint32_t>(ia.x) : 0u) | anytmo;
        if constexpr (MODE == MODE_PROBS) {
          const float s0 = warp_sum_f<8>(wl ? fa.x : 0.f);
          const float s1 = warp_sum_f<8>(wl ? fa.y : 0.f);
          const float m0 = warp_min_nan_f<8>(wl ? fa.z : kInfF);
          const float m1 = warp_min_nan_f<8>(wl ? fa.w : kInfF);
          if (lane == 0) {
            putf(0, s0);
            putf(1, s1);
            sm.myrec[2] = (tf ? 1u : 0u) | (m0 >= 0.f ? 0u : 2u) | (m1 >= 0.f ? 0u : 4u);
            sm.myrec[3] = 0u;
          }
          if (!send_recv(4)) anytmo = 1;
          if (!anytmo) {
            warp_converged();
            Zp.hi = warp_sum_f<16>(cl ? recf(lane, 0) : 0.f);
            Zq.hi = warp_sum_f<16>(cl ? recf(lane, 1) : 0.f);
            const uint32_t f = __reduce_or_sync(0xFFFFFFFFu, cl ? rec(lane, 2) : 0u);
            anytmo = f & 1u;
            badf = f;
          }
          Bp = sum_bound(Zp.hi, nadd);
          Bq = sum_bound(Zq.hi, nadd);
        } else {
          // warps -> CTA (one more rescale step)
          const float wmp = wl ? fa.x : -kInfF, wmq = wl ? fa.w : -kInfF;
          const float cmp = warp_max_f<8>(wmp), cmq = warp_max_f<8>(wmq);
          const float c6 = warp_max_nan_f<8>(wl ? fb.z : -kInfF);
          const float c7 = warp_max_nan_f<8>(wl ? fb.w : -kInfF);
          const int rr = warp_max_i<8>(wl ? ia.y : 0);
          float sp = 0.f, sq = 0.f, wp = 0.f, wq = 0.f;
          if (wmp > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(cmp, wmp), khi);
            const float f = ex2_ftz(-d);
            sp = __fmul_rn(fa.y, f);
            wp = __fmul_rn(__fmaf_rn(d, fa.y, fa.z), f);
          }
          if (wmq > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(cmq, wmq), khi);
            const float f = ex2_ftz(-d);
            sq = __fmul_rn(fb.x, f);
            wq = __fmul_rn(__fmaf_rn(d, fb.x, fb.y), f);
          }
          warp_converged();
          sp = warp_sum_f<8>(sp);
          sq = warp_sum_f<8>(sq);
          wp = warp_sum_f<8>(wp);
          wq = warp_sum_f<8>(wq);
          if (lane == 0) {
            putf(0, cmp);
            putf(1, cmq);
            putf(2, sp);
            putf(3, wp);
            putf(4, sq);
            putf(5, wq);
            sm.myrec[6] = static_cast<uint32_t>(rr);
            sm.myrec[7] = (tf ? 1u : 0u) | (c6 < kInfF ? 0u : 2u) | (c7 < kInfF ? 0u : 4u);
          }
          if (!send_recv(8)) anytmo = 1;
          mp = mq = -kInfF;
          if (!anytmo) {
            warp_converged();
            const float rmp = cl ? recf(lane, 0) : -kInfF, rmq = cl ? recf(lane, 1) : -kInfF;
            mp = warp_max_f<16>(rmp);
            mq = warp_max_f<16>(rmq);
            const int R = warp_max_i<16>(cl ? static_cast<int>(rec(lane, 6)) : 0);
            const uint32_t fl = __reduce_or_sync(0xFFFFFFFFu, cl ? rec(lane, 7) : 0u);
            anytmo = fl & 1u;
            badf = fl;
            // CTAs -> cluster (one more rescale step)
            float zp = 0.f, zq = 0.f, w1 = 0.f, w2 = 0.f;
            if (rmp > -kInfF) {
              const float d = __fmul_rn(__fsub_rn(mp, rmp), khi);
              const float f = ex2_ftz(-d);
              zp = __fmul_rn(recf(lane, 2), f);
              w1 = __fmul_rn(__fmaf_rn(d, recf(lane, 2), recf(lane, 3)), f);
            }
            if (rmq > -kInfF) {
              const float d = __fmul_rn(__fsub_rn(mq, rmq), khi);
              const float f = ex2_ftz(-d);
              zq = __fmul_rn(recf(lane, 4), f);
              w2 = __fmul_rn(__fmaf_rn(d, recf(lane, 4), recf(lane, 5)), f);
            }
            warp_converged();
            Zp.hi = warp_sum_f<16>(zp);
            Zq.hi = warp_sum_f<16>(zq);
            const float Wp = warp_sum_f<16>(w1), Wq = warp_sum_f<16>(w2);
            Bp = online_bound(Zp.hi, Wp, R + 1, nadd, fabsf(__fmul_rn(mp, khi))) + static_cast<float>(P.V) * 1.2e-38f;
            Bq = online_bound(Zq.hi, Wq, R + 1, nadd, fabsf(__fmul_rn(mq, khi))) + static_cast<float>(P.V) * 1.2e-38f;
          }
        }
        // ---- lane 0: the decision (input errors in the oracle's order, then
        // the accept test; the exact masses when the filter cannot decide)
        int act = ACT_CONTINUE;
        if (lane == 0) {
          int t = -1;
          float u = 0.f, gp = 0.f, gq = 0.f;
          if (i < kMaxGather) {
            u = sm.g_u[i];
            t = bonus ? -1 : sm.g_t[i];
            gp = sm.g_p[i];
            gq = sm.g_q[i];
          } else {
            u = P.uni[t0 + i];
            if (!bonus) {
              t = P.tok[d0 + i];
              if (t >= 0 && t < P.V) {
                gp = TR::to_f(tgt[(t0 + i) * P.stride + t]);
                gq = TR::to_f(drf[(d0 + i) * P.stride + t]);
              }
            }
          }
          const WarpT wfp = warp_p(i, mp), wfq = warp_q(i, mq, bonus);
          bool posted = false;  // dec[pb] handed over already (an exact pass followed)
          bool have_exact = false;
          double Zp_ex = 0.0, Zq_ex = 0.0;
          // hands the exact pass to the consumers and waits for its limbs
          auto run_exact = [&]() -> bool {
            Dec& dd = sm.dec[pb];
            dd.act = ACT_EXACT;
            dd.mp = mp;
            dd.mq = mq;
            if (!posted) mbar_arrive_local(&sm.dfull[pb]);
            posted = true;
            const bool okx = mbar_wait_bounded(&sm.xfull, static_cast<uint32_t>(xr & 1)) && sm.bi[5] != 0;
            ++xr;
            if (okx) {
              Zp_ex = limbs_to_double(sm.lp);
              Zq_ex = bonus ? 0.0 : limbs_to_double(sm.lq);
              have_exact = true;
            }
            return okx;
          };
          uint32_t err = 0;
          bool p_bad = false, q_bad = false, need_x = false;
          if (anytmo) {
            act = ACT_ABORT;
          } else {
            if (!bonus && (t < 0 || t >= P.V)) err = ST_BAD_TOKEN;
            if constexpr (MODE == MODE_PROBS) {
              p_bad = (badf & 2u) != 0u;  // NaN or a negative value
              q_bad = !bonus && (badf & 4u) != 0u;
              // a non-finite approximate mass means a +Inf element or an fp32
              // overflow of the partial sums: the exact pass tells them apart
              need_x = !err && !p_bad && !q_bad && (!(Zp.hi <= FLT_MAX) || (!bonus && !(Zq.hi <= FLT_MAX)));
            } else {
              // NaN or +Inf logit, or a NaN floor (an invalid filter parameter)
              p_bad = (badf & 2u) != 0u || wfp.lo != wfp.lo;
              q_bad = !bonus && ((badf & 4u) != 0u || wfq.lo != wfq.lo);
            }
            if (need_x) {
              if (run_exact()) {
                p_bad = p_bad || (sm.infl & 1u);
                q_bad = q_bad || (sm.infl & 2u);
              } else {
                act = ACT_ABORT;
              }
            }
          }
          if (act != ACT_ABORT) {
            if (!err && p_bad) err = ST_BAD_VALUE;
            if (!err && q_bad) err = ST_BAD_VALUE;
            if (!err && !(u >= 0.f && u < 1.f)) err = ST_BAD_VALUE;
            const bool p_zero = MODE == MODE_PROBS ? (have_exact ? Zp_ex == 0.0 : Zp.hi == 0.f) : mp == -kInfF;
            const bool q_zero = MODE == MODE_PROBS ? (have_exact ? Zq_ex == 0.0 : Zq.hi == 0.f) : mq == -kInfF;
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
              int dec = have_exact ? -1 : filter_decide(u, pt, qt, Zp, Bp, Zq, Bq);
              if (!have_exact && (force_exact || dec < 0) && !run_exact()) {
                act = ACT_ABORT;
              } else {
                if (have_exact) {
                  dec = exact_accept(u, pt, qt, sm.lp, sm.lq) ? 1 : 0;
                  st |= ST_EXACT;
                }
                act = dec ? ACT_CONTINUE : ACT_DRAW;
              }
            }
          }
          // ---- the outcome for the consumers
          Dec& dd = sm.dec[pb];
          dd.mp = mp;
          dd.mq = mq;
          if (act == ACT_DRAW) {
            const float ud = kb < kMaxGather ? sm.g_u[kb] : P.uni[t0 + kb];
            const float zp = have_exact ? static_cast<float>(Zp_ex) : Zp.hi;
            const float zq = bonus ? 1.f : (have_exact ? static_cast<float>(Zq_ex) : Zq.hi);
            if constexpr (MODE == MODE_LOGITS) {
              const DF mk = two_prod(mp, khi), qk = two_prod(mq, khi);
              sm.dpar[0] = -__fadd_rn(mk.hi, __fadd_rn(mk.lo, log2f(zp)));
              sm.dpar[1] = bonus ? 0.f : -__fadd_rn(qk.hi, __fadd_rn(qk.lo, log2f(zq)));
            } else {
              const double zpd = have_exact ? Zp_ex : static_cast<double>(zp);
              const double zqd = have_exact && !bonus ? Zq_ex : static_cast<double>(zq);
              norm_factors(zpd, sm.dpar[0], sm.dpar[1]);
              norm_factors(zqd, sm.dpar[2], sm.dpar[3]);
            }
            dd.u_draw = ud;
          }
          dd.st = st;
          dd.act = act;
          if (act == ACT_CONTINUE) sm.go_row = i + 1;
          else sm.stop = 1;  // the producer issues nothing more
          if (posted) {
            mbar_arrive_local(&sm.xdec);  // after an exact pass the consumers wait here
          } else {
            mbar_arrive_local(&sm.dfull[pb]);
          }
        }
        act = __shfl_sync(0xFFFFFFFFu, act, 0);
        xr = __shfl_sync(0xFFFFFFFFu, xr, 0);
        if (act != ACT_CONTINUE) break;
      }
    } else {
      // ================================================ consumer warps
      // pass over row i's chunks as they stream in; its partials go to the
      // decision warp.  With watch >= 0 the consumers cut the pass short,
      // all together (a barrier reduction at each chunk), once row `watch` is
      // decided against continuing, and tell the producer (sm.cut_row); every
      // warp consumes the same chunks, as the ring's slots are shared.
      // Returns false if the pass was cut.
      auto pass_row = [&](int i, int watch) -> bool {
        const bool bonus = i == kb;
        Acc ap, aq;
        Online op, oq;
        ap.init();
        aq.init();
        op.init();
        oq.init();
        float ep = MODE == MODE_PROBS ? kInfF : -kInfF;  // probs: min; logits: max (validity)
        float eq = ep;
        for (int part = 0; part < (bonus ? 1 : 2); ++part) {
          const float lo = MODE == MODE_LOGITS ? row_floor(part == 1, i) : -kInfF;
          for (int j = 0; j < nck; ++j) {
            if (watch >= 0) {
              int cut = 0;
              if (tid == 0 && mbar_test(&sm.dfull[watch & 1], static_cast<uint32_t>((watch >> 1) & 1))) {
                const int a = sm.dec[watch & 1].act;
                cut = (a == ACT_DRAW || a == ACT_STOP || a == ACT_ABORT) ? 1 : 0;
              }
              if (bar_consumers_or<kConsumers>(cut)) {
                if (tid == 0) sm.cut_row = i;
                return false;
              }
            }
            const T* s = acquire();
            const int n = j == nck - 1 ? last_n : ck_el;
            if constexpr (MODE == MODE_PROBS)
              chunk_mass_f32(reinterpret_cast<const float*>(s), n, part ? aq : ap, part ? eq : ep);
            else
              chunk_online<T, FL>(s, n, khi, lo, part ? oq : op, part ? eq : ep);
            release();  // the slot takes later chunks while rows are decided
          }
        }
        // ---- warp partials -> shared memory, then to the decision warp
        const int pb = i & 1;
        warp_converged();
        const uint32_t tm = __reduce_or_sync(0xFFFFFFFFu, tmo);
        if constexpr (MODE == MODE_PROBS) {
          const float s0 = warp_sum_f(ap.f), s1 = warp_sum_f(aq.f);
          const float m0 = warp_min_nan_f(ep), m1 = warp_min_nan_f(eq);
          if (lane == 0) {
            sm.wf2[pb][warp][0] = s0;
            sm.wf2[pb][warp][1] = s1;
            sm.wf2[pb][warp][2] = m0;
            sm.wf2[pb][warp][3] = m1;
            sm.wi2[pb][warp][0] = static_cast<int>(tm);
          }
        } else {
          // rescale each lane's sums to the warp maximum (one more rescale step)
          const float wmp = warp_max_f(op.m), wmq = warp_max_f(oq.m);
          float sp = 0.f, wp = 0.f, sq = 0.f, wq = 0.f;
          if (op.m > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(wmp, op.m), khi);
            const float f = ex2_ftz(-d);
            sp = __fmul_rn(op.s, f);
            wp = __fmul_rn(__fmaf_rn(d, op.s, op.w), f);
          }
          if (oq.m > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(wmq, oq.m), khi);
            const float f = ex2_ftz(-d);
            sq = __fmul_rn(oq.s, f);
            wq = __fmul_rn(__fmaf_rn(d, oq.s, oq.w), f);
          }
          sp = warp_sum_f(sp);
          wp = warp_sum_f(wp);
          sq = warp_sum_f(sq);
          wq = warp_sum_f(wq);
          const float vmp = warp_max_nan_f(ep), vmq = warp_max_nan_f(eq);
          const int rr = warp_max_i(max(op.r, oq.r));
          if (lane == 0) {
            sm.wf2[pb][warp][0] = wmp;
            sm.wf2[pb][warp][1] = sp;
            sm.wf2[pb][warp][2] = wp;
            sm.wf2[pb][warp][3] = wmq;
            sm.wf2[pb][warp][4] = sq;
            sm.wf2[pb][warp][5] = wq;
            sm.wf2[pb][warp][6] = vmp;
            sm.wf2[pb][warp][7] = vmq;
            sm.wi2[pb][warp][0] = static_cast<int>(tm);
            sm.wi2[pb][warp][1] = rr;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_local(&sm.pfull[pb]);
        return true;
      };

      int xr = 0;  // exact passes so far
      pass_row(0, -1);
      for (int i = 0;; ++i) {
        const bool bonus = i == kb;
        const int pb = i & 1;
        if (!bonus) pass_row(i + 1, i);  // speculative: row i + 1 while row i is decided
        int act = mbar_wait_bounded(&sm.dfull[pb], static_cast<uint32_t>((i >> 1) & 1)) ? sm.dec[pb].act
                                                                                        : ACT_ABORT;
        if (act == ACT_EXACT) {  // exact masses of row i, then the final outcome
          const WarpT wfp = warp_p(i, sm.dec[pb].mp), wfq = warp_q(i, sm.dec[pb].mq, bonus);
          exact_pass(i, !bonus, wfp, wfq);
          if (tid == 0) mbar_arrive_local(&sm.xfull);
          act = mbar_wait_bounded(&sm.xdec, static_cast<uint32_t>(xr & 1)) ? sm.dec[pb].act : ACT_ABORT;
          ++xr;
        }
        if (act == ACT_ABORT) {
          abort = true;
          break;
        }
        // warped weights of this row for the caller (testing aid)
        if (MODE == MODE_LOGITS && (P.wt_out || P.wd_out) && act != ACT_STOP) {
          const WarpT wfp = warp_p(i, sm.dec[pb].mp), wfq = warp_q(i, sm.dec[pb].mq, bonus);
          const T* p = row_slice(false, i);
          const T* q = row_slice(true, i);
          for (int e = tid; e < n_el; e += kConsumers) {
            if (P.wt_out) P.wt_out[(t0 + i) * static_cast<long long>(P.V) + v_lo + e] = wfp(gload<T>(p, e));
            if (P.wd_out && !bonus)
              P.wd_out[(d0 + i) * static_cast<long long>(P.V) + v_lo + e] = wfq(gload<T>(q, e));
          }
        }
        if (act == ACT_CONTINUE) continue;
        if (act == ACT_STOP) break;
        // ---- ACT_DRAW: the bonus from p_K, or the residual after the first rejection
        const uint32_t st_now = sm.dec[pb].st;
        const float u_draw = sm.dec[pb].u_draw;
        if (!bonus && !(u_draw >= 0.f && u_draw < 1.f)) {
          if (tid == 0 && rank == 0) finish(i, -1, st_now | ST_BAD_VALUE);
          break;
        }
        int code = draw(i, !bonus, bonus ? kb : i, st_now, u_draw);
        if (code == 1) code = draw(i, false, i, st_now | ST_ZERO_MASS, u_draw);
        if (code < 0) abort = true;
        break;
      }
    }
  }

  if (abort && tid == 0) finish(0, -1, ST_TIMEOUT);
  if (tid == 0) sm.stop = 1;  // the producer stops issuing and drains its copies
  }  // consumers and decision warp

  // Peers push records into this CTA's shared memory.  On the normal path
  // every CTA takes part in the same exchanges, but a CTA whose wait gave up
  // must not exit while a slower peer may still push into it: every thread
  // of the cluster meets here once (every wait above is bounded, so each
  // one arrives) before any CTA of the cluster exits.
  __syncwarp();
  cluster_sync_all();
}

}  // namespace svk
