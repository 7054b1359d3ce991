// Row-parallel verification: one thread-block cluster per (row, sequence).
//
// The chain kernel (sv_verify.cuh) walks the rows of a sequence one after
// another, so a batch whose sequences fit one wave of clusters waits on a
// chain of dependent row links.  Here every row i of every sequence b is an
// item of its own, processed by a cluster of C CTAs that hold their slices
// of target row i and draft row i in shared memory:
//   * items are numbered row-major (i * B + b), so row 0 of every sequence is
//     launched first; an item whose sequence has already posted a terminal
//     row before i (a rejection, an error, a miss) skips its loads and work;
//   * the cluster takes the row's decision exactly as the chain kernel does
//     (one online-softmax pass with the chain's error bound, the same defined
//     weights, the same exact predicate and fallback), and,
//     if the row ends its sequence by a rejection or is the bonus row, its
//     inverse-CDF draw from the resident slices (no second read of the row);
//   * each item writes a small record of its outcome to global scratch and
//     counts itself in; the last item of a sequence to arrive (an atomic
//     counter, no waiting) combines the records left to right, writes the
//     sequence's outputs, and resets the counter and the posted row for the
//     next launch.
// Nothing waits on another cluster: the only waits are on the CTA's own bulk
// copies and on the cluster's exchanges, all bounded.
#pragma once
#include "sv_topk.cuh"
#include "sv_verify.cuh"

namespace svk {

constexpr int kRowsThreads = 256;  // 8 warps, every one reduces
constexpr uint32_t kRecTerminal = 0x80000000u;
constexpr uint32_t kRecFallback = 0x40000000u;  // fused filters: this row needs the general path
constexpr int kRowsExchanges = 5;  // row statistics, (unused), exact limbs, draw, draw from p

struct RowsParams {
  Params p;
  int* seq_count;  // per sequence: items arrived (0 between launches)
  int* seq_first;  // per sequence: INT_MAX - (first terminal row posted), 0 when none
  uint4* rec;      // per target row: {status | kRecTerminal, next, n, 0}
  int* seq_flag;   // fused filters: per sequence 1 = handed to the fallback (NULL otherwise)
  const int* top_k;    // fused filters: per sequence top-k (NULL otherwise)
  const float* top_p;  // fused filters: per sequence top-p (NULL: none)
  int nadd;        // fp32 additions of any element inside its thread (mass bounds)
  int x_off;       // byte offset of the draft slice
  int vsum_off;    // byte offset of the draw's group sums / the exact buckets
  int tail_off;    // byte offset of RowsTail
};

struct __align__(16) RowsTail {
  uint32_t xr[4][kMaxCluster][8];  // records of exchanges 0, 3, 4 (slot 1 unused)
  uint32_t xe[kMaxCluster][32];    // records of exchange 2 (exact limbs)
  uint32_t my[32];                 // this CTA's outgoing record
  float wf[kWarps][8];             // per-warp partials
  uint64_t xbar[kRowsExchanges];
  uint64_t full;
  int wi[kWarps][4];
  unsigned long long wu[kWarps];
  uint32_t lp[kLimbs], lq[kLimbs], infl;
  // decision inputs of the item's row, loaded while the slices stream in
  int t;
  float u, ud, gp, gq, lo_p, lo_q;
  int skip;
  int kk;    // fused filters: the sequence's top-k and top-p
  float pp;
  // the cluster's view after an exchange (written by warp 0)
  float fv[6];
  uint32_t iv[4];
  float dpar[4];
  int bi[4];
  // rank 0: the drawn id and status pushed by the draw's owner
  int out_tok;
  uint32_t out_st;
};

// Draw weights of vector vi of a resident slice pair (q may be null): VEC
// entries, zero past the slice end; returns the number of real elements.
template <typename T, typename D>
__device__ __forceinline__ int smem_draw_weights(const T* p, const T* q, int n, int vi, const D& dw, float* r) {
  constexpr int VEC = ElemTraits<T>::kVec;
  const int e0 = vi * VEC;
  float xp[VEC], xq[VEC];
  int cnt = VEC;
  if (e0 + VEC <= n) {
    unpack_vec<T>(reinterpret_cast<const uint4*>(p)[vi], xp);
    if (q) unpack_vec<T>(reinterpret_cast<const uint4*>(q)[vi], xq);
  } else {
    cnt = n - e0;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      xp[k] = k < cnt ? ElemTraits<T>::to_f(p[e0 + k]) : 0.f;
      xq[k] = (q && k < cnt) ? ElemTraits<T>::to_f(q[e0 + k]) : 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < VEC; ++k) r[k] = k < cnt ? dw(xp[k], q ? xq[k] : 0.f) : 0.f;
  return cnt;
}

}  // namespace svk

namespace svk {

enum : int { OUT_ACCEPT = 0, OUT_TERM = 1, OUT_SKIP = 2, OUT_TIMEOUT = 3, OUT_DRAW = 4, OUT_FALLBACK = 5 };

// Warp 0 of an item's rank-0 CTA, after the item is decided: writes the
// item's record (unless it skipped), counts the item in, and, when it is the
// last of the sequence's kb + 1 items, combines the records into the
// sequence's outputs and returns the counter and the posted row to zero.
// Records are read 32 rows per load round; the first terminal record ends
// the walk and the statuses of the rows up to it are ORed.  A record marked
// kRecFallback ends the walk as well but hands the sequence to the general
// path (seq_flag[b] = 1, outputs left to it).
__device__ __forceinline__ void rows_record_combine(const RowsParams& R, int b, int i, int kb, long long t0,
                                                    bool write, uint4 rv) {
  const Params& P = R.p;
  const int lane = threadIdx.x & 31;
  int last = 0;
  if (lane == 0) {
    if (write) R.rec[t0 + i] = rv;
    __threadfence();
    last = atomicAdd(R.seq_count + b, 1) == kb ? 1 : 0;
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;  // every record of the sequence is written once the count is complete
  __threadfence();
  uint32_t st = 0u;
  int n = 0, nxt = -1;
  bool term = false, fb = false;
  for (int base = 0; base <= kb && !term; base += 32) {
    const int r = base + lane;
    const uint4 v = r <= kb ? __ldcg(R.rec + t0 + r) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t tm = __ballot_sync(0xFFFFFFFFu, r <= kb && (v.x & (kRecTerminal | kRecFallback)) != 0u);
    const int first = tm ? __ffs(tm) - 1 : 32;
    st |= __reduce_or_sync(0xFFFFFFFFu,
                           (lane <= first && r <= kb) ? (v.x & ~(kRecTerminal | kRecFallback)) : 0u);
    if (tm) {
      nxt = __shfl_sync(0xFFFFFFFFu, static_cast<int>(v.y), first);
      n = __shfl_sync(0xFFFFFFFFu, static_cast<int>(v.z), first);
      fb = (__shfl_sync(0xFFFFFFFFu, v.x, first) & kRecFallback) != 0u;
      term = true;
    }
  }
  if (lane == 0) {
    if (fb) {
      R.seq_flag[b] = 1;
    } else {
      if (!term || (st & ST_TIMEOUT)) {
        n = 0;
        nxt = -1;
        st = ST_TIMEOUT;
      }
      if (P.ext_err && *P.ext_err) {  // the producer of the rows gave up: they are invalid
        n = 0;
        nxt = -1;
        st |= ST_TIMEOUT;
      }
      P.n_out[b] = n;
      P.next_out[b] = nxt;
      P.st_out[b] = st;
      if (R.seq_flag) R.seq_flag[b] = 0;
    }
    R.seq_count[b] = 0;  // ready for the next launch
    R.seq_first[b] = 0;
  }
}

// TOPK: the sequences' top-k / top-p floors are computed here (16-bit logits,
// 1 <= top-k <= kTopKMax) instead of coming from the floors kernel.
template <int MODE, typename T, bool FL = false, bool TOPK = false>
__global__ void __launch_bounds__(kRowsThreads, 3) sv_rows_kernel(const __grid_constant__ RowsParams R) {
  static_assert(kRowsThreads == kConsumers, "the chunk passes stride by kConsumers threads");
  const Params& P = R.p;
  using TR = ElemTraits<T>;
  constexpr int VEC = TR::kVec;
  using WarpT =
      typename std::conditional<MODE == MODE_LOGITS, typename WarpOf<T>::type, NoWarp>::type;
  using DrawT = typename std::conditional<MODE == MODE_LOGITS, DrawLogits<FL>, DrawProbs>::type;

  extern __shared__ __align__(128) unsigned char smem[];
  T* sp = reinterpret_cast<T*>(smem);
  T* sq = reinterpret_cast<T*>(smem + R.x_off);
  unsigned long long* vsum = reinterpret_cast<unsigned long long*>(smem + R.vsum_off);
  RowsTail& sm = *reinterpret_cast<RowsTail*>(smem + R.tail_off);
  const int tid = threadIdx.x;
  const int warp = __shfl_sync(0xFFFFFFFFu, tid >> 5, 0);
  const int lane = tid & 31;
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const long long item = blockIdx.x / C;
  const int b = static_cast<int>(item % P.B);
  const int i = static_cast<int>(item / P.B);
  if (P.gate && !P.gate[b]) return;  // the whole cluster shares b

  // the item's scalar inputs, issued together (b < B indexes every
  // per-sequence array)
  const float temp_in = MODE == MODE_LOGITS ? P.temp[b] : 0.f;
  int first_in = 0, kk_in = 0;
  float pp_in = 1.f;
  if (tid == 0) {
    if (i > 0) first_in = *reinterpret_cast<const volatile int*>(R.seq_first + b);
    if constexpr (TOPK) {
      kk_in = R.top_k ? R.top_k[b] : 0;
      pp_in = R.top_p ? R.top_p[b] : 1.f;
    }
  }

  // ---------------------------------------------------------------- sequence layout
  int kb = P.K;
  long long t0 = static_cast<long long>(b) * (P.K + 1LL), d0 = static_cast<long long>(b) * P.K;
  bool layout_ok = true;
  if (P.cu_k) {
    const int lo = P.cu_k[b], hi = P.cu_k[b + 1];
    if (lo < 0 || hi < lo || hi > P.sum_k || hi - lo > P.K) {
      layout_ok = false;
    } else {
      kb = hi - lo;
      t0 = lo + static_cast<long long>(b);
      d0 = lo;
    }
  }
  bool sampling = MODE != MODE_GREEDY;
  float temp = 0.f;
  bool temp_ok = true;
  if (MODE == MODE_LOGITS && layout_ok) {
    temp = temp_in;
    temp_ok = temp >= 0.f && temp <= FLT_MAX;
    sampling = temp > 0.f;
  }
  if (!layout_ok || !temp_ok) {  // row 0's item reports it; no other item of b takes part
    if (i == 0 && rank == 0 && tid == 0) {
      P.n_out[b] = 0;
      P.next_out[b] = -1;
      P.st_out[b] = (layout_ok ? ST_BAD_VALUE : ST_BAD_LAYOUT) | (P.ext_err && *P.ext_err ? ST_TIMEOUT : 0u);
      if (R.seq_flag) R.seq_flag[b] = 0;
    }
    return;
  }
  if (i > kb) return;  // the whole cluster shares b and i
  const bool bonus = i == kb;
  const bool two = sampling && !bonus;  // the item also holds draft row i

  const T* tgt = static_cast<const T*>(P.tgt);
  const T* drf = static_cast<const T*>(P.drf);
  const int v_lo = static_cast<int>(rank) * P.slice;
  const int n_el = max(0, min(P.V, v_lo + P.slice) - v_lo);
  const T* rowp = tgt + (t0 + i) * P.stride + v_lo;
  const T* rowq = two ? drf + (d0 + i) * P.stride + v_lo : nullptr;

  if (tid == 0) {
    // an earlier row of b already ended the sequence
    int skip = (first_in != 0 && INT_MAX - first_in < i) ? 1 : 0;
    if constexpr (TOPK) {
      // a fused-filter row the candidate lists cannot decide (top-k outside
      // [1, kTopKMax]) or an invalid top-p needs no rows: load nothing
      if (sampling && (!(kk_in >= 1 && kk_in <= kTopKMax && kk_in < P.V) || !(pp_in > 0.f))) skip |= 2;
      sm.kk = kk_in;
      sm.pp = pp_in;
    }
    sm.skip = skip;
    for (int x = 0; x < kRowsExchanges; ++x) mbar_init(&sm.xbar[x], C);
    mbar_init(&sm.full, 1);
    sm.out_tok = INT_MIN;
    sm.out_st = 0u;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  const bool skip_mine = (sm.skip & 1) != 0;
  const bool no_rows = (sm.skip & 2) != 0;  // fused filters: this item decides without its rows
  if (TOPK && sampling && no_rows) {
    // the same for every CTA of the cluster (read from the same words): rank 0
    // records the row's outcome without rows, barriers or exchanges: a bad
    // draft id, else a NaN floor (invalid top-p), else the general path
    if (rank != 0) return;
    if (warp == 0) {
      uint32_t rs = ST_BAD_VALUE | kRecTerminal;
      if (!bonus) {
        const int t = P.tok[d0 + i];
        if (t < 0 || t >= P.V) rs = ST_BAD_TOKEN | kRecTerminal;
      }
      if (rs == (ST_BAD_VALUE | kRecTerminal) && sm.pp > 0.f) rs = kRecFallback;
      if (lane == 0) atomicMax(R.seq_first + b, INT_MAX - i);
      rows_record_combine(R, b, i, kb, t0, true, make_uint4(rs, 0xFFFFFFFFu, static_cast<uint32_t>(i), 0u));
    }
    return;
  }

  // ---------------------------------------------------------------- loads
  if (!skip_mine && !no_rows) {
    if (P.use_tma) {
      if (warp == 0) {
        const uint32_t bytes = static_cast<uint32_t>(n_el) * static_cast<uint32_t>(sizeof(T));
        const uint32_t tma = bytes & ~15u;
        for (int e = static_cast<int>(tma / sizeof(T)) + lane; e < n_el; e += 32) {
          sp[e] = rowp[e];
          if (two) sq[e] = rowq[e];
        }
        __syncwarp();
        if (lane == 0) {
          if (tma) {
            mbar_arrive_expect_tx(&sm.full, two ? 2u * tma : tma);
            bulk_g2s(sp, rowp, tma, &sm.full);
            if (two) bulk_g2s(sq, rowq, tma, &sm.full);
          } else {
            mbar_arrive_local(&sm.full);
          }
        }
      }
    } else {
      for (int e = tid; e < n_el; e += kRowsThreads) {
        sp[e] = rowp[e];
        if (two) sq[e] = rowq[e];
      }
    }
  }
  cluster_sync_all();  // every peer runs and its barriers exist before the first remote arrive
  if (!skip_mine) {
    if (tid == 32) {  // the row's decision inputs, while the slices stream in
      int t = -1;
      float gpv = 0.f, gqv = 0.f;
      if (!bonus) {
        t = ld_issue_s32(P.tok + d0 + i);
        if (sampling && t >= 0 && t < P.V) {
          gpv = TR::to_f(tgt[(t0 + i) * P.stride + t]);
          gqv = TR::to_f(drf[(d0 + i) * P.stride + t]);
        }
      }
      sm.t = t;
      sm.gp = gpv;
      sm.gq = gqv;
      sm.u = sampling ? P.uni[t0 + i] : 0.f;
      sm.ud = sampling ? P.uni[t0 + kb] : 0.f;
      float lp = -kInfF, lq = -kInfF;
      if constexpr (FL) {
        if (P.flo_t) lp = __ldg(P.flo_t + t0 + i);
        if (P.flo_d && two) lq = __ldg(P.flo_d + d0 + i);
      }
      sm.lo_p = lp;
      sm.lo_q = lq;
    }
  }
  int bad = 0;  // this CTA's wait for its own copies gave up
  if (!skip_mine && !no_rows && P.use_tma) bad = mbar_wait_bounded(&sm.full, 0u) ? 0 : 1;
  __syncthreads();

  // Exchange of sm.my with every CTA of the cluster through exchange slot x
  // (a collective of warp 0; each slot's barrier completes once per launch).
  auto exchange = [&](int x, int words) -> bool {
    warp_converged();
    __syncwarp();
    uint32_t* base = x == 2 ? &sm.xe[0][0] : &sm.xr[x < 2 ? x : x - 1][0][0];
    const int stride = x == 2 ? 32 : 8;
    if (lane < static_cast<int>(C)) {
      const uint32_t dst = dsmem_addr(base + rank * stride, static_cast<uint32_t>(lane));
      for (int w = 0; w < words; w += 4) dsmem_st_v4(dst + 4u * w, *reinterpret_cast<const uint4*>(&sm.my[w]));
      dsmem_arrive_release(dsmem_addr(&sm.xbar[x], static_cast<uint32_t>(lane)));
    }
    const bool ok =
        mbar_wait_cluster_bounded(&sm.xbar[x], 0u, (P.flags & FLAG_EXPIRE_EXCHANGE) ? 0u : kWaitPolls);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
  };
  auto xrec = [&](int x, int c, int w) -> uint32_t {
    return x == 2 ? sm.xe[c][w] : sm.xr[x < 2 ? x : x - 1][c][w];
  };
  auto xrecf = [&](int x, int c, int w) -> float { return __uint_as_float(xrec(x, c, w)); };
  auto post_terminal = [&]() {  // rank 0: later rows of b may skip
    if (rank == 0 && tid == 0) atomicMax(R.seq_first + b, INT_MAX - i);
  };

  int out = OUT_TIMEOUT;  // the item's outcome (the same in every CTA of the cluster)
  int o_n = 0, o_next = -1;
  uint32_t o_st = 0u;

  if (!sampling) {
    // ============================================================== greedy: argmax of target row i
    float bv = __int_as_float(0x7FFFFFFF);  // NaN: no candidate yet
    int bi = INT_MAX;
    uint32_t nanf = 0;
    if (!skip_mine) chunk_argmax<T>(sp, n_el, v_lo, bv, bi, nanf);
    if (bv != bv) bi = INT_MAX;
    warp_converged();
    warp_argmax(bv, bi);
    const uint32_t fl = __reduce_or_sync(0xFFFFFFFFu, nanf);
    if (lane == 0) {
      sm.wf[warp][0] = bv;
      sm.wi[warp][0] = bi;
      sm.wi[warp][1] = static_cast<int>(fl);
    }
    bad = __syncthreads_or(bad);
    if (warp == 0) {
      warp_converged();
      float v = lane < kWarps ? sm.wf[lane][0] : 0.f;
      int a = lane < kWarps ? sm.wi[lane][0] : INT_MAX;
      const uint32_t f = __reduce_or_sync(0xFFFFFFFFu, lane < kWarps ? static_cast<uint32_t>(sm.wi[lane][1]) : 0u);
      warp_argmax(v, a);
      if (lane == 0) {
        sm.my[0] = __float_as_uint(v);
        sm.my[1] = static_cast<uint32_t>(a);
        sm.my[2] = f | (bad ? 2u : 0u) | (skip_mine ? 4u : 0u);
        sm.my[3] = 0u;
      }
      uint32_t g = 2u;
      int ga = INT_MAX;
      if (exchange(0, 4)) {
        const bool cl = lane < static_cast<int>(C);
        v = cl ? xrecf(0, lane, 0) : 0.f;
        a = cl ? static_cast<int>(xrec(0, lane, 1)) : INT_MAX;
        g = __reduce_or_sync(0xFFFFFFFFu, cl ? xrec(0, lane, 2) : 0u);
        warp_argmax(v, a);
        ga = a;
      }
      if (lane == 0) {
        sm.iv[0] = g;
        sm.bi[0] = ga;
      }
    }
    __syncthreads();
    const uint32_t g = sm.iv[0];
    int a = sm.bi[0];
    if (g & 2u) {
      out = OUT_TIMEOUT;
    } else if (g & 4u) {
      out = OUT_SKIP;
    } else {
      if (a == INT_MAX) a = 0;  // an all-NaN row
      o_st = (g & 1u) ? ST_BAD_VALUE : 0u;
      o_next = a;
      out = OUT_TERM;
      if (bonus) {
        o_n = kb;
      } else {
        const int t = sm.t;
        o_n = i;
        if (t < 0 || t >= P.V) o_st |= ST_BAD_TOKEN;
        else if (t == a) out = OUT_ACCEPT;
      }
      if (out == OUT_TERM) post_terminal();
    }
  } else if constexpr (TOPK) {
    // ============================================================== sampling, fused top-k / top-p
    // Every CTA takes, per row, the keys of its slice at or above the
    // slice's k-th largest key (and possibly a few below it): the row's k-th
    // largest key is at least every slice's, so the union of these lists
    // holds every key the filters keep.
    // Rank 0 gathers the lists and finds the floors, the masses of the kept
    // tokens, the decision and the draw on them alone (a logit below the
    // floor weighs 0 everywhere).  A row outside what the lists can decide
    // (top-k outside [1, kTopKMax], a list or kept set over its capacity)
    // is recorded for the general path.
    static_assert(sizeof(T) == 2 && MODE == MODE_LOGITS && FL, "fused filters: 16-bit logits rows");
    using KY = Key16x<T>;
    using WT = typename WarpOf<T>::type;
    float khi = 0.f, klo = 0.f;
    log2e_over(temp, khi, klo);
    const int kk = sm.kk;
    const float pp = sm.pp;
    const bool p_ok = pp > 0.f;  // NaN or <= 0: invalid top-p, the floors are NaN
    const bool use_p = pp < 1.f;
    const bool fast = kk >= 1 && kk <= kTopKMax && kk < P.V;
    unsigned char* vsa = smem + R.vsum_off;
    uint2* lst = reinterpret_cast<uint2*>(vsa);                               // [2][kListCap]
    unsigned* hist = reinterpret_cast<unsigned*>(vsa + 2 * kListCap * 8);     // [2][256]
    int* misc = reinterpret_cast<int*>(vsa + 2 * kListCap * 8 + 2048);        // [16]
    bad = __syncthreads_or(bad);
    uint32_t fl = (bad ? 16u : 0u) | (skip_mine ? 8u : 0u);  // 1 / 2 row invalid, 4 list overflow
    int nl0 = 0, nl1 = 0;
    uint32_t smax = 0u;  // the slice maximum keys of the two rows (16 bits each; 0: none)
    if (!bad && !skip_mine && fast && p_ok) {
      // Both rows go through each pass before the pass's barrier.  (1) The
      // slice maxima, keeping each thread's own maximum key.  (2) Per row,
      // one warp takes the kk-th largest of the 256 per-thread maxima: they
      // are kk distinct logits of the slice, so it is at most the slice's
      // kk-th largest key.  (3) Every logit at or above it goes to the list
      // (a packed compare per pair, per-element work only in the rare
      // vectors that hold one): the keys at or above the slice's kk-th
      // largest and a few more, which is all rank 0 needs.
      const int nx = two ? 2 : 1;
      unsigned* tkey = hist;  // [2][kRowsThreads] per-thread maximum keys
      for (int x = 0; x < nx; ++x) {
        const float tm = slice_max_nan16<T>(x ? sq : sp, n_el);  // -Inf for a thread without elements
        uint32_t k = 0u;  // (a NaN makes the row invalid below)
        if constexpr (std::is_same<T, __nv_bfloat16>::value) KY::key(__float_as_uint(tm) >> 16, k);
        else KY::key(__half_as_ushort(__float2half_rn(tm)), k);
        tkey[x * kRowsThreads + tid] = k;
        const float mxn = warp_max_nan_f(tm);
        if (lane == 0) sm.wf[warp][x] = mxn;
      }
      __syncthreads();
      bool live[2] = {false, false};
      for (int x = 0; x < nx; ++x) {
        float cm = -kInfF;
        for (int w = 0; w < kWarps; ++w) cm = fmax_nan(cm, sm.wf[w][x]);
        if (!(cm < kInfF)) {  // a NaN or +Inf logit: the row is invalid, its list stays empty
          fl |= x ? 2u : 1u;
          continue;
        }
        live[x] = true;
        uint32_t k = 0u;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) KY::key(__float_as_uint(cm) >> 16, k);
        else KY::key(__half_as_ushort(__float2half_rn(cm)), k);
        smax |= k << (16 * x);
      }
      if (warp < nx && live[warp]) {
        const uint32_t L = kth_of_256(tkey + warp * kRowsThreads, static_cast<unsigned>(kk));
        if (lane == 0) misc[warp] = static_cast<int>(L);
      }
      __syncthreads();
      // this thread's count of list entries, an exclusive scan of the counts
      // over the CTA, then the entries at those offsets (no atomics)
      KeysAtLeast16<T> sel[2] = {KeysAtLeast16<T>(sp, n_el, static_cast<uint32_t>(misc[0])),
                                 KeysAtLeast16<T>(sq, n_el, static_cast<uint32_t>(misc[1]))};
      unsigned mine[2] = {0u, 0u};
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (x < nx && live[x]) mine[x] = sel[x].count();
      unsigned* wt = hist;  // [2][kWarps] (the per-thread maxima are no longer read)
      unsigned incl[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        unsigned v = mine[x];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned t = __shfl_up_sync(0xFFFFFFFFu, v, o);
          if (lane >= o) v += t;
        }
        incl[x] = v;
        if (lane == 31) wt[x * kWarps + warp] = v;
      }
      __syncthreads();
      unsigned cnt[2] = {0u, 0u};
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x >= nx) continue;
        unsigned base = 0u;
        for (int w = 0; w < kWarps; ++w) {
          const unsigned t = wt[x * kWarps + w];
          if (w < warp) base += t;
          cnt[x] += t;
        }
        if (!live[x]) continue;
        uint2* lx = lst + x * kListCap;
        unsigned at = base + incl[x] - mine[x];
        sel[x].visit([&](uint32_t k, int e) {
          if (at < static_cast<unsigned>(kListCap)) lx[at] = make_uint2(k, static_cast<uint32_t>(v_lo + e));
          ++at;
        });
      }
      if (cnt[0] > static_cast<unsigned>(kListCap) || cnt[1] > static_cast<unsigned>(kListCap)) fl |= 4u;
      nl0 = static_cast<int>(min(cnt[0], static_cast<unsigned>(kListCap)));
      nl1 = static_cast<int>(min(cnt[1], static_cast<unsigned>(kListCap)));
    }
    __syncthreads();
    cluster_sync_all();  // rank 0 no longer reads its slices: they become its receive area
    {
      // rank 0's receive area: [C] headers {n_0, n_1, flags, slice maximum keys},
      // then [C][2][kListCap] entries
      const uint32_t base = dsmem_addr(smem, 0u);
      if (tid == 0)
        dsmem_st_v4(base + rank * 16u, make_uint4(static_cast<uint32_t>(nl0), static_cast<uint32_t>(nl1), fl, smax));
      const uint32_t lbase = base + 256u + rank * (2u * kListCap * 8u);
      for (int j = tid; j < nl0 + nl1; j += kRowsThreads) {
        const int x = j < nl0 ? 0 : 1;
        const int q = x ? j - nl0 : j;
        dsmem_st_v2(lbase + static_cast<uint32_t>(x * kListCap + q) * 8u, lst[x * kListCap + q]);
      }
    }
    __syncthreads();
    cluster_sync_all();  // every list has reached rank 0
    // Nothing reaches another CTA's shared memory after this point: the
    // other CTAs leave now (their SM slots take later items) and rank 0
    // finishes the item alone, without the final cluster barrier.
    if (rank != 0) {
      if (bad && tid == 0) mbar_wait_bounded(&sm.full, 0u);  // no copy may land after exit
      return;
    }
    {
      const uint4* rh = reinterpret_cast<const uint4*>(smem);
      const uint2* rl = reinterpret_cast<const uint2*>(smem + 256);
      unsigned char* w0 = smem + 256 + static_cast<size_t>(C) * 2 * kListCap * 8;
      // rank 0's work space after the lists (kTopkScratch bytes)
      uint2* kept = reinterpret_cast<uint2*>(w0);                          // [2][kKeptCap]
      int* ord = reinterpret_cast<int*>(kept + 2 * kKeptCap);             // [kKeptCap] p's kept, by index
      float* lqa = reinterpret_cast<float*>(ord + kKeptCap);               // [kKeptCap] q's logit there
      unsigned* hist2 = reinterpret_cast<unsigned*>(lqa + kKeptCap);       // [2][256]
      uint32_t* tk = hist2 + 2 * 256;                                      // [2][kTopKMax]
      uint32_t* tko = tk + 2 * kTopKMax;                                   // [2][kTopKMax]
      unsigned long long* tkw = reinterpret_cast<unsigned long long*>(tko + 2 * kTopKMax);  // [2][kTopKMax]
      uint2* tke = reinterpret_cast<uint2*>(tkw + 2 * kTopKMax);          // [2][kTopKMax] top-k entries
      int* rs = reinterpret_cast<int*>(tke + 2 * kTopKMax);               // [32]
      float* rsf = reinterpret_cast<float*>(rs + 24);                      // [4] inside rs
      unsigned long long* bk = reinterpret_cast<unsigned long long*>(vsa);  // exact buckets (over the lists)
      if (tid == 0) {
        uint32_t Fa = 0u;
        for (uint32_t c = 0; c < C; ++c) Fa |= rh[c].z;
        rs[0] = static_cast<int>(Fa);
      }
      __syncthreads();
      const uint32_t F = static_cast<uint32_t>(rs[0]);
      const int t = sm.t;
      const float u = sm.u;
      uint32_t st = 0u;
      out = OUT_TERM;
      o_n = i;
      o_next = -1;
      if (F & 16u) {
        out = OUT_TIMEOUT;
      } else if (F & 8u) {
        out = OUT_SKIP;
      } else {
        // input errors in the general path's order (a NaN floor is an invalid row)
        uint32_t err = 0u;
        if (!bonus && (t < 0 || t >= P.V)) err = ST_BAD_TOKEN;
        if (!err && !p_ok) err = ST_BAD_VALUE;
        if (!err && !fast) {
          out = OUT_FALLBACK;
        } else {
          if (!err && (F & 1u)) err = ST_BAD_VALUE;
          if (!err && two && (F & 2u)) err = ST_BAD_VALUE;
          if (!err && !(u >= 0.f && u < 1.f)) err = ST_BAD_VALUE;
          if (err) {
            o_st = err;
          } else if (F & 4u) {
            out = OUT_FALLBACK;
          } else {
            // ---- per row, one warp each (warp 0 the target row, warp 1 the
            // draft row): the maximum, the top-k floor key, the top-p floor key
            // among the top-k set, and the kept tokens (keys at or above it)
            if (warp < (two ? 2 : 1)) {
              const int x = warp;
              unsigned* hx = hist2 + x * 256;
              uint32_t* tkx = tk + x * kTopKMax;
              // every lane runs the same trips; `ok` marks the lanes holding an entry
              auto each = [&](auto f) {
                for (uint32_t c = 0; c < C; ++c) {
                  const int cnt = static_cast<int>(x ? rh[c].y : rh[c].x);
                  for (int q0 = 0; q0 < cnt; q0 += 32) {
                    const int q = q0 + lane;
                    const bool ok = q < cnt;
                    f(ok ? rl[(c * 2 + x) * kListCap + q] : make_uint2(0u, 0u), ok);
                  }
                }
              };
              // the row maximum: the largest slice maximum in the headers
              uint32_t km = lane < static_cast<int>(C) ? (rh[lane].w >> (16 * x)) & 0xFFFFu : 0u;
              km = __reduce_max_sync(0xFFFFFFFFu, km);
              int fbx = km == 0u ? 1 : 0;  // no key listed: cannot happen for a valid row
              float mrow = -kInfF, flox = -kInfF;
              int nkx = 0;
              if (!fbx) mrow = KY::value(km);
              if (!fbx && mrow > -kInfF) {  // (every logit -Inf: zero mass, no floor)
                for (int j = lane; j < 256; j += 32) hx[j] = 0u;
                __syncwarp();
                each([&](uint2 e, bool ok) {
                  const uint32_t d = km - e.x;
                  if (ok && d < 256u) atomicAdd(&hx[255u - d], 1u);
                });
                __syncwarp();
                unsigned tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) tot += hx[lane * 8 + j];
                tot = __reduce_add_sync(0xFFFFFFFFu, tot);
                unsigned ab = 0;
                const int bin = tot >= static_cast<unsigned>(kk) ? pick_bin_count(hx, 0u, static_cast<unsigned>(kk), ab)
                                                                 : -1;
                if (bin < 0) {
                  fbx = 1;  // the k-th largest lies more than 255 keys below the maximum
                } else {
                  const uint32_t key_k = km - (255u - static_cast<uint32_t>(bin));
                  uint32_t key_f = key_k;
                  int n = -1;  // the top-k set's size, once gathered into tkx / tke
                  if (use_p && key_k < km) {
                    n = 0;
                    each([&](uint2 e, bool ok) {  // keys and entries of the top-k set
                      const bool pr = ok && e.x >= key_k;
                      const unsigned bl = __ballot_sync(0xFFFFFFFFu, pr);
                      const int at = n + __popc(bl & ((1u << lane) - 1u));
                      if (pr && at < kTopKMax) {
                        tkx[at] = e.x;
                        tke[x * kTopKMax + at] = e;
                      }
                      n += __popc(bl);
                    });
                    if (n > kTopKMax) {
                      fbx = 1;
                    } else {
                      WT wf;
                      wf.m = mrow;
                      wf.k = khi;
                      wf.lo = -kInfF;
                      auto weight = [&](uint32_t k) -> unsigned long long {
                        return floor_u64(__fmul_rn(wf(KY::value(k)), 0x1p40f));
                      };
                      __syncwarp();
                      unsigned long long z = 0ull;
                      for (int j = lane; j < n; j += 32) z += weight(tkx[j]);
                      z = warp_sum_u64(z);
                      key_f = top_p_walk(tkx, n, weight, static_cast<double>(pp) * static_cast<double>(z),
                                         tko + x * kTopKMax, tkw + x * kTopKMax);
                    }
                  }
                  if (!fbx) {
                    flox = KY::value(key_f);
                    int n2 = 0;
                    if (n >= 0) {  // the kept set lies within the gathered top-k set
                      __syncwarp();
                      for (int q0 = 0; q0 < n; q0 += 32) {
                        const int q = q0 + lane;
                        const uint2 e = q < n ? tke[x * kTopKMax + q] : make_uint2(0u, 0u);
                        warp_compact(q < n && e.x >= key_f, e, kept + x * kKeptCap, kKeptCap, n2);
                      }
                    } else {
                      each([&](uint2 e, bool ok) { warp_compact(ok && e.x >= key_f, e, kept + x * kKeptCap, kKeptCap, n2); });
                    }
                    nkx = n2;
                    if (n2 > kKeptCap) fbx = 1;
                  }
                }
              }
              if (lane == 0) {
                rs[16 + x] = fbx;
                rs[18 + x] = nkx;
                rsf[x] = mrow;
                rsf[2 + x] = flox;
              }
            }
            __syncthreads();
            const bool fb = rs[16] != 0 || (two && rs[17] != 0);
            const float m_row[2] = {rsf[0], two ? rsf[1] : -kInfF};
            const float flo[2] = {rsf[2], two ? rsf[3] : -kInfF};
            const int nk[2] = {rs[18], two ? rs[19] : 0};
            if (fb) {
              out = OUT_FALLBACK;
            } else if (!(m_row[0] > -kInfF) || (!bonus && !(m_row[1] > -kInfF))) {
              o_st = ST_ZERO_MASS;
            } else {
              WT wfp, wfq;
              wfp.m = m_row[0];
              wfp.k = khi;
              wfp.lo = flo[0];
              wfq.m = m_row[1];
              wfq.k = khi;
              wfq.lo = flo[1];
              // fp32 masses of the kept tokens (each lane adds at most 8, then a tree)
              if (warp == 0) {
                float zp = 0.f, zq = 0.f;
                for (int j = lane; j < nk[0]; j += 32) zp = __fadd_rn(zp, wfp(KY::value(kept[j].x)));
                for (int j = lane; j < nk[1]; j += 32) zq = __fadd_rn(zq, wfq(KY::value(kept[kKeptCap + j].x)));
                zp = warp_sum_f(zp);
                zq = warp_sum_f(zq);
                if (lane == 0) {
                  sm.fv[0] = zp;
                  sm.fv[1] = zq;
                }
              }
              __syncthreads();
              const DF Zp = {sm.fv[0], 0.f}, Zq = {sm.fv[1], 0.f};
              bool have_exact = false;
              double Zp_ex = 0.0, Zq_ex = 0.0;
              int dec = 0;
              if (!bonus) {
                const float pt = wfp(sm.gp), qt = wfq(sm.gq);
                dec = filter_decide(u, pt, qt, Zp, sum_bound(Zp.hi, (nk[0] + 31) / 32), Zq,
                                    sum_bound(Zq.hi, (nk[1] + 31) / 32));
                if ((P.flags & FLAG_FORCE_EXACT) || dec < 0) {
                  // the exact masses of the kept tokens (every other weight is 0)
                  for (int q = tid; q < 2 * kBuckets; q += kRowsThreads) bk[q] = 0ull;
                  __syncthreads();
                  for (int j = tid; j < nk[0]; j += kRowsThreads) bucket_add(bk, wfp(KY::value(kept[j].x)));
                  for (int j = tid; j < nk[1]; j += kRowsThreads)
                    bucket_add(bk + kBuckets, wfq(KY::value(kept[kKeptCap + j].x)));
                  __syncthreads();
                  if (tid == 0) {
                    buckets_to_limbs(bk, sm.lp);
                    buckets_to_limbs(bk + kBuckets, sm.lq);
                    sm.bi[3] = exact_accept(u, pt, qt, sm.lp, sm.lq) ? 1 : 0;
                  }
                  __syncthreads();
                  dec = sm.bi[3];
                  have_exact = true;
                  Zp_ex = limbs_to_double(sm.lp);
                  Zq_ex = limbs_to_double(sm.lq);
                  st |= ST_EXACT;
                }
              }
              if (!bonus && dec) {
                out = OUT_ACCEPT;
                o_st = st;
              } else {
                // ---- the bonus from p_K, or the residual after the rejection, with u_K
                const float ud = sm.ud;
                o_n = bonus ? kb : i;
                if (!bonus && !(ud >= 0.f && ud < 1.f)) {
                  o_st = st | ST_BAD_VALUE;
                } else {
                  DrawLogits<true> dw;
                  dw.scale = __uint_as_float(static_cast<uint32_t>(127 + P.fixed_shift) << 23);
                  dw.resid = bonus ? 0 : 1;
                  const float zp = have_exact ? static_cast<float>(Zp_ex) : Zp.hi;
                  const float zq = bonus ? 1.f : (have_exact ? static_cast<float>(Zq_ex) : Zq.hi);
                  dw.k = khi;
                  const DF mk = two_prod(m_row[0], khi), qk = two_prod(m_row[1], khi);
                  dw.cp = -__fadd_rn(mk.hi, __fadd_rn(mk.lo, log2f(zp)));
                  dw.cq = bonus ? 0.f : -__fadd_rn(qk.hi, __fadd_rn(qk.lo, log2f(zq)));
                  dw.lo_p = flo[0];
                  dw.lo_q = bonus ? -kInfF : flo[1];
                  // warp 0: the kept tokens of p in index order, their fixed-point
                  // draw weights, the inverse CDF (0 found, 1 empty residual,
                  // 2 p has no draw mass)
                  // p's kept tokens ranked by vocab index, one thread each (the
                  // indices are distinct), with the draft logit at each token
                  // when q keeps it (-Inf otherwise)
                  static_assert(kKeptCap <= kRowsThreads, "one thread per kept token");
                  {
                    const int n = nk[0], nq = bonus ? 0 : nk[1];
                    if (tid < n) {
                      const uint32_t vj = kept[tid].y;
                      int r = 0;
#pragma unroll 4
                      for (int m = 0; m < n; ++m) r += kept[m].y < vj ? 1 : 0;
                      float lq = -kInfF;
#pragma unroll 4
                      for (int m = 0; m < nq; ++m) {
                        const uint2 e = kept[kKeptCap + m];
                        if (e.y == vj) lq = KY::value(e.x);
                      }
                      ord[r] = tid;
                      lqa[r] = lq;
                    }
                    __syncthreads();
                  }
                  auto draw_kept = [&](bool resid, uint32_t st_in) -> int {
                    const int n = nk[0];
                    unsigned long long f[8];
                    unsigned long long tot = 0ull;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                      const int pos = lane * 8 + q;
                      f[q] = 0ull;
                      if (pos < n) {
                        const uint2 e = kept[ord[pos]];
                        f[q] = dw.fix(dw(KY::value(e.x), resid ? lqa[pos] : -kInfF));
                        tot += f[q];
                      }
                    }
                    unsigned long long inc = tot;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                      const unsigned long long v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                      if (lane >= o) inc += v;
                    }
                    const unsigned long long Rt = __shfl_sync(0xFFFFFFFFu, inc, 31);
                    if (Rt == 0ull) return resid ? 1 : 2;
                    const unsigned long long tau = tau_of(ud, Rt);
                    const unsigned long long ex = inc - tot;
                    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, tau >= ex && tau < inc);
                    int found = -1, near_b = 0;
                    if (hit) {
                      const int L = __ffs(hit) - 1;
                      if (lane == L) {
                        unsigned long long c = ex;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                          const int pos = lane * 8 + q;
                          const unsigned long long cur = c + f[q];
                          if (found < 0 && pos < n && tau < cur) {
                            const unsigned long long dlo = tau - c, dhi = cur - tau;
                            found = static_cast<int>(kept[ord[pos]].y);
                            near_b = static_cast<double>(dlo < dhi ? dlo : dhi) <= 1e-5 * static_cast<double>(Rt) ? 1 : 0;
                          }
                          c = cur;
                        }
                      }
                      found = __shfl_sync(0xFFFFFFFFu, found, L);
                      near_b = __shfl_sync(0xFFFFFFFFu, near_b, L);
                    }
                    if (lane == 0) {
                      sm.out_tok = found;
                      sm.out_st = found >= 0 ? (st_in | (near_b ? ST_NEAR : 0u)) : ST_TIMEOUT;
                    }
                    return 0;
                  };
                  if (warp == 0) {
                    int code = draw_kept(!bonus, st);
                    if (code == 1) {  // an empty residual: the draw falls back to p
                      dw.resid = 0;
                      code = draw_kept(false, st | ST_ZERO_MASS);
                    }
                    if (lane == 0) sm.bi[2] = code;
                  }
                  __syncthreads();
                  const int code = sm.bi[2];
                  if (code == 2) {
                    o_st = st | ST_ZERO_MASS;
                  } else {
                    out = OUT_DRAW;
                  }
                }
              }
            }
          }
        }
        if (out == OUT_TERM || out == OUT_DRAW || out == OUT_FALLBACK) post_terminal();
      }
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

    // ---- exact masses of the row from the resident slices (collective);
    // the summed limbs and +Inf flags land in sm.lp / sm.lq / sm.infl
    auto exact_pass = [&](const WarpT& fp, const WarpT& fq) -> bool {
      for (int k = tid; k < 2 * kBuckets; k += kRowsThreads) vsum[k] = 0ull;
      __syncthreads();
      int bp = 0, bq = 0;
      for (int e = tid; e < n_el; e += kRowsThreads) {
        const float x = fp(TR::to_f(sp[e]));
        if (!(x <= FLT_MAX)) bp = 1;  // +Inf (NaN and negatives were rejected before)
        else bucket_add(vsum, x);
        if (two) {
          const float y = fq(TR::to_f(sq[e]));
          if (!(y <= FLT_MAX)) bq = 1;
          else bucket_add(vsum + kBuckets, y);
        }
      }
      bp = __syncthreads_or(bp);
      bq = __syncthreads_or(bq);
      if (tid == 0) {
        buckets_to_limbs(vsum, &sm.my[0]);
        buckets_to_limbs(vsum + kBuckets, &sm.my[kLimbs]);
        sm.my[2 * kLimbs] = (bp ? 1u : 0u) | (bq ? 2u : 0u);
        sm.my[2 * kLimbs + 1] = sm.my[2 * kLimbs + 2] = sm.my[2 * kLimbs + 3] = 0u;
      }
      __syncthreads();
      if (warp == 0) {
        const bool ok = exchange(2, 2 * kLimbs + 4);
        if (lane == 0) {
          if (ok) {
            unsigned long long ap[kLimbs], aq[kLimbs];
            for (int k = 0; k < kLimbs; ++k) ap[k] = aq[k] = 0ull;
            uint32_t infl = 0;
            for (uint32_t c = 0; c < C; ++c) {
              for (int k = 0; k < kLimbs; ++k) {
                ap[k] += xrec(2, c, k);
                aq[k] += xrec(2, c, kLimbs + k);
              }
              infl |= xrec(2, c, 2 * kLimbs);
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
          sm.bi[1] = ok ? 1 : 0;
        }
      }
      __syncthreads();
      return sm.bi[1] != 0;
    };

    // ---- pass A: probabilities: masses and minima; logits: maxima
    uint32_t flags = 1u;  // cluster view: 1 a wait gave up, 2 / 4 target / draft row invalid, 8 skip
    float mp = -kInfF, mq = -kInfF;
    DF Zp = {0.f, 0.f}, Zq = {0.f, 0.f};
    float Bp = 0.f, Bq = 0.f;
    if constexpr (MODE == MODE_PROBS) {
      Acc ap, aq;
      ap.init();
      aq.init();
      float mnp = kInfF, mnq = kInfF;
      if (!skip_mine) {
        chunk_mass_f32(reinterpret_cast<const float*>(sp), n_el, ap, mnp);
        if (two) chunk_mass_f32(reinterpret_cast<const float*>(sq), n_el, aq, mnq);
      }
      warp_converged();
      const float s0 = warp_sum_f(ap.f), s1 = warp_sum_f(aq.f);
      const float m0 = warp_min_nan_f(mnp), m1 = warp_min_nan_f(mnq);
      if (lane == 0) {
        sm.wf[warp][0] = s0;
        sm.wf[warp][1] = s1;
        sm.wf[warp][2] = m0;
        sm.wf[warp][3] = m1;
      }
      bad = __syncthreads_or(bad);
      if (warp == 0) {
        warp_converged();
        const bool wl = lane < kWarps;
        const float c0 = warp_sum_f<8>(wl ? sm.wf[lane][0] : 0.f);
        const float c1 = warp_sum_f<8>(wl ? sm.wf[lane][1] : 0.f);
        const float n0 = warp_min_nan_f<8>(wl ? sm.wf[lane][2] : kInfF);
        const float n1 = warp_min_nan_f<8>(wl ? sm.wf[lane][3] : kInfF);
        if (lane == 0) {
          sm.my[0] = __float_as_uint(c0);
          sm.my[1] = __float_as_uint(c1);
          sm.my[2] = (bad ? 1u : 0u) | (n0 >= 0.f ? 0u : 2u) | (n1 >= 0.f ? 0u : 4u) | (skip_mine ? 8u : 0u);
          sm.my[3] = 0u;
        }
        float zp = 0.f, zq = 0.f;
        uint32_t f = 1u;
        if (exchange(0, 4)) {
          const bool cl = lane < static_cast<int>(C);
          zp = warp_sum_f<16>(cl ? xrecf(0, lane, 0) : 0.f);
          zq = warp_sum_f<16>(cl ? xrecf(0, lane, 1) : 0.f);
          f = __reduce_or_sync(0xFFFFFFFFu, cl ? xrec(0, lane, 2) : 0u);
        }
        if (lane == 0) {
          sm.fv[0] = zp;
          sm.fv[1] = zq;
          sm.iv[0] = f;
        }
      }
      __syncthreads();
      Zp.hi = sm.fv[0];
      Zq.hi = sm.fv[1];
      flags = sm.iv[0];
      Bp = sum_bound(Zp.hi, R.nadd);
      Bq = sum_bound(Zq.hi, R.nadd);
    } else {
      // one online-softmax pass per row (running maximum and weight sums with
      // a tracked error bound), merged lanes -> warp -> CTA -> cluster, each
      // merge one rescale step, as in the chain kernel
      Online op, oq;
      op.init();
      oq.init();
      float ep = -kInfF, eq = -kInfF;  // NaN-propagating maxima (validity)
      if (!skip_mine) {
        chunk_online<T, FL>(sp, n_el, khi, sm.lo_p, op, ep);
        if (two) chunk_online<T, FL>(sq, n_el, khi, sm.lo_q, oq, eq);
      }
      warp_converged();
      const float wmp = warp_max_f(op.m), wmq = warp_max_f(oq.m);
      float s0 = 0.f, w0 = 0.f, s1 = 0.f, w1 = 0.f;
      if (op.m > -kInfF) {
        const float d = __fmul_rn(__fsub_rn(wmp, op.m), khi);
        const float f = ex2_ftz(-d);
        s0 = __fmul_rn(op.s, f);
        w0 = __fmul_rn(__fmaf_rn(d, op.s, op.w), f);
      }
      if (oq.m > -kInfF) {
        const float d = __fmul_rn(__fsub_rn(wmq, oq.m), khi);
        const float f = ex2_ftz(-d);
        s1 = __fmul_rn(oq.s, f);
        w1 = __fmul_rn(__fmaf_rn(d, oq.s, oq.w), f);
      }
      s0 = warp_sum_f(s0);
      w0 = warp_sum_f(w0);
      s1 = warp_sum_f(s1);
      w1 = warp_sum_f(w1);
      const float vmp = warp_max_nan_f(ep), vmq = warp_max_nan_f(eq);
      const int rr = warp_max_i(max(op.r, oq.r));
      if (lane == 0) {
        sm.wf[warp][0] = wmp;
        sm.wf[warp][1] = s0;
        sm.wf[warp][2] = w0;
        sm.wf[warp][3] = wmq;
        sm.wf[warp][4] = s1;
        sm.wf[warp][5] = w1;
        sm.wf[warp][6] = vmp;
        sm.wf[warp][7] = vmq;
        sm.wi[warp][0] = rr;
      }
      bad = __syncthreads_or(bad);
      if (warp == 0) {
        warp_converged();
        static_assert(kWarps == 8 && kMaxCluster <= 16, "combine widths");
        const bool wl = lane < kWarps;
        const float4 fa = *reinterpret_cast<const float4*>(&sm.wf[lane & 7][0]);
        const float4 fb = *reinterpret_cast<const float4*>(&sm.wf[lane & 7][4]);
        // warps -> CTA (one more rescale step)
        const float xmp = wl ? fa.x : -kInfF, xmq = wl ? fa.w : -kInfF;
        const float cmp = warp_max_f<8>(xmp), cmq = warp_max_f<8>(xmq);
        const float c6 = warp_max_nan_f<8>(wl ? fb.z : -kInfF);
        const float c7 = warp_max_nan_f<8>(wl ? fb.w : -kInfF);
        const int cr = warp_max_i<8>(wl ? sm.wi[lane & 7][0] : 0);
        float cs0 = 0.f, cw0 = 0.f, cs1 = 0.f, cw1 = 0.f;
        if (xmp > -kInfF) {
          const float d = __fmul_rn(__fsub_rn(cmp, xmp), khi);
          const float f = ex2_ftz(-d);
          cs0 = __fmul_rn(fa.y, f);
          cw0 = __fmul_rn(__fmaf_rn(d, fa.y, fa.z), f);
        }
        if (xmq > -kInfF) {
          const float d = __fmul_rn(__fsub_rn(cmq, xmq), khi);
          const float f = ex2_ftz(-d);
          cs1 = __fmul_rn(fb.x, f);
          cw1 = __fmul_rn(__fmaf_rn(d, fb.x, fb.y), f);
        }
        warp_converged();
        cs0 = warp_sum_f<8>(cs0);
        cw0 = warp_sum_f<8>(cw0);
        cs1 = warp_sum_f<8>(cs1);
        cw1 = warp_sum_f<8>(cw1);
        if (lane == 0) {
          sm.my[0] = __float_as_uint(cmp);
          sm.my[1] = __float_as_uint(cmq);
          sm.my[2] = __float_as_uint(cs0);
          sm.my[3] = __float_as_uint(cw0);
          sm.my[4] = __float_as_uint(cs1);
          sm.my[5] = __float_as_uint(cw1);
          sm.my[6] = static_cast<uint32_t>(cr);
          sm.my[7] = (bad ? 1u : 0u) | (c6 < kInfF ? 0u : 2u) | (c7 < kInfF ? 0u : 4u) | (skip_mine ? 8u : 0u);
        }
        float gmp = -kInfF, gmq = -kInfF, zp = 0.f, zq = 0.f, gwp = 0.f, gwq = 0.f;
        int gr = 0;
        uint32_t f = 1u;
        if (exchange(0, 8)) {
          // CTAs -> cluster (one more rescale step)
          warp_converged();
          const bool cl = lane < static_cast<int>(C);
          const float rmp = cl ? xrecf(0, lane, 0) : -kInfF, rmq = cl ? xrecf(0, lane, 1) : -kInfF;
          gmp = warp_max_f<16>(rmp);
          gmq = warp_max_f<16>(rmq);
          gr = warp_max_i<16>(cl ? static_cast<int>(xrec(0, lane, 6)) : 0);
          f = __reduce_or_sync(0xFFFFFFFFu, cl ? xrec(0, lane, 7) : 0u);
          float z0 = 0.f, z1 = 0.f, v0 = 0.f, v1 = 0.f;
          if (rmp > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(gmp, rmp), khi);
            const float ff = ex2_ftz(-d);
            z0 = __fmul_rn(xrecf(0, lane, 2), ff);
            v0 = __fmul_rn(__fmaf_rn(d, xrecf(0, lane, 2), xrecf(0, lane, 3)), ff);
          }
          if (rmq > -kInfF) {
            const float d = __fmul_rn(__fsub_rn(gmq, rmq), khi);
            const float ff = ex2_ftz(-d);
            z1 = __fmul_rn(xrecf(0, lane, 4), ff);
            v1 = __fmul_rn(__fmaf_rn(d, xrecf(0, lane, 4), xrecf(0, lane, 5)), ff);
          }
          warp_converged();
          zp = warp_sum_f<16>(z0);
          zq = warp_sum_f<16>(z1);
          gwp = warp_sum_f<16>(v0);
          gwq = warp_sum_f<16>(v1);
        }
        if (lane == 0) {
          sm.fv[0] = gmp;
          sm.fv[1] = gmq;
          sm.fv[2] = zp;
          sm.fv[3] = zq;
          sm.fv[4] = gwp;
          sm.fv[5] = gwq;
          sm.iv[0] = f;
          sm.iv[1] = static_cast<uint32_t>(gr);
        }
      }
      __syncthreads();
      mp = sm.fv[0];
      mq = sm.fv[1];
      Zp.hi = sm.fv[2];
      Zq.hi = sm.fv[3];
      flags = sm.iv[0];
      const int Rs = static_cast<int>(sm.iv[1]);
      Bp = online_bound(Zp.hi, sm.fv[4], Rs + 1, R.nadd, fabsf(__fmul_rn(mp, khi))) + static_cast<float>(P.V) * 1.2e-38f;
      Bq = online_bound(Zq.hi, sm.fv[5], Rs + 1, R.nadd, fabsf(__fmul_rn(mq, khi))) + static_cast<float>(P.V) * 1.2e-38f;
    }

    // ---- inverse-CDF draw over the resident slices (collective).  Returns
    // 0 when done (the owner pushed the id to rank 0), 1 when the residual
    // is empty, 2 when p itself has no draw mass, -1 when an exchange gave up.
    auto draw = [&](const DrawT& dw, bool resid, int x, uint32_t st_in, float ud) -> int {
      const T* qs = resid ? sq : nullptr;
      const int nvt = (n_el + VEC - 1) / VEC;
      const int ng = (nvt + kGroupVecs - 1) / kGroupVecs;
      constexpr int U = 4;
      constexpr int LG = kGroupVecs / U;  // lanes per group
      static_assert(LG == 8, "group sums reduce over 8 lanes");
      unsigned long long mine = 0;
      for (int it = 0; it * kRowsThreads * U < nvt; ++it) {  // same trip count for every thread
        const int v0 = (it * kRowsThreads + tid) * U;
        unsigned long long fs = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int vi = v0 + u;
          if (vi < nvt) {
            float r[VEC];
            smem_draw_weights<T>(sp, qs, n_el, vi, dw, r);
            fs += dw.fix(seq_sum<VEC>(r));
          }
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
      __syncthreads();
      if (warp == 0) {
        warp_converged();
        const unsigned long long tot = warp_sum_u64(lane < kWarps ? sm.wu[lane] : 0ull);
        if (lane == 0) {
          sm.my[0] = static_cast<uint32_t>(tot);
          sm.my[1] = static_cast<uint32_t>(tot >> 32);
          sm.my[2] = sm.my[3] = 0u;
        }
        int code = -1;
        if (exchange(x, 4)) {
          warp_converged();
          const unsigned long long rc =
              lane < static_cast<int>(C)
                  ? (static_cast<unsigned long long>(xrec(x, lane, 0)) |
                     (static_cast<unsigned long long>(xrec(x, lane, 1)) << 32))
                  : 0ull;
          unsigned long long inc = rc;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += n;
          }
          const unsigned long long Rt = __shfl_sync(0xFFFFFFFFu, inc, 31);
          if (Rt == 0) {
            code = resid ? 1 : 2;
          } else {
            const unsigned long long tau = tau_of(ud, Rt);
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, lane < static_cast<int>(C) && tau < inc);
            const int owner = hit ? __ffs(hit) - 1 : -1;
            const unsigned long long before = owner >= 0 ? __shfl_sync(0xFFFFFFFFu, inc - rc, owner) : 0ull;
            if (owner < 0) {
              code = -1;  // cannot happen: tau < Rt
            } else if (owner == static_cast<int>(rank)) {
              code = 3;  // this CTA walks its slice
              if (lane == 0) {
                sm.wu[0] = tau - before;
                sm.wu[1] = Rt;
              }
            } else {
              code = 0;
            }
          }
        }
        if (lane == 0) sm.bi[0] = code;
      }
      __syncthreads();
      const int code = sm.bi[0];
      if (code != 3) return code;
      if (warp != 0) return 0;
      // ---- the owner's warp 0: a scan of the group sums (lane l takes a run
      // of consecutive groups), then the crossing group's vectors, then one
      // vector's elements, all from shared memory
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
          cnt = smem_draw_weights<T>(sp, qs, n_el, v, dw, r);
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
        const uint32_t sfin = found >= 0 ? (st_in | (near_b ? ST_NEAR : 0u)) : ST_TIMEOUT;
        dsmem_st_u32(dsmem_addr(&sm.out_tok, 0u), static_cast<uint32_t>(found));
        dsmem_st_u32(dsmem_addr(&sm.out_st, 0u), sfin);
      }
      return 0;
    };

    if (flags & 1u) {
      out = OUT_TIMEOUT;
    } else if (flags & 8u) {
      out = OUT_SKIP;
    } else {
      const int t = sm.t;
      const float u = sm.u;
      const WarpT wfp = make_warp(mp, sm.lo_p), wfq = make_warp(mq, sm.lo_q);
      uint32_t err = 0u;
      if (!bonus && (t < 0 || t >= P.V)) err = ST_BAD_TOKEN;
      bool p_bad = (flags & 2u) != 0u, q_bad = two && (flags & 4u) != 0u;
      if constexpr (MODE == MODE_LOGITS) {
        p_bad = p_bad || wfp.lo != wfp.lo;  // a NaN floor (an invalid filter parameter)
        q_bad = q_bad || (two && wfq.lo != wfq.lo);
      }
      bool have_exact = false, failed = false;
      double Zp_ex = 0.0, Zq_ex = 0.0;
      auto take_exact = [&]() {
        if (exact_pass(wfp, wfq)) {
          have_exact = true;
          Zp_ex = limbs_to_double(sm.lp);
          Zq_ex = two ? limbs_to_double(sm.lq) : 0.0;
        } else {
          failed = true;
        }
      };
      if constexpr (MODE == MODE_PROBS) {
        // a non-finite approximate mass means a +Inf element or an fp32
        // overflow of the partial sums: the exact pass tells them apart
        if (!err && !p_bad && !q_bad && (!(Zp.hi <= FLT_MAX) || (two && !(Zq.hi <= FLT_MAX)))) {
          take_exact();
          if (have_exact) {
            p_bad = p_bad || (sm.infl & 1u);
            q_bad = q_bad || (two && (sm.infl & 2u));
          }
        }
      }
      uint32_t st = 0u;
      if (!failed) {
        if (!err && p_bad) err = ST_BAD_VALUE;
        if (!err && q_bad) err = ST_BAD_VALUE;
        if (!err && !(u >= 0.f && u < 1.f)) err = ST_BAD_VALUE;
        const bool p_zero = MODE == MODE_PROBS ? (have_exact ? Zp_ex == 0.0 : Zp.hi == 0.f) : mp == -kInfF;
        const bool q_zero = MODE == MODE_PROBS ? (have_exact ? Zq_ex == 0.0 : Zq.hi == 0.f) : mq == -kInfF;
        out = OUT_TERM;
        o_n = i;
        o_next = -1;
        if (err) {
          o_st = err;
        } else if (p_zero) {
          o_st = ST_ZERO_MASS;
        } else if (!bonus && q_zero) {
          o_st = ST_ZERO_MASS;
        } else {
          if (!failed) {
            if (bonus) {
              out = OUT_DRAW;  // all K_b drafts accepted: the bonus comes from p_K
              o_n = kb;
            } else {
              const float pt = wfp(sm.gp), qt = wfq(sm.gq);
              int dec = have_exact ? -1 : filter_decide(u, pt, qt, Zp, Bp, Zq, Bq);
              if (!have_exact && ((P.flags & FLAG_FORCE_EXACT) || dec < 0)) take_exact();
              if (!failed) {
                if (have_exact) {
                  if (tid == 0) sm.bi[3] = exact_accept(u, pt, qt, sm.lp, sm.lq) ? 1 : 0;
                  __syncthreads();
                  dec = sm.bi[3];
                  st |= ST_EXACT;
                }
                out = dec ? OUT_ACCEPT : OUT_DRAW;
                o_st = st;
              }
            }
          }
        }
        if (!failed && (out == OUT_TERM || out == OUT_DRAW)) post_terminal();
      }
      if (failed) out = OUT_TIMEOUT;

      if (out == OUT_DRAW) {
        // ---- the bonus from p_K, or the residual after the rejection, with u_K
        const float ud = sm.ud;
        if (!bonus && !(ud >= 0.f && ud < 1.f)) {
          out = OUT_TERM;
          o_st = st | ST_BAD_VALUE;
        } else {
          DrawT dw;
          dw.scale = __uint_as_float(static_cast<uint32_t>(127 + P.fixed_shift) << 23);
          dw.resid = bonus ? 0 : 1;
          const float zp = have_exact ? static_cast<float>(Zp_ex) : Zp.hi;
          const float zq = bonus ? 1.f : (have_exact ? static_cast<float>(Zq_ex) : Zq.hi);
          if constexpr (MODE == MODE_LOGITS) {
            dw.k = khi;  // c = -m k - log2 Z, folded into one FMA per element
            const DF mk = two_prod(mp, khi), qk = two_prod(mq, khi);
            dw.cp = -__fadd_rn(mk.hi, __fadd_rn(mk.lo, log2f(zp)));
            dw.cq = bonus ? 0.f : -__fadd_rn(qk.hi, __fadd_rn(qk.lo, log2f(zq)));
            dw.lo_p = sm.lo_p;
            dw.lo_q = bonus ? -kInfF : sm.lo_q;
          } else {
            const double zpd = have_exact ? Zp_ex : static_cast<double>(zp);
            const double zqd = have_exact && !bonus ? Zq_ex : static_cast<double>(zq);
            norm_factors(zpd, dw.sp, dw.ap);
            norm_factors(zqd, dw.sq, dw.aq);
          }
          int code = draw(dw, !bonus, 3, st, ud);
          if (code == 1) {  // an empty residual: the draw falls back to p
            dw.resid = 0;
            st |= ST_ZERO_MASS;
            code = draw(dw, false, 4, st, ud);
          }
          if (code == 2) {
            out = OUT_TERM;
            o_st = st | ST_ZERO_MASS;
          } else if (code < 0) {
            out = OUT_TIMEOUT;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- record, count, combine
  if (bad && tid == 0) mbar_wait_bounded(&sm.full, 0u);  // no copy may land after exit
  __syncthreads();
  // Peers push records (and the draw's owner its id) into this CTA's shared
  // memory: every thread of the cluster meets here once before any CTA of
  // the cluster exits or rank 0 reads the drawn id.  (A fused-filter
  // sampling item has only rank 0 left here, with no exchange pending.)
  if (!(TOPK && sampling)) cluster_sync_all();
  if (rank == 0 && warp == 0) {
    uint4 rv = make_uint4(ST_TIMEOUT | kRecTerminal, 0xFFFFFFFFu, 0u, 0u);
    if (out == OUT_ACCEPT) {
      rv = make_uint4(o_st, 0u, 0u, 0u);
    } else if (out == OUT_TERM) {
      rv = make_uint4(o_st | kRecTerminal, static_cast<uint32_t>(o_next), static_cast<uint32_t>(o_n), 0u);
    } else if (out == OUT_DRAW && sm.out_tok != INT_MIN) {
      rv = make_uint4(sm.out_st | kRecTerminal, static_cast<uint32_t>(sm.out_tok), static_cast<uint32_t>(o_n), 0u);
    } else if (out == OUT_FALLBACK) {
      rv = make_uint4(kRecFallback, 0xFFFFFFFFu, 0u, 0u);
    }
    rows_record_combine(R, b, i, kb, t0, out != OUT_SKIP, rv);
  }
}

}  // namespace svk
