// Host side of the row-parallel plan (sv_rows.cuh): its shape rule, the
// device scratch its items count themselves into, and the launch.
//
// The scratch (per sequence an arrival counter and the first terminal row
// posted, per target row a 16-byte record) lives in file-scope device arrays
// that the module reserves once, zeroed; the last item of every sequence puts
// its words back to zero, so no call clears or allocates anything and a CUDA
// graph may capture the launch.  Launches that use one scratch slot must not
// overlap in time, so every stream gets a slot of its own (stream order then
// serialises the launches that share it); a call on a stream beyond the
// slots, or larger than a slot, takes the chain plan.
#include <cuda_runtime.h>

#include <mutex>

#include "sv_host.h"
#include "sv_rows.cuh"

namespace {

using svh::fail;

constexpr int kSlots = 4;
constexpr int kMaxSeq = 1 << 16;   // sequences per launch
constexpr int kMaxRows = 1 << 18;  // target rows per launch (sum_k + B)

static __device__ int g_count[kSlots][kMaxSeq];
static __device__ int g_first[kSlots][kMaxSeq];
static __device__ uint4 g_rec[kSlots][kMaxRows];
// the filtered verification: per sequence the fallback flag, per row the floor
static __device__ int g_flag[kSlots][kMaxSeq];
static __device__ float g_floor[kSlots][2][kMaxRows];

struct Slot {
  bool used;
  cudaStream_t stream;
  int* count;
  int* first;
  uint4* rec;
  int* flag;
  float* floor_t;
  float* floor_d;
};

std::mutex g_slot_mutex;
Slot g_slot[64][kSlots] = {};

// The scratch slot of `stream` on the current device (assigned on first use);
// false when every slot belongs to another stream or a lookup fails.
bool slot_for(cudaStream_t stream, Slot& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(g_slot_mutex);
  Slot* free_slot = nullptr;
  int free_idx = -1;
  for (int s = 0; s < kSlots; ++s) {
    Slot& sl = g_slot[dev][s];
    if (sl.used && sl.stream == stream) {
      out = sl;
      return true;
    }
    if (!sl.used && !free_slot) {
      free_slot = &sl;
      free_idx = s;
    }
  }
  if (!free_slot) return false;
  void *pc = nullptr, *pf = nullptr, *pr = nullptr, *pg = nullptr, *pl = nullptr;
  if (cudaGetSymbolAddress(&pc, g_count) != cudaSuccess || cudaGetSymbolAddress(&pf, g_first) != cudaSuccess ||
      cudaGetSymbolAddress(&pr, g_rec) != cudaSuccess || cudaGetSymbolAddress(&pg, g_flag) != cudaSuccess ||
      cudaGetSymbolAddress(&pl, g_floor) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  free_slot->used = true;
  free_slot->stream = stream;
  free_slot->count = static_cast<int*>(pc) + static_cast<size_t>(free_idx) * kMaxSeq;
  free_slot->first = static_cast<int*>(pf) + static_cast<size_t>(free_idx) * kMaxSeq;
  free_slot->rec = static_cast<uint4*>(pr) + static_cast<size_t>(free_idx) * kMaxRows;
  free_slot->flag = static_cast<int*>(pg) + static_cast<size_t>(free_idx) * kMaxSeq;
  free_slot->floor_t = static_cast<float*>(pl) + static_cast<size_t>(free_idx) * 2 * kMaxRows;
  free_slot->floor_d = free_slot->floor_t + kMaxRows;
  out = *free_slot;
  return true;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bytes of one row slice per CTA: two slices (target and draft) of 32 KB,
// or one greedy slice of 64 KB, leave room for three CTAs per SM.
constexpr long long kSampleSliceBytes = 32768;
constexpr long long kGreedySliceBytes = 65536;
constexpr size_t kSmemPerSM = 227 * 1024;

struct RowsPlan {
  int C, slice, nadd, x_off, vsum_off, tail_off;
  size_t smem;
};

// topk: the fused filters' plan (16-bit rows): room for the candidate lists
// and the radix histogram beside the draw sums, and for rank 0's receive area
// and work space inside the row slices.
bool rows_plan(bool sampling, int V, int elem, RowsPlan& p, bool topk = false) {
  const int vec = 16 / elem;
  const long long row_bytes = static_cast<long long>(V) * elem;
  const long long cap = sampling ? kSampleSliceBytes : kGreedySliceBytes;
  long long C = (row_bytes + cap - 1) / cap;
  if (C < 1) C = 1;
  if (C > svk::kMaxCluster) return false;
  long long slice = (V + C - 1) / C;
  slice = (slice + vec - 1) / vec * vec;
  p.C = static_cast<int>((V + slice - 1) / slice);
  p.slice = static_cast<int>(slice);
  const size_t sbytes = round_up(static_cast<size_t>(slice) * elem, 128);
  p.x_off = static_cast<int>(sbytes);
  const size_t rows = sampling ? 2 * sbytes : sbytes;
  const long long nvt = (slice + vec - 1) / vec;
  size_t vs = static_cast<size_t>((nvt + svk::kGroupVecs - 1) / svk::kGroupVecs) * 8;
  if (vs < 2 * svk::kBuckets * 8) vs = 2 * svk::kBuckets * 8;
  if (topk) {
    // lists [2][kListCap], histograms [2][256], 16 scalars
    if (vs < static_cast<size_t>(2 * svk::kListCap * 8 + 2048 + 64)) vs = 2 * svk::kListCap * 8 + 2048 + 64;
    const size_t recv = 256 + static_cast<size_t>(p.C) * 2 * svk::kListCap * 8 + svk::kTopkScratch;
    if (!sampling || recv > rows) return false;
  }
  p.vsum_off = static_cast<int>(rows);
  p.tail_off = static_cast<int>(round_up(rows + vs, 128));
  p.smem = p.tail_off + sizeof(svk::RowsTail);
  // fp32 additions of an element inside its thread: one per vector the
  // thread sums, one for a tail element, and the vector's pairwise tree
  int lg = 0;
  while ((1 << lg) < vec) ++lg;
  p.nadd = static_cast<int>((slice / vec + svk::kRowsThreads - 1) / svk::kRowsThreads) + 1 + lg;
  return p.smem <= kSmemPerSM;
}

struct Cache {
  size_t smem_set;
  bool cluster16;
  unsigned fits_mask;
  size_t smem_fit[svk::kMaxCluster + 1];
};

template <int MODE, typename T, bool FL, bool TOPK = false>
Cache& cache_of(int dev) {
  static Cache c[64] = {};
  return c[dev >= 0 && dev < 64 ? dev : 0];
}

template <int MODE, typename T, bool FL, bool TOPK = false>
sv_status launch_t(svk::RowsParams rp, const RowsPlan& pl, long long blocks, cudaStream_t stream) {
  auto kern = svk::sv_rows_kernel<MODE, T, FL, TOPK>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  Cache& kc = cache_of<MODE, T, FL, TOPK>(dev);
  cudaError_t e;
  if (kc.smem_set < pl.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.smem));
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "cudaFuncSetAttribute(smem, rows): %s", cudaGetErrorString(e));
    kc.smem_set = pl.smem;
  }
  if (pl.C > 8 && !kc.cluster16) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
      return fail(SV_ERR_CUDA, "cudaFuncSetAttribute(cluster, rows): %s", cudaGetErrorString(e));
    kc.cluster16 = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(svk::kRowsThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned bit = 1u << pl.C;
  if (!(kc.fits_mask & bit) || kc.smem_fit[pl.C] < pl.smem) {
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess)
      return fail(SV_ERR_CUDA, "cudaOccupancyMaxActiveClusters(rows): %s", cudaGetErrorString(e));
    if (clusters < 1)
      return fail(SV_ERR_UNSUPPORTED, "no cluster of %d CTAs with %zu B shared memory fits", pl.C, pl.smem);
    kc.fits_mask |= bit;
    kc.smem_fit[pl.C] = pl.smem;
  }
  e = cudaLaunchKernelEx(&cfg, kern, rp);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "rows kernel launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

template <int MODE, typename T>
sv_status launch_m(svk::RowsParams rp, const RowsPlan& pl, long long blocks, bool filtered, cudaStream_t st) {
  if constexpr (MODE == svk::MODE_LOGITS) {
    if (filtered) return launch_t<MODE, T, true>(rp, pl, blocks, st);
  }
  return launch_t<MODE, T, false>(rp, pl, blocks, st);
}

}  // namespace

int svh::rows_cluster_size(int mode, int elem, const svk::Params& p) {
  RowsPlan pl;
  if (p.B < 1 || p.B > kMaxSeq) return 0;
  if (static_cast<long long>(p.sum_k) + p.B > kMaxRows) return 0;
  if (p.wt_out || p.wd_out) return 0;  // the warped-row outputs come from the chain plan
  if (!rows_plan(mode != svk::MODE_GREEDY, p.V, elem, pl)) return 0;
  const long long blocks = static_cast<long long>(pl.C) * p.B * (p.K + 1LL);
  return blocks <= 0x7FFFFFFFLL ? pl.C : 0;
}

sv_status svh::launch_rows(int mode, sv_dtype dtype, const svk::Params& p, bool filtered, cudaStream_t stream) {
  const int elem = dtype == SV_F32 ? 4 : 2;
  RowsPlan pl;
  // greedy items of a logits batch hold only their target row, but share
  // the sampling items' launch shape
  if (!rows_plan(mode != svk::MODE_GREEDY, p.V, elem, pl))
    return fail(SV_ERR_UNSUPPORTED, "row-parallel plan: vocab %d too large", p.V);
  Slot sl;
  if (!slot_for(stream, sl)) return fail(SV_ERR_UNSUPPORTED, "row-parallel plan: no scratch slot for this stream");
  svk::RowsParams rp;
  rp.p = p;
  rp.p.slice = pl.slice;
  rp.seq_count = sl.count;
  rp.seq_first = sl.first;
  rp.rec = sl.rec;
  rp.seq_flag = nullptr;
  rp.top_k = nullptr;
  rp.top_p = nullptr;
  rp.nadd = pl.nadd;
  rp.x_off = pl.x_off;
  rp.vsum_off = pl.vsum_off;
  rp.tail_off = pl.tail_off;
  const long long blocks = static_cast<long long>(pl.C) * p.B * (p.K + 1LL);
  switch (mode) {
    case svk::MODE_GREEDY:
      if (dtype == SV_F32) return launch_m<svk::MODE_GREEDY, float>(rp, pl, blocks, false, stream);
      if (dtype == SV_BF16) return launch_m<svk::MODE_GREEDY, __nv_bfloat16>(rp, pl, blocks, false, stream);
      return launch_m<svk::MODE_GREEDY, __half>(rp, pl, blocks, false, stream);
    case svk::MODE_PROBS:
      return launch_m<svk::MODE_PROBS, float>(rp, pl, blocks, false, stream);
    default:
      if (dtype == SV_F32) return launch_m<svk::MODE_LOGITS, float>(rp, pl, blocks, filtered, stream);
      if (dtype == SV_BF16) return launch_m<svk::MODE_LOGITS, __nv_bfloat16>(rp, pl, blocks, filtered, stream);
      return launch_m<svk::MODE_LOGITS, __half>(rp, pl, blocks, filtered, stream);
  }
}

bool svh::rows_filter_scratch(cudaStream_t stream, int batch, int t_rows, int** flag, float** floor_t,
                              float** floor_d) {
  if (batch < 0 || batch > kMaxSeq || t_rows < 0 || t_rows > kMaxRows) return false;
  Slot sl;
  if (!slot_for(stream, sl)) return false;
  *flag = sl.flag;
  *floor_t = sl.floor_t;
  *floor_d = sl.floor_d;
  return true;
}

sv_status svh::launch_rows_topk(sv_dtype dtype, const svk::Params& p, const int32_t* top_k, const float* top_p,
                                cudaStream_t stream) {
  if (dtype == SV_F32 || !top_k) return fail(SV_ERR_UNSUPPORTED, "fused filters: 16-bit logits with top-k only");
  if (p.B < 1 || p.B > kMaxSeq || static_cast<long long>(p.sum_k) + p.B > kMaxRows || p.wt_out || p.wd_out)
    return fail(SV_ERR_UNSUPPORTED, "fused filters: shape beyond the scratch");
  RowsPlan pl;
  if (!rows_plan(true, p.V, 2, pl, true)) return fail(SV_ERR_UNSUPPORTED, "fused filters: vocab %d", p.V);
  const long long blocks = static_cast<long long>(pl.C) * p.B * (p.K + 1LL);
  if (blocks > 0x7FFFFFFFLL) return fail(SV_ERR_UNSUPPORTED, "fused filters: too many rows");
  Slot sl;
  if (!slot_for(stream, sl)) return fail(SV_ERR_UNSUPPORTED, "fused filters: no scratch slot for this stream");
  svk::RowsParams rp;
  rp.p = p;
  rp.p.slice = pl.slice;
  rp.seq_count = sl.count;
  rp.seq_first = sl.first;
  rp.rec = sl.rec;
  rp.seq_flag = sl.flag;
  rp.top_k = top_k;
  rp.top_p = top_p;
  rp.nadd = pl.nadd;
  rp.x_off = pl.x_off;
  rp.vsum_off = pl.vsum_off;
  rp.tail_off = pl.tail_off;
  if (dtype == SV_BF16) return launch_t<svk::MODE_LOGITS, __nv_bfloat16, true, true>(rp, pl, blocks, stream);
  return launch_t<svk::MODE_LOGITS, __half, true, true>(rp, pl, blocks, stream);
}
