// The LM head in front of verification: logits = H . W^T on the 5th-
// generation tensor cores, and the verification from hidden states built on
// it (llmstudio.ru, "Как работает speculative decoding и MTP при инференсе
// LLM", sections 21-22).
//
// Work units of 256 x 256 logits (two 128-row slabs of states against one
// 256-row projection tile); one persistent CTA per SM, six warps:
//   warps 0-3  epilogue: wait for a unit's accumulators, read them out of
//              tensor memory (warp w owns TMEM lanes 32w..32w+31, the slabs'
//              rows), store them as fp32 rows and hand them back;
//   warp 4     producer: TMA loads of the two H slabs (128 x 64 each) and the
//              W tile (256 x 64) of every K step into a 3-stage ring,
//              128-byte swizzled;
//   warp 5     allocates 2 x 256 TMEM columns (one accumulator per slab), one
//              thread issues the MMAs (M = 128, N = 256, K = 16, bf16 x bf16
//              -> fp32) and commits each stage back to the producer, then
//              frees TMEM.
// Consecutive units share their W tile (all slab pairs of one W tile first),
// so the CTAs working on a W tile at the same time read it once from HBM.
// Every mbarrier wait is bounded; a wait that gives up sets bit 0 of *err.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "../../include/sv_lm_head.h"
#include "sv_host.h"
#include "sv_ptx.cuh"

namespace svl {

using svk::mbar_arrive_expect_tx;
using svk::mbar_init;
using svk::mbar_wait_bounded;
using svk::smem_u32;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB: one 128-row slab of states
constexpr int B_BYTES = BN * BK * 2;  // 32 KB: 256 projection rows
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;  // two slabs share the projection tile
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;  // one fp32 accumulator: 128 lanes x 256 columns

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5), A and B
// bf16 (bits 7-9, 10-12), both K-major (bits 15, 16 clear), N / 8 (bits
// 17-22), M / 16 (bits 24-28).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(BN) >> 3) << 17) |
                            ((uint32_t(BM) >> 4) << 24);
// The same with M = 64, for a slab that holds at most 64 rows: its results
// occupy lanes 0-15 of each 32-lane quarter of tensor memory (row r in lane
// 32 (r / 16) + r % 16), and the MMA does half the work.
constexpr uint32_t kIdesc64 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(BN) >> 3) << 17) |
                              ((64u >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 64 bf16 (128 bytes), 8-row groups 1024 bytes apart (stride byte
// offset), descriptor version 1 (bit 46), swizzle mode 2 (bits 61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrives on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

struct __align__(8) Bars {
  uint64_t full[STAGES];   // producer -> MMA: the stage's tiles landed
  uint64_t empty[STAGES];  // MMA -> producer: the stage's MMAs have read it
  uint64_t acc_full;       // MMA -> epilogue: both accumulators are final
  uint64_t acc_empty;      // epilogue -> MMA: both accumulators were read out
  uint32_t tmem;
  volatile int abort;      // a wait gave up: every role skips its remaining work
};

constexpr int kSmemBytes = STAGES * STAGE_BYTES + 1024 + static_cast<int>(sizeof(Bars));

// Two row blocks share the launch (the target states, then the draft
// states): 128-row slabs 0..mt0-1 come from map a0 and go to out0, the
// rest from a1 to out1.  A work unit is a pair of slabs (2p, 2p + 1; the
// second may not exist) against one 256-column projection tile: unit u is
// pair u % pairs, N tile u / pairs.
struct Args {
  int rows0, rows1, mt0, mt, pairs;
  int vocab, nk, units;
  long long ld;
  float* out0;
  float* out1;
  unsigned* err;
};

// Rows of slab sl that hold data (at most BM).
__device__ __forceinline__ int slab_rows(const Args& g, int sl) {
  const bool second = sl >= g.mt0;
  const int left = (second ? g.rows1 : g.rows0) - (second ? sl - g.mt0 : sl) * BM;
  return left < BM ? left : BM;
}

// A bounded wait that also gives up at once once another role has.
__device__ __forceinline__ bool wait_or_abort(Bars& bars, uint64_t* bar, uint32_t parity, unsigned* err) {
  if (bars.abort) return false;
  if (svk::mbar_wait_bounded(bar, parity)) return true;
  bars.abort = 1;
  atomicOr(err, 1u);
  return false;
}

// Persistent: CTA c takes units c, c + gridDim.x, ...  Each K step loads two
// 128-row slabs of states and one 256-row projection tile (64 KB) and issues
// two MMAs that share the projection tile, into two 256-column accumulators
// (all 512 TMEM columns): half the shared-memory bytes per FLOP of a single
// slab, so three stages keep twice the work in flight.  The producer streams
// ahead into the next unit while the epilogue drains the accumulators.
__global__ void __launch_bounds__(THREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                   const __grid_constant__ CUtensorMap w, Args g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // stage tiles on 1024-byte boundaries (the 128-byte swizzle's atom)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.acc_empty, 4);  // one arrival per epilogue warp
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {  // the whole warp allocates both accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem)),
                 "r"(2 * TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = bars.tmem;

  if (warp == 4) {
    // ---- producer: one thread, every K step of every unit of this CTA
    if (lane == 0) {
      int gk = 0;  // K steps issued so far (stage gk % STAGES, use gk / STAGES)
      for (int u = blockIdx.x; u < g.units && !bars.abort; u += gridDim.x) {
        const int p = u % g.pairs, n0 = (u / g.pairs) * BN;
        const bool two = 2 * p + 1 < g.mt;
        const CUtensorMap* map[2];
        int m0[2];
        for (int h = 0; h < 2; ++h) {
          const int sl = 2 * p + h;
          const bool second = sl >= g.mt0;
          map[h] = second ? &a1 : &a0;
          m0[h] = (second ? sl - g.mt0 : sl) * BM;
        }
        for (int ks = 0; ks < g.nk; ++ks, ++gk) {
          const int s = gk % STAGES;
          if (gk >= STAGES && !wait_or_abort(bars, &bars.empty[s], ((gk / STAGES) - 1) & 1, g.err)) break;
          const uint32_t a = smem_u32(smem + s * STAGE_BYTES), b = a + 2 * A_BYTES;
          mbar_arrive_expect_tx(&bars.full[s], two ? STAGE_BYTES : STAGE_BYTES - A_BYTES);
          tma_load_2d(a, map[0], ks * BK, m0[0], &bars.full[s]);
          if (two) tma_load_2d(a + A_BYTES, map[1], ks * BK, m0[1], &bars.full[s]);
          tma_load_2d(b, &w, ks * BK, n0, &bars.full[s]);
        }
      }
      // no copy may still be writing shared memory at exit: the last load of
      // every stage has landed (the MMA thread normally saw it already)
      for (int k = gk - STAGES > 0 ? gk - STAGES : 0; k < gk; ++k)
        if (!svk::mbar_wait_bounded(&bars.full[k % STAGES], (k / STAGES) & 1)) atomicOr(g.err, 1u);
    }
  } else if (warp == 5) {
    // ---- MMA: one thread issues, the tensor core accumulates in TMEM
    if (lane == 0) {
      int gk = 0, j = 0;
      for (int u = blockIdx.x; u < g.units && !bars.abort; u += gridDim.x, ++j) {
        const int p0 = 2 * (u % g.pairs);
        const bool two = p0 + 1 < g.mt;
        const uint32_t id0 = slab_rows(g, p0) <= 64 ? kIdesc64 : kIdesc;
        const uint32_t id1 = two && slab_rows(g, p0 + 1) <= 64 ? kIdesc64 : kIdesc;
        if (j >= 1 && !wait_or_abort(bars, &bars.acc_empty, (j - 1) & 1, g.err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        bool ok = true;
        for (int ks = 0; ks < g.nk; ++ks, ++gk) {
          const int s = gk % STAGES;
          if (!wait_or_abort(bars, &bars.full[s], (gk / STAGES) & 1, g.err)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a = smem_u32(smem + s * STAGE_BYTES), b = a + 2 * A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {  // K = 16 per MMA: 32 bytes along the swizzled rows
            const uint64_t bd = desc_sw128(b + kk * 32);
            const uint32_t first = (ks | kk) ? 1u : 0u;
            mma_bf16(tmem, desc_sw128(a + kk * 32), bd, id0, first);
            if (two) mma_bf16(tmem + TMEM_COLS, desc_sw128(a + A_BYTES + kk * 32), bd, id1, first);
          }
          mma_commit(&bars.empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(&bars.acc_full);  // the accumulators are final once every MMA issued so far is
        if (!ok) break;
      }
    }
  } else {
    // ---- epilogue: warp w holds rows 32 w + lane of each slab
    int j = 0;
    for (int u = blockIdx.x; u < g.units; u += gridDim.x, ++j) {
      if (!wait_or_abort(bars, &bars.acc_full, j & 1, g.err)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int p = u % g.pairs, n0 = (u / g.pairs) * BN;
      for (int h = 0; h < 2; ++h) {
        const int sl = 2 * p + h;
        if (sl >= g.mt) break;
        const bool second = sl >= g.mt0;
        const bool m64 = slab_rows(g, sl) <= 64;  // rows in lanes 0-15 of each quarter
        const int row = (second ? sl - g.mt0 : sl) * BM + (m64 ? (lane < 16 ? warp * 16 + lane : BM) : warp * 32 + lane);
        const int rows = second ? g.rows1 : g.rows0;
        float* dst_row = (second ? g.out1 : g.out0) + static_cast<long long>(row) * g.ld;
        const uint32_t acc =
            tmem + static_cast<uint32_t>(h) * TMEM_COLS + (static_cast<uint32_t>(warp * 32) << 16);
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(acc + static_cast<uint32_t>(c * 32), v);
          const int col = n0 + c * 32;
          if (row < rows && col < g.vocab) {
            if (col + 32 <= g.vocab) {
              float4* d4 = reinterpret_cast<float4*>(dst_row + col);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
#pragma unroll
              for (int q = 0; q < 32; ++q)
                if (col + q < g.vocab) dst_row[col + q] = v[q];
            }
          }
        }
      }
      // this warp's reads are complete: hand the accumulators back to the MMAs
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) svk::mbar_arrive_local(&bars.acc_empty);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * TMEM_COLS)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A [rows, dim] bf16 row-major matrix as a 2-D tensor map with boxes of
// `box_rows` x 64 (128-byte rows, 128-byte swizzle); out-of-range boxes read 0.
bool encode(CUtensorMap* map, const void* base, int rows, int dim, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(dim) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One launch: rows0 rows of s0 into out0 and rows1 rows of s1 into out1
// (rows1 may be 0), every row `ld` floats apart.
sv_status launch(const void* s0, int rows0, const void* s1, int rows1, const void* proj, int vocab, int dim,
                 float* out0, float* out1, long long ld, unsigned* err, cudaStream_t stream) {
  if (!encoder()) return svh::fail(SV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  CUtensorMap m0, m1, mw;
  if (!encode(&m0, s0, rows0, dim, BM) || !encode(&mw, proj, vocab, dim, BN) ||
      !encode(&m1, rows1 ? s1 : s0, rows1 ? rows1 : rows0, dim, BM))
    return svh::fail(SV_ERR_ARG, "tensor map encoding failed (alignment or size)");
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set[dev] = true;
  }
  Args g;
  g.rows0 = rows0;
  g.rows1 = rows1;
  g.mt0 = (rows0 + BM - 1) / BM;
  g.mt = g.mt0 + (rows1 + BM - 1) / BM;
  g.pairs = (g.mt + 1) / 2;
  g.vocab = vocab;
  g.nk = (dim + BK - 1) / BK;
  const long long tiles = static_cast<long long>(g.pairs) * ((vocab + BN - 1) / BN);
  if (tiles > 0x7FFFFFFFLL) return svh::fail(SV_ERR_UNSUPPORTED, "too many tiles");
  g.units = static_cast<int>(tiles);
  g.ld = ld;
  g.out0 = out0;
  g.out1 = out1;
  g.err = err;
  // one CTA per SM (the ring takes most of its shared memory), each walking tiles
  static int sms[64] = {0};
  if (!sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    sms[dev] = n;
  }
  const unsigned grid = static_cast<unsigned>(tiles < sms[dev] ? tiles : sms[dev]);
  lm_head_kernel<<<grid, THREADS, kSmemBytes, stream>>>(m0, m1, mw, g);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

}  // namespace svl

extern "C" {

sv_status sv_lm_head_logits(const void* states, const void* proj, int32_t rows, int32_t vocab, int32_t dim,
                            float* logits, int64_t ld, uint32_t* err, void* stream) {
  svh::clear_error();
  if (rows < 0 || vocab < 1 || dim < 1) return svh::fail(SV_ERR_ARG, "rows, vocab, dim out of range");
  if (dim % 8) return svh::fail(SV_ERR_ARG, "dim (%d) must be a multiple of 8", dim);
  if (ld < vocab || ld % 4) return svh::fail(SV_ERR_ARG, "ld (%lld) must be >= vocab and a multiple of 4", (long long)ld);
  if (static_cast<long long>(vocab + svl::BN - 1) / svl::BN > 65535)
    return svh::fail(SV_ERR_UNSUPPORTED, "vocab %d too large", vocab);
  if (rows == 0) return SV_OK;
  if (!states || !proj || !logits) return svh::fail(SV_ERR_ARG, "a pointer is NULL");
  if (!svl::aligned16(states) || !svl::aligned16(proj) || !svl::aligned16(logits))
    return svh::fail(SV_ERR_ARG, "states, proj and logits must be 16-byte aligned");
  return svl::launch(states, rows, nullptr, 0, proj, vocab, dim, logits, nullptr, ld, err,
                     static_cast<cudaStream_t>(stream));
}

size_t sv_lm_head_workspace_size(int32_t batch, int32_t sum_k, int32_t vocab) {
  if (batch < 0 || sum_k < 0 || vocab < 1) return 0;
  const size_t ldv = (static_cast<size_t>(vocab) + 3) / 4 * 4;
  return 256 + (2 * static_cast<size_t>(sum_k) + batch) * ldv * 4;
}

sv_status sv_lm_head_verify(const void* target_states, const void* draft_states, const void* proj, int32_t dim,
                            const float* temperature, const int32_t* draft_tokens, const float* uniforms,
                            const int32_t* cu_k, int32_t batch, int32_t k, int32_t sum_k, int32_t vocab,
                            int32_t* n_accepted, int32_t* next_token, uint32_t* status, void* workspace,
                            size_t workspace_bytes, uint32_t flags, void* stream) {
  svh::clear_error();
  if (batch < 0 || sum_k < 0 || vocab < 1 || dim < 1) return svh::fail(SV_ERR_ARG, "size out of range");
  if (batch == 0) return SV_OK;
  if (dim % 8) return svh::fail(SV_ERR_ARG, "dim (%d) must be a multiple of 8", dim);
  if (static_cast<long long>(vocab + svl::BN - 1) / svl::BN > 65535)
    return svh::fail(SV_ERR_UNSUPPORTED, "vocab %d too large", vocab);
  if (static_cast<long long>(sum_k) + batch > 0x7FFFFFFFLL) return svh::fail(SV_ERR_ARG, "too many rows");
  if (!target_states || (sum_k > 0 && !draft_states) || !proj)
    return svh::fail(SV_ERR_ARG, "a states or proj pointer is NULL");
  if (!svl::aligned16(target_states) || (sum_k > 0 && !svl::aligned16(draft_states)) || !svl::aligned16(proj))
    return svh::fail(SV_ERR_ARG, "states and proj must be 16-byte aligned");
  const size_t need = sv_lm_head_workspace_size(batch, sum_k, vocab);
  if (!workspace || workspace_bytes < need)
    return svh::fail(SV_ERR_ARG, "workspace_bytes (%zu) < the %zu bytes sv_lm_head_workspace_size() asks for",
                     workspace_bytes, need);
  if (!svl::aligned16(workspace)) return svh::fail(SV_ERR_ARG, "workspace must be 16-byte aligned");
  const long long ldv = (static_cast<long long>(vocab) + 3) / 4 * 4;
  const int t_rows = sum_k + batch;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  float* lt = reinterpret_cast<float*>(ws + 256);
  float* ld = lt + static_cast<size_t>(t_rows) * ldv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the host-side checks of the verification first, so that nothing is
  // enqueued when they fail (a zero batch of the same arguments enqueues nothing)
  sv_status s = svh::accept_logits(lt, ld, SV_F32, ldv, temperature, draft_tokens, uniforms, cu_k, 0, k, 0,
                                   vocab, nullptr, nullptr, n_accepted, next_token, status, nullptr, nullptr,
                                   nullptr, flags, stream);
  if (s != SV_OK) return s;
  if (!cu_k && static_cast<long long>(batch) * k != sum_k)
    return svh::fail(SV_ERR_ARG, "without cu_k, sum_k must equal batch * k");
  if (!temperature || !uniforms || (sum_k > 0 && !draft_tokens) || !n_accepted || !next_token || !status)
    return svh::fail(SV_ERR_ARG, "a verification pointer is NULL");
  const cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return svh::fail(SV_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  s = svl::launch(target_states, t_rows, draft_states, sum_k, proj, vocab, dim, lt, ld, ldv, err, st);
  if (s != SV_OK) return s;
  return svh::accept_logits(lt, ld, SV_F32, ldv, temperature, draft_tokens, uniforms, cu_k, batch, k, sum_k,
                            vocab, nullptr, nullptr, n_accepted, next_token, status, nullptr, nullptr, err, flags,
                            stream);
}

}  // extern "C"
