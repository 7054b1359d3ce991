// The LM head in front of verification: logits = H . W^T on the 5th-
// generation tensor cores, and the verification from hidden states built on
// it (llmstudio.ru, "Как работает speculative decoding и MTP при инференсе
// LLM", sections 21-22).
//
// One CTA per 128 x 256 tile of logits, six warps:
//   warps 0-3  epilogue: wait for the accumulator, read it out of tensor
//              memory (warp w owns TMEM lanes 32w..32w+31, the tile's rows)
//              and store it as fp32 rows;
//   warp 4     producer: TMA loads of the H (128 x 64) and W (256 x 64) tiles
//              of every K step into a 4-stage ring, 128-byte swizzled;
//   warp 5     allocates 256 TMEM columns, one thread issues the MMAs
//              (M = 128, N = 256, K = 16, bf16 x bf16 -> fp32) and commits
//              each stage back to the producer, then frees TMEM.
// The grid walks the M tiles of one N tile together (blockIdx.x), so the
// CTAs that share a W tile run at the same time and read it once from HBM.
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

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;  // the fp32 accumulator: 128 lanes x 256 columns

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5), A and B
// bf16 (bits 7-9, 10-12), both K-major (bits 15, 16 clear), N / 8 (bits
// 17-22), M / 16 (bits 24-28).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(BN) >> 3) << 17) |
                            ((uint32_t(BM) >> 4) << 24);

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

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc)
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
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc;
  uint32_t tmem;
};

constexpr int kSmemBytes = STAGES * STAGE_BYTES + 1024 + static_cast<int>(sizeof(Bars));

// Two row blocks share the launch (the target states, then the draft
// states): M tiles 0..mt0-1 read map a0 and write out0, the rest a1 / out1.
struct Args {
  int rows0, rows1, mt0;
  int vocab, nk;
  long long ld;
  float* out0;
  float* out1;
  unsigned* err;
};

__global__ void __launch_bounds__(THREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                   const __grid_constant__ CUtensorMap w, Args g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // stage tiles on 1024-byte boundaries (the 128-byte swizzle's atom)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool second = static_cast<int>(blockIdx.x) >= g.mt0;
  const int m0 = (second ? static_cast<int>(blockIdx.x) - g.mt0 : static_cast<int>(blockIdx.x)) * BM;
  const int n0 = static_cast<int>(blockIdx.y) * BN;
  const CUtensorMap* amap = second ? &a1 : &a0;
  const int rows = second ? g.rows1 : g.rows0;
  float* out = second ? g.out1 : g.out0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.acc, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {  // the whole warp allocates
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = bars.tmem;

  if (warp == 4) {
    if (lane == 0) {
      int issued = 0;
      for (int ks = 0; ks < g.nk; ++ks) {
        const int s = ks % STAGES;
        if (ks >= STAGES && !mbar_wait_bounded(&bars.empty[s], ((ks / STAGES) - 1) & 1)) {
          atomicOr(g.err, 1u);
          break;
        }
        const uint32_t a = smem_u32(smem + s * STAGE_BYTES), b = a + A_BYTES;
        mbar_arrive_expect_tx(&bars.full[s], STAGE_BYTES);
        tma_load_2d(a, amap, ks * BK, m0, &bars.full[s]);
        tma_load_2d(b, &w, ks * BK, n0, &bars.full[s]);
        ++issued;
      }
      // no copy may still be writing shared memory at exit: the last loads
      // of every stage have landed (the MMA warp normally saw them already)
      for (int ks = issued - STAGES > 0 ? issued - STAGES : 0; ks < issued; ++ks)
        if (!mbar_wait_bounded(&bars.full[ks % STAGES], (ks / STAGES) & 1)) atomicOr(g.err, 1u);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      for (int ks = 0; ks < g.nk; ++ks) {
        const int s = ks % STAGES;
        if (!mbar_wait_bounded(&bars.full[s], (ks / STAGES) & 1)) {
          atomicOr(g.err, 1u);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a = smem_u32(smem + s * STAGE_BYTES), b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled rows
          mma_bf16(tmem, desc_sw128(a + kk * 32), desc_sw128(b + kk * 32), (ks | kk) ? 1u : 0u);
        mma_commit(&bars.empty[s]);  // the stage is free once these MMAs have read it
      }
      mma_commit(&bars.acc);  // the accumulator is final once every MMA issued so far is
    }
  } else {
    // epilogue: warp w holds rows m0 + 32 w + lane
    if (!mbar_wait_bounded(&bars.acc, 0)) {
      if (lane == 0) atomicOr(g.err, 1u);
    } else {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int row = m0 + warp * 32 + lane;
      float* dst_row = out + static_cast<long long>(row) * g.ld;
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(c * 32), v);
        const int col = n0 + c * 32;
        if (row < rows && col < g.vocab) {
          if (col + 32 <= g.vocab) {
            float4* d4 = reinterpret_cast<float4*>(dst_row + col);
#pragma unroll
            for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col + j < g.vocab) dst_row[col + j] = v[j];
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
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
  g.vocab = vocab;
  g.nk = (dim + BK - 1) / BK;
  g.ld = ld;
  g.out0 = out0;
  g.out1 = out1;
  g.err = err;
  const dim3 grid(static_cast<unsigned>(g.mt0 + (rows1 + BM - 1) / BM), static_cast<unsigned>((vocab + BN - 1) / BN));
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
