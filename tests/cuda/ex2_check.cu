// Measures the relative error of ex2.approx.ftz.f32 (the special-function
// unit's 2^x, used by the logits warp) against CUDA's double-precision exp2,
// on EVERY f32 argument in [-126, 0]: all bit patterns from -0 (0x80000000)
// to -126 (0xC2FC0000), and +0.  Test helper only.
#include <cuda_runtime.h>
#include <cstdint>

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

constexpr unsigned kFirst = 0x80000000u;        // -0
constexpr unsigned kLast = 0xC2FC0000u;         // -126
constexpr unsigned long long kCount = kLast - kFirst + 2ull;  // + the +0 argument

// worst[0]: the largest relative error (as ordered bits of a non-negative
// double), worst[1]: the argument's bits.
__global__ void ex2_err_kernel(unsigned long long* worst) {
  double mine = 0.0;
  unsigned arg = 0;
  const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
  for (unsigned long long i = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x; i < kCount;
       i += stride) {
    const unsigned bits = i + 1 == kCount ? 0u : kFirst + static_cast<unsigned>(i);
    const float x = __uint_as_float(bits);
    const double ref = exp2(static_cast<double>(x));
    const double rel = fabs(static_cast<double>(ex2_approx(x)) - ref) / ref;
    if (rel > mine) {
      mine = rel;
      arg = bits;
    }
  }
  // non-negative doubles order like their bit patterns
  const unsigned long long key = static_cast<unsigned long long>(__double_as_longlong(mine));
  const unsigned long long prev = atomicMax(worst, key);
  if (key > prev) atomicExch(worst + 1, static_cast<unsigned long long>(arg));
}

// out[0] = the largest relative error, out[1] = its argument, out[2] = the
// number of arguments checked.
extern "C" int ex2_max_rel_err(double* out) {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(*d)) != cudaSuccess) return 1;
  cudaMemset(d, 0, 2 * sizeof(*d));
  ex2_err_kernel<<<152 * 8, 256>>>(d);
  unsigned long long h[2] = {0, 0};
  const cudaError_t e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return 2;
  double v;
  static_assert(sizeof(v) == sizeof(h[0]), "");
  __builtin_memcpy(&v, &h[0], sizeof(v));
  float a;
  const unsigned ab = static_cast<unsigned>(h[1]);
  __builtin_memcpy(&a, &ab, sizeof(a));
  out[0] = v;
  out[1] = a;
  out[2] = static_cast<double>(kCount);
  return 0;
}
