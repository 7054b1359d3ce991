// Measures the relative error of ex2.approx.ftz.f32 (the special-function
// unit's 2^x, used by the logits warp) against CUDA's double-precision exp2,
// over a sample of arguments in [-126, 0].  Test helper only.
#include <cuda_runtime.h>
#include <cstdint>

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__global__ void ex2_err_kernel(unsigned long long n, unsigned long long* worst_bits) {
  const unsigned long long i = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
  if (i >= n) return;
  // two sweeps: [-126, 0] uniformly, and [-1, 0] densely
  const double frac = static_cast<double>(i >> 1) / static_cast<double>(n >> 1);
  const float x = (i & 1) ? static_cast<float>(-126.0 * frac) : static_cast<float>(-frac);
  const double ref = exp2(static_cast<double>(x));
  const double got = static_cast<double>(ex2_approx(x));
  const double rel = fabs(got - ref) / ref;
  // non-negative doubles order like their bit patterns
  atomicMax(worst_bits, static_cast<unsigned long long>(__double_as_longlong(rel)));
}

extern "C" int ex2_max_rel_err(unsigned long long n, double* out) {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, sizeof(*d)) != cudaSuccess) return 1;
  cudaMemset(d, 0, sizeof(*d));
  const unsigned threads = 256;
  ex2_err_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads>>>(n, d);
  unsigned long long bits = 0;
  const cudaError_t e = cudaMemcpy(&bits, d, sizeof(bits), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return 2;
  double v;
  static_assert(sizeof(v) == sizeof(bits), "");
  __builtin_memcpy(&v, &bits, sizeof(v));
  *out = v;
  return 0;
}
