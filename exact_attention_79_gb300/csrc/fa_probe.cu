// Throughput of the exponential instruction the softmax runs (ex2.approx),
// measured on the device at hand: the second ceiling of the forward besides
// the tensor cores. The forward takes one exponential per 4 d of its
// floating-point operations, and work off the matrix units runs at a small
// fraction of their rate ("FlashAttention v2相比于v1有哪些更新", sections 2
// and 3, "CUDA Core vs. Tensor Core": up to 16 times lower), so at small d
// the exponentials can bound it.
//
// One CTA per SM, 512 threads (four warps per scheduler), each running eight
// independent chains x <- 2^-x, which stay in (0, 1]. Every CTA records the
// cycles between two block barriers around the loop; there are no waits on
// anything but those barriers.
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

__device__ unsigned long long g_ex2_cycles[kEx2MaxSms];
__device__ float g_ex2_sink;

__global__ void __launch_bounds__(kEx2Threads, 1) ex2_rate_kernel(int iters) {
  __syncthreads();
  const long long t0 = clock64();
  // start values that the compiler cannot know, so no part of the loop moves
  // above the first clock read
  const float seed = static_cast<float>(t0 & 1) * 1e-30f + 0.05f * static_cast<float>(threadIdx.x & 7);
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = seed + 0.01f * static_cast<float>(k);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = ex2_approx(-x[k]);
  }
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) acc += x[k];
  asm volatile("" :: "f"(acc));                // the chains complete before the second clock read
  __syncthreads();
  const long long t1 = clock64();
  if (acc < 0.f) g_ex2_sink = acc;              // never true (2^-x > 0); keeps the chains
  if (threadIdx.x == 0) g_ex2_cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
}

cudaError_t measure_ex2_rate(int num_sms, int iters, double* per_sm_per_cycle, cudaStream_t stream) {
  if (num_sms < 1 || num_sms > kEx2MaxSms || iters < 1) return cudaErrorInvalidValue;
  ex2_rate_kernel<<<num_sms, kEx2Threads, 0, stream>>>(iters);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unsigned long long cycles[kEx2MaxSms];
  e = cudaMemcpyFromSymbolAsync(cycles, g_ex2_cycles, sizeof(unsigned long long) * num_sms, 0,
                                cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const double per_cta = static_cast<double>(kEx2Threads) * iters * 8.0;
  double sum = 0.0;
  for (int i = 0; i < num_sms; ++i) sum += per_cta / static_cast<double>(cycles[i] > 0 ? cycles[i] : 1);
  *per_sm_per_cycle = sum / num_sms;
  return cudaSuccess;
}

}  // namespace fa
