// probe_kernel.cuh -- throughput probe of the special-function unit's exp2
// (ex2.approx.ftz.f32), the instruction that the online softmax issues once per
// unmasked score.  The exp term of the attention roofline divides the exp
// count by this rate.
//
// Each thread runs 8 independent chains; one link of a chain is four
// dependent ex2 followed by one subtraction that keeps the value bounded
// (x in [-12, 0] -> 2^x in (0, 1] -> ... -> [4, 16] -> minus 16), so the FMA
// pipe sees one instruction per four ex2 and the issue slots stay free.
#pragma once

#include <cstdint>

namespace gb300 {

constexpr int PROBE_CHAINS = 8;
constexpr int PROBE_EX2_PER_LINK = 4;

__device__ __forceinline__ float probe_ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned long long probe_globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// timing[2 b] = SM clock cycles and timing[2 b + 1] = nanoseconds that CTA b
// spent in its loop, both between the same two CTA barriers
__global__ void __launch_bounds__(1024) ex2_probe_kernel(int iters, unsigned long long* timing,
                                                         float* sink) {
  float x[PROBE_CHAINS];
#pragma unroll
  for (int c = 0; c < PROBE_CHAINS; ++c)
    x[c] = -0.001f * static_cast<float>((threadIdx.x + 37 * c) & 1023);
  __syncthreads();
  const unsigned long long t0 = clock64();
  const unsigned long long n0 = probe_globaltimer();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < PROBE_CHAINS; ++c) {
      float y = probe_ex2(x[c]);
      y = probe_ex2(y);
      y = probe_ex2(y);
      y = probe_ex2(y);
      x[c] = y - 16.0f;
    }
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  const unsigned long long n1 = probe_globaltimer();
  if (threadIdx.x == 0) {
    timing[2 * blockIdx.x] = t1 - t0;
    timing[2 * blockIdx.x + 1] = n1 - n0;
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < PROBE_CHAINS; ++c) s += x[c];
  // every chain stays in [-12, 0]: the store never happens, but the compiler
  // cannot prove it, so the chains stay live
  if (s > 1.0e30f) *sink = s;
}

}  // namespace gb300
