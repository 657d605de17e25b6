// Device helpers shared by the scan kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "scan_plan.h"

namespace mscan {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32). Here x <= 0 always, so the
// result lies in [0, 1]; very negative x flushes to 0.
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(g) = 1 / (1 + 2^(-g*log2 e)). For g << 0 the denominator overflows to +inf and the
// quotient is 0; for g >> 0 it is 1.
__device__ __forceinline__ float sigmoid_fast(float g) {
  return __fdividef(1.0f, 1.0f + ex2_sfu(-g * kLog2e));
}

// Read-only, streamed-once global load.
__device__ __forceinline__ float ld_stream(const float* p) { return __ldg(p); }

// Sum over the G lanes that share a channel group (they differ in the low log2(G) lane bits).
template <int G>
__device__ __forceinline__ float sum_over_state_lanes(float v) {
#pragma unroll
  for (int off = 1; off < G; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Sum over the channel groups of a warp (lanes that differ in the bits above log2(G)).
template <int G>
__device__ __forceinline__ float sum_over_channel_lanes(float v) {
#pragma unroll
  for (int off = G; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

}  // namespace mscan
