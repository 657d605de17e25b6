// Internal (not part of the C ABI): parameters of the conv1d + SiLU kernels (conv1d.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mscan {

constexpr int kConvRun = 32;    // consecutive steps per thread
constexpr int kConvMaxK = 8;    // largest kernel size

struct ConvParams {
  const float* x; const float* w; const float* bias;
  float* u;                         // forward output
  const float* d_u;                 // backward input
  float* d_x; float* d_w; float* d_bias;
  float* part_w; float* part_b;     // scratch: per (batch row, run) weight-gradient partials
  int batch, T, Di, K, nruns;
};

// runs along T, and the scratch floats the backward needs (per-run partials of d_w, d_bias)
inline int conv_nruns(int64_t T) { return (int)((T + kConvRun - 1) / kConvRun); }
inline size_t conv_part_w_floats(int64_t batch, int64_t T, int64_t Di, int64_t K) {
  return (size_t)batch * conv_nruns(T) * Di * K;
}
inline size_t conv_part_b_floats(int64_t batch, int64_t T, int64_t Di) {
  return (size_t)batch * conv_nruns(T) * Di;
}

// Enqueues the forward (1 kernel) or the backward (2 kernels); returns that count or -1.
int launch_conv(const ConvParams& p, bool bwd, cudaStream_t stream);

}  // namespace mscan
