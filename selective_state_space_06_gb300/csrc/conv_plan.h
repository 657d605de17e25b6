// Internal (not part of the C ABI): parameters of the conv1d + SiLU kernels (conv1d.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mscan {

constexpr int kConvRun = 32;    // fewest consecutive steps per thread (the scratch is sized for it)
constexpr int kConvRunMax = 256;
constexpr int kConvMaxK = 8;    // largest kernel size

struct ConvParams {
  const float* x; const float* w; const float* bias;
  float* u;                         // forward output
  const float* d_u;                 // backward input
  float* d_x; float* d_w; float* d_bias;
  float* part_w; float* part_b;     // scratch: per (batch row, run) weight-gradient partials
  int batch, T, Di, K;
  int run;                          // steps per thread, chosen per launch (>= kConvRun)
  int nruns, ngroups;               // ceil(T / run), ceil(nruns / kConvRunsPerCta)
};

// The backward's CTA holds 8 warps: 8 consecutive runs of the same 32 channel groups. It sums
// their weight gradients in shared memory, so there is one partial per (batch row, 8 runs).
constexpr int kConvRunsPerCta = 8;

// runs along T, groups of 8 runs, and the scratch floats the backward needs (per-group partials
// of d_w, d_bias), all at the shortest run, which has the most partials
inline int conv_nruns(int64_t T) { return (int)((T + kConvRun - 1) / kConvRun); }
inline int conv_ngroups(int64_t T) {
  return (conv_nruns(T) + kConvRunsPerCta - 1) / kConvRunsPerCta;
}
inline size_t conv_part_w_floats(int64_t batch, int64_t T, int64_t Di, int64_t K) {
  return (size_t)batch * conv_ngroups(T) * Di * K;
}
inline size_t conv_part_b_floats(int64_t batch, int64_t T, int64_t Di) {
  return (size_t)batch * conv_ngroups(T) * Di;
}

// Enqueues the forward (1 kernel) or the backward (2 kernels); returns that count or -1.
int launch_conv(const ConvParams& p, bool bwd, cudaStream_t stream);

}  // namespace mscan
