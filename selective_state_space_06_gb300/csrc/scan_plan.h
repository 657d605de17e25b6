// Internal (not part of the C ABI): launch plan and kernel parameter blocks shared by the
// host entry points (mamba_scan_abi.cu) and the kernel launchers (scan_fwd.cu, scan_bwd.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mscan {

// Thread mapping of both scan kernels (see scan_fwd.cu for the picture):
//   a thread owns kDPT consecutive channels d and NPT = states_per_thread(NP) consecutive
//   states n; G = NP / NPT lanes of a warp share the same channels and split the states
//   between them; a warp therefore covers (32 / G) * kDPT channels; a CTA has kWarps warps.
constexpr int kDPT = 2;     // channels per thread
#ifndef MSCAN_NPT
#define MSCAN_NPT 4
#endif
// states per thread (2 or 4) for d_state padded to NP
__host__ __device__ constexpr int states_per_thread(int NP) {
  return NP < MSCAN_NPT ? NP : MSCAN_NPT;
}
constexpr int kWarps = 4;   // warps per CTA
constexpr int kChunk = 16;  // time steps per chunk (= checkpoint interval)
constexpr int kMaxState = 64;

struct Plan {
  int64_t batch = 0, T = 0, Di = 0, N = 0;
  int NP = 0;        // d_state padded to 4, 8, 16, 32 or 64
  int G = 0;         // lanes per channel group
  int DC = 0;        // channels per CTA
  int nblk = 0;      // CTAs along d_inner
  int nchunks = 0;   // chunks along T
  size_t ckpt_elems = 0;
  // scratch layout (float offsets, each region 256-byte aligned)
  size_t off_partB = 0, off_partC = 0, off_partA = 0, off_partD = 0, scratch_elems = 0;
};

// Returns false when the sizes are outside what the kernels support.
bool make_plan(int64_t batch, int64_t T, int64_t Di, int64_t N, Plan* plan);

struct FwdParams {
  const float* delta; const float* u; const float* B; const float* C; const float* gate;
  const float* A_log; const float* D;
  float* out; float* y; float* ckpt;
  int batch, T, Di, N, nchunks;
};

struct BwdParams {
  const float* delta; const float* u; const float* B; const float* C; const float* gate;
  const float* A_log; const float* D; const float* dy; const float* ckpt;
  float* d_delta; float* d_u; float* d_gate;
  float* partB; float* partC; float* partA; float* partD;   // scratch
  float* d_B; float* d_C; float* d_A_log; float* d_D;
  int batch, T, Di, N, nchunks, nblk;
};

// Each returns the number of kernels enqueued (>= 1) or -1 on a launch error.
int launch_fwd(const Plan& plan, const FwdParams& p, cudaStream_t stream);
int launch_bwd(const Plan& plan, const BwdParams& p, cudaStream_t stream);

}  // namespace mscan
