// Forward selective scan (sm_103a).
//
// What it computes, for every row (b, d) and state n (h_{-1} = 0, A = -exp(A_log)):
//   h_t = exp(delta_t * A) * h_{t-1} + delta_t * u_t * B_t[n]
//   y_t = sum_n C_t[n] * h_t + D * u_t,     out_t = y_t * SiLU(gate_t)
// This is the recurrence whose derivatives are the SSM BPTT of mamba-rs
// src/mamba_ssm/cpu/backward.rs (Phase B3). That page precomputes a_neg = -exp(A_log) (its
// "O3") to avoid a transcendental per step. Here the same happens in registers, with the
// log2(e) factor folded in, so each step costs one ex2.
//
// Mapping. grid = (ceil(d_inner / DC), batch). A CTA owns one batch row b and DC consecutive
// channels, and runs the whole time axis for them.
//   lane = dg * G + ng :  ng picks the state group [ng*4, ng*4+4), and dg picks the pair of
//                         channels [2*dg, 2*dg+2) inside the warp's 2*(32/G) channels.
// So each thread carries 2 x 4 states in registers. The reduction of C*h over n is 4 in-thread
// FMAs followed by a log2(G)-step xor butterfly. Loads of delta/u/gate are coalesced along d,
// and all lanes of a state group load the same B/C words (broadcast).
//
// Every kChunk steps the state is written to the checkpoint buffer [batch][chunk][d][n]
// (chunk = 0 .. nchunks-2, the state after that chunk). The backward restarts each chunk from
// these states.
#include "scan_common.cuh"

namespace mscan {

template <int NP>
__global__ void __launch_bounds__(kWarps * 32)
scan_fwd_kernel(const FwdParams p) {
  constexpr int G = NP / kNPT;
  constexpr int DW = (32 / G) * kDPT;
  constexpr int DC = kWarps * DW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int d0 = blockIdx.x * DC + warp * DW + dg * kDPT;
  const int n0 = ng * kNPT;
  const int Di = p.Di, N = p.N, T = p.T;

  bool dv[kDPT];
  float a2[kDPT][kNPT], h[kDPT][kNPT], Dd[kDPT];
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    dv[j] = d < Di;
    Dd[j] = dv[j] ? p.D[d] : 0.f;
#pragma unroll
    for (int k = 0; k < kNPT; ++k) {
      const int n = n0 + k;
      a2[j][k] = (dv[j] && n < N) ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
      h[j][k] = 0.f;
    }
  }
  // lane that finishes channel j (after the butterfly every lane of the group holds y)
  const bool owner[kDPT] = {ng == 0, ng == (G > 1 ? 1 : 0)};

  const size_t row0 = (size_t)b * T;
  for (int c = 0; c < p.nchunks; ++c) {
    const int t0 = c * kChunk;
    const int len = min(kChunk, T - t0);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (i < len) {
        const size_t xo = (row0 + t0 + i) * Di;
        const size_t bo = (row0 + t0 + i) * N;
        float dl[kDPT], uu[kDPT], Bn[kNPT], Cn[kNPT], yp[kDPT];
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          dl[j] = dv[j] ? ld_stream(p.delta + xo + d0 + j) : 0.f;
          uu[j] = dv[j] ? ld_stream(p.u + xo + d0 + j) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kNPT; ++k) {
          Bn[k] = (n0 + k < N) ? ld_stream(p.B + bo + n0 + k) : 0.f;
          Cn[k] = (n0 + k < N) ? ld_stream(p.C + bo + n0 + k) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          const float du = dl[j] * uu[j];
          yp[j] = 0.f;
#pragma unroll
          for (int k = 0; k < kNPT; ++k) {
            const float da = ex2_sfu(dl[j] * a2[j][k]);
            h[j][k] = fmaf(da, h[j][k], du * Bn[k]);
            yp[j] = fmaf(Cn[k], h[j][k], yp[j]);
          }
          yp[j] = sum_over_state_lanes<G>(yp[j]);
        }
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          if (dv[j] && owner[j]) {
            const float g = ld_stream(p.gate + xo + d0 + j);
            const float y = fmaf(Dd[j], uu[j], yp[j]);
            p.out[xo + d0 + j] = y * (g * sigmoid_fast(g));
            if (p.y) p.y[xo + d0 + j] = y;
          }
        }
      }
    }
    if (c + 1 < p.nchunks) {
      float* ck = p.ckpt + ((size_t)b * (p.nchunks - 1) + c) * (size_t)Di * N;
#pragma unroll
      for (int j = 0; j < kDPT; ++j)
#pragma unroll
        for (int k = 0; k < kNPT; ++k)
          if (dv[j] && n0 + k < N) ck[(size_t)(d0 + j) * N + n0 + k] = h[j][k];
    }
  }
}

template <int NP>
static void launch_np(const Plan& plan, const FwdParams& p, cudaStream_t s) {
  dim3 grid(plan.nblk, (unsigned)plan.batch);
  scan_fwd_kernel<NP><<<grid, kWarps * 32, 0, s>>>(p);
}

int launch_fwd(const Plan& plan, const FwdParams& p, cudaStream_t s) {
  switch (plan.NP) {
    case 4: launch_np<4>(plan, p, s); break;
    case 8: launch_np<8>(plan, p, s); break;
    case 16: launch_np<16>(plan, p, s); break;
    case 32: launch_np<32>(plan, p, s); break;
    case 64: launch_np<64>(plan, p, s); break;
    default: return -1;
  }
  return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace mscan
