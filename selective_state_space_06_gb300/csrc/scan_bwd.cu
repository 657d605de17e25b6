// Backward selective scan (sm_103a): the gating backward and the reverse-time SSM BPTT of
// mamba-rs src/mamba_ssm/cpu/backward.rs (Phases B2 and B3), with h recomputed per chunk from
// the forward's checkpoints instead of being stored for every t.
//
// Per row (b, d), walking the chunks from last to first:
//   1. recompute: restart from the chunk's checkpoint (zero for chunk 0) and run the forward
//      recurrence over the chunk, keeping h_t for the chunk's kChunk steps in registers;
//   2. reverse: for t = last .. first of the chunk
//        y = sum_n C*h_t + D*u                              (recomputed, for d_gate)
//        d_y = dy*SiLU(g),  d_gate = dy*y*s*(1 + g*(1-s))  (Phase B2)
//        d_h = d_h + d_y*C                                  (Phase B3, in the page's order)
//        d_delta = sum_n d_h*(A*da*h_{t-1} + u*B),  d_u = d_y*D + sum_n d_h*delta*B
//        d_B[t,n] += d_h*delta*u,  d_C[t,n] += d_y*h_t    (summed over d)
//        d_A_log += d_h*da*delta*A*h_{t-1},  d_D += d_y*u (summed over b, t)
//        d_h = da*d_h
//   The code uses r = (da*d_h)*h_{t-1}, so the A-term of d_delta is ln2 * sum_n a2*r and
//   d_A_log = ln2 * a2 * sum_t delta*r, where a2 = A*log2(e) is the register constant of ex2.
// Reductions, all in a fixed order (deterministic):
//   d_B, d_C over d: in-thread over the thread's 2 channels, then an xor butterfly over the
//   warp's channel lanes, then the CTA's warps summed through shared memory. That gives one
//   partial per CTA, written to scratch [blk][b][t][n]. scan_reduce_kernel then sums the
//   partials over blk in index order.
//   d_A_log, d_D over (b, t): register accumulators over t, then one partial per b in
//   scratch, summed over b in index order by scan_reduce_kernel.
#include "scan_common.cuh"

namespace mscan {

template <int NP>
__global__ void __launch_bounds__(kWarps * 32)
scan_bwd_kernel(const BwdParams p) {
  constexpr int G = NP / kNPT;
  constexpr int DW = (32 / G) * kDPT;
  constexpr int DC = kWarps * DW;
  __shared__ float redB[kWarps][kChunk][NP];
  __shared__ float redC[kWarps][kChunk][NP];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int d0 = blockIdx.x * DC + warp * DW + dg * kDPT;
  const int n0 = ng * kNPT;
  const int Di = p.Di, N = p.N, T = p.T;

  bool dv[kDPT];
  float a2[kDPT][kNPT], dh[kDPT][kNPT], accA[kDPT][kNPT], Dd[kDPT], dD[kDPT];
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    dv[j] = d < Di;
    Dd[j] = dv[j] ? p.D[d] : 0.f;
    dD[j] = 0.f;
#pragma unroll
    for (int k = 0; k < kNPT; ++k) {
      const int n = n0 + k;
      a2[j][k] = (dv[j] && n < N) ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
      dh[j][k] = 0.f;
      accA[j][k] = 0.f;
    }
  }
  const bool owner[kDPT] = {ng == 0, ng == (G > 1 ? 1 : 0)};
  const size_t row0 = (size_t)b * T;

  for (int c = p.nchunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk;
    const int len = min(kChunk, T - t0);
    const float* ck = (c > 0) ? p.ckpt + ((size_t)b * (p.nchunks - 1) + (c - 1)) * (size_t)Di * N
                              : nullptr;

    // ---- 1. recompute h over the chunk --------------------------------------------------
    float hs[kChunk][kDPT][kNPT];
    {
      float hc[kDPT][kNPT];
#pragma unroll
      for (int j = 0; j < kDPT; ++j)
#pragma unroll
        for (int k = 0; k < kNPT; ++k)
          hc[j][k] = (ck && dv[j] && n0 + k < N) ? ck[(size_t)(d0 + j) * N + n0 + k] : 0.f;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        if (i < len) {
          const size_t xo = (row0 + t0 + i) * Di;
          const size_t bo = (row0 + t0 + i) * N;
          float dl[kDPT], uu[kDPT], Bn[kNPT];
#pragma unroll
          for (int j = 0; j < kDPT; ++j) {
            dl[j] = dv[j] ? ld_stream(p.delta + xo + d0 + j) : 0.f;
            uu[j] = dv[j] ? ld_stream(p.u + xo + d0 + j) : 0.f;
          }
#pragma unroll
          for (int k = 0; k < kNPT; ++k) Bn[k] = (n0 + k < N) ? ld_stream(p.B + bo + n0 + k) : 0.f;
#pragma unroll
          for (int j = 0; j < kDPT; ++j) {
            const float du = dl[j] * uu[j];
#pragma unroll
            for (int k = 0; k < kNPT; ++k) {
              const float da = ex2_sfu(dl[j] * a2[j][k]);
              hc[j][k] = fmaf(da, hc[j][k], du * Bn[k]);
              hs[i][j][k] = hc[j][k];
            }
          }
        }
      }
    }

    // ---- 2. reverse recurrence over the chunk -------------------------------------------
#pragma unroll
    for (int ii = 0; ii < kChunk; ++ii) {
      const int i = kChunk - 1 - ii;
      if (i < len) {
        const size_t xo = (row0 + t0 + i) * Di;
        const size_t bo = (row0 + t0 + i) * N;
        float dl[kDPT], uu[kDPT], gt[kDPT], go[kDPT], Bn[kNPT], Cn[kNPT];
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          dl[j] = dv[j] ? ld_stream(p.delta + xo + d0 + j) : 0.f;
          uu[j] = dv[j] ? ld_stream(p.u + xo + d0 + j) : 0.f;
          gt[j] = dv[j] ? ld_stream(p.gate + xo + d0 + j) : 0.f;
          go[j] = dv[j] ? ld_stream(p.dy + xo + d0 + j) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kNPT; ++k) {
          Bn[k] = (n0 + k < N) ? ld_stream(p.B + bo + n0 + k) : 0.f;
          Cn[k] = (n0 + k < N) ? ld_stream(p.C + bo + n0 + k) : 0.f;
        }
        // state before step i: the previous stash entry, or the chunk's checkpoint
        float hp[kDPT][kNPT];
#pragma unroll
        for (int j = 0; j < kDPT; ++j)
#pragma unroll
          for (int k = 0; k < kNPT; ++k) {
            if (i > 0) hp[j][k] = hs[i > 0 ? i - 1 : 0][j][k];
            else hp[j][k] = (ck && dv[j] && n0 + k < N) ? ck[(size_t)(d0 + j) * N + n0 + k] : 0.f;
          }

        float y[kDPT], s[kDPT], d_y[kDPT];
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          float yp = 0.f;
#pragma unroll
          for (int k = 0; k < kNPT; ++k) yp = fmaf(Cn[k], hs[i][j][k], yp);
          y[j] = fmaf(Dd[j], uu[j], sum_over_state_lanes<G>(yp));
          s[j] = sigmoid_fast(gt[j]);
          d_y[j] = go[j] * (gt[j] * s[j]);
        }

        float sA[kDPT], sB[kDPT], xb[kNPT], xc[kNPT];
#pragma unroll
        for (int k = 0; k < kNPT; ++k) { xb[k] = 0.f; xc[k] = 0.f; }
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          const float du = dl[j] * uu[j];
          sA[j] = 0.f;
          sB[j] = 0.f;
#pragma unroll
          for (int k = 0; k < kNPT; ++k) {
            const float da = ex2_sfu(dl[j] * a2[j][k]);
            const float gh = fmaf(d_y[j], Cn[k], dh[j][k]);   // d_h += d_y*C
            const float cr = da * gh;                          // carry to t-1
            const float r = cr * hp[j][k];                     // d_h*da*h_{t-1}
            accA[j][k] = fmaf(r, dl[j], accA[j][k]);
            sA[j] = fmaf(a2[j][k], r, sA[j]);
            sB[j] = fmaf(gh, Bn[k], sB[j]);
            xb[k] = fmaf(gh, du, xb[k]);
            xc[k] = fmaf(d_y[j], hs[i][j][k], xc[k]);
            dh[j][k] = cr;
          }
          sA[j] = sum_over_state_lanes<G>(sA[j]);
          sB[j] = sum_over_state_lanes<G>(sB[j]);
          dD[j] = fmaf(d_y[j], uu[j], dD[j]);
        }
#pragma unroll
        for (int j = 0; j < kDPT; ++j) {
          if (dv[j] && owner[j]) {
            p.d_delta[xo + d0 + j] = fmaf(sA[j], kLn2, uu[j] * sB[j]);
            p.d_u[xo + d0 + j] = fmaf(d_y[j], Dd[j], dl[j] * sB[j]);
            p.d_gate[xo + d0 + j] = go[j] * y[j] * (s[j] * fmaf(gt[j], 1.f - s[j], 1.f));
          }
        }
#pragma unroll
        for (int k = 0; k < kNPT; ++k) {
          xb[k] = sum_over_channel_lanes<G>(xb[k]);
          xc[k] = sum_over_channel_lanes<G>(xc[k]);
          if (dg == 0) {
            redB[warp][i][n0 + k] = xb[k];
            redC[warp][i][n0 + k] = xc[k];
          }
        }
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kChunk * NP; idx += kWarps * 32) {
      const int i = idx / NP, n = idx % NP;
      if (i < len && n < N) {
        float sb = 0.f, sc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          sb += redB[w][i][n];
          sc += redC[w][i][n];
        }
        const size_t o = (((size_t)blockIdx.x * p.batch + b) * T + t0 + i) * N + n;
        p.partB[o] = sb;
        p.partC[o] = sc;
      }
    }
    __syncthreads();
  }

  // per-batch partials of d_A_log (= A * sum_t delta*r = ln2*a2*accA) and d_D
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    if (!dv[j]) continue;
#pragma unroll
    for (int k = 0; k < kNPT; ++k)
      if (n0 + k < N)
        p.partA[((size_t)b * Di + d0 + j) * N + n0 + k] = kLn2 * a2[j][k] * accA[j][k];
    if (ng == 0) p.partD[(size_t)b * Di + d0 + j] = dD[j];
  }
}

// Fixed-order sums of the partials: d_B/d_C over CTAs along d, d_A_log/d_D over batch.
__global__ void scan_reduce_kernel(const BwdParams p) {
  const size_t btn = (size_t)p.batch * p.T * p.N;
  const size_t dn = (size_t)p.Di * p.N;
  const size_t total = btn + dn + (size_t)p.Di;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    if (e < btn) {
      float sb = 0.f, sc = 0.f;
      for (int k = 0; k < p.nblk; ++k) {
        sb += p.partB[(size_t)k * btn + e];
        sc += p.partC[(size_t)k * btn + e];
      }
      p.d_B[e] = sb;
      p.d_C[e] = sc;
    } else if (e < btn + dn) {
      const size_t q = e - btn;
      float sa = 0.f;
      for (int bb = 0; bb < p.batch; ++bb) sa += p.partA[(size_t)bb * dn + q];
      p.d_A_log[q] = sa;
    } else {
      const size_t q = e - btn - dn;
      float sd = 0.f;
      for (int bb = 0; bb < p.batch; ++bb) sd += p.partD[(size_t)bb * p.Di + q];
      p.d_D[q] = sd;
    }
  }
}

template <int NP>
static void launch_np(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  dim3 grid(plan.nblk, (unsigned)plan.batch);
  scan_bwd_kernel<NP><<<grid, kWarps * 32, 0, s>>>(p);
}

int launch_bwd(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  switch (plan.NP) {
    case 4: launch_np<4>(plan, p, s); break;
    case 8: launch_np<8>(plan, p, s); break;
    case 16: launch_np<16>(plan, p, s); break;
    case 32: launch_np<32>(plan, p, s); break;
    case 64: launch_np<64>(plan, p, s); break;
    default: return -1;
  }
  if (cudaPeekAtLastError() != cudaSuccess) return -1;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  scan_reduce_kernel<<<sms * 4, 256, 0, s>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? 2 : -1;
}

}  // namespace mscan
