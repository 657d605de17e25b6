// Causal depthwise conv1d + SiLU, the step before the scan (sm_103a): its forward, and the
// backward of Phase B6 of mamba-rs src/mamba_ssm/cpu/backward.rs.
//   pre[b,t,d] = bias[d] + sum_{j<K} w[d,j] * x[b, t-(K-1)+j, d]   (x = 0 before t = 0)
//   u = pre * sigmoid(pre)
// The page walks the backward in reverse time with a shift-register carry of the later steps'
// taps. On the GPU the same sums are a stencil: d_x[t] = sum_{m<K} d_pre[t+m] * w[d, K-1-m].
// A thread owns VW consecutive channels (4 when d_inner is a multiple of 4, else 1) of one
// batch row and a run of kConvRun consecutive steps. It slides a register window along the run,
// so that every element is loaded once plus a halo of K-1 steps per run. The weight gradients
// are summed per thread over its run, and a fixed-order kernel adds the runs' partials.
#include "scan_common.cuh"
#include "conv_plan.h"

namespace mscan {

template <int VW>
struct Vec;
template <>
struct Vec<4> {
  using T = float4;
  static __device__ __forceinline__ float4 load(const float* p) {
    return *reinterpret_cast<const float4*>(p);
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  static __device__ __forceinline__ void unpack(const float4& a, float (&v)[4]) {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  }
};
template <>
struct Vec<1> {
  using T = float;
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, const float (&v)[1]) { *p = v[0]; }
  static __device__ __forceinline__ void unpack(const float& a, float (&v)[1]) { v[0] = a; }
};

// thread -> (b, run, channel group); neighbouring threads take neighbouring channel groups
struct ConvThread {
  int b, t0, t1, d0;
  bool valid;
};
__device__ __forceinline__ ConvThread conv_thread(const ConvParams& p, int VW) {
  const int ncg = p.Di / VW;
  const long long gid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  ConvThread c;
  const long long total = (long long)p.batch * p.nruns * ncg;
  c.valid = gid < total;
  const long long g = c.valid ? gid : 0;
  const int cg = (int)(g % ncg);
  const long long rest = g / ncg;
  const int r = (int)(rest % p.nruns);
  c.b = (int)(rest / p.nruns);
  c.d0 = cg * VW;
  c.t0 = r * kConvRun;
  c.t1 = min(p.T, c.t0 + kConvRun);
  return c;
}

__device__ __forceinline__ float silu_f(float p) { return p * sigmoid_fast(p); }

template <int K, int VW>
__global__ void __launch_bounds__(256) conv_fwd_kernel(const ConvParams p) {
  using V = Vec<VW>;
  const ConvThread c = conv_thread(p, VW);
  if (!c.valid) return;
  float w[K][VW], bias[VW];
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    bias[v] = p.bias[c.d0 + v];
#pragma unroll
    for (int j = 0; j < K; ++j) w[j][v] = p.w[(size_t)(c.d0 + v) * K + j];
  }
  const size_t row = (size_t)c.b * p.T;
  // window of the K-1 previous inputs (zeros before t = 0)
  float win[K > 1 ? K - 1 : 1][VW];
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int ts = c.t0 - (K - 1) + j;
    if (ts >= 0) {
      V::unpack(V::load(p.x + (row + ts) * p.Di + c.d0), win[j]);
    } else {
#pragma unroll
      for (int v = 0; v < VW; ++v) win[j][v] = 0.f;
    }
  }
#pragma unroll 4
  for (int t = c.t0; t < c.t1; ++t) {
    float xv[VW], out[VW];
    V::unpack(V::load(p.x + (row + t) * p.Di + c.d0), xv);
#pragma unroll
    for (int v = 0; v < VW; ++v) {
      float acc = fmaf(w[K - 1][v], xv[v], bias[v]);
#pragma unroll
      for (int j = 0; j < K - 1; ++j) acc = fmaf(w[j][v], win[j][v], acc);
      out[v] = silu_f(acc);
    }
    V::store(p.u + (row + t) * p.Di + c.d0, out);
#pragma unroll
    for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
      for (int v = 0; v < VW; ++v) win[j][v] = win[j + 1][v];
    if constexpr (K > 1) {
#pragma unroll
      for (int v = 0; v < VW; ++v) win[K - 2][v] = xv[v];
    }
  }
}

// Backward. Walking t forward from the run's start, d_pre[t] is formed from the recomputed
// pre[t]; d_x[t-(K-1)] is complete once d_pre[t] is known (its taps are d_pre[t-(K-1) .. t]).
// The walk runs K-1 steps past the run (d_pre = 0 past T).
template <int K, int VW>
__global__ void __launch_bounds__(256) conv_bwd_kernel(const ConvParams p) {
  using V = Vec<VW>;
  const ConvThread c = conv_thread(p, VW);
  if (!c.valid) return;
  float w[K][VW], bias[VW];
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    bias[v] = p.bias[c.d0 + v];
#pragma unroll
    for (int j = 0; j < K; ++j) w[j][v] = p.w[(size_t)(c.d0 + v) * K + j];
  }
  const size_t row = (size_t)c.b * p.T;
  float xwin[K][VW];    // x[t-(K-1) .. t] (slot K-1 filled at each step)
  float dpw[K][VW];     // d_pre[t-(K-1) .. t]
  float gw[K][VW], gb[VW];
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int v = 0; v < VW; ++v) {
      dpw[j][v] = 0.f;
      gw[j][v] = 0.f;
    }
#pragma unroll
  for (int v = 0; v < VW; ++v) gb[v] = 0.f;
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int ts = c.t0 - (K - 1) + j;
    if (ts >= 0) {
      V::unpack(V::load(p.x + (row + ts) * p.Di + c.d0), xwin[j]);
    } else {
#pragma unroll
      for (int v = 0; v < VW; ++v) xwin[j][v] = 0.f;
    }
  }
  const int t_end = c.t1 + (K - 1);
#pragma unroll 2
  for (int t = c.t0; t < t_end; ++t) {
    const bool in = t < p.T;
    float dp[VW];
    if (in) {
      float xv[VW], du[VW];
      V::unpack(V::load(p.x + (row + t) * p.Di + c.d0), xv);
      V::unpack(V::load(p.d_u + (row + t) * p.Di + c.d0), du);
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        xwin[K - 1][v] = xv[v];
        float pre = bias[v];
#pragma unroll
        for (int j = 0; j < K; ++j) pre = fmaf(w[j][v], xwin[j][v], pre);
        const float s = sigmoid_fast(pre);
        dp[v] = du[v] * (s * fmaf(pre, 1.f - s, 1.f));
      }
    } else {
#pragma unroll
      for (int v = 0; v < VW; ++v) dp[v] = 0.f;
    }
    // this thread's weight gradients: steps of its own run only
    if (t < c.t1) {
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        gb[v] += dp[v];
#pragma unroll
        for (int j = 0; j < K; ++j) gw[j][v] = fmaf(dp[v], xwin[j][v], gw[j][v]);
      }
    }
    // shift the d_pre window and complete d_x[t - (K-1)]
#pragma unroll
    for (int j = 0; j + 1 < K; ++j)
#pragma unroll
      for (int v = 0; v < VW; ++v) dpw[j][v] = dpw[j + 1][v];
#pragma unroll
    for (int v = 0; v < VW; ++v) dpw[K - 1][v] = dp[v];
    const int to = t - (K - 1);
    if (to >= c.t0) {
      float dx[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < K; ++m) acc = fmaf(dpw[m][v], w[K - 1 - m][v], acc);
        dx[v] = acc;
      }
      V::store(p.d_x + (row + to) * p.Di + c.d0, dx);
    }
#pragma unroll
    for (int j = 0; j + 1 < K; ++j)
#pragma unroll
      for (int v = 0; v < VW; ++v) xwin[j][v] = xwin[j + 1][v];
  }
  // partials of this (batch row, run): [b * nruns + run][d][K] and [b * nruns + run][d]
  const size_t part = (size_t)c.b * p.nruns + c.t0 / kConvRun;
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    p.part_b[part * p.Di + c.d0 + v] = gb[v];
#pragma unroll
    for (int j = 0; j < K; ++j) p.part_w[(part * p.Di + c.d0 + v) * K + j] = gw[j][v];
  }
}

// d_w and d_bias: the runs' partials summed in index order (eight loads in flight at a time).
__global__ void conv_reduce_kernel(const ConvParams p) {
  const size_t nw = (size_t)p.Di * p.K;
  const size_t total = nw + (size_t)p.Di;
  const int nk = p.batch * p.nruns;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const bool is_w = e < nw;
    const size_t q = is_w ? e : e - nw;
    const size_t stride = is_w ? nw : (size_t)p.Di;
    const float* part = is_w ? p.part_w : p.part_b;
    float acc = 0.f;
    for (int k0 = 0; k0 < nk; k0 += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = k0 + k < nk ? part[(size_t)(k0 + k) * stride + q] : 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc += v[k];
    }
    (is_w ? p.d_w : p.d_bias)[q] = acc;
  }
}

template <int K>
static int launch_k(const ConvParams& p, bool bwd, cudaStream_t s) {
  const bool vec = p.Di % 4 == 0;
  const int VW = vec ? 4 : 1;
  const long long threads = (long long)p.batch * p.nruns * (p.Di / VW);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (!bwd) {
    if (vec) conv_fwd_kernel<K, 4><<<blocks, 256, 0, s>>>(p);
    else conv_fwd_kernel<K, 1><<<blocks, 256, 0, s>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
  }
  if (vec) conv_bwd_kernel<K, 4><<<blocks, 256, 0, s>>>(p);
  else conv_bwd_kernel<K, 1><<<blocks, 256, 0, s>>>(p);
  if (cudaPeekAtLastError() != cudaSuccess) return -1;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  conv_reduce_kernel<<<sms * 2, 256, 0, s>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? 2 : -1;
}

int launch_conv(const ConvParams& p, bool bwd, cudaStream_t s) {
  switch (p.K) {
    case 1: return launch_k<1>(p, bwd, s);
    case 2: return launch_k<2>(p, bwd, s);
    case 3: return launch_k<3>(p, bwd, s);
    case 4: return launch_k<4>(p, bwd, s);
    case 5: return launch_k<5>(p, bwd, s);
    case 6: return launch_k<6>(p, bwd, s);
    case 7: return launch_k<7>(p, bwd, s);
    case 8: return launch_k<8>(p, bwd, s);
    default: return -1;
  }
}

}  // namespace mscan
