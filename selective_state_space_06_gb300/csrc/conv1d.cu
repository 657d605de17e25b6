// Causal depthwise conv1d + SiLU, the step before the scan (sm_103a): its forward, and the
// backward of Phase B6 of mamba-rs src/mamba_ssm/cpu/backward.rs.
//   pre[b,t,d] = bias[d] + sum_{j<K} w[d,j] * x[b, t-(K-1)+j, d]   (x = 0 before t = 0)
//   u = pre * sigmoid(pre)
// The page walks the backward in reverse time with a shift-register carry of the later steps'
// taps. On the GPU the same sums are a stencil: d_x[t] = sum_{m<K} d_pre[t+m] * w[d, K-1-m].
// A thread owns VW consecutive channels (2 when d_inner is even, else 1) of one
// batch row and a run of consecutive steps (32 or more, picked per launch). It slides a register window along the run,
// so that every element is loaded once plus a halo of K-1 steps per run. The weight gradients
// are summed per thread over its run, then over the 8 runs of its CTA in shared memory, and a
// fixed-order kernel adds the CTAs' partials.
#include <algorithm>

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
struct Vec<2> {
  using T = float2;
  static __device__ __forceinline__ float2 load(const float* p) {
    return *reinterpret_cast<const float2*>(p);
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
  static __device__ __forceinline__ void unpack(const float2& a, float (&v)[2]) {
    v[0] = a.x; v[1] = a.y;
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
  c.t0 = r * p.run;
  c.t1 = min(p.T, c.t0 + p.run);
  return c;
}

__device__ __forceinline__ float silu_f(float p) { return p * sigmoid_fast(p); }

// base + off for a load of n elements; in the bounds-checked build an access outside the first
// len elements is recorded and redirected to the buffer's first element
__device__ __forceinline__ const float* at(const float* base, size_t off, size_t n, size_t len) {
  return inb(off, n, len) ? base + off : base;
}

// The register windows are rings of K slots indexed by (t - t0) mod K. Steps go in batches of
// K, so inside a batch every slot index is a compile-time constant and nothing is shifted; the
// loads of a batch are issued together, ahead of its arithmetic.
template <int K, int VW>
__global__ void __launch_bounds__(256) conv_fwd_kernel(const ConvParams p) {
  using V = Vec<VW>;
  pdl_wait();      // the previous kernel's writes are visible
  pdl_release();   // the next kernel may take the room the last wave leaves
  const ConvThread c = conv_thread(p, VW);
  if (!c.valid) return;
  float w[K][VW], bias[VW];
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    bias[v] = inb(c.d0 + v, 1, p.Di) ? p.bias[c.d0 + v] : 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j)
      w[j][v] = inb((size_t)(c.d0 + v) * K + j, 1, (size_t)p.Di * K)
                    ? p.w[(size_t)(c.d0 + v) * K + j] : 0.f;
  }
  const size_t row = (size_t)c.b * p.T;
  const size_t nx = (size_t)p.batch * p.T * p.Di;
  const float* __restrict__ xg = p.x;
  float* __restrict__ ug = p.u;
  float ring[K][VW];   // x[t'] at slot (t' - t0) mod K; the K-1 steps before t0 first (0 before t = 0)
#pragma unroll
  for (int s = 1; s < K; ++s) {
    const int ts = c.t0 - K + s;
    if (ts >= 0) {
      V::unpack(V::load(at(xg, (row + ts) * p.Di + c.d0, VW, nx)), ring[s]);
    } else {
#pragma unroll
      for (int v = 0; v < VW; ++v) ring[s][v] = 0.f;
    }
  }
  for (int tb = c.t0; tb < c.t1; tb += K) {
    float xb[K][VW];
#pragma unroll
    for (int q = 0; q < K; ++q)   // past the run: a repeated in-range load, unused
      V::unpack(V::load(at(xg, (row + min(tb + q, c.t1 - 1)) * p.Di + c.d0, VW, nx)), xb[q]);
#pragma unroll
    for (int q = 0; q < K; ++q) {
      const int t = tb + q;
#pragma unroll
      for (int v = 0; v < VW; ++v) ring[q][v] = xb[q][v];
      float out[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        float acc = bias[v];
#pragma unroll
        for (int j = 0; j < K; ++j) acc = fmaf(w[j][v], ring[(q + 1 + j) % K][v], acc);
        out[v] = silu_f(acc);
      }
      if (t < c.t1 && inb((row + t) * p.Di + c.d0, VW, nx)) V::store(ug + (row + t) * p.Di + c.d0, out);
    }
  }
}

// Backward. Walking t forward from the run's start, d_pre[t] is formed from the recomputed
// pre[t]; d_x[t-(K-1)] is complete once d_pre[t] is known (its taps are d_pre[t-(K-1) .. t]).
// The walk runs K-1 steps past the run (d_pre = 0 past T).
template <int K, int VW>
__global__ void __launch_bounds__(256) conv_bwd_kernel(const ConvParams p) {
  using V = Vec<VW>;
  // CTA = (batch row, group of 8 runs, 32 channel groups); warp = run, lane = channel group
  __shared__ float s_red[kConvRunsPerCta][32][(K + 1) * VW];
  pdl_wait();      // the previous kernel's writes are visible
  pdl_release();   // the reduction may take the room this kernel leaves
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncg = p.Di / VW;
  const int ncgb = (ncg + 31) / 32;
  const int cgb = blockIdx.x % ncgb;
  const int rg = (blockIdx.x / ncgb) % p.ngroups;
  ConvThread c;
  c.b = blockIdx.x / (ncgb * p.ngroups);
  const int cg = cgb * 32 + lane;
  const int run = rg * kConvRunsPerCta + warp;
  c.valid = cg < ncg && run < p.nruns;
  c.d0 = (cg < ncg ? cg : 0) * VW;
  c.t0 = run * p.run;
  c.t1 = c.valid ? min(p.T, c.t0 + p.run) : c.t0;
  float w[K][VW], bias[VW];
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    bias[v] = inb(c.d0 + v, 1, p.Di) ? p.bias[c.d0 + v] : 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j)
      w[j][v] = inb((size_t)(c.d0 + v) * K + j, 1, (size_t)p.Di * K)
                    ? p.w[(size_t)(c.d0 + v) * K + j] : 0.f;
  }
  const size_t row = (size_t)c.b * p.T;
  const size_t nx = (size_t)p.batch * p.T * p.Di;
  const float* __restrict__ xg = p.x;
  const float* __restrict__ dug = p.d_u;
  float* __restrict__ dxg = p.d_x;
  float xr[K][VW];    // x[t'] at slot (t' - t0) mod K
  float dr[K][VW];    // d_pre[t'] at slot (t' - t0) mod K
  float gw[K][VW], gb[VW];
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int v = 0; v < VW; ++v) {
      dr[j][v] = 0.f;
      gw[j][v] = 0.f;
    }
#pragma unroll
  for (int v = 0; v < VW; ++v) gb[v] = 0.f;
#pragma unroll
  for (int s = 1; s < K; ++s) {
    const int ts = c.t0 - K + s;
    if (c.valid && ts >= 0) {
      V::unpack(V::load(at(xg, (row + ts) * p.Di + c.d0, VW, nx)), xr[s]);
    } else {
#pragma unroll
      for (int v = 0; v < VW; ++v) xr[s][v] = 0.f;
    }
  }
  const int t_end = c.valid ? c.t1 + (K - 1) : c.t0;   // an invalid thread loads nothing
  const int t_last = min(t_end, p.T) - 1;   // the last step that exists
  for (int tb = c.t0; tb < t_end; tb += K) {
    float xb[K][VW], db[K][VW];
#pragma unroll
    for (int q = 0; q < K; ++q) {   // past the end: a repeated in-range load, unused
      const int t = min(tb + q, t_last);
      V::unpack(V::load(at(xg, (row + t) * p.Di + c.d0, VW, nx)), xb[q]);
      V::unpack(V::load(at(dug, (row + t) * p.Di + c.d0, VW, nx)), db[q]);
    }
#pragma unroll
    for (int q = 0; q < K; ++q) {
      const int t = tb + q;
      const bool in = t < p.T;
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        xr[q][v] = xb[q][v];
        float pre = bias[v];
#pragma unroll
        for (int j = 0; j < K; ++j) pre = fmaf(w[j][v], xr[(q + 1 + j) % K][v], pre);
        const float sg = sigmoid_fast(pre);
        dr[q][v] = in ? db[q][v] * (sg * fmaf(pre, 1.f - sg, 1.f)) : 0.f;
      }
      // this thread's weight gradients: steps of its own run only
      if (t < c.t1) {
#pragma unroll
        for (int v = 0; v < VW; ++v) {
          gb[v] += dr[q][v];
#pragma unroll
          for (int j = 0; j < K; ++j) gw[j][v] = fmaf(dr[q][v], xr[(q + 1 + j) % K][v], gw[j][v]);
        }
      }
      // d_x[t-(K-1)] = sum_m d_pre[t-(K-1)+m] * w[K-1-m]
      const int to = t - (K - 1);
      if (to >= c.t0 && to < c.t1) {
        float dx[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) {
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < K; ++m) acc = fmaf(dr[(q + 1 + m) % K][v], w[K - 1 - m][v], acc);
          dx[v] = acc;
        }
        if (inb((row + to) * p.Di + c.d0, VW, nx)) V::store(dxg + (row + to) * p.Di + c.d0, dx);
      }
    }
  }
  // the CTA's 8 runs summed in shared memory in run order (invalid threads hold zeros), then one
  // partial per (batch row, run group): [b * ngroups + group][d][K] and [..][d]
#pragma unroll
  for (int v = 0; v < VW; ++v) {
    s_red[warp][lane][K * VW + v] = gb[v];
#pragma unroll
    for (int j = 0; j < K; ++j) s_red[warp][lane][j * VW + v] = gw[j][v];
  }
  __syncthreads();
  if (warp == 0 && cg < ncg) {
    const size_t part = (size_t)c.b * p.ngroups + rg;
#pragma unroll
    for (int i = 0; i < (K + 1) * VW; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < kConvRunsPerCta; ++r) acc += s_red[r][lane][i];
      const int v = i % VW, j = i / VW;
      const size_t nparts = (size_t)p.batch * p.ngroups;
      if (j < K) {
        if (inb((part * p.Di + c.d0 + v) * K + j, 1, nparts * p.Di * K))
          p.part_w[(part * p.Di + c.d0 + v) * K + j] = acc;
      } else if (inb(part * p.Di + c.d0 + v, 1, nparts * p.Di)) {
        p.part_b[part * p.Di + c.d0 + v] = acc;
      }
    }
  }
}

// d_w and d_bias: one warp per output sums the run groups' partials in a fixed order: lane l takes
// runs l, l+32, ... in turn, then the lanes are added by a fixed butterfly (deterministic).
__global__ void conv_reduce_kernel(const ConvParams p) {
  pdl_wait();   // the backward's partials are visible
  const size_t nw = (size_t)p.Di * p.K;
  const size_t total = nw + (size_t)p.Di;
  const int nk = p.batch * p.ngroups;
  const int lane = threadIdx.x & 31;
  const size_t warps = (size_t)gridDim.x * (blockDim.x / 32);
  for (size_t e = blockIdx.x * (size_t)(blockDim.x / 32) + (threadIdx.x >> 5); e < total;
       e += warps) {
    const bool is_w = e < nw;
    const size_t q = is_w ? e : e - nw;
    const size_t stride = is_w ? nw : (size_t)p.Di;
    const float* part = is_w ? p.part_w : p.part_b;
    float acc = 0.f;
    for (int k0 = lane; k0 < nk; k0 += 32 * 8) {   // eight loads in flight per lane
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + 32 * i;
        v[i] = (k < nk && inb((size_t)k * stride + q, 1, (size_t)nk * stride))
                   ? part[(size_t)k * stride + q] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += v[i];
    }
#pragma unroll
    for (int m = 16; m >= 1; m /= 2) acc += __shfl_xor_sync(kFull, acc, m);
    if (lane == 0) (is_w ? p.d_w : p.d_bias)[q] = acc;
  }
}

// Run length. A launch of c CTAs with `slots` resident CTAs per GPU takes ceil(c / slots) waves
// of about (run + K - 1) steps each, so the run length minimises that product; a run of 32
// steps at mamba130m's size, for instance, would leave a second wave of 8 CTAs. Shortest run
// on ties (more CTAs in flight). Never shorter than kConvRun, which sizes the scratch.
template <typename CtaCount>
static int pick_run(const ConvParams& p, long long slots, CtaCount ctas) {
  int best = kConvRun;
  long long best_cost = -1;
  const int hi = std::max(kConvRun, std::min(p.T, kConvRunMax));
  for (int r = kConvRun; r <= hi; ++r) {
    const int nruns = (p.T + r - 1) / r;
    if (r > kConvRun && (p.T + r - 2) / (r - 1) == nruns) continue;   // same runs, longer
    const long long waves = (ctas(nruns) + slots - 1) / slots;
    const long long cost = waves * (r + p.K - 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = r;
    }
  }
  return best;
}

static long long resident_slots(const void* kern, int threads) {
  int sms = 152, dev = 0, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return (long long)sms * per_sm;
}

template <int K>
static int launch_k(const ConvParams& p0, bool bwd, cudaStream_t s) {
  // 2 channels per thread (8-byte loads: still one 256-byte segment per warp row) keep the
  // register windows small enough for high occupancy
  const bool vec = p0.Di % 2 == 0;
  const int VW = vec ? 2 : 1;
  const long long ncg = p0.Di / VW;
  ConvParams p = p0;
  if (!bwd) {
    auto kern = vec ? conv_fwd_kernel<K, 2> : conv_fwd_kernel<K, 1>;
    const long long slots = resident_slots((const void*)kern, 256);
    p.run = pick_run(p, slots, [&](int nruns) { return (p.batch * nruns * ncg + 255) / 256; });
    p.nruns = (p.T + p.run - 1) / p.run;
    const unsigned blocks = (unsigned)(((long long)p.batch * p.nruns * ncg + 255) / 256);
    return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, p) == cudaSuccess ? 1 : -1;
  }
  const long long ncgb = (ncg + 31) / 32;
  auto bkern = vec ? conv_bwd_kernel<K, 2> : conv_bwd_kernel<K, 1>;
  const long long slots = resident_slots((const void*)bkern, 256);
  p.run = pick_run(p, slots, [&](int nruns) {
    return (long long)p.batch * ((nruns + kConvRunsPerCta - 1) / kConvRunsPerCta) * ncgb;
  });
  p.nruns = (p.T + p.run - 1) / p.run;
  p.ngroups = (p.nruns + kConvRunsPerCta - 1) / kConvRunsPerCta;   // <= the scratch's count
  const unsigned bblocks = (unsigned)((long long)p.batch * p.ngroups * ncgb);
  if (launch_pdl(bkern, dim3(bblocks), dim3(256), 0, s, p) != cudaSuccess) return -1;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t outs = (size_t)p.Di * (p.K + 1);
  const unsigned rblocks = (unsigned)std::min<size_t>((outs + 7) / 8, (size_t)sms * 16);
  return launch_pdl(conv_reduce_kernel, dim3(rblocks), dim3(256), 0, s, p) == cudaSuccess ? 2
                                                                                         : -1;
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

MSCAN_OOB_HOOKS(conv)

}  // namespace mscan
