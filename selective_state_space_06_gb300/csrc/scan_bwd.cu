// Backward selective scan (sm_103a). This is the gating backward and the reverse-time SSM
// BPTT of mamba-rs src/mamba_ssm/cpu/backward.rs (Phases B2 and B3). h is recomputed per chunk
// from the forward's checkpoints instead of being stored for every t.
//
// Per row (b, d), the chunks are walked from last to first (thread mapping as in the forward:
// 2 channels x NPT states per thread, G lanes per channel group):
//   0. gating (Phase B2), once per (t, d) of the chunk and cooperatively:
//        d_y = dy * g * s  (into the staged gate tile) and d_gate = dy * y * s * (1 + g*(1 - s))
//      (stored at once), s = sigmoid(g), with the y the forward kept.
//   1. recompute: restart from the chunk's checkpoint (zero for chunk 0) and run the forward
//      recurrence over the chunk, kSub steps at a time, keeping those h_t in registers;
//   2. reverse (Phase B3, in the page's order), for t = last .. first of the chunk:
//        d_h += d_y*C
//        d_delta = sum_n d_h*(A*da*h_{t-1} + u*B),  d_u = d_y*D + sum_n d_h*delta*B
//        d_B[t,n] += d_h*delta*u,  d_C[t,n] += d_y*h_t           (over d)
//        d_A_log += d_h*da*delta*A*h_{t-1},  d_D += d_y*u         (over b, t)
//        d_h = da*d_h
//      The code forms r = (da*d_h)*h_{t-1}. With a2 = A*log2(e), the register constant of ex2,
//      the A-term of d_delta is ln2 * sum_n a2*r and d_A_log = ln2 * a2 * sum_t delta*r.
// Reductions, all in a fixed order (deterministic):
//   * sum over n (the A-term, the B-term): in-thread, then a butterfly reduce-scatter over
//     the G state lanes, batched over P = G/2 steps. Each lane ends with one (step, channel),
//     and stores d_delta and d_u for it.
//   * d_B, d_C over d: in-thread over the thread's 2 channels, then a reduce-scatter over the
//     warp's channel lanes, then the warps summed through shared memory. That gives one partial
//     per CTA, written to scratch [blk][b][t][n]; scan_reduce_kernel sums the partials over blk
//     in index order.
//   * d_A_log, d_D over (b, t): register accumulators over t, then one partial per batch row in
//     scratch, summed over b in index order by scan_reduce_kernel.
#include "scan_common.cuh"

namespace mscan {

constexpr int kBwdStages = 2;

template <int NP>
struct BwdShape {
  static constexpr int NPT = states_per_thread_bwd(NP);
  static constexpr int NPR = NPT / 2;
  static constexpr int kSub = 32 / NPT;         // steps kept in registers at a time (64 floats)
  static constexpr int kNSub = kChunk / kSub;
  static constexpr int G = NP / NPT;
  static constexpr int DW = (32 / G) * kDPT;
  static constexpr int DC = kWarps * DW;
  static constexpr int P = G >= 2 ? G / 2 : 1;
  // per stage: delta, u, gate, dy [kChunk][DC]; B, C [kChunk][NP]; the chunk's starting
  // checkpoint [DC][N] (N <= NP); the forward's y [kChunk][DC]
  static constexpr int kStageFloats = kChunk * (5 * DC + 2 * NP) + DC * NP;
  static constexpr int kRedFloats = kWarps * kChunk * 2 * NP;   // per-warp d_B/d_C sums
  static constexpr size_t kSmemBytes =
      ((size_t)kBwdStages * kStageFloats + kRedFloats) * sizeof(float);
};

template <int NP, bool VEC>
__device__ __forceinline__ void bwd_load_chunk(const BwdParams& p, float* st, int c, int b,
                                               int dblk0) {
  using S = BwdShape<NP>;
  constexpr int DC = S::DC, NTH = kWarps * 32;
  // layout: delta, u, gate, dy [kChunk][DC]; B, C [kChunk][NP]; checkpoint row [DC][N]
  float* s_dl = st;
  float* s_u = st + kChunk * DC;
  float* s_g = st + 2 * kChunk * DC;
  float* s_dy = st + 3 * kChunk * DC;
  float* s_B = st + 4 * kChunk * DC;
  float* s_C = s_B + kChunk * NP;
  const int t0 = c * kChunk;
  const size_t rowb = (size_t)b * p.T;
  if constexpr (VEC) {
    for (int q = threadIdx.x; q < kChunk * DC / 4; q += NTH) {
      const int i = q / (DC / 4), col = (q % (DC / 4)) * 4;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di && inb((rowb + t) * p.Di + d, 4, p.n_io());
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async16(s_dl + i * DC + col, p.delta + go, v);
      cp_async16(s_u + i * DC + col, p.u + go, v);
      cp_async16(s_g + i * DC + col, p.gate + go, v);
      cp_async16(s_dy + i * DC + col, p.dy + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP / 4; q += NTH) {
      const int i = q / (NP / 4), n = (q % (NP / 4)) * 4;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N && inb((rowb + t) * p.N + n, 4, p.n_bc());
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async16(s_B + i * NP + n, p.B + go, v);
      cp_async16(s_C + i * NP + n, p.C + go, v);
    }
  } else {
    for (int q = threadIdx.x; q < kChunk * DC; q += NTH) {
      const int i = q / DC, col = q % DC;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di && inb((rowb + t) * p.Di + d, 1, p.n_io());
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async4(s_dl + i * DC + col, p.delta + go, v);
      cp_async4(s_u + i * DC + col, p.u + go, v);
      cp_async4(s_g + i * DC + col, p.gate + go, v);
      cp_async4(s_dy + i * DC + col, p.dy + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP; q += NTH) {
      const int i = q / NP, n = q % NP;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N && inb((rowb + t) * p.N + n, 1, p.n_bc());
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async4(s_B + i * NP + n, p.B + go, v);
      cp_async4(s_C + i * NP + n, p.C + go, v);
    }
  }
  stage_tile<DC, NTH, VEC>(s_C + kChunk * NP + DC * NP, p.y_ck, (size_t)b * p.T, t0, p.T, p.Di,
                           dblk0, p.n_io());
  {
    // state entering chunk c (checkpoint slot c-1); zeros for the first chunk
    float* s_h0 = s_C + kChunk * NP;
    const bool have = c > 0;
    const size_t src0 = have ? (((size_t)b * (p.nchunks - 1) + (c - 1)) * p.Di + dblk0) * p.N : 0;
    const float* src = p.ckpt + src0;
    const int rowlen = DC * p.N;
    if constexpr (VEC) {
      for (int q = threadIdx.x * 4; q < rowlen; q += NTH * 4) {
        const bool v = have && (dblk0 + q / p.N < p.Di) && inb(src0 + q, 4, p.n_ck());
        cp_async16(s_h0 + q, v ? src + q : p.delta, v);
      }
    } else {
      for (int q = threadIdx.x; q < rowlen; q += NTH) {
        const bool v = have && (dblk0 + q / p.N < p.Di) && inb(src0 + q, 1, p.n_ck());
        cp_async4(s_h0 + q, v ? src + q : p.delta, v);
      }
    }
  }
  cp_async_commit();
}

// Segment pre-pass of the backward: for every segment but the first, run the d_h recurrence of
// Phase B3 from a zero carry at the segment's end back to its start. That gives the local
// prefix L = sum_t (prod_{s<=t} exp(delta_s*A)) * d_y_t * C_t[n] (products from the segment's
// first step to t), plus the segment's sum of delta. The carry leaving a segment towards
// earlier time is L + exp(A * sum(delta)) * (carry entering it from later time), so the
// segments compose exactly (scan_bwd_compose_kernel). The sum is accumulated in forward order,
// and the product is taken as exp(A * running sum of delta), which leaves no serial multiply
// chain. A CTA covers kAggWarps warps of channels and one sub-segment (a segment may be split
// into nsub sub-segments, which compose the same way, to give the pre-pass more CTAs).
template <int NP>
struct BwdAggShape {
  using S = BwdShape<NP>;
  static constexpr int AW = kAggWarps;
  static constexpr int DC = AW * S::DW;
  static constexpr int NTH = AW * 32;
  static constexpr int kStages = 4;
  static constexpr int kStageFloats = kChunk * (3 * DC + NP);   // delta, gate, dy, C
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageFloats * sizeof(float);
};

template <int NP, bool VEC>
__global__ void __launch_bounds__(kAggWarps * 32)
scan_bwd_agg_kernel(const BwdParams p) {
  using S = BwdShape<NP>;
  using A = BwdAggShape<NP>;
  constexpr int G = S::G, DW = S::DW, NPT = S::NPT, NPR = S::NPR, DC = A::DC, NTH = A::NTH;
  extern __shared__ __align__(16) float smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int nblk_a = (p.Di + DC - 1) / DC;
  const int blk = blockIdx.x % nblk_a, grp = blockIdx.x / nblk_a;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * kDPT;
  const int d0 = dblk0 + cl;
  const int n0 = ng * NPT;
  const int Di = p.Di, N = p.N, T = p.T;
  // segments 1 .. nseg-1 need aggregates; sub-segment j of segment sg (may be empty)
  const int sg = 1 + grp / p.nsub, j_sub = grp % p.nsub;
  const int slot = sg * p.nsub + j_sub;
  const int c_begin = sg * p.seg_chunks + j_sub * p.sub_chunks;
  const int c_end = min(min(p.nchunks, (sg + 1) * p.seg_chunks), c_begin + p.sub_chunks);
  const size_t row0 = (size_t)b * T;

  float2 a2[kDPT][NPR], L[kDPT][NPR];
  float sd[kDPT] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    const bool dv = d < Di;
    float t4[NPT];
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      const int n = n0 + k;
      t4[k] = (dv && n < N && inb((size_t)d * N + n, 1, (size_t)Di * N))
                  ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NPR; ++q) {
      a2[j][q] = make_float2(t4[2 * q], t4[2 * q + 1]);
      L[j][q] = make_float2(0.f, 0.f);
    }
  }

  auto load = [&](int stage, int c) {
    float* st = smem + stage * A::kStageFloats;
    stage_tile<DC, NTH, VEC>(st, p.delta, row0, c * kChunk, T, Di, dblk0, p.n_io());
    stage_tile<DC, NTH, VEC>(st + kChunk * DC, p.gate, row0, c * kChunk, T, Di, dblk0, p.n_io());
    stage_tile<DC, NTH, VEC>(st + 2 * kChunk * DC, p.dy, row0, c * kChunk, T, Di, dblk0, p.n_io());
    stage_tile<NP, NTH, VEC>(st + 3 * kChunk * DC, p.C, row0, c * kChunk, T, N, 0, p.n_bc());
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < A::kStages - 1; ++s) {
    if (c_begin + s < c_end) load(s, c_begin + s);
    else cp_async_commit();
  }
  for (int c = c_begin; c < c_end; ++c) {
    const int it = c - c_begin;
    cp_async_wait<A::kStages - 2>();
    __syncthreads();
    if (c + A::kStages - 1 < c_end) load((it + A::kStages - 1) % A::kStages, c + A::kStages - 1);
    else cp_async_commit();
    float* st = smem + (it % A::kStages) * A::kStageFloats;
    const float* s_dl = st;
    float* s_g = st + kChunk * DC;          // becomes d_y
    const float* s_dy = st + 2 * kChunk * DC;
    const float* s_C = st + 3 * kChunk * DC;
    for (int e = threadIdx.x; e < kChunk * DC; e += NTH) {
      const float g = s_g[e];
      s_g[e] = s_dy[e] * (g * sigmoid_fast(g));
    }
    if (p.softplus) softplus_tile<DC, NTH>(st, T - c * kChunk, Di - dblk0);   // raw -> delta
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const float2 dlv = lds2(s_dl + i * DC + cl);
      const float2 dyv = lds2(s_g + i * DC + cl);
      float2 Cp[NPR];
      lds_pairs<NPR>(s_C + i * NP + n0, Cp);
#pragma unroll
      for (int j = 0; j < kDPT; ++j) {
        sd[j] += j ? dlv.y : dlv.x;
        const float2 sd2 = splat2(sd[j]), dy2 = splat2(j ? dyv.y : dyv.x);
#pragma unroll
        for (int q = 0; q < NPR; ++q) {
          // prod_{s<=t} exp(delta_s*A) = exp(A * sum_{s<=t} delta_s): no serial product chain
          const float2 cum = ex2_2(mul2(sd2, a2[j][q]));
          L[j][q] = fma2(cum, mul2(dy2, Cp[q]), L[j][q]);
        }
      }
    }
  }
  cp_async_wait<0>();
  // emit the sub-segment's aggregate (zeros for an empty one)
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    const size_t row = ((size_t)b * p.nseg * p.nsub + slot) * Di + d;
    if (d < Di && inb(row, 1, p.n_agg_sd()) && inb(row * N, N, p.n_agg_l())) {
      if (ng == 0) p.agg_sd[row] = sd[j];
      if constexpr (VEC) {
        if (n0 < N) st_pairs<NPR>(p.agg_L + row * N + n0, L[j]);   // N % 4 == 0 here
      } else {
#pragma unroll
        for (int k = 0; k < NPT; ++k)
          if (n0 + k < N) p.agg_L[row * N + n0 + k] = (k & 1) ? L[j][k >> 1].y : L[j][k >> 1].x;
      }
    }
  }
}

// Composition of the backward segment aggregates, in place: for every (b, d, n), walking the
// sub-segments from last to first, carry <- L + exp(A * sum_delta) * carry. The carry entering
// segment s from later time (zero for the last) replaces the aggregate in the first sub-slot
// of s; slot 0 receives the carry entering segment 0.
__global__ void scan_bwd_compose_kernel(const BwdParams p) {
  pdl_wait();   // the pre-pass's aggregates are visible
  const size_t dn = (size_t)p.Di * p.N;
  const size_t total = (size_t)p.batch * dn;
  const int nslot = p.nseg * p.nsub;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t b = e / dn, q = e % dn;
    const size_t d = q / p.N;
    const float a2 = inb(q, 1, dn) ? -expf(p.A_log[q]) * kLog2e : 0.f;
    float carry = 0.f;
    for (int sg = p.nseg - 1; sg >= 1; --sg) {
      const float carry_in = carry;
      // eight sub-slots at a time: their loads do not depend on the carry, so they are all in
      // flight together (a missing slot reads as L = 0, sum 0: the identity)
      for (int j0 = p.nsub - 1; j0 >= 0; j0 -= 8) {
        float Lv[8], sv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int j = j0 - k;
          const size_t row = b * nslot + (size_t)sg * p.nsub + (j >= 0 ? j : 0);
          const bool in = j >= 0 && inb(row * dn + q, 1, p.n_agg_l()) &&
                          inb(row * p.Di + d, 1, p.n_agg_sd());
          Lv[k] = in ? p.agg_L[row * dn + q] : 0.f;
          sv[k] = in ? p.agg_sd[row * p.Di + d] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) carry = fmaf(ex2_sfu(sv[k] * a2), carry, Lv[k]);
      }
      const size_t o = (b * nslot + (size_t)sg * p.nsub) * dn + q;
      if (inb(o, 1, p.n_agg_l())) p.agg_L[o] = carry_in;
    }
    if (inb((b * nslot) * dn + q, 1, p.n_agg_l())) p.agg_L[(b * nslot) * dn + q] = carry;
  }
}

// Forward recurrence of step i of the staged chunk on the thread's 2 x 4 states hc.
template <int NP, int DC, int NPR>
__device__ __forceinline__ void bwd_step_fwd(int i, const float* s_dl, const float* s_u,
                                             const float* s_B, int cl, int n0,
                                             const float2 (&a2)[kDPT][NPR],
                                             float2 (&hc)[kDPT][NPR]) {
  const float2 dlv = lds2(s_dl + i * DC + cl);
  const float2 uv = lds2(s_u + i * DC + cl);
  float2 Bp[NPR];
  lds_pairs<NPR>(s_B + i * NP + n0, Bp);
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const float dl = j ? dlv.y : dlv.x;
    const float uu = j ? uv.y : uv.x;
    const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
#pragma unroll
    for (int pp = 0; pp < NPR; ++pp) {
      const float2 da = ex2_2(mul2(dl2, a2[j][pp]));
      hc[j][pp] = fma2(da, hc[j][pp], mul2(du2, Bp[pp]));
    }
  }
}

template <int NP, bool VEC>
__global__ void __launch_bounds__(kWarps * 32)
scan_bwd_kernel(const BwdParams p) {
  using S = BwdShape<NP>;
  constexpr int G = S::G, DW = S::DW, DC = S::DC, P = S::P, NTH = kWarps * 32;
  constexpr int NPT = S::NPT, NPR = S::NPR, kSub = S::kSub, kNSub = S::kNSub;
  extern __shared__ __align__(16) float smem[];
  float* red = smem + kBwdStages * S::kStageFloats;   // [kWarps][kChunk][2*NP]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int blk = blockIdx.x % p.nblk, seg = blockIdx.x / p.nblk;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * kDPT;
  const int d0 = dblk0 + cl;
  const int n0 = ng * NPT;
  const int Di = p.Di, N = p.N, T = p.T;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(p.nchunks, c_begin + p.seg_chunks);

  float2 a2[kDPT][NPR], dh[kDPT][NPR], accA[kDPT][NPR];
  float Dd[kDPT], dD[kDPT];
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    const bool dv = d < Di;
    Dd[j] = (dv && inb(d, 1, Di)) ? p.D[d] : 0.f;
    dD[j] = 0.f;
    float t4[NPT];
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      const int n = n0 + k;
      t4[k] = (dv && n < N && inb((size_t)d * N + n, 1, (size_t)Di * N))
                  ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NPR; ++q) {
      a2[j][q] = make_float2(t4[2 * q], t4[2 * q + 1]);
      dh[j][q] = accA[j][q] = make_float2(0.f, 0.f);
    }
  }

  using RSn = ReduceScatter<4 * P, G / 2, 1>;    // (A-term, B-term) x 2 channels x P steps
  using RSd = ReduceScatter<2 * NPT, 16, G>;      // (d_B x NPT, d_C x NPT) over channel lanes
  const int nbase = RSn::base(lane);
  constexpr int kN = RSn::kept();
  const int dbase = RSd::base(lane);
  const bool dwriter = RSd::writer(lane);
  constexpr int kD = RSd::kept();
  const size_t rowb = (size_t)b * T;
  const int last = c_end - 1;           // chunks of this segment, walked last to first
  const int nck = c_end - c_begin;

#pragma unroll
  for (int s = 0; s < kBwdStages - 1; ++s) {
    if (s < nck) bwd_load_chunk<NP, VEC>(p, smem + s * S::kStageFloats, last - s, b, dblk0);
    else cp_async_commit();
  }

  // d_h entering the segment from the future: compose the later segments' aggregates,
  // d_h <- L + exp(A * sum(delta)) * d_h, from the last segment down to seg + 1
  for (int sp = p.nseg - 1; sp > seg; --sp) {
#pragma unroll
    for (int j = 0; j < kDPT; ++j) {
      const int d = d0 + j;
      const size_t row = ((size_t)b * p.nseg + sp) * Di + d;
      if (d >= Di || !inb(row, 1, p.n_agg_sd()) || !inb(row * N, N, p.n_agg_l())) continue;
      const float sd = p.agg_sd[row];
      float2 Lv[NPR];
      if constexpr (VEC) {
        if (n0 < N) {
          ld_pairs<NPR>(p.agg_L + row * N + n0, Lv);
        } else {
#pragma unroll
          for (int q = 0; q < NPR; ++q) Lv[q] = make_float2(0.f, 0.f);
        }
      } else {
#pragma unroll
        for (int q = 0; q < NPR; ++q) {
          const int n = n0 + 2 * q;
          Lv[q] = make_float2(n < N ? p.agg_L[row * N + n] : 0.f,
                              n + 1 < N ? p.agg_L[row * N + n + 1] : 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < NPR; ++q)
        dh[j][q] = fma2(ex2_2(mul2(splat2(sd), a2[j][q])), dh[j][q], Lv[q]);
    }
  }

  for (int it = 0; it < nck; ++it) {
    const int c = last - it;
    cp_async_wait<kBwdStages - 2>();
    __syncthreads();
    {
      const int itn = it + kBwdStages - 1;
      if (itn < nck)
        bwd_load_chunk<NP, VEC>(p, smem + (itn % kBwdStages) * S::kStageFloats, last - itn, b,
                                dblk0);
      else
        cp_async_commit();
    }
    float* st = smem + (it % kBwdStages) * S::kStageFloats;
    float* const s_dlw = st;
    const float* s_dl = st;
    const float* s_u = st + kChunk * DC;
    float* s_g = st + 2 * kChunk * DC;    // becomes d_y
    float* s_dy = st + 3 * kChunk * DC;   // becomes d_delta/d_raw (softplus variant)
    const float* s_B = st + 4 * kChunk * DC;
    const float* s_C = s_B + kChunk * NP;
    const float* s_y = s_C + kChunk * NP + DC * NP;
    const int t0 = c * kChunk;

    // ---- 0. gating backward (Phase B2) for the whole chunk tile: d_y into the gate tile, and
    // d_gate = dy * y * s * (1 + g*(1 - s)) straight to global memory, with the y the forward
    // kept (coalesced along d)
    static_assert((kChunk * DC) % NTH == 0, "tile must split evenly over the CTA");
#pragma unroll
    for (int k = 0; k < kChunk * DC / NTH; ++k) {
      const int e = k * NTH + threadIdx.x;
      const int i = e / DC, col = e % DC;
      const size_t o = (rowb + t0 + i) * Di + dblk0 + col;
      const bool ok = (t0 + i < T) && (dblk0 + col < Di) && inb(o, 1, p.n_io());
      const float yv = s_y[e];
      const float g = s_g[e], go = s_dy[e];
      const float s = sigmoid_fast(g);
      s_g[e] = go * (g * s);
      st_global_if(p.d_gate + o, go * yv * (s * fmaf(g, 1.f - s, 1.f)), ok);
      if (p.softplus && ok) {   // raw -> delta, and the factor d_raw / d_delta
        softplus_both(s_dlw[e], s_dlw[e], s_dy[e]);
      }
    }
    __syncthreads();

    // ---- 1./2. recompute + reverse, one sub-block of kSub steps at a time ----------------
    // The sub-block start states come from one recompute pass without stash. Then, for each
    // sub-block from last to first, the states are recomputed into registers and walked in
    // reverse. That is 1.5x the recompute work of a full-chunk stash, but half the registers.
    // the chunk's starting state, staged with the chunk (zeros for chunk 0)
    const float* s_h0 = s_C + kChunk * NP;
    float2 hsub[kNSub][kDPT][NPR];
#pragma unroll
    for (int j = 0; j < kDPT; ++j) {
      const int e = (cl + j) * N + n0;
      if constexpr (VEC) {
        if (n0 < N) {
          lds_pairs<NPR>(s_h0 + e, hsub[0][j]);
        } else {
#pragma unroll
          for (int q = 0; q < NPR; ++q) hsub[0][j][q] = make_float2(0.f, 0.f);
        }
      } else {
        float hv[NPT];
#pragma unroll
        for (int k = 0; k < NPT; ++k) hv[k] = (n0 + k < N && d0 + j < Di) ? s_h0[e + k] : 0.f;
#pragma unroll
        for (int q = 0; q < NPR; ++q) hsub[0][j][q] = make_float2(hv[2 * q], hv[2 * q + 1]);
      }
    }
    {
      float2 hc[kDPT][NPR];
#pragma unroll
      for (int j = 0; j < kDPT; ++j)
#pragma unroll
        for (int q = 0; q < NPR; ++q) hc[j][q] = hsub[0][j][q];
#pragma unroll
      for (int sb = 1; sb < kNSub; ++sb) {
#pragma unroll 1
        for (int q = 0; q < kSub; ++q)   // no stash here: a rolled loop keeps the code small
          bwd_step_fwd<NP, DC, NPR>((sb - 1) * kSub + q, s_dl, s_u, s_B, cl, n0, a2, hc);
#pragma unroll
        for (int j = 0; j < kDPT; ++j)
#pragma unroll
          for (int q = 0; q < NPR; ++q) hsub[sb][j][q] = hc[j][q];
      }
    }

#pragma unroll
    for (int sq = 0; sq < kNSub; ++sq) {
      const int sb = kNSub - 1 - sq;
      float2 hs[kSub][kDPT][NPR];
      {
        float2 hc[kDPT][NPR];
#pragma unroll
        for (int j = 0; j < kDPT; ++j)
#pragma unroll
          for (int q = 0; q < NPR; ++q) hc[j][q] = hsub[sb][j][q];
#pragma unroll
        for (int q = 0; q < kSub; ++q) {
          bwd_step_fwd<NP, DC, NPR>(sb * kSub + q, s_dl, s_u, s_B, cl, n0, a2, hc);
#pragma unroll
          for (int j = 0; j < kDPT; ++j)
#pragma unroll
            for (int qq = 0; qq < NPR; ++qq) hs[q][j][qq] = hc[j][qq];
        }
      }
#pragma unroll
      for (int gq = 0; gq < kSub / P; ++gq) {
        const int gl = kSub / P - 1 - gq;          // group inside the sub-block
        float vn[4 * P];
#pragma unroll
        for (int tq = 0; tq < P; ++tq) {
          const int tt = P - 1 - tq;
          const int q = gl * P + tt;               // step inside the sub-block
          const int i = sb * kSub + q;             // step inside the chunk
          const float2 dlv = lds2(s_dl + i * DC + cl);
          const float2 uv = lds2(s_u + i * DC + cl);
          const float2 dyv = lds2(s_g + i * DC + cl);
          float2 Bp[NPR], Cp[NPR], xb[NPR], xc[NPR];
          lds_pairs<NPR>(s_B + i * NP + n0, Bp);
          lds_pairs<NPR>(s_C + i * NP + n0, Cp);
#pragma unroll
          for (int pp = 0; pp < NPR; ++pp) xb[pp] = xc[pp] = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < kDPT; ++j) {
            const float dl = j ? dlv.y : dlv.x;
            const float uu = j ? uv.y : uv.x;
            const float dyj = j ? dyv.y : dyv.x;
            const float2 dl2 = splat2(dl), du2 = splat2(dl * uu), dy2 = splat2(dyj);
            float2 sa = make_float2(0.f, 0.f), sb2 = sa;
#pragma unroll
            for (int pp = 0; pp < NPR; ++pp) {
              const float2 hcur = hs[q][j][pp];
              const float2 hprev = (q > 0) ? hs[q > 0 ? q - 1 : 0][j][pp] : hsub[sb][j][pp];
              const float2 da = ex2_2(mul2(dl2, a2[j][pp]));
              const float2 gh = fma2(dy2, Cp[pp], dh[j][pp]);   // d_h += d_y*C
              const float2 cr = mul2(da, gh);                    // carried to t-1
              const float2 r = mul2(cr, hprev);                  // d_h*da*h_{t-1}
              accA[j][pp] = fma2(r, dl2, accA[j][pp]);
              sa = fma2(a2[j][pp], r, sa);
              sb2 = fma2(gh, Bp[pp], sb2);
              xb[pp] = fma2(gh, du2, xb[pp]);
              xc[pp] = fma2(dy2, hcur, xc[pp]);
              dh[j][pp] = cr;
            }
            vn[(tt * 2 + j) * 2 + 0] = sa.x + sa.y;
            vn[(tt * 2 + j) * 2 + 1] = sb2.x + sb2.y;
            dD[j] = fmaf(dyj, uu, dD[j]);
          }
          // d_B / d_C of this step: sum over the warp's channels
          float vd[2 * NPT];
#pragma unroll
          for (int pp = 0; pp < NPR; ++pp) {
            vd[2 * pp] = xb[pp].x;
            vd[2 * pp + 1] = xb[pp].y;
            vd[NPT + 2 * pp] = xc[pp].x;
            vd[NPT + 2 * pp + 1] = xc[pp].y;
          }
          RSd::run(vd, lane);
#pragma unroll
          for (int r = 0; r < kD; ++r) {
            const int idx = dbase + r;   // < NPT: d_B of state n0+idx, else d_C of n0+idx-NPT
            st_shared_if(red + (warp * kChunk + i) * 2 * NP + (idx / NPT) * NP + n0 + (idx % NPT),
                         vd[r], dwriter);
          }
        }
        // sums over n, scattered so that each lane finishes one (step, channel)
        RSn::run(vn, lane);
#pragma unroll
        for (int r = 0; r < kN / 2; ++r) {
          const int qq = nbase / 2 + r;
          const int tt = qq >> 1, j = qq & 1;
          const int i = sb * kSub + gl * P + tt;
          const int t = t0 + i, d = d0 + j;
          const int e = i * DC + cl + j;
          const float uu = s_u[e], dl = s_dl[e], dyj = s_g[e];
          const float Dj = j ? Dd[1] : Dd[0];
          const float sA = vn[2 * r], sB = vn[2 * r + 1];
          const size_t o = (rowb + t) * Di + d;
          const bool ok = (t < T) && (d < Di) && inb(o, 1, p.n_io());
          const float fac = p.softplus ? s_dy[e] : 1.f;
          st_global_if(p.d_delta + o, fmaf(sA, kLn2, uu * sB) * fac, ok);
          st_global_if(p.d_u + o, fmaf(dyj, Dj, dl * sB), ok);
        }
      }
    }
    __syncthreads();
    // CTA partial of d_B / d_C for this chunk: fixed-order sum over the warps
    for (int e = threadIdx.x; e < kChunk * 2 * NP; e += NTH) {
      const int i = e / (2 * NP), kn = e % (2 * NP);
      const int kind = kn / NP, n = kn % NP;
      const int t = t0 + i;
      if (t < T && n < N) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[(w * kChunk + i) * 2 * NP + kn];
        const size_t o = (((size_t)blk * p.batch + b) * T + t) * N + n;
        if (inb(o, 1, p.n_part_bc())) (kind ? p.partC : p.partB)[o] = sum;
      }
    }
  }
  cp_async_wait<0>();

  // per-(batch, segment) partials of d_A_log (= A * sum_t delta*r = ln2*a2*accA) and d_D
#pragma unroll
  for (int j = 0; j < kDPT; ++j) {
    const int d = d0 + j;
    const size_t row = ((size_t)b * p.nseg + seg) * Di + d;
    if (d >= Di || !inb(row, 1, p.n_part_d()) || !inb(row * N, N, p.n_part_a())) continue;
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      const float2 aa = a2[j][k >> 1], ac = accA[j][k >> 1];
      if (n0 + k < N) p.partA[row * N + n0 + k] = kLn2 * ((k & 1) ? aa.y * ac.y : aa.x * ac.x);
    }
    if (ng == 0) p.partD[row] = dD[j];
  }
}

// Fixed-order sums of the partials: d_B/d_C over CTAs along d, d_A_log/d_D over
// (batch, segment).
__global__ void scan_reduce_kernel(const BwdParams p) {
  pdl_wait();   // the backward's partials are visible
  const size_t btn = (size_t)p.batch * p.T * p.N;
  const size_t dn = (size_t)p.Di * p.N;
  const size_t total = btn + dn + (size_t)p.Di;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    if (e < btn) {
      float sb = 0.f, sc = 0.f;
      for (int k = 0; k < p.nblk; ++k) {
        if (!inb((size_t)k * btn + e, 1, p.n_part_bc())) break;
        sb += p.partB[(size_t)k * btn + e];
        sc += p.partC[(size_t)k * btn + e];
      }
      if (p.io_bf16) {   // the fused bf16 call: d_B, d_C in bf16 (rounded to nearest even)
        const uint32_t w = pack_bf16x2(sb, sc);
        reinterpret_cast<uint16_t*>(p.d_B)[e] = (uint16_t)(w & 0xffffu);
        reinterpret_cast<uint16_t*>(p.d_C)[e] = (uint16_t)(w >> 16);
      } else {
        p.d_B[e] = sb;
        p.d_C[e] = sc;
      }
    } else if (e < btn + dn) {
      const size_t q = e - btn;
      float sa = 0.f;
      for (int k = 0; k < p.batch * p.nseg; ++k)
        if (inb((size_t)k * dn + q, 1, p.n_part_a())) sa += p.partA[(size_t)k * dn + q];
      p.d_A_log[q] = sa;
    } else {
      const size_t q = e - btn - dn;
      float sd = 0.f;
      for (int k = 0; k < p.batch * p.nseg; ++k)
        if (inb((size_t)k * p.Di + q, 1, p.n_part_d())) sd += p.partD[(size_t)k * p.Di + q];
      p.d_D[q] = sd;
    }
  }
}

template <int NP, bool VEC>
static int launch_np(const Plan& plan, const BwdParams& p0, cudaStream_t s) {
  BwdParams p = p0;
  using S = BwdShape<NP>;
  if (cudaFuncSetAttribute(scan_bwd_kernel<NP, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)S::kSmemBytes) != cudaSuccess)
    return -1;
  int n = 0;
  if (plan.bwd.nseg > 1) {
    using A = BwdAggShape<NP>;
    if (cudaFuncSetAttribute(scan_bwd_agg_kernel<NP, VEC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)A::kSmemBytes) != cudaSuccess)
      return -1;
    const int nblk_a = (int)((plan.Di + A::DC - 1) / A::DC);
    const int ngrp = (plan.bwd.nseg - 1) * plan.bwd.nsub;
    dim3 ga((unsigned)(nblk_a * ngrp), (unsigned)plan.batch);
    scan_bwd_agg_kernel<NP, VEC><<<ga, A::NTH, A::kSmemBytes, s>>>(p);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    ++n;
  }
  dim3 grid((unsigned)(plan.bwd.nblk * plan.bwd.nseg), (unsigned)plan.batch);
  scan_bwd_kernel<NP, VEC><<<grid, kWarps * 32, S::kSmemBytes, s>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? n + 1 : -1;
}

// d_state > 8: the pre-pass of scan_bwd_tmem.cu, the composition of its aggregates, then the
// tensor-memory main kernel.
template <int NP>
static int launch_agg_tmem(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  int na = launch_bwd_agg_tmem(plan, p, s);
  if (na < 0) return -1;
  if (plan.bwd.nseg > 1) {
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (launch_pdl(scan_bwd_compose_kernel, dim3(sms * 4), dim3(256), 0, s, p) != cudaSuccess)
      return -1;
    ++na;
  }
  const int nm = launch_bwd_main_tmem(plan, p, s);
  return nm < 0 ? -1 : na + nm;
}

template <int NP>
static int launch_vec(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  const bool vec = (plan.Di % 4 == 0) && (plan.N % 4 == 0);
  return vec ? launch_np<NP, true>(plan, p, s) : launch_np<NP, false>(plan, p, s);
}

// d_state 9..64: the segment pre-pass and the composition of its aggregates into carries
// (they read only inputs), and then, separately, the backward and the reduction.
int launch_bwd_carries(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  if (plan.NP < kTmemMinNP) return -1;
  int n = launch_bwd_agg_tmem(plan, p, s);
  if (n < 0) return -1;
  if (plan.bwd.nseg > 1) {
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (launch_pdl(scan_bwd_compose_kernel, dim3(sms * 4), dim3(256), 0, s, p) != cudaSuccess)
      return -1;
    ++n;
  }
  return n;
}

int launch_bwd_after_carries(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  if (plan.NP < kTmemMinNP) return -1;
  const int nm = launch_bwd_main_tmem(plan, p, s);
  if (nm < 0) return -1;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (launch_pdl(scan_reduce_kernel, dim3(sms * 4), dim3(256), 0, s, p) != cudaSuccess)
    return -1;
  return nm + 1;
}

int launch_bwd(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  int n;
  switch (plan.NP) {
    case 4: n = launch_vec<4>(plan, p, s); break;
    case 8: n = launch_vec<8>(plan, p, s); break;
    case 16: n = launch_agg_tmem<16>(plan, p, s); break;
    case 32: n = launch_agg_tmem<32>(plan, p, s); break;
    case 64: n = launch_agg_tmem<64>(plan, p, s); break;
    default: return -1;
  }
  if (n < 0) return -1;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (launch_pdl(scan_reduce_kernel, dim3(sms * 4), dim3(256), 0, s, p) != cudaSuccess)
    return -1;
  return cudaPeekAtLastError() == cudaSuccess ? n + 1 : -1;
}

MSCAN_OOB_HOOKS(bwd)

}  // namespace mscan
