// Forward selective scan (sm_103a).
//
// What it computes, for every row (b, d) and state n (h_{-1} = 0, A = -exp(A_log)):
//   h_t = exp(delta_t * A) * h_{t-1} + delta_t * u_t * B_t[n]
//   y_t = sum_n C_t[n] * h_t + D * u_t,     out_t = y_t * SiLU(gate_t)
// The Phase B3 SSM BPTT of mamba-rs src/mamba_ssm/cpu/backward.rs is the derivative of this
// recurrence. That page precomputes a_neg = -exp(A_log) (its "O3"). Here the same constant
// lives in registers with log2(e) folded in (a2), so a step costs one ex2 per state.
//
// Mapping. grid = (ceil(d_inner / DC), batch). A CTA owns one batch row b and DC consecutive
// channels, and walks the whole time axis for them in chunks of kChunk steps.
//   lane = dg * G + ng :  ng picks the states [NPT*ng, NPT*ng+NPT), and dg picks the DPT
//                         channels [DPT*dg, DPT*dg+DPT) of the warp's DPT*(32/G) channels.
// A thread keeps DPT channels (2, or 4 at d_state 64) x NPT states in registers as float2 pairs
// of states and updates them with packed fp32x2 FMAs.
//
// Staging. Each chunk's tiles (delta, u and gate [kChunk][DC]; B and C [kChunk][NP]) go
// global -> shared with cp.async, STAGES chunks ahead of the compute. Rows past T and channels
// past d_inner arrive as zeros. For those the recurrence is an exact no-op (decay 1, input 0),
// so the control flow needs no tail special cases.
//
// y = sum_n C*h. In-thread FMAs first, then a butterfly reduce-scatter over the G state
// lanes, batched over P = G/DPT steps. It leaves each lane the complete y of one (step,
// channel) (two when G < DPT). That lane then applies D*u and the SiLU gate and stores out. So no
// sigmoid is computed twice.
//
// Every kChunk steps the state goes to the checkpoint buffer [batch][chunk][d][n] (the state
// after chunk 0 .. nchunks-2). The backward restarts each chunk from these states.
#include "scan_common.cuh"

namespace mscan {

constexpr int kFwdStages = 4;

// The DPT consecutive channels of a thread from one staged row (8- or 16-byte aligned).
template <int DPT>
__device__ __forceinline__ void lds_chan(const float* p, float (&v)[DPT]) {
  static_assert(DPT == 2 || DPT == 4, "2 or 4 channels per thread");
  if constexpr (DPT == 2) {
    const float2 t = lds2(p);
    v[0] = t.x;
    v[1] = t.y;
  } else {
    const float4 t = lds4(p);
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
  }
}

template <int NP>
struct FwdShape {
  static constexpr int NPT = states_per_thread_fwd(NP);    // states per thread
  static constexpr int NPR = NPT / 2;                  // float2 pairs of states per thread
  static constexpr int DPT = fwd_channels_per_thread(NP);   // channels per thread
  static constexpr int G = NP / NPT;                   // lanes per channel group
  static constexpr int DW = (32 / G) * DPT;            // channels per warp
  static constexpr int DC = kFwdWarps * DW;            // channels per CTA
  static constexpr int P = G >= DPT ? G / DPT : 1;     // steps per output group
  static constexpr int kStageFloats = kChunk * (3 * DC + 2 * NP);
  static constexpr size_t kSmemBytes = (size_t)kFwdStages * kStageFloats * sizeof(float);
};

template <int NP, bool VEC, bool ST = false, bool BF = false>
__device__ __forceinline__ void fwd_load_chunk(const FwdParams& p, float* st, int c, int b,
                                               int dblk0) {
  using S = FwdShape<NP>;
  constexpr int DC = S::DC, NTH = kFwdWarps * 32;
  float* s_dl = st;
  float* s_u = st + kChunk * DC;
  float* s_g = st + 2 * kChunk * DC;
  float* s_B = st + 3 * kChunk * DC;
  float* s_C = s_B + kChunk * NP;
  const int t0 = c * kChunk;
  const size_t rowb = (size_t)b * p.T;
  if constexpr (BF) {
    // bf16 tiles into the slots the states-only forward leaves unused: delta and u share the
    // gate slot (a half each), B takes the first half of the C slot; they are widened into
    // their own slots after the wait
    static_assert(ST && VEC, "bf16 input is taken by the states-only forward");
    stage_tile_bf16<DC, NTH>(s_g, reinterpret_cast<const uint16_t*>(p.delta), rowb, t0, p.T,
                             p.Di, dblk0);
    stage_tile_bf16<DC, NTH>(s_g + kChunk * DC / 2, reinterpret_cast<const uint16_t*>(p.u), rowb,
                             t0, p.T, p.Di, dblk0);
    stage_tile_bf16<NP, NTH>(s_C, reinterpret_cast<const uint16_t*>(p.B), rowb, t0, p.T, p.N, 0);
  } else if constexpr (VEC) {
    for (int q = threadIdx.x; q < kChunk * DC / 4; q += NTH) {
      const int i = q / (DC / 4), col = (q % (DC / 4)) * 4;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di;
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async16(s_dl + i * DC + col, p.delta + go, v);
      cp_async16(s_u + i * DC + col, p.u + go, v);
      if constexpr (!ST) cp_async16(s_g + i * DC + col, p.gate + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP / 4; q += NTH) {
      const int i = q / (NP / 4), n = (q % (NP / 4)) * 4;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N;
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async16(s_B + i * NP + n, p.B + go, v);
      if constexpr (!ST) cp_async16(s_C + i * NP + n, p.C + go, v);
    }
  } else {
    for (int q = threadIdx.x; q < kChunk * DC; q += NTH) {
      const int i = q / DC, col = q % DC;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di;
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async4(s_dl + i * DC + col, p.delta + go, v);
      cp_async4(s_u + i * DC + col, p.u + go, v);
      if constexpr (!ST) cp_async4(s_g + i * DC + col, p.gate + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP; q += NTH) {
      const int i = q / NP, n = q % NP;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N;
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async4(s_B + i * NP + n, p.B + go, v);
      if constexpr (!ST) cp_async4(s_C + i * NP + n, p.C + go, v);
    }
  }
  cp_async_commit();
}

// Segment pre-pass of the forward: for every segment but the last, run the recurrence from a
// zero state and keep the end state and the sum of delta over the segment, per (b, d, n).
// Since h_end = exp(A * sum(delta)) * h_start + h_end(from zero), the main kernel composes these
// to obtain the exact state entering each segment. A CTA covers kAggWarps warps of
// channels and agg_k consecutive segments, with the chunk pipeline running straight through the
// segment boundaries.
template <int NP>
struct FwdAggShape {
  using S = FwdShape<NP>;
  static constexpr int AW = kAggWarps;
  static constexpr int DC = AW * S::DW;
  static constexpr int NTH = AW * 32;
  static constexpr int kStages = 4;
  static constexpr int kStageFloats = kChunk * (2 * DC + NP);   // delta, u, B
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageFloats * sizeof(float);
};

template <int NP, bool VEC, bool BF = false>
__global__ void __launch_bounds__(kAggWarps * 32)
scan_fwd_agg_kernel(const FwdParams p) {
  using S = FwdShape<NP>;
  using A = FwdAggShape<NP>;
  constexpr int G = S::G, DW = S::DW, NPT = S::NPT, NPR = S::NPR, DC = A::DC, NTH = A::NTH;
  constexpr int DPT = S::DPT;
  extern __shared__ __align__(16) float smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int nblk_a = (p.Di + DC - 1) / DC;
  const int blk = blockIdx.x % nblk_a, grp = blockIdx.x / nblk_a;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * DPT;
  const int d0 = dblk0 + cl;
  const int n0 = ng * NPT;
  const int Di = p.Di, N = p.N, T = p.T;
  const int seg_lo = grp * p.agg_k;                       // segments 0 .. nseg-2 need aggregates
  const int seg_hi = min(p.nseg - 1, seg_lo + p.agg_k);
  const int c_begin = seg_lo * p.seg_chunks;
  const int c_end = min(p.nchunks, seg_hi * p.seg_chunks);
  const size_t row0 = (size_t)b * T;

  float2 a2[DPT][NPR], h[DPT][NPR];
  float sd[DPT];
#pragma unroll
  for (int j = 0; j < DPT; ++j) {
    const int d = d0 + j;
    const bool dv = d < Di;
    sd[j] = 0.f;
    float t4[NPT];
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      const int n = n0 + k;
      t4[k] = (dv && n < N) ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NPR; ++q) {
      a2[j][q] = make_float2(t4[2 * q], t4[2 * q + 1]);
      h[j][q] = make_float2(0.f, 0.f);
    }
  }

  auto load = [&](int stage, int c) {
    float* st = smem + stage * A::kStageFloats;
    if constexpr (BF) {   // bf16 tiles into the first half of each slot
      stage_tile_bf16<DC, NTH>(st, reinterpret_cast<const uint16_t*>(p.delta), row0, c * kChunk,
                               T, Di, dblk0);
      stage_tile_bf16<DC, NTH>(st + kChunk * DC, reinterpret_cast<const uint16_t*>(p.u), row0,
                               c * kChunk, T, Di, dblk0);
      stage_tile_bf16<NP, NTH>(st + 2 * kChunk * DC, reinterpret_cast<const uint16_t*>(p.B),
                               row0, c * kChunk, T, N, 0);
    } else {
      stage_tile<DC, NTH, VEC>(st, p.delta, row0, c * kChunk, T, Di, dblk0);
      stage_tile<DC, NTH, VEC>(st + kChunk * DC, p.u, row0, c * kChunk, T, Di, dblk0);
      stage_tile<NP, NTH, VEC>(st + 2 * kChunk * DC, p.B, row0, c * kChunk, T, N, 0);
    }
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
    if constexpr (BF) {   // widen the bf16 tiles in place
      BfTile<kChunk * DC, NTH> wdl, wu;
      BfTile<kChunk * NP, NTH> wB;
      wdl.read(st);
      wu.read(st + kChunk * DC);
      wB.read(st + 2 * kChunk * DC);
      __syncthreads();
      wdl.write(st);
      wu.write(st + kChunk * DC);
      wB.write(st + 2 * kChunk * DC);
      __syncthreads();
    }
    if (p.softplus) {   // raw delta -> delta in shared memory, once per element
      softplus_tile<DC, NTH>(st, T - c * kChunk, Di - dblk0);
      __syncthreads();
    }
    const float* s_dl = st;
    const float* s_u = st + kChunk * DC;
    const float* s_B = st + 2 * kChunk * DC;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      float dlv[DPT], uv[DPT];
      lds_chan<DPT>(s_dl + i * DC + cl, dlv);
      lds_chan<DPT>(s_u + i * DC + cl, uv);
      float2 Bp[NPR];
      lds_pairs<NPR>(s_B + i * NP + n0, Bp);
#pragma unroll
      for (int j = 0; j < DPT; ++j) {
        const float dl = dlv[j];
        const float uu = uv[j];
        sd[j] += dl;
        const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
#pragma unroll
        for (int q = 0; q < NPR; ++q) {
          const float2 da = ex2_2(mul2(dl2, a2[j][q]));
          h[j][q] = fma2(da, h[j][q], mul2(du2, Bp[q]));
        }
      }
    }
    if ((c + 1) % p.seg_chunks == 0) {   // the last chunk of a segment: emit, then restart
      const int seg = c / p.seg_chunks;
#pragma unroll
      for (int j = 0; j < DPT; ++j) {
        const int d = d0 + j;
        if (d < Di) {
          const size_t row = ((size_t)b * p.nseg + seg) * Di + d;
          if (ng == 0) p.agg_sd[row] = sd[j];
          if constexpr (VEC) {
            st_pairs_row<NPR>(p.agg_h + row * N, n0, N, h[j]);   // N % 4 == 0 here
          } else {
#pragma unroll
            for (int k = 0; k < NPT; ++k)
              if (n0 + k < N)
                p.agg_h[row * N + n0 + k] = (k & 1) ? h[j][k >> 1].y : h[j][k >> 1].x;
          }
        }
        sd[j] = 0.f;
#pragma unroll
        for (int q = 0; q < NPR; ++q) h[j][q] = make_float2(0.f, 0.f);
      }
    }
  }
  cp_async_wait<0>();
}

// ST (states only, for the fused forward + backward call): the recurrence and the checkpoints
// alone; the backward then recomputes y from the states and writes out.
// BF (with ST): delta, u and B arrive as bf16 and are widened in shared memory.
template <int NP, bool VEC, bool WITH_Y, bool SP, bool ST, bool BF = false>
__global__ void __launch_bounds__(kFwdWarps * 32)
scan_fwd_kernel(const FwdParams p) {
  static_assert(!(ST && (SP || WITH_Y)), "the states-only forward takes the plain delta");
  static_assert(!BF || ST, "bf16 input is taken by the states-only forward");
  using S = FwdShape<NP>;
  constexpr int G = S::G, DW = S::DW, DC = S::DC, P = S::P, NPT = S::NPT, NPR = S::NPR;
  constexpr int DPT = S::DPT;
  extern __shared__ __align__(16) float smem[];
  pdl_wait();      // the previous kernel's writes (inputs, workspace) are visible
  pdl_release();   // one wave: the next kernel may take the room this one leaves

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane % G, dg = lane / G;
  const int b = blockIdx.y;
  const int blk = blockIdx.x % p.nblk, seg = blockIdx.x / p.nblk;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * DPT;    // first channel of this thread inside the CTA tile
  const int d0 = dblk0 + cl;
  const int n0 = ng * NPT;
  const int Di = p.Di, N = p.N, T = p.T;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(p.nchunks, c_begin + p.seg_chunks);

  float2 a2[DPT][NPR], h[DPT][NPR];
  float Dd[DPT];
#pragma unroll
  for (int j = 0; j < DPT; ++j) {
    const int d = d0 + j;
    const bool dv = d < Di;
    Dd[j] = dv ? p.D[d] : 0.f;
    float t4[NPT];
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      const int n = n0 + k;
      t4[k] = (dv && n < N) ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NPR; ++q) {
      a2[j][q] = make_float2(t4[2 * q], t4[2 * q + 1]);
      h[j][q] = make_float2(0.f, 0.f);
    }
  }

  using RSy = ReduceScatter<DPT * P, G / 2, 1>;
  const int ybase = RSy::base(lane);
  constexpr int kY = RSy::kept();
  const size_t rowb = (size_t)b * T;

#pragma unroll
  for (int s = 0; s < kFwdStages - 1; ++s) {
    if (c_begin + s < c_end)
      fwd_load_chunk<NP, VEC, ST, BF>(p, smem + s * S::kStageFloats, c_begin + s, b, dblk0);
    else
      cp_async_commit();
  }

  // state entering the segment: compose the earlier segments' aggregates,
  // h <- exp(A * sum(delta)) * h + (segment end state from zero)
  for (int sp = 0; sp < seg; ++sp) {
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      const int d = d0 + j;
      if (d >= Di) continue;
      const size_t row = ((size_t)b * p.nseg + sp) * Di + d;
      const float sd = p.agg_sd[row];
      float2 hl[NPR];
      if constexpr (VEC) {
        ld_pairs_row<NPR>(p.agg_h + row * N, n0, N, hl);
      } else {
#pragma unroll
        for (int q = 0; q < NPR; ++q) {
          const int n = n0 + 2 * q;
          hl[q] = make_float2(n < N ? p.agg_h[row * N + n] : 0.f,
                              n + 1 < N ? p.agg_h[row * N + n + 1] : 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < NPR; ++q)
        h[j][q] = fma2(ex2_2(mul2(splat2(sd), a2[j][q])), h[j][q], hl[q]);
    }
  }

  for (int c = c_begin; c < c_end; ++c) {
    const int it = c - c_begin;
    cp_async_wait<kFwdStages - 2>();
    __syncthreads();
    {
      const int cn = c + kFwdStages - 1;
      if (cn < c_end)
        fwd_load_chunk<NP, VEC, ST, BF>(
            p, smem + ((it + kFwdStages - 1) % kFwdStages) * S::kStageFloats, cn, b, dblk0);
      else
        cp_async_commit();
    }
    float* st = smem + (it % kFwdStages) * S::kStageFloats;
    if constexpr (BF) {   // widen the bf16 tiles into their slots (no overlap: one barrier)
      BfTile<kChunk * DC, kFwdWarps * 32> wdl, wu;
      BfTile<kChunk * NP, kFwdWarps * 32> wB;
      wdl.read(st + 2 * kChunk * DC);
      wu.read(st + 2 * kChunk * DC + kChunk * DC / 2);
      wB.read(st + 3 * kChunk * DC + kChunk * NP);
      wdl.write(st);
      wu.write(st + kChunk * DC);
      wB.write(st + 3 * kChunk * DC);
      __syncthreads();
    }
    if constexpr (SP) {   // raw delta -> delta in shared memory, once per element
      softplus_tile<DC, kFwdWarps * 32>(st, p.T - c * kChunk, p.Di - dblk0);
      __syncthreads();
    }
    const float* s_dl = st;
    const float* s_u = st + kChunk * DC;
    const float* s_g = st + 2 * kChunk * DC;
    const float* s_B = st + 3 * kChunk * DC;
    const float* s_C = s_B + kChunk * NP;
    const int t0 = c * kChunk;

    if constexpr (ST) {
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        float dlv[DPT], uv[DPT];
        lds_chan<DPT>(s_dl + i * DC + cl, dlv);
        lds_chan<DPT>(s_u + i * DC + cl, uv);
        float2 Bp[NPR];
        lds_pairs<NPR>(s_B + i * NP + n0, Bp);
#pragma unroll
        for (int j = 0; j < DPT; ++j) {
          const float dl = dlv[j];
          const float uu = uv[j];
          const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
#pragma unroll
          for (int pp = 0; pp < NPR; ++pp)
            h[j][pp] = fma2(ex2_2(mul2(dl2, a2[j][pp])), h[j][pp], mul2(du2, Bp[pp]));
        }
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < kChunk / P; ++gi) {
        float yv[DPT * P];
#pragma unroll
        for (int tt = 0; tt < P; ++tt) {
          const int i = gi * P + tt;
          float dlv[DPT], uv[DPT];
          lds_chan<DPT>(s_dl + i * DC + cl, dlv);
          lds_chan<DPT>(s_u + i * DC + cl, uv);
          float2 Bp[NPR], Cp[NPR];
          lds_pairs<NPR>(s_B + i * NP + n0, Bp);
          lds_pairs<NPR>(s_C + i * NP + n0, Cp);
#pragma unroll
          for (int j = 0; j < DPT; ++j) {
            const float dl = dlv[j];
            const float uu = uv[j];
            const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
            float2 ya = make_float2(0.f, 0.f);
#pragma unroll
            for (int pp = 0; pp < NPR; ++pp) {
              const float2 da = ex2_2(mul2(dl2, a2[j][pp]));
              h[j][pp] = fma2(da, h[j][pp], mul2(du2, Bp[pp]));
              ya = fma2(Cp[pp], h[j][pp], ya);
            }
            yv[tt * DPT + j] = ya.x + ya.y;
          }
        }
        RSy::run(yv, lane);
#pragma unroll
        for (int r = 0; r < kY; ++r) {
          const int idx = ybase + r;
          const int tt = idx / DPT, j = idx % DPT;
          const int i = gi * P + tt;
          const int t = t0 + i, d = d0 + j;
          const float uu = s_u[i * DC + cl + j];
          const float g = s_g[i * DC + cl + j];
          float Dj = Dd[0];   // Dd[j] without a dynamically indexed register array
#pragma unroll
          for (int k = 1; k < DPT; ++k) Dj = j == k ? Dd[k] : Dj;
          const float y = fmaf(Dj, uu, yv[r]);
          const bool ok = (t < T) && (d < Di);
          const size_t o = (rowb + t) * Di + d;
          st_global_if(p.out + o, y * (g * sigmoid_fast(g)), ok);
          st_global_if(p.y_ck + o, y, ok);            // kept for the backward's d_gate
          if constexpr (WITH_Y) st_global_if(p.y + o, y, ok);
        }
      }
    }

    if (c + 1 < p.nchunks) {
      float* ck = p.ckpt + ((size_t)b * (p.nchunks - 1) + c) * (size_t)Di * N;
#pragma unroll
      for (int j = 0; j < DPT; ++j) {
        const int d = d0 + j;
        if (d >= Di) continue;
        if constexpr (VEC) {
          st_pairs_row<NPR>(ck + (size_t)d * N, n0, N, h[j]);
        } else {
#pragma unroll
          for (int k = 0; k < NPT; ++k)
            if (n0 + k < N) ck[(size_t)d * N + n0 + k] = (k & 1) ? h[j][k >> 1].y : h[j][k >> 1].x;
        }
      }
    }
  }
  cp_async_wait<0>();
}

template <int NP, bool VEC, bool WITH_Y>
static int launch_np(const Plan& plan, const FwdParams& p0, cudaStream_t s) {
  FwdParams p = p0;
  using S = FwdShape<NP>;
  auto kern = p0.states_only ? scan_fwd_kernel<NP, VEC, false, false, true>
             : p0.softplus   ? scan_fwd_kernel<NP, VEC, WITH_Y, true, false>
                             : scan_fwd_kernel<NP, VEC, WITH_Y, false, false>;
  auto agg = scan_fwd_agg_kernel<NP, VEC>;
  if constexpr (NP >= kTmemMinNP && VEC && !WITH_Y && S::DC % 8 == 0) {   // bf16 fused call
    if (p0.io_bf16) {
      kern = scan_fwd_kernel<NP, true, false, false, true, true>;
      agg = scan_fwd_agg_kernel<NP, true, true>;
    }
  } else {
    if (p0.io_bf16) return -1;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)S::kSmemBytes) != cudaSuccess)
    return -1;
  int n = 0;
  if (plan.fwd.nseg > 1) {
    using A = FwdAggShape<NP>;
    if (cudaFuncSetAttribute(agg, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)A::kSmemBytes) != cudaSuccess)
      return -1;
    const int nblk_a = (int)((plan.Di + A::DC - 1) / A::DC);
    p.agg_k = 1;   // one segment per CTA measured fastest (the kernel accepts more)
    const int ngrp = (plan.fwd.nseg - 1 + p.agg_k - 1) / p.agg_k;
    dim3 ga((unsigned)(nblk_a * ngrp), (unsigned)plan.batch);
    agg<<<ga, A::NTH, A::kSmemBytes, s>>>(p);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    ++n;
  }
  dim3 grid((unsigned)(plan.fwd.nblk * plan.fwd.nseg), (unsigned)plan.batch);
  if (launch_pdl(kern, grid, dim3(kFwdWarps * 32), S::kSmemBytes, s, p) != cudaSuccess)
    return -1;
  return n + 1;
}

template <int NP>
static int launch_vec(const Plan& plan, const FwdParams& p, cudaStream_t s) {
  const bool vec = (plan.Di % 4 == 0) && (plan.N % 4 == 0);
  if (p.y) return vec ? launch_np<NP, true, true>(plan, p, s) : launch_np<NP, false, true>(plan, p, s);
  return vec ? launch_np<NP, true, false>(plan, p, s) : launch_np<NP, false, false>(plan, p, s);
}

int launch_fwd(const Plan& plan, const FwdParams& p, cudaStream_t s) {
  switch (plan.NP) {
    case 4: return launch_vec<4>(plan, p, s);
    case 8: return launch_vec<8>(plan, p, s);
    case 16: return launch_vec<16>(plan, p, s);
    case 32: return launch_vec<32>(plan, p, s);
    case 64: return launch_vec<64>(plan, p, s);
    default: return -1;
  }
}

}  // namespace mscan
