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
// of channels, x[q][s] = (channel 2q, channel 2q+1) of state s, and updates them with packed
// fp32x2 FMAs: the per-channel delta*u and the sums over n then come out as channel pairs with
// no scalar multiply or horizontal add.
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
#include <string.h>

#include <mutex>

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

// The NPT/2 state pairs of channel k (0 or 1) of a channel pair x[s], s < NPT, for the row
// stores (checkpoints, aggregates) whose rows hold one channel's states.
template <int NPT>
__device__ __forceinline__ void chan_states(const float2 (&x)[NPT], int k, float2 (&out)[NPT / 2]) {
#pragma unroll
  for (int pp = 0; pp < NPT / 2; ++pp)
    out[pp] = k ? make_float2(x[2 * pp].y, x[2 * pp + 1].y) : make_float2(x[2 * pp].x, x[2 * pp + 1].x);
}

// element s of a float2 pair array (s compile-time)
__device__ __forceinline__ float pair_el(const float2* v, int s) {
  return (s & 1) ? v[s >> 1].y : v[s >> 1].x;
}

// a2[q][s] = A[d, n] * log2(e) = -exp(A_log[d, n]) * log2(e) for the channels d0 + 2q,
// d0 + 2q + 1 and the states n0 + s; zero outside d_inner x d_state (a no-op decay there).
template <int DP, int NPT>
__device__ __forceinline__ void load_a2(const FwdParams& p, int d0, int n0,
                                        float2 (&a2)[DP][NPT]) {
  const int Di = p.Di, N = p.N;
#pragma unroll
  for (int q = 0; q < DP; ++q)
#pragma unroll
    for (int s = 0; s < NPT; ++s) {
      float v[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int d = d0 + 2 * q + k, n = n0 + s;
        v[k] = (d < Di && n < N && inb((size_t)d * N + n, 1, (size_t)Di * N))
                   ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
      }
      a2[q][s] = make_float2(v[0], v[1]);
    }
}

// One step of the recurrence on the thread's channel pairs, h = exp(delta*A)*h + delta*u*B,
// from the step's delta and u of its 2*DP channels and the B pairs of its NPT states; dl2
// receives the delta pairs.
template <int DP, int NPT>
__device__ __forceinline__ void fwd_step(const float (&dlv)[2 * DP], const float (&uv)[2 * DP],
                                         const float2 (&Bp)[NPT / 2], const float2 (&a2)[DP][NPT],
                                         float2 (&h)[DP][NPT], float2 (&dl2)[DP]) {
#pragma unroll
  for (int q = 0; q < DP; ++q) {
    dl2[q] = make_float2(dlv[2 * q], dlv[2 * q + 1]);
    const float2 du2 = mul2(dl2[q], make_float2(uv[2 * q], uv[2 * q + 1]));
#pragma unroll
    for (int s = 0; s < NPT; ++s)
      h[q][s] = fma2(ex2_2(mul2(dl2[q], a2[q][s])), h[q][s], mul2(du2, splat2(pair_el(Bp, s))));
  }
}

template <int NP>
struct FwdShape {
  static constexpr int NPT = states_per_thread_fwd(NP);    // states per thread
  static constexpr int NPR = NPT / 2;                  // float2 pairs of states per thread
  static constexpr int DPT = fwd_channels_per_thread(NP);   // channels per thread
  static constexpr int G = NP / NPT;                   // lanes per channel group
  static constexpr int DW = (32 / G) * DPT;            // channels per warp
  static constexpr int NW = fwd_warps(NP);             // warps per CTA
  static constexpr int DC = NW * DW;                   // channels per CTA
  static constexpr int P = G >= DPT ? G / DPT : 1;     // steps per output group
  static constexpr int kStageFloats = kChunk * (3 * DC + 2 * NP);
  static constexpr size_t kSmemBytes = (size_t)kFwdStages * kStageFloats * sizeof(float);
  // TMA staging: 3 stages and their barriers (the 4 of the cp.async ring fill the shared memory
  // of 4 CTAs per SM at d_state 64 exactly, leaving no room for the barriers)
  static constexpr int kStagesTma = 3;
  static constexpr size_t kSmemBytesTma =
      (size_t)kStagesTma * kStageFloats * sizeof(float) + 8 * kStagesTma;
};

static __device__ unsigned int g_fwd_fault;   // set when a bounded copy wait gave up

// TMA staging (d_state 64, d_inner a multiple of 4, fp32): one thread issues the
// chunk's tiles into a stage laid out as the cp.async path lays it out (delta, u, gate tiles of
// [kChunk][DC], then B, C tiles of [kChunk][NP]; dst_g and dst_C null when not read), and the
// stage's barrier counts their bytes. Rows past T, channels past d_inner and states past
// d_state arrive as zeros.
template <int NP>
__device__ __forceinline__ void fwd_tma_tiles(const FwdMaps& maps, uint64_t* bar, int c, int b,
                                              int dblk0, float* dst_dl, float* dst_u,
                                              float* dst_g, float* dst_B, float* dst_C) {
  constexpr uint32_t kTile = (uint32_t)(kChunk * FwdShape<NP>::DC * 4), kBC = kChunk * NP * 4;
  if (threadIdx.x != 0) return;
  mbar_expect_tx(bar, 2 * kTile + (dst_g ? kTile : 0u) + kBC + (dst_C ? kBC : 0u));
  const int t0 = c * kChunk;
  tma_load_3d(dst_dl, &maps.delta, bar, dblk0, t0, b);
  tma_load_3d(dst_u, &maps.u, bar, dblk0, t0, b);
  if (dst_g) tma_load_3d(dst_g, &maps.gate, bar, dblk0, t0, b);
  tma_load_3d(dst_B, &maps.B, bar, 0, t0, b);
  if (dst_C) tma_load_3d(dst_C, &maps.C, bar, 0, t0, b);
}

// Waits until stage `stage` of a TMA ring holds chunk use number `use` (bounded; a wait that
// gives up sets the fault word and the kernel runs on with the stale stage).
__device__ __forceinline__ void fwd_tma_wait(uint64_t* bars, int stages, int it,
                                             unsigned long long limit_ns) {
  if (!mbar_wait(bars + it % stages, (uint32_t)((it / stages) & 1),
                 limit_ns ? limit_ns : kWaitLimitNs))
    atomicOr(&g_fwd_fault, 1u);
}

template <int NP, bool VEC, bool ST = false, bool BF = false>
__device__ __forceinline__ void fwd_load_chunk(const FwdParams& p, float* st, int c, int b,
                                               int dblk0) {
  using S = FwdShape<NP>;
  constexpr int DC = S::DC, NTH = S::NW * 32;
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
                             p.Di, dblk0, p.n_io());
    stage_tile_bf16<DC, NTH>(s_g + kChunk * DC / 2, reinterpret_cast<const uint16_t*>(p.u), rowb,
                             t0, p.T, p.Di, dblk0, p.n_io());
    stage_tile_bf16<NP, NTH>(s_C, reinterpret_cast<const uint16_t*>(p.B), rowb, t0, p.T, p.N, 0,
                             p.n_bc());
  } else if constexpr (VEC) {
    for (int q = threadIdx.x; q < kChunk * DC / 4; q += NTH) {
      const int i = q / (DC / 4), col = (q % (DC / 4)) * 4;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di && inb((rowb + t) * p.Di + d, 4, p.n_io());
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async16(s_dl + i * DC + col, p.delta + go, v);
      cp_async16(s_u + i * DC + col, p.u + go, v);
      if constexpr (!ST) cp_async16(s_g + i * DC + col, p.gate + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP / 4; q += NTH) {
      const int i = q / (NP / 4), n = (q % (NP / 4)) * 4;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N && inb((rowb + t) * p.N + n, 4, p.n_bc());
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async16(s_B + i * NP + n, p.B + go, v);
      if constexpr (!ST) cp_async16(s_C + i * NP + n, p.C + go, v);
    }
  } else {
    for (int q = threadIdx.x; q < kChunk * DC; q += NTH) {
      const int i = q / DC, col = q % DC;
      const int t = t0 + i, d = dblk0 + col;
      const bool v = t < p.T && d < p.Di && inb((rowb + t) * p.Di + d, 1, p.n_io());
      const size_t go = v ? (rowb + t) * p.Di + d : 0;
      cp_async4(s_dl + i * DC + col, p.delta + go, v);
      cp_async4(s_u + i * DC + col, p.u + go, v);
      if constexpr (!ST) cp_async4(s_g + i * DC + col, p.gate + go, v);
    }
    for (int q = threadIdx.x; q < kChunk * NP; q += NTH) {
      const int i = q / NP, n = q % NP;
      const int t = t0 + i;
      const bool v = t < p.T && n < p.N && inb((rowb + t) * p.N + n, 1, p.n_bc());
      const size_t go = v ? (rowb + t) * p.N + n : 0;
      cp_async4(s_B + i * NP + n, p.B + go, v);
      if constexpr (!ST) cp_async4(s_C + i * NP + n, p.C + go, v);
    }
  }
  cp_async_commit();
}

// Segment pre-pass of the forward: for every segment but the last, run the recurrence from a
// zero state and keep the end state and the sum of delta over the segment, per (b, d, n).
// Since h_end = exp(A * sum(delta)) * h_start + h_end(from zero), scan_fwd_compose_kernel
// composes these into the exact state entering each segment. A CTA has the main kernel's warps
// and channels (its tensor-copy boxes are the main kernel's) and agg_k consecutive segments,
// with the chunk pipeline running straight through the segment boundaries.
template <int NP>
struct FwdAggShape {
  using S = FwdShape<NP>;
  static constexpr int AW = S::NW;   // the main kernel's CTA shape
  static constexpr int DC = AW * S::DW;
  static constexpr int NTH = AW * 32;
  // 3 stages: at d_state 64 the pre-pass then keeps 7 CTAs per SM (its registers' limit)
  // instead of 6 (its shared memory's with 4 stages); measured on GB300, the longseq forward
  // call took 3.65 ms against 3.67 with 4 stages (and 3.65 with 2)
  static constexpr int kStages = 3;
  static constexpr int kStageFloats = kChunk * (2 * DC + NP);   // delta, u, B
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageFloats * sizeof(float);
  static constexpr size_t kSmemBytesTma = kSmemBytes + 8 * kStages;   // + the barriers
  static_assert(DC == S::DC, "the pre-pass shares the main kernel's channel blocks (TMA boxes)");
};

template <int NP, bool VEC, bool BF = false, bool TMA = false>
__global__ void __launch_bounds__(fwd_warps(NP) * 32)
scan_fwd_agg_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p) {
  static_assert(!TMA || (VEC && !BF), "TMA staging takes fp32 tiles of whole 16-byte groups");
  using S = FwdShape<NP>;
  using A = FwdAggShape<NP>;
  constexpr int G = S::G, DW = S::DW, NPT = S::NPT, NPR = S::NPR, DC = A::DC, NTH = A::NTH;
  constexpr int DPT = S::DPT;
  extern __shared__ __align__(128) float smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + A::kStages * A::kStageFloats);   // (TMA)
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

  constexpr int DP = DPT / 2;
  float2 a2[DP][NPT], h[DP][NPT], sd2[DP];   // channel pairs (see the file comment)
  load_a2<DP, NPT>(p, d0, n0, a2);
#pragma unroll
  for (int q = 0; q < DP; ++q) {
    sd2[q] = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < NPT; ++s) h[q][s] = make_float2(0.f, 0.f);
  }

  auto load = [&](int stage, int c) {
    float* st = smem + stage * A::kStageFloats;
    if constexpr (TMA) {
      fwd_tma_tiles<NP>(maps, bars + stage, c, b, dblk0, st, st + kChunk * DC, nullptr,
                        st + 2 * kChunk * DC, nullptr);
      return;
    }
    if constexpr (BF) {   // bf16 tiles into the first half of each slot
      stage_tile_bf16<DC, NTH>(st, reinterpret_cast<const uint16_t*>(p.delta), row0, c * kChunk,
                               T, Di, dblk0, p.n_io());
      stage_tile_bf16<DC, NTH>(st + kChunk * DC, reinterpret_cast<const uint16_t*>(p.u), row0,
                               c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile_bf16<NP, NTH>(st + 2 * kChunk * DC, reinterpret_cast<const uint16_t*>(p.B),
                               row0, c * kChunk, T, N, 0, p.n_bc());
    } else {
      stage_tile<DC, NTH, VEC>(st, p.delta, row0, c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile<DC, NTH, VEC>(st + kChunk * DC, p.u, row0, c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile<NP, NTH, VEC>(st + 2 * kChunk * DC, p.B, row0, c * kChunk, T, N, 0, p.n_bc());
    }
    cp_async_commit();
  };
  if constexpr (TMA) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int s = 0; s < A::kStages; ++s) mbar_init(bars + s, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
#pragma unroll
  for (int s = 0; s < A::kStages - 1; ++s) {
    if (c_begin + s < c_end) load(s, c_begin + s);
    else if constexpr (!TMA) cp_async_commit();
  }
  for (int c = c_begin; c < c_end; ++c) {
    const int it = c - c_begin;
    if constexpr (TMA) fwd_tma_wait(bars, A::kStages, it, p.wait_limit_ns);
    else cp_async_wait<A::kStages - 2>();
    __syncthreads();
    if (c + A::kStages - 1 < c_end) load((it + A::kStages - 1) % A::kStages, c + A::kStages - 1);
    else if constexpr (!TMA) cp_async_commit();
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
      float2 Bp[NPR], dl2[DP];
      lds_pairs<NPR>(s_B + i * NP + n0, Bp);
      fwd_step<DP, NPT>(dlv, uv, Bp, a2, h, dl2);
#pragma unroll
      for (int q = 0; q < DP; ++q) sd2[q] = add2(sd2[q], dl2[q]);
    }
    if ((c + 1) % p.seg_chunks == 0) {   // the last chunk of a segment: emit, then restart
      const int seg = c / p.seg_chunks;
#pragma unroll
      for (int j = 0; j < DPT; ++j) {
        const int d = d0 + j, q = j >> 1, k = j & 1;
        const size_t row = ((size_t)b * p.nseg + seg) * Di + d;
        if (d < Di && inb(row, 1, p.n_agg_sd()) && inb(row * N, N, p.n_agg_h())) {
          if (ng == 0) p.agg_sd[row] = k ? sd2[q].y : sd2[q].x;
          float2 hs[NPR];
          chan_states<NPT>(h[q], k, hs);
          if constexpr (VEC) {
            st_pairs_row<NPR>(p.agg_h + row * N, n0, N, hs);   // N % 4 == 0 here
          } else {
#pragma unroll
            for (int s = 0; s < NPT; ++s)
              if (n0 + s < N) p.agg_h[row * N + n0 + s] = pair_el(hs, s);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < DP; ++q) {
        sd2[q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int s = 0; s < NPT; ++s) h[q][s] = make_float2(0.f, 0.f);
      }
    }
    // (TMA) this thread's shared-memory writes (softplus, bf16 widening) come before the copy
    // that refills the stage
    if constexpr (TMA) fence_proxy_async_smem();
  }
  if constexpr (!TMA) cp_async_wait<0>();
}

// ST (states only, for the fused forward + backward call): the recurrence and the checkpoints
// alone; the backward then recomputes y from the states and writes out.
// BF (with ST): delta, u and B arrive as bf16 and are widened in shared memory.
// TMA: the tiles arrive by tensor copies (FwdMaps) into a ring of kStagesTma stages; its shared
// memory leaves room for 5 CTAs per SM, and the register bound keeps that many resident (the
// segment plan counts on it).
template <int NP, bool VEC, bool WITH_Y, bool SP, bool ST, bool BF = false, bool TMA = false>
__global__ void __launch_bounds__(fwd_warps(NP) * 32, TMA ? kFwdSlots64 / kSMs : 1)
scan_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p) {
  static_assert(!(ST && (SP || WITH_Y)), "the states-only forward takes the plain delta");
  static_assert(!BF || ST, "bf16 input is taken by the states-only forward");
  static_assert(!TMA || (VEC && !BF), "TMA staging takes fp32 tiles of whole 16-byte groups");
  using S = FwdShape<NP>;
  constexpr int G = S::G, DW = S::DW, DC = S::DC, P = S::P, NPT = S::NPT, NPR = S::NPR;
  constexpr int DPT = S::DPT;
  constexpr int NS = TMA ? S::kStagesTma : kFwdStages;   // stages of the ring
  extern __shared__ __align__(128) float smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * S::kStageFloats);   // (TMA)
  pdl_wait();      // the previous kernel's writes (inputs, workspace) are visible
  pdl_release();   // the next kernel may take the room the last wave leaves

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

  constexpr int DP = DPT / 2;
  float2 a2[DP][NPT], h[DP][NPT];   // channel pairs (see the file comment)
  float Dd[DPT];
  load_a2<DP, NPT>(p, d0, n0, a2);
#pragma unroll
  for (int j = 0; j < DPT; ++j) {
    const int d = d0 + j;
    Dd[j] = (d < Di && inb(d, 1, Di)) ? p.D[d] : 0.f;
  }
#pragma unroll
  for (int q = 0; q < DP; ++q)
#pragma unroll
    for (int s = 0; s < NPT; ++s) h[q][s] = make_float2(0.f, 0.f);

  using RSy = ReduceScatter<DPT * P, G / 2, 1>;
  const int ybase = RSy::base(lane);
  constexpr int kY = RSy::kept();
  const size_t rowb = (size_t)b * T;

  auto issue = [&](int stage, int c) {
    float* st = smem + stage * S::kStageFloats;
    if constexpr (TMA) {
      // the failure-path test leaves the CTA's last chunk without copies
      if (p.test_skip_last_copy && c == c_end - 1) return;
      fwd_tma_tiles<NP>(maps, bars + stage, c, b, dblk0, st, st + kChunk * DC,
                        ST ? nullptr : st + 2 * kChunk * DC, st + 3 * kChunk * DC,
                        ST ? nullptr : st + 3 * kChunk * DC + kChunk * NP);
    } else {
      fwd_load_chunk<NP, VEC, ST, BF>(p, st, c, b, dblk0);
    }
  };
  if constexpr (TMA) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int s = 0; s < NS; ++s) mbar_init(bars + s, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
#pragma unroll
  for (int s = 0; s < NS - 1; ++s) {
    if (c_begin + s < c_end) issue(s, c_begin + s);
    else if constexpr (!TMA) cp_async_commit();
  }

  // state entering the segment: scan_fwd_compose_kernel left it in the slot of the previous
  // segment's aggregate (a channel past d_inner starts from 0)
  if (seg > 0) {
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      const int d = d0 + j;
      const size_t row = ((size_t)b * p.nseg + seg - 1) * Di + d;
      if (d >= Di || !inb(row * N, N, p.n_agg_h())) continue;
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
      for (int s = 0; s < NPT; ++s) {
        if (j & 1) h[j >> 1][s].y = pair_el(hl, s);
        else h[j >> 1][s].x = pair_el(hl, s);
      }
    }
  }

  for (int c = c_begin; c < c_end; ++c) {
    const int it = c - c_begin;
    if constexpr (TMA) fwd_tma_wait(bars, NS, it, p.wait_limit_ns);
    else cp_async_wait<NS - 2>();
    __syncthreads();
    {
      const int cn = c + NS - 1;
      if (cn < c_end) issue((it + NS - 1) % NS, cn);
      else if constexpr (!TMA) cp_async_commit();
    }
    float* st = smem + (it % NS) * S::kStageFloats;
    if constexpr (BF) {   // widen the bf16 tiles into their slots (no overlap: one barrier)
      BfTile<kChunk * DC, S::NW * 32> wdl, wu;
      BfTile<kChunk * NP, S::NW * 32> wB;
      wdl.read(st + 2 * kChunk * DC);
      wu.read(st + 2 * kChunk * DC + kChunk * DC / 2);
      wB.read(st + 3 * kChunk * DC + kChunk * NP);
      wdl.write(st);
      wu.write(st + kChunk * DC);
      wB.write(st + 3 * kChunk * DC);
      __syncthreads();
    }
    if constexpr (SP) {   // raw delta -> delta in shared memory, once per element
      softplus_tile<DC, S::NW * 32>(st, p.T - c * kChunk, p.Di - dblk0);
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
        float2 Bp[NPR], dl2[DP];
        lds_pairs<NPR>(s_B + i * NP + n0, Bp);
        fwd_step<DP, NPT>(dlv, uv, Bp, a2, h, dl2);
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
          float2 Bp[NPR], Cp[NPR], dl2[DP];
          lds_pairs<NPR>(s_B + i * NP + n0, Bp);
          lds_pairs<NPR>(s_C + i * NP + n0, Cp);
          fwd_step<DP, NPT>(dlv, uv, Bp, a2, h, dl2);
#pragma unroll
          for (int q = 0; q < DP; ++q) {   // y of the channel pair: sum over the states
            float2 ya = mul2(splat2(Cp[0].x), h[q][0]);
#pragma unroll
            for (int s = 1; s < NPT; ++s) ya = fma2(splat2(pair_el(Cp, s)), h[q][s], ya);
            yv[tt * DPT + 2 * q] = ya.x;
            yv[tt * DPT + 2 * q + 1] = ya.y;
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
          const size_t o = (rowb + t) * Di + d;
          const bool ok = (t < T) && (d < Di) && inb(o, 1, p.n_io());
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
        if (d >= Di || !inb((size_t)(ck - p.ckpt) + (size_t)d * N, N, p.n_ck())) continue;
        float2 hs[NPR];
        chan_states<NPT>(h[j >> 1], j & 1, hs);
        if constexpr (VEC) {
          st_pairs_row<NPR>(ck + (size_t)d * N, n0, N, hs);
        } else {
#pragma unroll
          for (int s = 0; s < NPT; ++s)
            if (n0 + s < N) ck[(size_t)d * N + n0 + s] = pair_el(hs, s);
        }
      }
    }
    // (TMA) this thread's shared-memory writes (softplus in place) come before the copy that
    // refills the stage
    if constexpr (TMA) fence_proxy_async_smem();
  }
  if constexpr (!TMA) cp_async_wait<0>();
}

// The state entering every segment but the first, from the pre-pass's aggregates, composed in
// segment order: h <- exp(A * sum(delta)) * h + (segment end state from zero). One thread walks
// the segments of one (batch row, channel, state); the state after segment s overwrites the
// aggregate of segment s, which nothing reads afterwards, and is the state entering segment
// s + 1. The arithmetic is the main kernel's own per step (ex2 of the product, one fma).
__global__ void scan_fwd_compose_kernel(const FwdParams p) {
  pdl_wait();   // the pre-pass's aggregates are visible
  const size_t dn = (size_t)p.Di * p.N;
  const size_t total = (size_t)p.batch * dn;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t b = e / dn, q = e % dn;
    const size_t d = q / p.N;
    const float a2 = inb(q, 1, dn) ? -expf(p.A_log[q]) * kLog2e : 0.f;
    float h = 0.f;
    // eight segments at a time: their loads do not depend on h, so they are all in flight
    for (int s0 = 0; s0 < p.nseg - 1; s0 += 8) {
      float Lv[8], sv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int sg = s0 + k;
        const size_t row = b * p.nseg + (sg < p.nseg - 1 ? sg : 0);
        const bool in = sg < p.nseg - 1 && inb(row * dn + q, 1, p.n_agg_h()) &&
                        inb(row * p.Di + d, 1, p.n_agg_sd());
        Lv[k] = in ? p.agg_h[row * dn + q] : 0.f;
        sv[k] = in ? p.agg_sd[row * p.Di + d] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int sg = s0 + k;
        if (sg >= p.nseg - 1) break;
        h = fmaf(ex2_sfu(sv[k] * a2), h, Lv[k]);
        const size_t o = (b * p.nseg + sg) * dn + q;
        if (inb(o, 1, p.n_agg_h())) p.agg_h[o] = h;
      }
    }
  }
}

// the composition between the pre-pass and the main kernel (when there are segments)
static int launch_compose(const FwdParams& p, cudaStream_t s) {
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(scan_fwd_compose_kernel, dim3(sms * 4), dim3(256), 0, s, p) == cudaSuccess
             ? 1
             : -1;
}

// ---- host side ---------------------------------------------------------------------------------

unsigned fwd_take_fault() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_fault, sizeof(v)) != cudaSuccess) return 0;
  if (v) {
    const unsigned zero = 0;
    cudaMemcpyToSymbol(g_fwd_fault, &zero, sizeof(zero));
  }
  return v;
}

// The tensor maps of one call; the last call's maps are reused while its pointers and sizes
// stay the same.
template <int NP>
static bool make_fwd_maps(const Plan& plan, const FwdParams& p, FwdMaps* m) {
  using S = FwdShape<NP>;
  struct Key {
    const void* ptr[5];
    int64_t dims[4];
  };
  static std::mutex mu;
  static Key last_key;
  static FwdMaps last_maps;
  static bool have_last = false;
  const void* gate = p.states_only ? (const void*)p.delta : (const void*)p.gate;
  const void* Cp = p.states_only ? (const void*)p.B : (const void*)p.C;
  Key key;
  memset(&key, 0, sizeof(key));
  const void* ptrs[5] = {p.delta, p.u, gate, p.B, Cp};
  memcpy(key.ptr, ptrs, sizeof(ptrs));
  const int64_t dims[4] = {plan.batch, plan.T, plan.Di, plan.N};
  memcpy(key.dims, dims, sizeof(dims));
  std::lock_guard<std::mutex> lock(mu);
  if (have_last && memcmp(&key, &last_key, sizeof(Key)) == 0) {
    *m = last_maps;
    return true;
  }
  const cuuint64_t Di = plan.Di, T = plan.T, Bt = plan.batch, N = plan.N;
  const cuuint64_t dTD[3] = {Di, T, Bt}, sTD[2] = {Di * 4, T * Di * 4};
  const cuuint32_t bTD[3] = {(cuuint32_t)S::DC, (cuuint32_t)kChunk, 1};
  const cuuint64_t dTN[3] = {N, T, Bt}, sTN[2] = {N * 4, T * N * 4};
  const cuuint32_t bTN[3] = {(cuuint32_t)NP, (cuuint32_t)kChunk, 1};
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  FwdMaps mm;
  memset(&mm, 0, sizeof(mm));
  const bool ok = encode_tiled(&mm.delta, f32, p.delta, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.u, f32, p.u, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.gate, f32, gate, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.B, f32, p.B, 3, dTN, sTN, bTN) &&
                  encode_tiled(&mm.C, f32, Cp, 3, dTN, sTN, bTN);
  if (!ok) return false;
  *m = mm;
  last_key = key;
  last_maps = mm;
  have_last = true;
  return true;
}

// d_state 64 with d_inner a multiple of 4 and fp32 inputs: tiles by TMA.
template <int NP, bool WITH_Y>
static int launch_np_tma(const Plan& plan, const FwdParams& p0, cudaStream_t s) {
  FwdParams p = p0;
  using S = FwdShape<NP>;
  using A = FwdAggShape<NP>;
  FwdMaps maps;
  if (!make_fwd_maps<NP>(plan, p, &maps)) return -1;
  auto kern = p0.states_only ? scan_fwd_kernel<NP, true, false, false, true, false, true>
             : p0.softplus   ? scan_fwd_kernel<NP, true, WITH_Y, true, false, false, true>
                             : scan_fwd_kernel<NP, true, WITH_Y, false, false, false, true>;
  auto agg = scan_fwd_agg_kernel<NP, true, false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)S::kSmemBytesTma) != cudaSuccess)
    return -1;
  int n = 0;
  if (plan.fwd.nseg > 1) {
    if (cudaFuncSetAttribute(agg, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)A::kSmemBytesTma) != cudaSuccess)
      return -1;
    const int nblk_a = (int)((plan.Di + A::DC - 1) / A::DC);
    p.agg_k = 1;
    const int ngrp = (plan.fwd.nseg - 1 + p.agg_k - 1) / p.agg_k;
    dim3 ga((unsigned)(nblk_a * ngrp), (unsigned)plan.batch);
    agg<<<ga, A::NTH, A::kSmemBytesTma, s>>>(maps, p);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    if (launch_compose(p, s) < 0) return -1;
    n += 2;
  }
  dim3 grid((unsigned)(plan.fwd.nblk * plan.fwd.nseg), (unsigned)plan.batch);
  if (launch_pdl(kern, grid, dim3(S::NW * 32), S::kSmemBytesTma, s, maps, p) != cudaSuccess)
    return -1;
  return n + 1;
}

// TMA staging at d_state 64 only. Measured against the cp.async ring: longseq's forward call
// 4.14 -> 3.82 ms; at d_state 16 the TMA forward issued 6 % fewer instructions for the same
// time at mamba370m and ran 3 % slower at mamba130m (its shorter chunks expose the barrier
// waits), since that kernel is bound by the shared-memory data path, not by the staging.
constexpr int kFwdTmaMinNP = 64;

template <int NP, bool VEC, bool WITH_Y>
static int launch_np(const Plan& plan, const FwdParams& p0, cudaStream_t s) {
  if constexpr (NP >= kFwdTmaMinNP && VEC) {
    if (!p0.io_bf16) return launch_np_tma<NP, WITH_Y>(plan, p0, s);
  }
  FwdParams p = p0;
  using S = FwdShape<NP>;
  FwdMaps none;   // the cp.async kernels take no tensor maps
  memset(&none, 0, sizeof(none));
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
    agg<<<ga, A::NTH, A::kSmemBytes, s>>>(none, p);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    if (launch_compose(p, s) < 0) return -1;
    n += 2;
  }
  dim3 grid((unsigned)(plan.fwd.nblk * plan.fwd.nseg), (unsigned)plan.batch);
  if (launch_pdl(kern, grid, dim3(S::NW * 32), S::kSmemBytes, s, none, p) != cudaSuccess)
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

MSCAN_OOB_HOOKS(fwd)

}  // namespace mscan
