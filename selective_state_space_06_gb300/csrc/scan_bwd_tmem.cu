// Backward selective scan for d_state 16, 32 and 64 (sm_103a), with the per-chunk states kept
// in tensor memory. It computes the same Phases B2 (gating) and B3 (reverse-time BPTT) of
// mamba-rs src/mamba_ssm/cpu/backward.rs as scan_bwd_kernel, with the same outputs and
// partials; only the work layout differs.
//
// Mapping. A thread owns 4 channels x 4 states. The channels are packed as two float2 pairs
// (so the per-channel scalars delta, u, d_y come straight from shared memory as pairs) and the
// per-state scalars B, C are staged duplicated ({B, B}) for the packed multiplies.
//   lane = dg * G + ng, G = d_state_padded / 4 state lanes, LD = 32 / G channel lanes
//   ng picks the states 4*ng .. 4*ng+3, dg picks the channels 4*dg .. 4*dg+3 of the warp.
//
// Chunk walk (chunks of 16 steps, last to first):
//   0. gating: d_y into the gate tile, d_gate to global memory (as in scan_bwd_kernel), and
//      the duplicated B / C tiles for the packed multiplies;
//   1. forward recompute of the chunk from its checkpoint. The state before every step goes
//      to tensor memory: 16 steps x 16 floats = 256 columns per thread lane;
//   2. reverse walk: the state before the step comes back from tensor memory; the state after
//      it is the one read for the later step. No step is recomputed twice. A step's d_delta
//      and d_u go into its (then dead) rows of the delta and u tiles, and the whole chunk is
//      stored as coalesced rows after the walk.
// When the y tile is free after the gating step (d_state 32 and 64, unfused), the gating step
// also leaves delta*u there, so the recompute and the reverse walk load it instead of forming
// it per step.
// Variants (template flags): SP takes the raw delta and applies the softplus in shared memory;
// FY (the fused forward + backward call) forms y = sum_n C*h + D*u during step 1 and runs step
// 0's gating after it, writing out as well; BF (FY with bf16 I/O) receives its tiles as bf16
// in shared memory the fused path leaves idle and stores bf16 outputs.
//
// Reductions without select instructions where possible. A butterfly level that halves the
// values a lane keeps normally needs two selects per exchanged value (which half to keep,
// which to send). Here each lane stores its channels and states in a lane-dependent order,
// chosen so that at those levels every lane keeps its first half and sends its second:
//   * over states (d_delta, d_u): the lane with bit G/2 set holds its two channel pairs
//     swapped, so the first level keeps the first pair; the second level (inside a pair) uses
//     selects; further levels are plain all-reduce steps;
//   * over channels (d_B, d_C): the lane with bit 16 set holds its two state pairs swapped, and
//     the lane with bit 8 set (when it takes part) holds the states of each pair swapped (it
//     reads B, C from a pair-swapped copy); the last level (B or C) uses selects.
#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled
#include <string.h>

#include <mutex>

#include "scan_common.cuh"

namespace mscan {

constexpr int kTmemStages = 2;   // cp.async pipeline depth

template <int NP>
struct BwdTmemShape {
  static constexpr int DPT = 4, NPT = 4;
  static constexpr int G = NP / NPT;                     // state lanes: 4, 8, 16
  static constexpr int LG = G == 4 ? 2 : G == 8 ? 3 : 4;
  static constexpr int LD = 32 / G;                      // channel lanes: 8, 4, 2
  static constexpr int DW = LD * DPT;                    // channels per warp
  static constexpr int DC = kWarps * DW;                 // channels per CTA: 128, 64, 32
  static constexpr bool SWAP = LD >= 4;                  // channel reduction splits inside pairs
  static constexpr bool KIND = LD >= 8;                  // ... and on B / C
  static constexpr int TILE = kChunk * DC;
  // per stage: delta, u, gate (-> d_y), dy, y [kChunk][DC]; B, C [kChunk][NP]; the chunk's
  // starting checkpoint [DC][NP] (states past d_state are zeros or unused)
  static constexpr int kStageFloats = 5 * TILE + 2 * kChunk * NP + DC * NP;
  static constexpr uint32_t kStageBytes = kStageFloats * sizeof(float);
  // duplicated B, C [kChunk][NP][2] (and their pair-swapped copies)
  static constexpr int kDupFloats = kChunk * NP * 2 * (SWAP ? 4 : 2);
  // per-warp d_B / d_C sums of the chunk [kWarps][kChunk][2][NP]; they fit in the y tile of
  // the current stage (dead after the gating step) when d_state is 16. (The dy tile then holds
  // the softplus variant's factor d_raw / d_delta.)
  static constexpr int kRedFloats = kWarps * kChunk * 2 * NP;
  static constexpr bool RED_ALIAS = kRedFloats <= TILE;
  static constexpr size_t kDataFloats =
      (size_t)kTmemStages * kStageFloats + kDupFloats + (RED_ALIAS ? 0 : kRedFloats);
  // + the stage barriers, + slack to align the base to 128 bytes (TMA destinations)
  static constexpr size_t kSmemBytes = kDataFloats * sizeof(float) + 8 * kTmemStages + 128;
  static constexpr uint32_t kTmemCols = kChunk * DPT * NPT;   // 256
  // tensor memory holds 512 columns per SM: at most two CTAs may be resident
  static_assert(3 * (kSmemBytes + 1024) > 228 * 1024, "shared memory must cap CTAs per SM at 2");
  static_assert(kStageBytes % 128 == 0 && (TILE * 4) % 128 == 0 && (kChunk * NP * 4) % 128 == 0,
                "TMA destinations must stay 128-byte aligned");
};

static __device__ unsigned int g_bwd_fault;   // set when a bounded wait gave up

// Stage layout: delta, u, gate, dy, y tiles, then B, C, then the checkpoint row. FY (the fused
// call) leaves the y tile to the kernel, which fills it from the recomputed states.
template <int NP, bool VEC, bool TMA, bool FY = false, bool BF = false>
__device__ __forceinline__ void bwd_tmem_load_chunk(const BwdMaps& maps, const BwdParams& p,
                                                    float* st, uint64_t* bar, int c, int b,
                                                    int dblk0) {
  using S = BwdTmemShape<NP>;
  constexpr int DC = S::DC, NTH = kWarps * 32, TILE = S::TILE;
  const int t0 = c * kChunk;
  float* s_h0 = st + 5 * TILE + 2 * kChunk * NP;
  if constexpr (TMA) {
    // one thread issues the whole stage; rows past T, channels past d_inner, states past
    // d_state and the (absent) checkpoint before chunk 0 arrive as zeros. With BF (fused call)
    // the tiles are bf16 and land where the fused path has room until it needs it: delta and u
    // in the halves of the y slot (widened into their own slots before the recompute fills y),
    // gate and dy in the halves of the gate slot (read as bf16), B and C in the first halves of
    // their slots (read as bf16 when duplicated). The checkpoint row stays fp32.
    constexpr uint32_t kEl = BF ? 2u : 4u;
    constexpr uint32_t kBytes = (4u * TILE + (FY ? 0u : TILE) + 2u * kChunk * NP) * kEl +
                                (uint32_t)(DC * NP) * 4u;
    static_assert(BF || kBytes == S::kStageBytes - (FY ? TILE * 4u : 0u), "stage bytes");
    if (threadIdx.x == 0) {
      mbar_expect_tx(bar, kBytes);
      if constexpr (BF) {
        tma_load_3d(st + 4 * TILE, &maps.delta, bar, dblk0, t0, b);
        tma_load_3d(st + 4 * TILE + TILE / 2, &maps.u, bar, dblk0, t0, b);
        tma_load_3d(st + 2 * TILE, &maps.gate, bar, dblk0, t0, b);
        tma_load_3d(st + 2 * TILE + TILE / 2, &maps.dy, bar, dblk0, t0, b);
      } else {
        tma_load_3d(st, &maps.delta, bar, dblk0, t0, b);
        tma_load_3d(st + TILE, &maps.u, bar, dblk0, t0, b);
        tma_load_3d(st + 2 * TILE, &maps.gate, bar, dblk0, t0, b);
        tma_load_3d(st + 3 * TILE, &maps.dy, bar, dblk0, t0, b);
      }
      if constexpr (!FY) tma_load_3d(st + 4 * TILE, &maps.y, bar, dblk0, t0, b);
      tma_load_3d(st + 5 * TILE, &maps.B, bar, 0, t0, b);
      tma_load_3d(st + 5 * TILE + kChunk * NP, &maps.C, bar, 0, t0, b);
      tma_load_4d(s_h0, &maps.ckpt, bar, 0, dblk0, c - 1, b);
    }
  } else {
    const size_t row0 = (size_t)b * p.T;
    const size_t nio = p.n_io(), nbc = p.n_bc();
    stage_tile<DC, NTH, VEC>(st, p.delta, row0, t0, p.T, p.Di, dblk0, nio);
    stage_tile<DC, NTH, VEC>(st + TILE, p.u, row0, t0, p.T, p.Di, dblk0, nio);
    stage_tile<DC, NTH, VEC>(st + 2 * TILE, p.gate, row0, t0, p.T, p.Di, dblk0, nio);
    stage_tile<DC, NTH, VEC>(st + 3 * TILE, p.dy, row0, t0, p.T, p.Di, dblk0, nio);
    if constexpr (!FY)
      stage_tile<DC, NTH, VEC>(st + 4 * TILE, p.y_ck, row0, t0, p.T, p.Di, dblk0, nio);
    stage_tile<NP, NTH, VEC>(st + 5 * TILE, p.B, row0, t0, p.T, p.N, 0, nbc);
    stage_tile<NP, NTH, VEC>(st + 5 * TILE + kChunk * NP, p.C, row0, t0, p.T, p.N, 0, nbc);
    // state entering chunk c (checkpoint slot c-1), rows of N states at a stride of NP;
    // zeros for the first chunk and for channels past d_inner
    const bool have = c > 0;
    const size_t src0 = have ? (((size_t)b * (p.nchunks - 1) + (c - 1)) * p.Di + dblk0) * p.N : 0;
    const float* src = p.ckpt + src0;
    const int rowlen = DC * p.N;
    if constexpr (VEC) {
      for (int q = threadIdx.x * 4; q < rowlen; q += NTH * 4) {
        const int row = q / p.N, col = q % p.N;
        const bool v = have && (dblk0 + row < p.Di) && inb(src0 + q, 4, p.n_ck());
        cp_async16(s_h0 + row * NP + col, v ? src + q : p.delta, v);
      }
    } else {
      for (int q = threadIdx.x; q < rowlen; q += NTH) {
        const int row = q / p.N, col = q % p.N;
        const bool v = have && (dblk0 + row < p.Di) && inb(src0 + q, 1, p.n_ck());
        cp_async4(s_h0 + row * NP + col, v ? src + q : p.delta, v);
      }
    }
    cp_async_commit();
  }
}

// Waits until stage `stage` (its use number `use`) has landed in shared memory.
template <bool TMA>
__device__ __forceinline__ void bwd_tmem_wait_stage(uint64_t* bars, int stage, int use,
                                                    uint64_t limit_ns) {
  if constexpr (TMA) {
    if (!mbar_wait(bars + stage, (uint32_t)(use & 1), limit_ns)) atomicOr(&g_bwd_fault, 1u);
  } else {
    cp_async_wait<kTmemStages - 2>();
  }
}

// FY: the fused forward + backward call. The forward wrote only the checkpoints, so the
// recompute also forms y = sum_n C*h + D*u (a reduce-scatter over the state lanes, as for the
// d_delta sums) into the y tile, and the gating step runs after it and writes out as well.
// BF (fused bf16 call): delta, u, gate, dy, B, C arrive as bf16 and are widened in shared
// memory; out, d_gate, d_delta and d_u are stored as bf16.
template <int NP, bool VEC, bool TMA, bool SP, bool FY, bool BF = false>
__global__ void __launch_bounds__(kWarps * 32, 2)
scan_bwd_tmem_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p) {
  static_assert(!(SP && FY), "the fused call takes the plain delta");
  static_assert(!BF || (FY && TMA && VEC), "bf16 I/O is the fused call's, with TMA staging");
  using S = BwdTmemShape<NP>;
  constexpr int G = S::G, LG = S::LG, DW = S::DW, DC = S::DC, TILE = S::TILE;
  constexpr int NTH = kWarps * 32;
  // Without the intra-pair state swap (fewer than 4 channel lanes) and with fp32 tiles, the
  // lanes read their B and C pairs straight from the stage and splat them in registers: half
  // the shared-memory bytes of a duplicated {B, B} copy, and no copy to write.
  constexpr bool DBC = !S::SWAP && !BF;
  // delta*u formed once per element by the gating step, into a tile that is free after it: the
  // raw dy tile when nothing reads it later (fp32 without softplus), else the y tile unless it
  // holds the warps' d_B / d_C rows. Not in the fused call, whose gating follows the recompute.
  constexpr int DU_TILE = FY ? 0 : (!SP && !BF) ? 3 : !S::RED_ALIAS ? 4 : 0;
  constexpr bool DU = DU_TILE != 0;
  // d_delta / d_u staged in shared memory and stored as whole rows after the walk (below) at
  // d_state 32 and 64. At d_state 16 a CTA covers 128 channels, and writing its staged chunk
  // out after the walk measured slower (404 against 397 us at mamba370m) than one predicated
  // store per lane and step, which the walk hides among its arithmetic.
  constexpr bool STAGE = DC <= 64;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint32_t s_tmem;
  float* smem = reinterpret_cast<float*>(
      smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u));   // 128-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kDataFloats);
  pdl_wait();      // the previous kernel's writes (carries, checkpoints) are visible
  pdl_release();   // the reduction may take the room the last wave leaves

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane & (G - 1), dg = lane >> LG;
  const int b = blockIdx.y;
  const int blk = blockIdx.x % p.nblk, seg = blockIdx.x / p.nblk;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * 4;     // first channel of the thread inside the CTA block
  const int d0 = dblk0 + cl;
  const int n0 = ng * 4;
  const int Di = p.Di, N = p.N, T = p.T;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(p.nchunks, c_begin + p.seg_chunks);
  const int last = c_end - 1;
  const int nck = c_end - c_begin;

  // the first stage's copies go out before anything else, to overlap the set-up below
  if constexpr (TMA) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int s = 0; s < kTmemStages; ++s) mbar_init(bars + s, 1);
      fence_mbar_init();
    }
  }
  // the failure-path test leaves the copies of the CTA's last chunk (use nck - 1) unissued
  const int skip_use = (TMA && p.test_skip_last_copy) ? nck - 1 : -1;
#pragma unroll
  for (int s = 0; s < kTmemStages - 1; ++s) {
    if (s < nck && s != skip_use)
      bwd_tmem_load_chunk<NP, VEC, TMA, FY, BF>(maps, p, smem + s * S::kStageFloats, bars + s,
                                                last - s, b, dblk0);
    else if constexpr (!TMA)
      cp_async_commit();
  }

  // lane-dependent storage order (see the file comment)
  const int mc = (lane >> (LG - 1)) & 1;               // channel pairs swapped
  const int mx = (lane >> (LG - 2)) & 1;               // channel inside the pair after the reduction
  const int m1 = (lane >> 4) & 1;                      // state pairs swapped
  const int m0 = S::SWAP ? (lane >> 3) & 1 : 0;        // states inside each pair swapped
  const int mk = S::KIND ? (lane >> 2) & 1 : 0;        // keeps C (1) or B (0) after the reduction
  // channel of physical pair q, element k: d0 + 2*(q ^ mc) + k
  // state of physical slot s = 2*pp + e:   n0 + 2*(pp ^ m1) + (e ^ m0)
  auto chan = [&](int q, int k) { return 2 * (q ^ mc) + k; };
  auto state = [&](int s) { return n0 + 2 * ((s >> 1) ^ m1) + ((s & 1) ^ m0); };

  // the channel whose d_delta / d_u this lane stores after the reduction over states
  const int j_out = 2 * mc + mx;
  const int d_out = d0 + j_out;
  const int wsel = lane & (G / 4 - 1);
  const bool w_delta = wsel == 0;
  const bool w_u = (G == 4) ? true : wsel == 1;
  const float D_out = (d_out < Di && inb(d_out, 1, Di)) ? p.D[d_out] : 0.f;
  float dD_out = 0.f;

  float2 a2[2][4], dh[2][4], accA[2][4];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int n = state(s);
      float v[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int d = d0 + chan(q, k);
        v[k] = (d < Di && n < N && inb((size_t)d * N + n, 1, (size_t)Di * N))
                   ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
      }
      a2[q][s] = make_float2(v[0], v[1]);
      dh[q][s] = accA[q][s] = make_float2(0.f, 0.f);
    }
  // d_h entering the segment from the future: the composed carry of the later segments
  // (scan_bwd_compose_kernel), zero for the last segment
  if (seg + 1 < p.nseg) {
    const size_t rowbase = ((size_t)b * p.nseg * p.nsub + (size_t)seg * p.nsub) * Di;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int n = state(s);
        float L[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int d = d0 + chan(q, k);
          L[k] = (d < Di && n < N && inb((rowbase + d) * N + n, 1, p.n_agg_l()))
                     ? p.agg_L[(rowbase + d) * N + n] : 0.f;
        }
        dh[q][s] = make_float2(L[0], L[1]);
      }
  }

  if (warp == 0) tmem_alloc(&s_tmem, S::kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t taddr = s_tmem + ((uint32_t)(32 * warp) << 16);

  float* dup = smem + kTmemStages * S::kStageFloats;
  float* const s_Bw = dup;                         // {B, B} per (step, state)
  float* const s_Cw = dup + kChunk * NP * 2;
  float* const s_Bsw = dup + 2 * kChunk * NP * 2;  // pair-swapped copies (SWAP only)
  float* const s_Csw = dup + 3 * kChunk * NP * 2;
  const float* Bsrc = (S::SWAP && m0) ? s_Bsw : s_Bw;
  const float* Csrc = (S::SWAP && m0) ? s_Csw : s_Cw;
  float* const red_fixed = dup + S::kDupFloats;

  const size_t rowb = (size_t)b * T;
  int offc[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) offc[q] = cl + chan(q, 0);
  int offn[2];
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) offn[pp] = (n0 + 2 * (pp ^ m1)) * 2;
  // where this lane's reduced d_B / d_C values go inside a [2][NP] row of the warp's sums
  const int n_res = n0 + 2 * m1 + m0;
  const float4* pB[2] = {reinterpret_cast<const float4*>(Bsrc + offn[0]),
                         reinterpret_cast<const float4*>(Bsrc + offn[1])};
  const float4* pC[2] = {reinterpret_cast<const float4*>(Csrc + offn[0]),
                         reinterpret_cast<const float4*>(Csrc + offn[1])};

  for (int it = 0; it < nck; ++it) {
    const int c = last - it;
    bwd_tmem_wait_stage<TMA>(bars, it % kTmemStages, it / kTmemStages, p.wait_limit_ns);
    __syncthreads();
    {
      const int itn = it + kTmemStages - 1;
      if (itn < nck && itn != skip_use)
        bwd_tmem_load_chunk<NP, VEC, TMA, FY, BF>(maps, p,
                                                  smem + (itn % kTmemStages) * S::kStageFloats,
                                                  bars + itn % kTmemStages, last - itn, b, dblk0);
      else if constexpr (!TMA)
        cp_async_commit();
    }
    float* st = smem + (it % kTmemStages) * S::kStageFloats;
    if constexpr (BF) {   // delta and u: bf16 halves of the y slot -> their fp32 slots
      BfTile<TILE, NTH> wdl, wu;
      wdl.read(st + 4 * TILE);
      wu.read(st + 4 * TILE + TILE / 2);
      wdl.write(st);
      wu.write(st + TILE);
    }
    const float* s_dl = st;
    const float* s_u = st + TILE;
    float* s_g = st + 2 * TILE;          // becomes d_y (BF: gate and dy as bf16 halves)
    const float* s_dy = st + 3 * TILE;   // (BF: receives d_y)
    float* s_y = st + 4 * TILE;   // y: loaded, or formed by the recompute (FY)
    float* const s_du = st + (DU ? DU_TILE : 4) * TILE;   // delta*u (DU)
    const float* s_B = st + 5 * TILE;
    const float* s_C = s_B + kChunk * NP;
    const float* s_h0 = s_C + kChunk * NP;
    // (DBC) this lane's state pairs pp = 0, 1 of B and C in the stage: states n0 + 2*(pp ^ m1)
    const float2* qB[2] = {reinterpret_cast<const float2*>(s_B + n0 + 2 * m1),
                           reinterpret_cast<const float2*>(s_B + n0 + 2 * (1 - m1))};
    const float2* qC[2] = {reinterpret_cast<const float2*>(s_C + n0 + 2 * m1),
                           reinterpret_cast<const float2*>(s_C + n0 + 2 * (1 - m1))};
    float* red = S::RED_ALIAS ? st + 4 * TILE : red_fixed;
    float* const red_lane = red + warp * kChunk * 2 * NP + (S::KIND ? mk * NP : 0) + n_res;
    const int t0 = c * kChunk;

    // ---- 0. gating backward (Phase B2) and the duplicated B / C tiles --------------------
    // d_y = dy*g*s into the gate tile, d_gate = dy*y*s*(1 + g*(1-s)) straight to global memory
    // (and, in the fused call, out = y*g*s). The fused call runs it after the recompute, which
    // forms y.
    auto gating = [&]() {
      if constexpr (VEC) {   // four consecutive channels at a time (all inside d_inner or none)
        static_assert(TILE % (4 * NTH) == 0, "tile must split evenly over the CTA");
#pragma unroll 2
        for (int k = 0; k < TILE / (4 * NTH); ++k) {
          const int e = 4 * (k * NTH + threadIdx.x);
          const int i = e / DC, col = e % DC;
          const bool ok = (t0 + i < T) && (dblk0 + col < Di) &&
                          inb((rowb + t0 + i) * Di + dblk0 + col, 4, p.n_io());
          const float4 yv = *reinterpret_cast<const float4*>(s_y + e);
          float4 g, go;
          if constexpr (BF) {   // 4 bf16 of gate and of dy from the halves of the gate slot
            const uint16_t* gd = reinterpret_cast<const uint16_t*>(s_g);
            const uint2 gw = *reinterpret_cast<const uint2*>(gd + e);
            const uint2 dw = *reinterpret_cast<const uint2*>(gd + TILE + e);
            g = make_float4(bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y));
            go = make_float4(bf16_lo(dw.x), bf16_hi(dw.x), bf16_lo(dw.y), bf16_hi(dw.y));
          } else {
            g = *reinterpret_cast<const float4*>(s_g + e);
            go = *reinterpret_cast<const float4*>(s_dy + e);
          }
          float4 dyo, dgo;
          {
            const float s0 = sigmoid_fast(g.x), s1 = sigmoid_fast(g.y);
            const float s2 = sigmoid_fast(g.z), s3 = sigmoid_fast(g.w);
            dyo = make_float4(go.x * (g.x * s0), go.y * (g.y * s1), go.z * (g.z * s2),
                              go.w * (g.w * s3));
            dgo = make_float4(go.x * yv.x * (s0 * fmaf(g.x, 1.f - s0, 1.f)),
                              go.y * yv.y * (s1 * fmaf(g.y, 1.f - s1, 1.f)),
                              go.z * yv.z * (s2 * fmaf(g.z, 1.f - s2, 1.f)),
                              go.w * yv.w * (s3 * fmaf(g.w, 1.f - s3, 1.f)));
            if constexpr (FY) {
              const float4 ov = make_float4(yv.x * (g.x * s0), yv.y * (g.y * s1),
                                            yv.z * (g.z * s2), yv.w * (g.w * s3));
              const size_t o = (rowb + t0 + i) * Di + dblk0 + col;
              if constexpr (BF) st_global_bf16x4_if(reinterpret_cast<uint16_t*>(p.out) + o, ov, ok);
              else st_global4_if(p.out + o, ov, ok);
            }
          }
          // d_y: into the gate tile, or (BF, where the gate slot holds bf16 still being read
          // by other threads) into the dy slot
          *reinterpret_cast<float4*>((BF ? const_cast<float*>(s_dy) : s_g) + e) = dyo;
          if constexpr (BF)
            st_global_bf16x4_if(reinterpret_cast<uint16_t*>(p.d_gate) + (rowb + t0 + i) * Di +
                                    dblk0 + col, dgo, ok);
          else
            st_global4_if(p.d_gate + (rowb + t0 + i) * Di + dblk0 + col, dgo, ok);
          if (SP && ok) {   // raw -> delta, and the factor d_raw / d_delta
            float* dl = const_cast<float*>(s_dl) + e;
            float* fac = const_cast<float*>(s_dy) + e;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) softplus_both(dl[k4], dl[k4], fac[k4]);
          }
          if constexpr (DU) {   // delta*u over the y values just read (this thread's own)
            const float4 d4 = *reinterpret_cast<const float4*>(s_dl + e);
            const float4 u4 = *reinterpret_cast<const float4*>(s_u + e);
            *reinterpret_cast<float4*>(s_du + e) =
                make_float4(d4.x * u4.x, d4.y * u4.y, d4.z * u4.z, d4.w * u4.w);
          }
        }
      } else {
        static_assert(TILE % NTH == 0, "tile must split evenly over the CTA");
#pragma unroll 4
        for (int k = 0; k < TILE / NTH; ++k) {
          const int e = k * NTH + threadIdx.x;
          const int i = e / DC, col = e % DC;
          const size_t o = (rowb + t0 + i) * Di + dblk0 + col;
          const bool ok = (t0 + i < T) && (dblk0 + col < Di) && inb(o, 1, p.n_io());
          const float yv = s_y[e];
          const float g = s_g[e], go = s_dy[e];
          const float sg = sigmoid_fast(g);
          s_g[e] = go * (g * sg);
          st_global_if(p.d_gate + o, go * yv * (sg * fmaf(g, 1.f - sg, 1.f)), ok);
          if constexpr (FY) st_global_if(p.out + o, yv * (g * sg), ok);
          if (SP && ok) {   // raw -> delta, and the factor d_raw / d_delta
            softplus_both(s_dl[e], const_cast<float*>(s_dl)[e], const_cast<float*>(s_dy)[e]);
          }
          if constexpr (DU) s_du[e] = s_dl[e] * s_u[e];
        }
      }
    };
    if constexpr (!FY) gating();
    for (int e = threadIdx.x; e < (DBC ? 0 : kChunk * NP); e += NTH) {
      float bv, cv;
      if constexpr (BF) {   // bf16 B and C in the first halves of their slots
        bv = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(s_B)[e] << 16);
        cv = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(s_C)[e] << 16);
      } else {
        bv = s_B[e];
        cv = s_C[e];
      }
      *reinterpret_cast<float2*>(s_Bw + 2 * e) = make_float2(bv, bv);
      *reinterpret_cast<float2*>(s_Cw + 2 * e) = make_float2(cv, cv);
      if constexpr (S::SWAP) {
        const int es = e ^ 1;   // (step, state ^ 1)
        *reinterpret_cast<float2*>(s_Bsw + 2 * es) = make_float2(bv, bv);
        *reinterpret_cast<float2*>(s_Csw + 2 * es) = make_float2(cv, cv);
      }
    }
    __syncthreads();

    // ---- 1. forward recompute; the state before each step goes to tensor memory ---------
    float2 h[2][4];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int n = state(s);
        float v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k)
          v[k] = (TMA || n < N) ? s_h0[(cl + chan(q, k)) * NP + n] : 0.f;
        h[q][s] = make_float2(v[0], v[1]);
      }
    // per-thread views of the staged tiles (measured: the recompute loop fully unrolled, the
    // reverse walk by four; both fit the 255 registers a thread may have)
    const float2* pdl[2] = {reinterpret_cast<const float2*>(s_dl + offc[0]),
                            reinterpret_cast<const float2*>(s_dl + offc[1])};
    const float2* pu[2] = {reinterpret_cast<const float2*>(s_u + offc[0]),
                           reinterpret_cast<const float2*>(s_u + offc[1])};
    const float* s_dyv = BF ? s_dy : s_g;   // d_y
    const float2* pdy[2] = {reinterpret_cast<const float2*>(s_dyv + offc[0]),
                            reinterpret_cast<const float2*>(s_dyv + offc[1])};
    const float2* pdu[2] = {reinterpret_cast<const float2*>(s_du + offc[0]),
                            reinterpret_cast<const float2*>(s_du + offc[1])};
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      step_fence();
      tmem_st16(taddr + 16 * i, reinterpret_cast<const float2(&)[8]>(h));
      float2 dl2[2], u2[2], du2[2], B2[4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        dl2[q] = pdl[q][i * DC / 2];
        if constexpr (DU) {
          du2[q] = pdu[q][i * DC / 2];
        } else {
          u2[q] = pu[q][i * DC / 2];
          du2[q] = mul2(dl2[q], u2[q]);
        }
      }
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if constexpr (DBC) {
          const float2 v = qB[pp][i * NP / 2];
          B2[2 * pp] = splat2(v.x);
          B2[2 * pp + 1] = splat2(v.y);
        } else {
          const float4 v = pB[pp][i * NP / 2];
          B2[2 * pp] = make_float2(v.x, v.y);
          B2[2 * pp + 1] = make_float2(v.z, v.w);
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float2 da = ex2_2(mul2(dl2[q], a2[q][s]));
          h[q][s] = fma2(da, h[q][s], mul2(du2[q], B2[s]));
        }
      if constexpr (FY) {   // y of this step: sum over n of C*h, then + D*u
        float2 C2[4];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          if constexpr (DBC) {
            const float2 v = qC[pp][i * NP / 2];
            C2[2 * pp] = splat2(v.x);
            C2[2 * pp + 1] = splat2(v.y);
          } else {
            const float4 v = pC[pp][i * NP / 2];
            C2[2 * pp] = make_float2(v.x, v.y);
            C2[2 * pp + 1] = make_float2(v.z, v.w);
          }
        }
        float2 ya[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          ya[q] = mul2(C2[0], h[q][0]);
#pragma unroll
          for (int s = 1; s < 4; ++s) ya[q] = fma2(C2[s], h[q][s], ya[q]);
        }
        // same reduce-scatter as the d_delta sums: level G/2 over the channel pairs, level G/4
        // inside the pair, then the remaining state lanes
        ya[0] = add2(ya[0], make_float2(__shfl_xor_sync(kFull, ya[1].x, G / 2),
                                        __shfl_xor_sync(kFull, ya[1].y, G / 2)));
        float yv = (mx ? ya[0].y : ya[0].x) +
                   __shfl_xor_sync(kFull, mx ? ya[0].x : ya[0].y, G / 4);
#pragma unroll
        for (int m = G / 8; m >= 1; m /= 2) yv += __shfl_xor_sync(kFull, yv, m);
        if (w_delta) s_y[i * DC + cl + j_out] = fmaf(D_out, mx ? u2[0].y : u2[0].x, yv);
      }
    }
    tmem_wait_st();
    if constexpr (FY) {
      __syncthreads();   // the y tile is complete
      gating();
      __syncthreads();   // d_y is in the gate tile
    }

    // ---- 2. reverse walk (Phase B3) ------------------------------------------------------
    // The lane's d_delta and d_u of step i overwrite row i of the delta tile and of the d_y
    // tile. d_delta is a sum over the state lanes of terms formed from each lane's delta of the
    // step, and d_u one of terms formed from each lane's d_y, so neither store can issue before
    // every lane's loads of the row it overwrites have returned; no later step reads row i.
    // The stores of step i are issued in step i-1, behind that step's shared-memory loads:
    // shared-memory accesses of a warp are served in order, and a store issued at the end of
    // its own step would hold the next step's loads behind the step's reductions.
    float* const row_dd = const_cast<float*>(s_dl) + cl + j_out;
    float* const row_du = const_cast<float*>(s_dyv) + cl + j_out;
    const float* const row_u = s_u + cl + j_out;
    float pend_dd = 0.f, pend_du = 0.f;   // the previous step's d_delta and d_u
    // without staging: this lane's output rows of the chunk; rows at or past T are not stored
    const size_t o_row = (rowb + t0) * Di + d_out;
    const bool o_ok = d_out < Di && inb((rowb + min(T, t0 + kChunk) - 1) * Di + d_out, 1, p.n_io());
    const int lim_dd = (w_delta && o_ok) ? T - t0 : 0;
    const int lim_du = (w_u && o_ok) ? T - t0 : 0;
#pragma unroll 4
    for (int ii = 0; ii < kChunk; ++ii) {
      const int i = kChunk - 1 - ii;
      step_fence();
      float2 hp[2][4];   // state before step i
      tmem_ld16(taddr + 16 * i, reinterpret_cast<float2(&)[8]>(hp));
      float2 dl2[2], u2[2], dy2[2], du2[2], B2[4], C2[4];
      float u_lane = 0.f;   // (DU) u of the lane's output channel, for d_delta
      if constexpr (DU) u_lane = row_u[i * DC];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        dl2[q] = pdl[q][i * DC / 2];
        dy2[q] = pdy[q][i * DC / 2];
        if constexpr (DU) {
          du2[q] = pdu[q][i * DC / 2];
        } else {
          u2[q] = pu[q][i * DC / 2];
          du2[q] = mul2(dl2[q], u2[q]);
        }
      }
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if constexpr (DBC) {
          const float2 vb = qB[pp][i * NP / 2];
          const float2 vc = qC[pp][i * NP / 2];
          B2[2 * pp] = splat2(vb.x);
          B2[2 * pp + 1] = splat2(vb.y);
          C2[2 * pp] = splat2(vc.x);
          C2[2 * pp + 1] = splat2(vc.y);
        } else {
          const float4 vb = pB[pp][i * NP / 2];
          const float4 vc = pC[pp][i * NP / 2];
          B2[2 * pp] = make_float2(vb.x, vb.y);
          B2[2 * pp + 1] = make_float2(vb.z, vb.w);
          C2[2 * pp] = make_float2(vc.x, vc.y);
          C2[2 * pp + 1] = make_float2(vc.z, vc.w);
        }
      }
      if constexpr (STAGE) {   // (row i + 1: for ii = 0 the predicate is off, nothing accessed)
        st_shared_if(row_dd + (i + 1) * DC, pend_dd, w_delta && ii > 0);
        st_shared_if(row_du + (i + 1) * DC, pend_du, w_u && ii > 0);
      }
      tmem_wait_ld(reinterpret_cast<float2(&)[8]>(hp));
      float2 sa2[2], sb2[2], xb2[4], xc2[4];
#pragma unroll
      for (int q = 0; q < 2; ++q) sa2[q] = sb2[q] = make_float2(0.f, 0.f);
#pragma unroll
      for (int s = 0; s < 4; ++s) xb2[s] = xc2[s] = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float2 da = ex2_2(mul2(dl2[q], a2[q][s]));
          const float2 gh = fma2(dy2[q], C2[s], dh[q][s]);   // d_h += d_y*C
          const float2 cr = mul2(da, gh);                      // carried to t-1
          const float2 r = mul2(cr, hp[q][s]);                 // d_h*da*h_{t-1}
          accA[q][s] = fma2(r, dl2[q], accA[q][s]);
          sa2[q] = fma2(a2[q][s], r, sa2[q]);
          sb2[q] = fma2(gh, B2[s], sb2[q]);
          xb2[s] = fma2(gh, du2[q], xb2[s]);
          xc2[s] = fma2(dy2[q], h[q][s], xc2[s]);
          dh[q][s] = cr;
        }
      // d_B / d_C of this step: sum over the warp's channels
      float v[8];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        v[s] = xb2[s].x + xb2[s].y;
        v[4 + s] = xc2[s].x + xc2[s].y;
      }
      // level 16: the state pairs (lanes with bit 16 hold them swapped)
      v[0] += __shfl_xor_sync(kFull, v[2], 16);
      v[1] += __shfl_xor_sync(kFull, v[3], 16);
      v[4] += __shfl_xor_sync(kFull, v[6], 16);
      v[5] += __shfl_xor_sync(kFull, v[7], 16);
      if constexpr (S::SWAP) {   // level 8: inside the pair (lanes with bit 8 hold it swapped)
        v[0] += __shfl_xor_sync(kFull, v[1], 8);
        v[4] += __shfl_xor_sync(kFull, v[5], 8);
      }
      float* rrow = red_lane + i * 2 * NP;
      if constexpr (S::KIND) {   // level 4: B or C
        const float send = mk ? v[0] : v[4];
        const float keep = mk ? v[4] : v[0];
        rrow[0] = keep + __shfl_xor_sync(kFull, send, 4);
      } else if constexpr (S::SWAP) {
        rrow[0] = v[0];
        rrow[NP] = v[4];
      } else {
        *reinterpret_cast<float2*>(rrow) = make_float2(v[0], v[1]);
        *reinterpret_cast<float2*>(rrow + NP) = make_float2(v[4], v[5]);
      }
      // sums over n: level G/2 over the channel pairs (lanes with that bit hold them swapped)
      sa2[0] = add2(sa2[0], make_float2(__shfl_xor_sync(kFull, sa2[1].x, G / 2),
                                        __shfl_xor_sync(kFull, sa2[1].y, G / 2)));
      sb2[0] = add2(sb2[0], make_float2(__shfl_xor_sync(kFull, sb2[1].x, G / 2),
                                        __shfl_xor_sync(kFull, sb2[1].y, G / 2)));
      // level G/4: inside the pair, with selects
      float sA = (mx ? sa2[0].y : sa2[0].x) +
                 __shfl_xor_sync(kFull, mx ? sa2[0].x : sa2[0].y, G / 4);
      float sB = (mx ? sb2[0].y : sb2[0].x) +
                 __shfl_xor_sync(kFull, mx ? sb2[0].x : sb2[0].y, G / 4);
#pragma unroll
      for (int m = G / 8; m >= 1; m /= 2) {
        sA += __shfl_xor_sync(kFull, sA, m);
        sB += __shfl_xor_sync(kFull, sB, m);
      }
      {
        float uo;
        if constexpr (DU) uo = u_lane;
        else uo = mx ? u2[0].y : u2[0].x;
        const float dlo = mx ? dl2[0].y : dl2[0].x;
        const float dyo = mx ? dy2[0].y : dy2[0].x;
        dD_out = fmaf(dyo, uo, dD_out);
        float ddo = fmaf(sA, kLn2, uo * sB);
        if constexpr (SP) ddo *= s_dy[i * DC + cl + j_out];   // d_raw = d_delta * softplus'
        const float duo = fmaf(dyo, D_out, dlo * sB);
        if constexpr (STAGE) {
          pend_dd = ddo;
          pend_du = duo;
        } else if constexpr (BF) {
          uint16_t* const o16 = reinterpret_cast<uint16_t*>(p.d_delta) + o_row + (size_t)i * Di;
          st_global_bf16_lt(o16, ddo, i, lim_dd);
          st_global_bf16_lt(reinterpret_cast<uint16_t*>(p.d_u) + o_row + (size_t)i * Di, duo, i,
                            lim_du);
        } else {
          st_global_lt(p.d_delta + o_row + (size_t)i * Di, ddo, i, lim_dd);
          st_global_lt(p.d_u + o_row + (size_t)i * Di, duo, i, lim_du);
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int s = 0; s < 4; ++s) h[q][s] = hp[q][s];
    }
    if constexpr (STAGE) {
      st_shared_if(row_dd, pend_dd, w_delta);   // step 0
      st_shared_if(row_du, pend_du, w_u);
    }
    __syncthreads();
    // d_delta and d_u of the chunk, out of the tiles the walk left them in, as whole rows
    const float* const s_duo = s_dyv;
    if constexpr (!STAGE) {
    } else if constexpr (VEC) {   // four consecutive channels at a time (all inside d_inner or none)
#pragma unroll
      for (int k = 0; k < TILE / (4 * NTH); ++k) {
        const int e = 4 * (k * NTH + threadIdx.x);
        const int i = e / DC, col = e % DC;
        const size_t o = (rowb + t0 + i) * Di + dblk0 + col;
        const bool ok = (t0 + i < T) && (dblk0 + col < Di) && inb(o, 4, p.n_io());
        const float4 vd = lds4(s_dl + e), vu = lds4(s_duo + e);
        if constexpr (BF) {
          st_global_bf16x4_if(reinterpret_cast<uint16_t*>(p.d_delta) + o, vd, ok);
          st_global_bf16x4_if(reinterpret_cast<uint16_t*>(p.d_u) + o, vu, ok);
        } else {
          st_global4_if(p.d_delta + o, vd, ok);
          st_global4_if(p.d_u + o, vu, ok);
        }
      }
    } else {
      for (int e = threadIdx.x; e < TILE; e += NTH) {
        const int i = e / DC, col = e % DC;
        const size_t o = (rowb + t0 + i) * Di + dblk0 + col;
        const bool ok = (t0 + i < T) && (dblk0 + col < Di) && inb(o, 1, p.n_io());
        st_global_if(p.d_delta + o, s_dl[e], ok);
        st_global_if(p.d_u + o, s_duo[e], ok);
      }
    }
    // CTA partial of d_B / d_C for this chunk: fixed-order sum over the warps
    if constexpr (VEC) {   // four consecutive states at a time (d_state % 4 == 0)
      for (int e = 4 * threadIdx.x; e < kChunk * 2 * NP; e += 4 * NTH) {
        const int i = e / (2 * NP), kn = e % (2 * NP);
        const int kind = kn / NP, n = kn % NP;
        const int t = t0 + i;
        float4 sum = *reinterpret_cast<const float4*>(red + i * 2 * NP + kn);
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(red + (w * kChunk + i) * 2 * NP + kn);
          sum = make_float4(sum.x + v.x, sum.y + v.y, sum.z + v.z, sum.w + v.w);
        }
        const size_t o = (((size_t)blk * p.batch + b) * T + t) * N + n;
        st_global4_if((kind ? p.partC : p.partB) + o, sum,
                      t < T && n < N && inb(o, 4, p.n_part_bc()));
      }
    } else {
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
    // this thread's shared-memory writes (d_y, the warp sums) come before the copies that
    // refill the stage
    if constexpr (TMA) fence_proxy_async_smem();
  }
  if constexpr (!TMA) cp_async_wait<0>();

  // per-(batch, segment) partials of d_A_log (= A * sum_t delta*r = ln2*a2*accA) and d_D
  {
    const size_t rowbase = ((size_t)b * p.nseg + seg) * Di;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int n = state(s);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int d = d0 + chan(q, k);
          const float aa = k ? a2[q][s].y : a2[q][s].x;
          const float ac = k ? accA[q][s].y : accA[q][s].x;
          if (d < Di && n < N && inb((rowbase + d) * N + n, 1, p.n_part_a()))
            p.partA[(rowbase + d) * N + n] = kLn2 * aa * ac;
        }
      }
    if (w_delta && d_out < Di && inb(rowbase + d_out, 1, p.n_part_d()))
      p.partD[rowbase + d_out] = dD_out;
  }

  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(s_tmem, S::kTmemCols);
}

// Segment pre-pass with the main kernel's channel blocks (the same aggregates as
// scan_bwd_agg_kernel: L = sum_t exp(A * sum_{s<=t} delta_s) * d_y_t * C_t[n] and the sum of
// delta over one sub-segment). A thread owns 4 channels x 4 states, channel-packed; its four
// states of C come as one plain quad and are splatted in registers, and nothing crosses lanes.
template <int NP>
struct BwdAgg4Shape {
  using S = BwdTmemShape<NP>;
  static constexpr int kStages = 2;
  // per stage: delta, gate (-> d_y), dy [kChunk][DC]; C [kChunk][NP]
  static constexpr int kStageFloats = 3 * S::TILE + kChunk * NP;
  static constexpr uint32_t kStageBytes = kStageFloats * sizeof(float);
  static constexpr size_t kDataFloats = (size_t)kStages * kStageFloats;
  static constexpr size_t kSmemBytes = kDataFloats * sizeof(float) + 8 * kStages + 128;
  static_assert(kStageBytes % 128 == 0, "TMA destinations must stay 128-byte aligned");
};

template <int NP, bool VEC, bool TMA, bool BF = false>
__global__ void __launch_bounds__(kWarps * 32)
scan_bwd_agg4_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p) {
  static_assert(!BF || TMA, "bf16 tiles come by TMA");
  using S = BwdTmemShape<NP>;
  using A = BwdAgg4Shape<NP>;
  constexpr int G = S::G, LG = S::LG, DW = S::DW, DC = S::DC, TILE = S::TILE;
  constexpr int NTH = kWarps * 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* smem = reinterpret_cast<float*>(
      smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u));   // 128-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + A::kDataFloats);
  pdl_wait();   // the previous kernel's writes are visible
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = lane & (G - 1), dg = lane >> LG;
  const int b = blockIdx.y;
  const int blk = blockIdx.x % p.nblk, grp = blockIdx.x / p.nblk;
  const int dblk0 = blk * DC;
  const int cl = warp * DW + dg * 4;
  const int d0 = dblk0 + cl;
  const int n0 = ng * 4;
  const int Di = p.Di, N = p.N, T = p.T;
  // segments 1 .. nseg-1 need aggregates; sub-segment j of segment sg (may be empty)
  const int sg = 1 + grp / p.nsub, j_sub = grp % p.nsub;
  const int slot = sg * p.nsub + j_sub;
  const int c_begin = sg * p.seg_chunks + j_sub * p.sub_chunks;
  const int c_end = min(min(p.nchunks, (sg + 1) * p.seg_chunks), c_begin + p.sub_chunks);
  const size_t row0 = (size_t)b * T;

  auto load = [&](int stage, int c) {
    float* st = smem + stage * A::kStageFloats;
    if constexpr (TMA) {
      if (threadIdx.x == 0) {
        uint64_t* bar = bars + stage;
        mbar_expect_tx(bar, BF ? A::kStageBytes / 2 : A::kStageBytes);
        tma_load_3d(st, &maps.delta, bar, dblk0, c * kChunk, b);
        tma_load_3d(st + TILE, &maps.gate, bar, dblk0, c * kChunk, b);
        tma_load_3d(st + 2 * TILE, &maps.dy, bar, dblk0, c * kChunk, b);
        tma_load_3d(st + 3 * TILE, &maps.C, bar, 0, c * kChunk, b);
      }
    } else {
      stage_tile<DC, NTH, VEC>(st, p.delta, row0, c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile<DC, NTH, VEC>(st + TILE, p.gate, row0, c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile<DC, NTH, VEC>(st + 2 * TILE, p.dy, row0, c * kChunk, T, Di, dblk0, p.n_io());
      stage_tile<NP, NTH, VEC>(st + 3 * TILE, p.C, row0, c * kChunk, T, N, 0, p.n_bc());
      cp_async_commit();
    }
  };
  // the first stage's copies go out before the set-up below
  if constexpr (TMA) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int s = 0; s < A::kStages; ++s) mbar_init(bars + s, 1);
      fence_mbar_init();
    }
  }
#pragma unroll
  for (int s = 0; s < A::kStages - 1; ++s) {
    if (c_begin + s < c_end) load(s, c_begin + s);
    else if constexpr (!TMA) cp_async_commit();
  }
  if constexpr (TMA) __syncthreads();   // the barriers are initialised before anyone waits

  float2 a2[2][4], L[2][4];
  float2 P2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // running sums of delta
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int n = n0 + s;
      float v[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int d = d0 + 2 * q + k;
        v[k] = (d < Di && n < N && inb((size_t)d * N + n, 1, (size_t)Di * N))
                   ? -expf(p.A_log[(size_t)d * N + n]) * kLog2e : 0.f;
      }
      a2[q][s] = make_float2(v[0], v[1]);
      L[q][s] = make_float2(0.f, 0.f);
    }

  for (int c = c_begin; c < c_end; ++c) {
    const int it = c - c_begin;
    if constexpr (TMA) {
      if (!mbar_wait(bars + it % A::kStages, (uint32_t)((it / A::kStages) & 1), p.wait_limit_ns))
        atomicOr(&g_bwd_fault, 2u);
    } else {
      cp_async_wait<A::kStages - 2>();
    }
    __syncthreads();
    if (c + A::kStages - 1 < c_end) load((it + A::kStages - 1) % A::kStages, c + A::kStages - 1);
    else if constexpr (!TMA) cp_async_commit();
    float* st = smem + (it % A::kStages) * A::kStageFloats;
    if constexpr (BF) {   // widen the bf16 tiles in place
      BfTile<TILE, NTH> wdl, wg, wdy;
      BfTile<kChunk * NP, NTH> wC;
      wdl.read(st);
      wg.read(st + TILE);
      wdy.read(st + 2 * TILE);
      wC.read(st + 3 * TILE);
      __syncthreads();
      wdl.write(st);
      wg.write(st + TILE);
      wdy.write(st + 2 * TILE);
      wC.write(st + 3 * TILE);
      __syncthreads();
    }
    const float* s_dl = st;
    float* s_g = st + TILE;             // becomes d_y
    const float* s_dy = st + 2 * TILE;
    const float* s_C = st + 3 * TILE;
    if constexpr (VEC) {
#pragma unroll
      for (int e = 4 * threadIdx.x; e < TILE; e += 4 * NTH) {
        const float4 g = *reinterpret_cast<const float4*>(s_g + e);
        const float4 go = *reinterpret_cast<const float4*>(s_dy + e);
        *reinterpret_cast<float4*>(s_g + e) =
            make_float4(go.x * (g.x * sigmoid_fast(g.x)), go.y * (g.y * sigmoid_fast(g.y)),
                        go.z * (g.z * sigmoid_fast(g.z)), go.w * (g.w * sigmoid_fast(g.w)));
      }
    } else {
#pragma unroll 4
      for (int e = threadIdx.x; e < TILE; e += NTH) {
        const float g = s_g[e];
        s_g[e] = s_dy[e] * (g * sigmoid_fast(g));
      }
    }
    if (p.softplus) softplus_tile<DC, NTH>(st, T - c * kChunk, Di - dblk0);   // raw -> delta
    __syncthreads();
    const float4* pdl = reinterpret_cast<const float4*>(s_dl + cl);
    const float4* pdy = reinterpret_cast<const float4*>(s_g + cl);
    const float4* pcq = reinterpret_cast<const float4*>(s_C + n0);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const float4 dl = pdl[i * DC / 4];
      const float4 dy = pdy[i * DC / 4];
      P2[0] = __fadd2_rn(P2[0], make_float2(dl.x, dl.y));
      P2[1] = __fadd2_rn(P2[1], make_float2(dl.z, dl.w));
      const float2 dy2[2] = {make_float2(dy.x, dy.y), make_float2(dy.z, dy.w)};
      // the thread's four states of C, splatted in registers (loading a duplicated {C, C}
      // copy instead doubles the shared-memory bytes of a path bound by them)
      const float4 cq = pcq[i * NP / 4];
      const float2 C2[4] = {splat2(cq.x), splat2(cq.y), splat2(cq.z), splat2(cq.w)};
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float2 cum = ex2_2(mul2(P2[q], a2[q][s]));
          L[q][s] = fma2(cum, mul2(dy2[q], C2[s]), L[q][s]);
        }
    }
    // the d_y writes above come before the copies that refill this stage
    if constexpr (TMA) fence_proxy_async_smem();
  }
  if constexpr (!TMA) cp_async_wait<0>();
  // emit the sub-segment's aggregate (zeros for an empty one)
  const size_t rowbase = ((size_t)b * p.nseg * p.nsub + slot) * Di;
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int d = d0 + 2 * q + k;
      if (d >= Di || !inb(rowbase + d, 1, p.n_agg_sd()) || !inb((rowbase + d) * N, N, p.n_agg_l()))
        continue;
      if (ng == 0) p.agg_sd[rowbase + d] = k ? P2[q].y : P2[q].x;
      float v[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) v[s] = k ? L[q][s].y : L[q][s].x;
      float* dst = p.agg_L + (rowbase + d) * N + n0;
      if constexpr (VEC) {
        if (n0 < N) *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (n0 + s < N) dst[s] = v[s];
      }
    }
}

// ---- host side: tensor maps ------------------------------------------------------------------
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType ty, const void* base, cuuint32_t rank,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  const EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return f(m, ty, rank, const_cast<void*>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode_f32(CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box) {
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rank, dims, strides, box);
}

// The maps of one call; the last call's maps are kept and reused when nothing changed.
template <int NP>
static bool make_maps(const Plan& plan, const BwdParams& p, BwdMaps* m) {
  using S = BwdTmemShape<NP>;
  struct Key {
    const void* ptr[8];
    int64_t dims[5];   // batch, T, d_inner, d_state, bf16 I/O
  };
  static std::mutex mu;
  static Key last_key;
  static BwdMaps last_maps;
  static bool have_last = false;
  const Key key = {{p.delta, p.u, p.gate, p.dy, p.y_ck, p.B, p.C, p.ckpt},
                   {plan.batch, plan.T, plan.Di, plan.N, (int64_t)p.io_bf16}};
  std::lock_guard<std::mutex> lock(mu);
  if (have_last && memcmp(&key, &last_key, sizeof(Key)) == 0) {
    *m = last_maps;
    return true;
  }
  const cuuint64_t Di = plan.Di, T = plan.T, Bt = plan.batch, N = plan.N;
  const cuuint64_t nck = plan.nchunks - 1;
  // the I/O tensors' element size: 2 for the fused bf16 call (the checkpoints stay fp32)
  const cuuint64_t es = p.io_bf16 ? 2 : 4;
  const CUtensorMapDataType io =
      p.io_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t dTD[3] = {Di, T, Bt}, sTD[2] = {Di * es, T * Di * es};
  const cuuint32_t bTD[3] = {(cuuint32_t)S::DC, (cuuint32_t)kChunk, 1};
  const cuuint64_t dTN[3] = {N, T, Bt}, sTN[2] = {N * es, T * N * es};
  const cuuint32_t bTN[3] = {(cuuint32_t)NP, (cuuint32_t)kChunk, 1};
  const cuuint64_t dCK[4] = {N, Di, nck, Bt}, sCK[3] = {N * 4, Di * N * 4, nck * Di * N * 4};
  const cuuint32_t bCK[4] = {(cuuint32_t)NP, (cuuint32_t)S::DC, 1, 1};
  BwdMaps mm;
  memset(&mm, 0, sizeof(mm));
  const bool ok = encode_tiled(&mm.delta, io, p.delta, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.u, io, p.u, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.gate, io, p.gate, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.dy, io, p.dy, 3, dTD, sTD, bTD) &&
                  // the fused call has no stored y: its map is never used
                  encode_tiled(&mm.y, io, p.y_ck ? p.y_ck : p.delta, 3, dTD, sTD, bTD) &&
                  encode_tiled(&mm.B, io, p.B, 3, dTN, sTN, bTN) &&
                  encode_tiled(&mm.C, io, p.C, 3, dTN, sTN, bTN) &&
                  encode_f32(&mm.ckpt, p.ckpt, 4, dCK, sCK, bCK);
  if (!ok) return false;
  *m = mm;
  last_key = key;
  last_maps = mm;
  have_last = true;
  return true;
}

unsigned bwd_take_fault() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwd_fault, sizeof(v)) != cudaSuccess) return 0;
  if (v) {
    const unsigned zero = 0;
    cudaMemcpyToSymbol(g_bwd_fault, &zero, sizeof(zero));
  }
  return v;
}

template <int NP, bool VEC, bool TMA>
static int launch_main(const Plan& plan, const BwdMaps& maps, const BwdParams& p,
                       cudaStream_t s) {
  using S = BwdTmemShape<NP>;
  auto kern = p.out        ? scan_bwd_tmem_kernel<NP, VEC, TMA, false, true>
              : p.softplus ? scan_bwd_tmem_kernel<NP, VEC, TMA, true, false>
                           : scan_bwd_tmem_kernel<NP, VEC, TMA, false, false>;
  if constexpr (VEC && TMA) {
    if (p.io_bf16) kern = scan_bwd_tmem_kernel<NP, true, true, false, true, true>;
  } else {
    if (p.io_bf16) return -1;   // bf16 tiles need the TMA path
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)S::kSmemBytes) != cudaSuccess)
    return -1;
  dim3 grid((unsigned)(plan.bwd.nblk * plan.bwd.nseg), (unsigned)plan.batch);
  return launch_pdl(kern, grid, dim3(kWarps * 32), S::kSmemBytes, s, maps, p) == cudaSuccess
             ? 1
             : -1;
}

// TMA needs 16-byte strides (d_inner and d_state multiples of 4) and a checkpoint tensor
// (T > 16); otherwise the stages are filled with cp.async.
template <int NP>
static int launch_np(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  const bool vec = (plan.Di % 4 == 0) && (plan.N % 4 == 0);
  BwdMaps maps;
  if (vec && plan.nchunks >= 2 && make_maps<NP>(plan, p, &maps))
    return launch_main<NP, true, true>(plan, maps, p, s);
  if (p.io_bf16) return -1;
  memset(&maps, 0, sizeof(maps));
  return vec ? launch_main<NP, true, false>(plan, maps, p, s)
             : launch_main<NP, false, false>(plan, maps, p, s);
}

template <int NP, bool VEC, bool TMA>
static int launch_agg4(const Plan& plan, const BwdMaps& maps, const BwdParams& p,
                       cudaStream_t s) {
  using A = BwdAgg4Shape<NP>;
  auto kern = scan_bwd_agg4_kernel<NP, VEC, TMA>;
  if constexpr (VEC && TMA) {
    if (p.io_bf16) kern = scan_bwd_agg4_kernel<NP, true, true, true>;
  } else {
    if (p.io_bf16) return -1;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)A::kSmemBytes) != cudaSuccess)
    return -1;
  dim3 grid((unsigned)(plan.bwd.nblk * (plan.bwd.nseg - 1) * plan.bwd.nsub),
            (unsigned)plan.batch);
  if (launch_pdl(kern, grid, dim3(kWarps * 32), A::kSmemBytes, s, maps, p) != cudaSuccess)
    return -1;
  return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

template <int NP>
static int launch_agg_np(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  const bool vec = (plan.Di % 4 == 0) && (plan.N % 4 == 0);
  BwdMaps maps;
  if (vec && plan.nchunks >= 2 && make_maps<NP>(plan, p, &maps))
    return launch_agg4<NP, true, true>(plan, maps, p, s);
  if (p.io_bf16) return -1;
  memset(&maps, 0, sizeof(maps));
  return vec ? launch_agg4<NP, true, false>(plan, maps, p, s)
             : launch_agg4<NP, false, false>(plan, maps, p, s);
}

int launch_bwd_agg_tmem(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  if (plan.bwd.nseg <= 1) return 0;
  switch (plan.NP) {
    case 16: return launch_agg_np<16>(plan, p, s);
    case 32: return launch_agg_np<32>(plan, p, s);
    case 64: return launch_agg_np<64>(plan, p, s);
    default: return -1;
  }
}

int launch_bwd_main_tmem(const Plan& plan, const BwdParams& p, cudaStream_t s) {
  switch (plan.NP) {
    case 16: return launch_np<16>(plan, p, s);
    case 32: return launch_np<32>(plan, p, s);
    case 64: return launch_np<64>(plan, p, s);
    default: return -1;
  }
}

MSCAN_OOB_HOOKS(tmem)

}  // namespace mscan
